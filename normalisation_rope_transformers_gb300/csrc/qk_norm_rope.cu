// Per-head Q/K RMSNorm fused with NeoX rotary embedding, for sm_103a.
//
// Computes what the vllm.cpp page src/vt/cuda/cuda_ops.cu gives in its fused
// attention-preamble section (RMSNorm over head_dim per (token, head), then
// the rotation, no rounding in between) with the angles of its NeoX RoPE
// section (freq_i = theta^(-2i/D), angle = pos * freq_i, pairs (i, i + D/2)).
//
// Design (not the page's, which runs one 256-thread block per (token, head)
// and reads a precomputed f32 cos/sin table from global memory):
//  * A group of L lanes owns one head row.  Lane l loads one 128-bit vector
//    from each half of the row -- elements [l*N, l*N+N) and the same slots
//    shifted by D/2 -- so both members of every rotated pair sit in the same
//    lane and the rotation needs no data exchange.  The row's sum of squares
//    is a butterfly over the L lanes.
//  * A warp owns whole tokens (all their Q and K heads), persistently: warp w
//    of W takes tokens w, w + W, ..., so at any moment the warps work on one
//    contiguous window of tokens.  Its head rows form one flat stream of
//    iterations (32/L rows per iteration) that crosses token boundaries; each
//    lane copies its vectors RING iterations ahead into a per-warp
//    shared-memory ring with cp.async, so several iterations are in flight
//    without holding registers.  There is no block-level barrier after the
//    weights are staged, so warps never wait for each other.
//  * Each (token, pair) angle is computed once per warp (a few sincospif per
//    lane) into a per-warp shared-memory table and reused by all the token's
//    heads.  The angle pos*freq_i is reduced modulo one turn exactly, as
//    (pos * turn_i) mod 2^64 with turn_i = frac(freq_i / 2pi) * 2^64 prepared
//    on the host in double; the top 32 bits feed sincospif.  No f64 math runs
//    on the device and no cos/sin table is read from HBM.
//  * Head rows are read once and written once (in place allowed).
#include <atomic>
#include <map>
#include <mutex>
#include <type_traits>
#include <utility>

#include "nr_common.cuh"
#include "nr_internal.h"

namespace nr {
namespace {

// Iterations in flight per warp (shared-memory ring slots); a build-time knob.
#ifndef NR_QK_RING
#define NR_QK_RING 5
#endif

constexpr int kQkThreads = 128;
constexpr int kQkWarps = kQkThreads / kWarp;

template <typename WT>
__device__ __forceinline__ float load_w(const WT* w, int i);
template <>
__device__ __forceinline__ float load_w<float>(const float* w, int i) {
  return __ldg(w + i);
}
template <>
__device__ __forceinline__ float load_w<__nv_bfloat16>(const __nv_bfloat16* w, int i) {
  return __bfloat162float(w[i]);
}

struct QkArgs {
  void* q_out;
  void* k_out;
  const void* q;
  const void* k;
  const void* wq;
  const void* wk;
  const int32_t* pos;
  int64_t tokens;
  int64_t q_stride;  // elements between consecutive tokens
  int64_t k_stride;
  int hq;
  int hk;
  float eps;
  float inv_d;
  float w_add;
  // RoPE variants (the general kernel only)
  int rot_vec;             // 128-bit vectors of the row that are rotated (rotary_dim / N)
  int interleaved;         // 0: rotate-half pairs (i, i + rot/2); 1: GPT-J pairs (2i, 2i + 1)
  int mrope;               // 1: three position rows, pair i uses row axis[i]
  int64_t pos_row_stride;  // elements between the position rows (= tokens)
  unsigned* status;        // the device status word (bounded waits that ran out)
};

// T: storage dtype of q/k; WT: weight dtype; L: lanes per head row
// (head_dim = 2 * L * N with N = 128-bit vector width in elements);
// RING: iterations kept in flight per warp (shared-memory ring slots).
template <typename T, int L>
struct QkSmem {
  static constexpr int N = Vec<T>::N;
  static constexpr int HALF = L * N;
  static constexpr int D = 2 * HALF;
  // per warp: RING slots x 32 lanes x ((a, b) vectors + npos positions), one angle table
  static constexpr size_t per_warp(int ring, int npos) {
    return static_cast<size_t>(ring) * kWarp * (2 * sizeof(uint4) + npos * sizeof(int)) +
           HALF * sizeof(float2);
  }
  static constexpr size_t bytes(int ring, int npos) {
    return kQkWarps * per_warp(ring, npos) + 2 * D * sizeof(float) +
           HALF * sizeof(unsigned long long) + HALF;
  }
};

// GEN = false: the rotary dimension is the whole head and pairs are
// rotate-half (the benchmark path).  GEN = true adds, at run time: a rotary
// dimension below head_dim (lanes past the rotated block carry two normed,
// unrotated vectors), GPT-J interleaved pairs (both members inside one vector)
// and M-RoPE (three position rows; pair i takes row axis[i]).
template <typename T, typename WT, int L, int RING, bool GEN>
__global__ void __launch_bounds__(kQkThreads) qk_norm_rope_kernel(const QkArgs a,
                                                                  const RopeTurns turns) {
  pdl_enter();  // before any global read: the previous kernel may still run
  using S = QkSmem<T, L>;
  constexpr int N = Vec<T>::N;
  constexpr int HALF = S::HALF;
  constexpr int D = S::D;
  constexpr int GW = kWarp / L;  // head rows per warp iteration
  constexpr int NPOS = GEN ? 3 : 1;

  extern __shared__ __align__(16) unsigned char smem[];
  const int warp = threadIdx.x / kWarp;
  const int lane32 = threadIdx.x % kWarp;
  unsigned char* wbase = smem + warp * S::per_warp(RING, NPOS);
  uint4* ring_a = reinterpret_cast<uint4*>(wbase);                   // [RING][32]
  uint4* ring_b = ring_a + RING * kWarp;                             // [RING][32]
  int* ring_pos = reinterpret_cast<int*>(ring_b + RING * kWarp);     // [RING][32][NPOS]
  float2* trig = reinterpret_cast<float2*>(ring_pos + RING * kWarp * NPOS);  // [HALF]
  float* wsm = reinterpret_cast<float*>(smem + kQkWarps * S::per_warp(RING, NPOS));  // [2D]
  unsigned long long* turn_sm = reinterpret_cast<unsigned long long*>(wsm + 2 * D);  // [HALF]
  unsigned char* axis_sm = reinterpret_cast<unsigned char*>(turn_sm + HALF);         // [HALF]

  const WT* wq = static_cast<const WT*>(a.wq);
  const WT* wk = static_cast<const WT*>(a.wk);
  for (int i = threadIdx.x; i < 2 * D; i += kQkThreads) {
    float wv = 0.0f;
    if (i < D)
      wv = load_w<WT>(wq, i);
    else if (a.hk > 0)
      wv = load_w<WT>(wk, i - D);
    wsm[i] = wv + a.w_add;
  }
  for (int i = threadIdx.x; i < HALF; i += kQkThreads) {
    turn_sm[i] = turns.turn[i];
    if (GEN) axis_sm[i] = turns.axis[i];
  }
  __syncthreads();  // the only block-level barrier

  const int g = lane32 / L;  // head row within the iteration
  const int l = lane32 % L;  // this lane's slot in the row
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kQkWarps + warp;
  const int64_t W = static_cast<int64_t>(gridDim.x) * kQkWarps;
  if (gw >= a.tokens) return;
  const int H = a.hq + a.hk;
  const int IT = (H + GW - 1) / GW;  // iterations per token

  // The two vectors of the row this lane owns.  Rotate-half: vector l and its
  // partner l + R/2 of the rotated block (R = 2L when the whole head rotates);
  // lanes past the rotated block take two unrotated vectors.  Interleaved:
  // vectors l and l + L (pairs never straddle vectors).
  int va_vec = l, vb_vec = l + L;
  bool rotates = true;  // rotate-half lane of the rotated block
  const int half_rot = GEN ? a.rot_vec / 2 : L;
  const int rot_pairs = GEN ? a.rot_vec * N / 2 : HALF;
  if (GEN && !a.interleaved) {
    if (l < half_rot) {
      vb_vec = l + half_rot;
    } else {
      va_vec = a.rot_vec + 2 * (l - half_rot);
      vb_vec = va_vec + 1;
      rotates = false;
    }
  }

  // A cursor walks this warp's iterations: token gw, gw + W, ... and, within
  // a token, iterations 0 .. IT-1 (rows it*GW .. it*GW + GW-1).  The copy
  // cursor runs RING iterations ahead of the compute cursor.
  struct Cursor {
    int64_t tok;
    int it;
  };
  auto advance = [&](Cursor& c) {
    if (++c.it == IT) {
      c.it = 0;
      c.tok += W;
    }
  };
  // Element offset of this lane's row of the cursor's iteration, and whether
  // it is a Q row; false when the iteration has no row for this lane.
  auto locate = [&](const Cursor& c, int64_t& off, bool& is_q) -> bool {
    const int row = c.it * GW + g;
    if (row >= H) return false;
    is_q = row < a.hq;
    off = is_q ? c.tok * a.q_stride + static_cast<int64_t>(row) * D
               : c.tok * a.k_stride + static_cast<int64_t>(row - a.hq) * D;
    return true;
  };

  Cursor cp{gw, 0}, cc{gw, 0};
  // Start the copies of the copy cursor's iteration into `slot`, one group.
  auto issue = [&](int slot) {
    if (cp.tok < a.tokens) {
      int64_t off;
      bool is_q;
      if (locate(cp, off, is_q)) {
        const T* src = static_cast<const T*>(is_q ? a.q : a.k) + off;
        const uint4* v = reinterpret_cast<const uint4*>(src);
        cp_async16(smem_addr(ring_a + slot * kWarp + lane32), v + va_vec);
        cp_async16(smem_addr(ring_b + slot * kWarp + lane32), v + vb_vec);
      }
      if (cp.it == 0) {
#pragma unroll
        for (int ax = 0; ax < NPOS; ax++)
          if (ax == 0 || (GEN && a.mrope))
            cp_async4(smem_addr(ring_pos + (slot * kWarp + lane32) * NPOS + ax),
                      a.pos + ax * a.pos_row_stride + cp.tok);
      }
      advance(cp);
    }
    cp_async_commit();  // possibly empty: keeps one group per iteration
  };

  for (int s = 0; s < RING; s++) issue(s);

  float2 cs[N];  // (cos, sin) of this lane's pairs for the current token
  int slot = 0;
  while (cc.tok < a.tokens) {
    cp_async_wait<RING - 1>();  // this iteration's group has landed
    int64_t off;
    bool is_q;
    const bool valid = locate(cc, off, is_q);
    if (cc.it == 0) {
      // New token: its angles, once per warp, then this lane's pairs.
      long long p[NPOS];
#pragma unroll
      for (int ax = 0; ax < NPOS; ax++)
        p[ax] = (ax == 0 || (GEN && a.mrope)) ? ring_pos[(slot * kWarp + lane32) * NPOS + ax] : 0;
      __syncwarp();
      for (int i = lane32; i < rot_pairs; i += kWarp) {
        const long long pi = (GEN && a.mrope) ? (axis_sm[i] == 0 ? p[0] : axis_sm[i] == 1
                                                     ? p[NPOS > 1 ? 1 : 0] : p[NPOS > 2 ? 2 : 0])
                                              : p[0];
        // the angle in turns, mod 1: exact for any int32 position
        const unsigned long long prod = static_cast<unsigned long long>(pi) * turn_sm[i];
        const int hi = static_cast<int>(prod >> 32);  // signed turn fraction * 2^32
        float sn, cn;
        sincospif(static_cast<float>(hi) * 0x1p-31f, &sn, &cn);  // angle = pi * hi / 2^31
        trig[i] = make_float2(cn, sn);
      }
      __syncwarp();
      if (!GEN || !a.interleaved) {
        if (rotates) {
#pragma unroll
          for (int e = 0; e < N; e++) cs[e] = trig[l * N + e];
        }
      } else {
#pragma unroll
        for (int j = 0; j < N / 2; j++) {
          if (va_vec < a.rot_vec) cs[j] = trig[va_vec * (N / 2) + j];
          if (vb_vec < a.rot_vec) cs[N / 2 + j] = trig[vb_vec * (N / 2) + j];
        }
      }
    }
    float xa[N], xb[N];
    float ss = 0.0f;
    if (valid) {
      Vec<T>::unpack(lds128(ring_a + slot * kWarp + lane32), xa);
      Vec<T>::unpack(lds128(ring_b + slot * kWarp + lane32), xb);
#pragma unroll
      for (int e = 0; e < N; e++) {
        ss = fmaf(xa[e], xa[e], ss);
        ss = fmaf(xb[e], xb[e], ss);
      }
    }
    // The slot's data is in registers: refill it RING iterations ahead.
    issue(slot);
    // Every lane joins the butterfly (full-warp shuffles), valid or not.
    ss = group_sum<L>(ss);
    if (valid) {
      const float inv = rsqrtf(ss * a.inv_d + a.eps);
      const float* w = wsm + (is_q ? 0 : D);
      const float* wa = w + va_vec * N;
      const float* wb = w + vb_vec * N;
      float oa[N], ob[N];
      if (!GEN || (!a.interleaved && rotates)) {
#pragma unroll
        for (int e = 0; e < N; e++) {
          const float na = xa[e] * inv * wa[e];
          const float nb = xb[e] * inv * wb[e];
          oa[e] = fmaf(na, cs[e].x, -nb * cs[e].y);
          ob[e] = fmaf(na, cs[e].y, nb * cs[e].x);
        }
      } else {
#pragma unroll
        for (int e = 0; e < N; e++) {
          oa[e] = xa[e] * inv * wa[e];
          ob[e] = xb[e] * inv * wb[e];
        }
        if (a.interleaved) {
#pragma unroll
          for (int j = 0; j < N / 2; j++) {
            if (va_vec < a.rot_vec) {
              const float x0 = oa[2 * j], x1 = oa[2 * j + 1];
              oa[2 * j] = fmaf(x0, cs[j].x, -x1 * cs[j].y);
              oa[2 * j + 1] = fmaf(x0, cs[j].y, x1 * cs[j].x);
            }
            if (vb_vec < a.rot_vec) {
              const float x0 = ob[2 * j], x1 = ob[2 * j + 1];
              ob[2 * j] = fmaf(x0, cs[N / 2 + j].x, -x1 * cs[N / 2 + j].y);
              ob[2 * j + 1] = fmaf(x0, cs[N / 2 + j].y, x1 * cs[N / 2 + j].x);
            }
          }
        }
      }
      uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(is_q ? a.q_out : a.k_out) + off);
      st_stream(dst + va_vec, Vec<T>::pack(oa));
      st_stream(dst + vb_vec, Vec<T>::pack(ob));
    }
    advance(cc);
    slot = slot + 1 == RING ? 0 : slot + 1;
  }
  cp_async_wait<0>();  // nothing may land after the block's shared memory is released
}

// ---------------------------------------------------------------------------
// Bulk-copy variant (full-head NeoX rotation): whole tokens move through
// shared memory by the TMA engine.
//
// A block of 4 warps owns tokens c, c + C, c + 2C, ... (C = grid size, so the
// blocks sweep one contiguous window of tokens).  Each token's Q rows and K
// rows are each one contiguous block of memory, so one bulk copy per tensor
// brings a token into a shared-memory stage; NST stages keep NST - 1 tokens
// in flight while one is computed.  The four warps split the token's head rows
// (lanes map to rows exactly as in the ring kernel), normalise and rotate them
// in place in the stage, and one thread writes the stage back with two bulk
// stores.  The next token's angle table is computed while the current token's
// rows are processed (double-buffered), so each token costs one block
// barrier.  Loads complete on a per-stage mbarrier; every wait on it is
// bounded and, if it runs out, sets a bit in the device status word and the
// block winds down (waiting, again bounded, for its copies in flight).
// ---------------------------------------------------------------------------
#ifndef NR_QKB_STAGES
#define NR_QKB_STAGES 3
#endif
// Kernel for the full-head NeoX case: 0 ring, 1 bulk copies (a build-time
// knob for comparisons).
#ifndef NR_QK_PATH
#define NR_QK_PATH 1
#endif
// L2 evict-first policy on the bulk loads (bit 0) and stores (bit 1); a
// build-time knob.  Both (3): the token blocks are touched once, and written
// lines leave L2 during this kernel instead of being written back while the
// next kernel runs (measured: this kernel 0.9 us faster, a following
// LayerNorm 1.7 us faster).
#ifndef NR_QKB_HINT
#define NR_QKB_HINT 3
#endif

// 1: each lane keeps its Q and K weights in registers (16 + 16 floats for
// head_dim 128 bf16) instead of reading them from shared memory for every
// head row; a build-time knob.
#ifndef NR_QKB_WREG
#define NR_QKB_WREG 1
#endif
// Upper bound on the bulk kernels' resident blocks per SM used to size the
// grid (a build-time knob; 0: as many as fit).
#ifndef NR_QKB_MAXB
#define NR_QKB_MAXB 0
#endif

// Minimum resident blocks per SM asked of the compiler for the full-head bulk
// kernel (a build-time knob; 0: none asked; shared memory allows 5 at 24 + 24
// heads of 128).
#ifndef NR_QKB_MINB
#define NR_QKB_MINB 0
#endif
#if NR_QKB_MINB > 0
#define NR_QKB_BOUNDS __launch_bounds__(kBulkThreads, NR_QKB_MINB)
#else
#define NR_QKB_BOUNDS __launch_bounds__(kBulkThreads)
#endif

// Warps per block (they split each token's head rows); a build-time knob.
#ifndef NR_QKB_WARPS
#define NR_QKB_WARPS 4
#endif
constexpr int kBulkWarps = NR_QKB_WARPS;
constexpr int kBulkThreads = kBulkWarps * kWarp;
constexpr long long kWaitLimitCycles = 1LL << 31;  // about one second

__device__ __forceinline__ void record_status(unsigned* word, unsigned bit) { atomicOr(word, bit); }

struct BulkGeom {
  unsigned q_bytes;      // one token's Q rows
  unsigned k_bytes;      // one token's K rows
  unsigned stage_bytes;  // q_bytes + k_bytes rounded up to 128
};

template <typename T, int L>
struct BulkSmem {
  static constexpr int N = Vec<T>::N;
  static constexpr int HALF = L * N;
  static constexpr int D = 2 * HALF;
  // [NST stages][2 angle tables of HALF float2][2D weights][HALF turns][NST mbarriers][flag]
  static size_t bytes(int nst, unsigned stage_bytes) {
    return static_cast<size_t>(nst) * stage_bytes + 2 * HALF * sizeof(float2) +
           2 * D * sizeof(float) + HALF * sizeof(unsigned long long) +
           nst * sizeof(unsigned long long) + 16;
  }
};

template <typename T, typename WT, int L, int NST, bool MROPE>
__global__ void NR_QKB_BOUNDS qk_norm_rope_bulk_kernel(const QkArgs a,
                                                                       const RopeTurns turns,
                                                                       const BulkGeom geo) {
  using S = BulkSmem<T, L>;
  constexpr int N = Vec<T>::N;
  constexpr int HALF = S::HALF;
  constexpr int D = S::D;
  constexpr int GW = kWarp / L;  // head rows per warp pass

  // bulk copies need 16-byte aligned shared addresses: the stages start at the
  // (16-byte aligned) base and every stage and K block offset is a multiple of 16
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char* stages = smem;
  float2* table = reinterpret_cast<float2*>(stages + static_cast<size_t>(NST) * geo.stage_bytes);
  float* wsm = reinterpret_cast<float*>(table + 2 * HALF);
  unsigned long long* turn_sm = reinterpret_cast<unsigned long long*>(wsm + 2 * D);
  unsigned long long* bars = turn_sm + HALF;
  int* abort_flag = reinterpret_cast<int*>(bars + NST);

  const int tid = threadIdx.x;
  const int warp = tid / kWarp;
  const int lane32 = tid % kWarp;
  const WT* wq = static_cast<const WT*>(a.wq);
  const WT* wk = static_cast<const WT*>(a.wk);
  // Set-up from kernel parameters into shared memory (no global read), before
  // the wait for the previous kernel: the rotary turns and the barriers.
  for (int i = tid; i < HALF; i += kBulkThreads) turn_sm[i] = turns.turn[i];
  if (tid == 0) {
    for (int st = 0; st < NST; st++) mbar_init(smem_addr(bars + st), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }

  const int64_t C = gridDim.x;
  const int64_t t0 = blockIdx.x;
  const int64_t ntok = t0 < a.tokens ? (a.tokens - 1 - t0) / C + 1 : 0;  // this block's tokens
  const int H = a.hq + a.hk;
  const int IT = (H + GW - 1) / GW;
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  T* q_out = static_cast<T*>(a.q_out);
  T* k_out = static_cast<T*>(a.k_out);
  auto stage = [&](int64_t j) { return stages + (j % NST) * geo.stage_bytes; };

  // Producer (thread 0): bring local token j into its stage.
  int64_t issued = 0;
  const uint64_t policy = NR_QKB_HINT ? l2_evict_first_policy() : 0;
  auto issue = [&](int64_t j) {
    const int64_t tok = t0 + j * C;
    const unsigned bar = smem_addr(bars + j % NST);
    mbar_arrive_expect_tx(bar, geo.q_bytes + geo.k_bytes);
    if (NR_QKB_HINT & 1) {
      bulk_load_hint(smem_addr(stage(j)), q + tok * a.q_stride, geo.q_bytes, bar, policy);
      if (geo.k_bytes)
        bulk_load_hint(smem_addr(stage(j) + geo.q_bytes), k + tok * a.k_stride, geo.k_bytes, bar,
                       policy);
    } else {
      bulk_load(smem_addr(stage(j)), q + tok * a.q_stride, geo.q_bytes, bar);
      if (geo.k_bytes) bulk_load(smem_addr(stage(j) + geo.q_bytes), k + tok * a.k_stride,
                                 geo.k_bytes, bar);
    }
    issued = j + 1;
  };
  pdl_enter();  // before any global read: the previous kernel may still run
  // The first tokens' loads go out before the weights are read, so their
  // latency overlaps the rest of the set-up.
  if (tid == 0)
    for (int64_t j = 0; j < NST - 1 && j < ntok; j++) issue(j);
  for (int i = tid; i < 2 * D; i += kBulkThreads) {
    float wv = 0.0f;
    if (i < D)
      wv = load_w<WT>(wq, i);
    else if (a.hk > 0)
      wv = load_w<WT>(wk, i - D);
    wsm[i] = wv + a.w_add;
  }
  __syncthreads();  // weights, turns and barriers visible to every thread

  // Angle table of a token into table buffer b (threads < HALF, strided).
  auto angles = [&](int b, int p) {
    for (int i = tid; i < HALF; i += kBulkThreads) {
      const unsigned long long prod = static_cast<unsigned long long>(static_cast<long long>(p)) *
                                      turn_sm[i];
      const int hi = static_cast<int>(prod >> 32);  // signed turn fraction * 2^32
      float sn, cn;
      sincospif(static_cast<float>(hi) * 0x1p-31f, &sn, &cn);  // angle = pi * hi / 2^31
      table[b * HALF + i] = make_float2(cn, sn);
    }
  };
  // M-RoPE (MROPE): thread i computes pair i's angle from position row
  // axis[i] (the launcher ensures one pair per thread); otherwise row 0.
  const int64_t pos_row = (MROPE && tid < HALF) ? turns.axis[tid] * a.pos_row_stride : 0;
  int pos_next = 0;  // position of local token j + 1, loaded one token ahead
  if (ntok > 0) {
    if (tid < HALF) {
      angles(0, a.pos[pos_row + t0]);
      if (ntok > 1) pos_next = a.pos[pos_row + t0 + C];
    }
  }
  __syncthreads();

  const int g = lane32 / L;
  const int l = lane32 % L;
  // This lane's weights (it always owns vectors l and l + L of a row), kept
  // in registers when NR_QKB_WREG is set instead of read from shared memory
  // for every head row.
  float wqa[NR_QKB_WREG ? N : 1], wqb[NR_QKB_WREG ? N : 1];
  float wka[NR_QKB_WREG ? N : 1], wkb[NR_QKB_WREG ? N : 1];
  if (NR_QKB_WREG) {
#pragma unroll
    for (int e = 0; e < (NR_QKB_WREG ? N : 1); e++) {
      wqa[e] = wsm[l * N + e];
      wqb[e] = wsm[HALF + l * N + e];
      wka[e] = wsm[D + l * N + e];
      wkb[e] = wsm[D + HALF + l * N + e];
    }
  }
  int64_t j = 0;
  for (; j < ntok; j++) {
    const int64_t tok = t0 + j * C;
    unsigned char* st = stage(j);
    if (!mbar_wait_bounded(smem_addr(bars + j % NST), static_cast<unsigned>((j / NST) & 1),
                           kWaitLimitCycles)) {
      record_status(a.status, kStatusBitQkBulkWait);
      *abort_flag = 1;
    }
    // this lane's (cos, sin) for the token
    float2 cs[N];
#pragma unroll
    for (int e = 0; e < N; e++) cs[e] = table[(j & 1) * HALF + l * N + e];
    // The stage holds the token's Q rows and then its K rows, contiguously,
    // so head row `row` (Q rows first) starts at row * D elements.
    auto row_ptr = [&](int row) {
      return reinterpret_cast<uint4*>(st + static_cast<size_t>(row) * D * sizeof(T));
    };
    // One pass: head rows it*GW .. it*GW + GW - 1, one per lane group.  KIND 0:
    // every row of the pass is a Q head, 1: every row a K head (the lane's
    // weights are then fixed for the pass); 2: a pass that straddles the Q/K
    // boundary or runs past the last head (each lane group picks its own).
    auto pass = [&](auto kind, int it) {
      constexpr int KIND = decltype(kind)::value;
      const int row = it * GW + g;
      // Lanes of a row past the last head carry zeros but still join the
      // butterfly: the shuffles take the full warp.
      const bool valid = KIND != 2 || row < H;
      const bool is_q = KIND == 0 || (KIND == 2 && row < a.hq);
      uint4* r = row_ptr(valid ? row : 0);
      float xa[N], xb[N];
      float ss = 0.0f;
      if (valid) {
        Vec<T>::unpack(r[l], xa);
        Vec<T>::unpack(r[l + L], xb);
#pragma unroll
        for (int e = 0; e < N; e++) {
          ss = fmaf(xa[e], xa[e], ss);
          ss = fmaf(xb[e], xb[e], ss);
        }
      }
      ss = group_sum<L>(ss);
      if (!valid) return;
      const float inv = rsqrtf(ss * a.inv_d + a.eps);
      const float* wa = wsm + (is_q ? 0 : D) + l * N;
      const float* wb = wa + HALF;
      float oa[N], ob[N];
#pragma unroll
      for (int e = 0; e < N; e++) {
        constexpr int E = NR_QKB_WREG ? 1 : 0;
        const float we_a = !NR_QKB_WREG ? wa[e]
                           : KIND == 0  ? wqa[E * e]
                           : KIND == 1  ? wka[E * e]
                                        : (is_q ? wqa[E * e] : wka[E * e]);
        const float we_b = !NR_QKB_WREG ? wb[e]
                           : KIND == 0  ? wqb[E * e]
                           : KIND == 1  ? wkb[E * e]
                                        : (is_q ? wqb[E * e] : wkb[E * e]);
        const float na = xa[e] * inv * we_a;
        const float nb = xb[e] * inv * we_b;
        oa[e] = fmaf(na, cs[e].x, -nb * cs[e].y);
        ob[e] = fmaf(na, cs[e].y, nb * cs[e].x);
      }
      r[l] = Vec<T>::pack(oa);
      r[l + L] = Vec<T>::pack(ob);
    };
    for (int it = warp; it < IT; it += kBulkWarps) {  // uniform across the warp
      const int first = it * GW;
      if (first + GW <= a.hq)
        pass(std::integral_constant<int, 0>(), it);
      else if (first >= a.hq && first + GW <= H)
        pass(std::integral_constant<int, 1>(), it);
      else
        pass(std::integral_constant<int, 2>(), it);
    }
    // the next token's angles, into the other table buffer
    if (tid < HALF && j + 1 < ntok) {
      angles(static_cast<int>((j + 1) & 1), pos_next);
      if (j + 2 < ntok) pos_next = a.pos[pos_row + t0 + (j + 2) * C];
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (*abort_flag) break;
    if (tid == 0) {
      if (NR_QKB_HINT & 2) {
        bulk_store_hint(q_out + tok * a.q_stride, smem_addr(st), geo.q_bytes, policy);
        if (geo.k_bytes) bulk_store_hint(k_out + tok * a.k_stride, smem_addr(st + geo.q_bytes),
                                         geo.k_bytes, policy);
      } else {
        bulk_store(q_out + tok * a.q_stride, smem_addr(st), geo.q_bytes);
        if (geo.k_bytes) bulk_store(k_out + tok * a.k_stride, smem_addr(st + geo.q_bytes),
                                    geo.k_bytes);
      }
      bulk_commit();
      if (j + NST - 1 < ntok) {
        bulk_wait_read<1>();  // the stage of token j - 1 has been read out
        issue(j + NST - 1);
      }
    }
  }
  if (tid == 0) {
    bulk_wait<0>();  // every store has landed before the block's shared memory is released
    // After an abandoned wait (at token j), let the loads still in flight
    // finish (bounded); after a normal finish there are none (j == issued).
    for (int64_t m = j; m < issued; m++)
      if (!mbar_wait_bounded(smem_addr(bars + m % NST), static_cast<unsigned>((m / NST) & 1),
                             kWaitLimitCycles))
        break;
  }
}

// The bulk-copy kernel for two RoPE variants (kept as its own kernel so the
// full-head NeoX kernel above is compiled exactly as measured): a rotary
// dimension below head_dim (lanes past the rotated block carry two normed,
// unrotated vectors) and GPT-J interleaved pairs.  The stages, the producer
// and the bounded waits are those of the kernel above.  (M-RoPE over the
// whole head runs the kernel above with MROPE set; other M-RoPE layouts run
// the ring kernel.)
template <typename T, typename WT, int L, int NST>
// Minimum resident blocks per SM asked of the compiler for the variant kernel
// (a build-time knob; 0: none asked).  With the weights in shared memory a
// cap of 7 (72 registers) ran GPT-J pairs with a 64-dim rotary part at
// [26598, 24 + 24, 128] in 105.1 µs instead of 112.4 µs (79 registers); with
// the weights in registers (NR_QKV_WREG) no cap (120 registers) runs it in
// 102.2 µs against 104.4 µs for the capped shared-memory build.
#ifndef NR_QKV_MINB
#define NR_QKV_MINB 0
#endif
#if NR_QKV_MINB > 0
#define NR_QKV_BOUNDS __launch_bounds__(kBulkThreads, NR_QKV_MINB)
#else
#define NR_QKV_BOUNDS __launch_bounds__(kBulkThreads)
#endif
// 1: the variant kernel keeps each lane's weights in registers (a build-time
// knob, as NR_QKB_WREG for the full-head kernel).
#ifndef NR_QKV_WREG
#define NR_QKV_WREG 1
#endif
__global__ void NR_QKV_BOUNDS qk_norm_rope_bulk_var_kernel(const QkArgs a,
                                                                       const RopeTurns turns,
                                                                       const BulkGeom geo) {
  using S = BulkSmem<T, L>;
  constexpr int N = Vec<T>::N;
  constexpr int HALF = S::HALF;
  constexpr int D = S::D;
  constexpr int GW = kWarp / L;  // head rows per warp pass

  // bulk copies need 16-byte aligned shared addresses: the stages start at the
  // (16-byte aligned) base and every stage and K block offset is a multiple of 16
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char* stages = smem;
  float2* table = reinterpret_cast<float2*>(stages + static_cast<size_t>(NST) * geo.stage_bytes);
  float* wsm = reinterpret_cast<float*>(table + 2 * HALF);
  unsigned long long* turn_sm = reinterpret_cast<unsigned long long*>(wsm + 2 * D);
  unsigned long long* bars = turn_sm + HALF;
  int* abort_flag = reinterpret_cast<int*>(bars + NST);

  const int tid = threadIdx.x;
  const int warp = tid / kWarp;
  const int lane32 = tid % kWarp;
  const WT* wq = static_cast<const WT*>(a.wq);
  const WT* wk = static_cast<const WT*>(a.wk);
  // Set-up from kernel parameters into shared memory (no global read), before
  // the wait for the previous kernel: the rotary turns and the barriers.
  for (int i = tid; i < HALF; i += kBulkThreads) turn_sm[i] = turns.turn[i];
  if (tid == 0) {
    for (int st = 0; st < NST; st++) mbar_init(smem_addr(bars + st), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }

  const int64_t C = gridDim.x;
  const int64_t t0 = blockIdx.x;
  const int64_t ntok = t0 < a.tokens ? (a.tokens - 1 - t0) / C + 1 : 0;  // this block's tokens
  const int H = a.hq + a.hk;
  const int IT = (H + GW - 1) / GW;
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  T* q_out = static_cast<T*>(a.q_out);
  T* k_out = static_cast<T*>(a.k_out);
  auto stage = [&](int64_t j) { return stages + (j % NST) * geo.stage_bytes; };

  // Producer (thread 0): bring local token j into its stage.
  int64_t issued = 0;
  const uint64_t policy = NR_QKB_HINT ? l2_evict_first_policy() : 0;
  auto issue = [&](int64_t j) {
    const int64_t tok = t0 + j * C;
    const unsigned bar = smem_addr(bars + j % NST);
    mbar_arrive_expect_tx(bar, geo.q_bytes + geo.k_bytes);
    if (NR_QKB_HINT & 1) {
      bulk_load_hint(smem_addr(stage(j)), q + tok * a.q_stride, geo.q_bytes, bar, policy);
      if (geo.k_bytes)
        bulk_load_hint(smem_addr(stage(j) + geo.q_bytes), k + tok * a.k_stride, geo.k_bytes, bar,
                       policy);
    } else {
      bulk_load(smem_addr(stage(j)), q + tok * a.q_stride, geo.q_bytes, bar);
      if (geo.k_bytes) bulk_load(smem_addr(stage(j) + geo.q_bytes), k + tok * a.k_stride,
                                 geo.k_bytes, bar);
    }
    issued = j + 1;
  };
  pdl_enter();  // before any global read: the previous kernel may still run
  // The first tokens' loads go out before the weights are read, so their
  // latency overlaps the rest of the set-up.
  if (tid == 0)
    for (int64_t j = 0; j < NST - 1 && j < ntok; j++) issue(j);
  for (int i = tid; i < 2 * D; i += kBulkThreads) {
    float wv = 0.0f;
    if (i < D)
      wv = load_w<WT>(wq, i);
    else if (a.hk > 0)
      wv = load_w<WT>(wk, i - D);
    wsm[i] = wv + a.w_add;
  }
  __syncthreads();  // weights, turns and barriers visible to every thread

  // Angle table of a token into table buffer b: pairs of the rotated block.
  const int rot_pairs = a.rot_vec * N / 2;
  auto angles = [&](int b, int p) {
    for (int i = tid; i < rot_pairs; i += kBulkThreads) {
      const unsigned long long prod = static_cast<unsigned long long>(static_cast<long long>(p)) *
                                      turn_sm[i];
      const int hi = static_cast<int>(prod >> 32);  // signed turn fraction * 2^32
      float sn, cn;
      sincospif(static_cast<float>(hi) * 0x1p-31f, &sn, &cn);  // angle = pi * hi / 2^31
      table[b * HALF + i] = make_float2(cn, sn);
    }
  };
  int pos_next = 0;  // position of local token j + 1, loaded one token ahead
  if (ntok > 0) {
    if (tid < rot_pairs) {
      angles(0, a.pos[t0]);
      if (ntok > 1) pos_next = a.pos[t0 + C];
    }
  }
  __syncthreads();

  const int g = lane32 / L;
  const int l = lane32 % L;
  // The two vectors of the row this lane owns, as in the ring kernel:
  // rotate-half lanes of the rotated block take vector l and its partner
  // l + R/2; lanes past it take two unrotated vectors; interleaved: l, l + L.
  int va_vec = l, vb_vec = l + L;
  bool rotates = true;
  if (!a.interleaved) {
    const int half_rot = a.rot_vec / 2;
    if (l < half_rot) {
      vb_vec = l + half_rot;
    } else {
      va_vec = a.rot_vec + 2 * (l - half_rot);
      vb_vec = va_vec + 1;
      rotates = false;
    }
  }
#if NR_QKV_WREG
  float wqa[N], wqb[N], wka[N], wkb[N];
#pragma unroll
  for (int e = 0; e < N; e++) {
    wqa[e] = wsm[va_vec * N + e];
    wqb[e] = wsm[vb_vec * N + e];
    wka[e] = wsm[D + va_vec * N + e];
    wkb[e] = wsm[D + vb_vec * N + e];
  }
#endif
  int64_t j = 0;
  for (; j < ntok; j++) {
    const int64_t tok = t0 + j * C;
    unsigned char* st = stage(j);
    if (!mbar_wait_bounded(smem_addr(bars + j % NST), static_cast<unsigned>((j / NST) & 1),
                           kWaitLimitCycles)) {
      record_status(a.status, kStatusBitQkBulkWait);
      *abort_flag = 1;
    }
    // this lane's (cos, sin) for the token
    float2 cs[N];
    const float2* tb = table + (j & 1) * HALF;
    if (!a.interleaved) {
      if (rotates) {
#pragma unroll
        for (int e = 0; e < N; e++) cs[e] = tb[l * N + e];
      }
    } else {
#pragma unroll
      for (int h = 0; h < N / 2; h++) {
        if (va_vec < a.rot_vec) cs[h] = tb[va_vec * (N / 2) + h];
        if (vb_vec < a.rot_vec) cs[N / 2 + h] = tb[vb_vec * (N / 2) + h];
      }
    }
    for (int it = warp; it < IT; it += kBulkWarps) {  // uniform across the warp
      const int row = it * GW + g;
      // Lanes of a row past the last head carry zeros but still join the
      // butterfly: the shuffles take the full warp.
      const bool valid = row < H;
      const bool is_q = row < a.hq;
      uint4* r = reinterpret_cast<uint4*>(
          st + (is_q ? 0u : geo.q_bytes) +
          static_cast<size_t>(valid ? (is_q ? row : row - a.hq) : 0) * D * sizeof(T));
      float xa[N], xb[N];
      float ss = 0.0f;
      if (valid) {
        Vec<T>::unpack(r[va_vec], xa);
        Vec<T>::unpack(r[vb_vec], xb);
#pragma unroll
        for (int e = 0; e < N; e++) {
          ss = fmaf(xa[e], xa[e], ss);
          ss = fmaf(xb[e], xb[e], ss);
        }
      }
      ss = group_sum<L>(ss);
      if (!valid) continue;
      const float inv = rsqrtf(ss * a.inv_d + a.eps);
#if NR_QKV_WREG
      float wa[N], wb[N];
#pragma unroll
      for (int e = 0; e < N; e++) {
        wa[e] = is_q ? wqa[e] : wka[e];
        wb[e] = is_q ? wqb[e] : wkb[e];
      }
#else
      const float* w = wsm + (is_q ? 0 : D);
      const float* wa = w + va_vec * N;
      const float* wb = w + vb_vec * N;
#endif
      float oa[N], ob[N];
      if (!a.interleaved && rotates) {
#pragma unroll
        for (int e = 0; e < N; e++) {
          const float na = xa[e] * inv * wa[e];
          const float nb = xb[e] * inv * wb[e];
          oa[e] = fmaf(na, cs[e].x, -nb * cs[e].y);
          ob[e] = fmaf(na, cs[e].y, nb * cs[e].x);
        }
      } else {
#pragma unroll
        for (int e = 0; e < N; e++) {
          oa[e] = xa[e] * inv * wa[e];
          ob[e] = xb[e] * inv * wb[e];
        }
        if (a.interleaved) {
#pragma unroll
          for (int h = 0; h < N / 2; h++) {
            if (va_vec < a.rot_vec) {
              const float x0 = oa[2 * h], x1 = oa[2 * h + 1];
              oa[2 * h] = fmaf(x0, cs[h].x, -x1 * cs[h].y);
              oa[2 * h + 1] = fmaf(x0, cs[h].y, x1 * cs[h].x);
            }
            if (vb_vec < a.rot_vec) {
              const float x0 = ob[2 * h], x1 = ob[2 * h + 1];
              ob[2 * h] = fmaf(x0, cs[N / 2 + h].x, -x1 * cs[N / 2 + h].y);
              ob[2 * h + 1] = fmaf(x0, cs[N / 2 + h].y, x1 * cs[N / 2 + h].x);
            }
          }
        }
      }
      r[va_vec] = Vec<T>::pack(oa);
      r[vb_vec] = Vec<T>::pack(ob);
    }
    // the next token's angles, into the other table buffer
    if (tid < rot_pairs && j + 1 < ntok) {
      angles(static_cast<int>((j + 1) & 1), pos_next);
      if (j + 2 < ntok) pos_next = a.pos[t0 + (j + 2) * C];
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (*abort_flag) break;
    if (tid == 0) {
      if (NR_QKB_HINT & 2) {
        bulk_store_hint(q_out + tok * a.q_stride, smem_addr(st), geo.q_bytes, policy);
        if (geo.k_bytes) bulk_store_hint(k_out + tok * a.k_stride, smem_addr(st + geo.q_bytes),
                                         geo.k_bytes, policy);
      } else {
        bulk_store(q_out + tok * a.q_stride, smem_addr(st), geo.q_bytes);
        if (geo.k_bytes) bulk_store(k_out + tok * a.k_stride, smem_addr(st + geo.q_bytes),
                                    geo.k_bytes);
      }
      bulk_commit();
      if (j + NST - 1 < ntok) {
        bulk_wait_read<1>();  // the stage of token j - 1 has been read out
        issue(j + NST - 1);
      }
    }
  }
  if (tid == 0) {
    bulk_wait<0>();  // every store has landed before the block's shared memory is released
    // After an abandoned wait (at token j), let the loads still in flight
    // finish (bounded); after a normal finish there are none (j == issued).
    for (int64_t m = j; m < issued; m++)
      if (!mbar_wait_bounded(smem_addr(bars + m % NST), static_cast<unsigned>((m / NST) & 1),
                             kWaitLimitCycles))
        break;
  }
}

// Resident blocks per SM of one kernel instantiation (with its dynamic shared
// memory), cached per device; also raises the kernel's shared-memory limit.
// (The host-side caches below may be filled by several threads at once; each
// entry is an atomic, and a racing thread at worst repeats the query.)
template <typename T, typename WT, int L, int RING, bool GEN>
int blocks_per_sm(int device) {
  static std::atomic<int> cached[64];
  if (device < 0 || device >= 64) return 1;
  int n = cached[device].load(std::memory_order_relaxed);
  if (n == 0) {
    const size_t smem = QkSmem<T, L>::bytes(RING, GEN ? 3 : 1);
    cudaFuncSetAttribute(qk_norm_rope_kernel<T, WT, L, RING, GEN>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, qk_norm_rope_kernel<T, WT, L, RING, GEN>,
                                                      kQkThreads, smem) != cudaSuccess ||
        n < 1)
      n = 1;
    cached[device].store(n, std::memory_order_relaxed);
  }
  return n;
}

int sm_count(int device) {
  static std::atomic<int> cached[64];
  if (device < 0 || device >= 64) return 1;
  int n = cached[device].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n < 1)
      n = 1;
    cached[device].store(n, std::memory_order_relaxed);
  }
  return n;
}

template <typename T, typename WT, int L, bool GEN>
cudaError_t launch_g(const QkArgs& a, const RopeTurns& turns, cudaStream_t s) {
  constexpr int RING = NR_QK_RING;
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  const int64_t resident =
      static_cast<int64_t>(sm_count(device)) * blocks_per_sm<T, WT, L, RING, GEN>(device);
  const int64_t needed = (a.tokens + kQkWarps - 1) / kQkWarps;  // one warp per token at most
  const int64_t blocks = needed < resident ? needed : resident;
  return launch_pdl(qk_norm_rope_kernel<T, WT, L, RING, GEN>, dim3(static_cast<unsigned>(blocks)),
                    dim3(kQkThreads), QkSmem<T, L>::bytes(RING, GEN ? 3 : 1), s, a, turns);
}

// 1: M-RoPE over the whole head runs the full-head bulk kernel (a build-time
// knob; 0: the ring kernel).  Measured at [26598, 24+24, 128], sections
// (16, 24, 24): 100.4 us against 107.0 us on the ring kernel.
#ifndef NR_MROPE_BULK
#define NR_MROPE_BULK 1
#endif

// Largest shared memory the bulk variant may take per block (stages plus
// tables): beyond it (very many heads per token) the ring kernel runs.
constexpr size_t kBulkMaxSmem = 112 * 1024;

template <typename T, typename WT, int L, bool VAR, bool MROPE>
cudaError_t launch_bulk(const QkArgs& a, const RopeTurns& turns, const BulkGeom& geo,
                        size_t smem, cudaStream_t s) {
  constexpr int NST = NR_QKB_STAGES;
  auto kernel = VAR ? qk_norm_rope_bulk_var_kernel<T, WT, L, NST>
                    : qk_norm_rope_bulk_kernel<T, WT, L, NST, MROPE>;
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  // Per device: raise the shared-memory limit once; cache the occupancy per
  // shared-memory size (a few distinct head layouts at most).
  static std::mutex mu;
  static std::map<std::pair<int, size_t>, int> occupancy;
  static std::atomic<int> limit_set[64];
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  if (!limit_set[device].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kBulkMaxSmem));
    if (e != cudaSuccess) return e;
    limit_set[device].store(1, std::memory_order_release);
  }
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = occupancy.find({device, smem});
    if (it != occupancy.end()) per_sm = it->second;
  }
  if (per_sm == 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kBulkThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    std::lock_guard<std::mutex> lock(mu);
    occupancy[{device, smem}] = per_sm;
  }
  if (NR_QKB_MAXB > 0 && per_sm > NR_QKB_MAXB) per_sm = NR_QKB_MAXB;
  const int64_t resident = static_cast<int64_t>(sm_count(device)) * per_sm;
  const int64_t blocks = a.tokens < resident ? a.tokens : resident;
  return launch_pdl(kernel, dim3(static_cast<unsigned>(blocks)), dim3(kBulkThreads), smem, s, a,
                    turns, geo);
}

template <typename T, typename WT, int L>
cudaError_t launch_l(const QkArgs& a, const RopeTurns& turns, cudaStream_t s) {
  const bool general = a.rot_vec != 2 * L || a.interleaved || a.mrope;
  // M-RoPE over the whole head with rotate-half pairs, one pair per thread:
  // the full-head bulk kernel, each thread reading its pair's position row;
  // any other M-RoPE: the ring kernel.
  constexpr int HALF = L * Vec<T>::N;
  const bool mrope_bulk = NR_MROPE_BULK && a.mrope && a.rot_vec == 2 * L && !a.interleaved &&
                          HALF <= kBulkThreads;
  if (a.mrope && !mrope_bulk) return launch_g<T, WT, L, true>(a, turns, s);
  // Whole tokens through shared memory when a token's rows fit the stages.
  constexpr int D = 2 * L * Vec<T>::N;
  BulkGeom geo;
  geo.q_bytes = static_cast<unsigned>(a.hq * D * sizeof(T));
  geo.k_bytes = static_cast<unsigned>(a.hk * D * sizeof(T));
  geo.stage_bytes = (geo.q_bytes + geo.k_bytes + 127u) & ~127u;
  const size_t smem = BulkSmem<T, L>::bytes(NR_QKB_STAGES, geo.stage_bytes);
  if (NR_QK_PATH == 1 && smem <= kBulkMaxSmem) {
    if (mrope_bulk) return launch_bulk<T, WT, L, false, true>(a, turns, geo, smem, s);
    return general ? launch_bulk<T, WT, L, true, false>(a, turns, geo, smem, s)
                   : launch_bulk<T, WT, L, false, false>(a, turns, geo, smem, s);
  }
  return general ? launch_g<T, WT, L, true>(a, turns, s) : launch_g<T, WT, L, false>(a, turns, s);
}

template <typename T, typename WT>
cudaError_t launch_w(const QkArgs& a, int lanes, const RopeTurns& turns, cudaStream_t s) {
  switch (lanes) {
    case 1: return launch_l<T, WT, 1>(a, turns, s);
    case 2: return launch_l<T, WT, 2>(a, turns, s);
    case 4: return launch_l<T, WT, 4>(a, turns, s);
    case 8: return launch_l<T, WT, 8>(a, turns, s);
    case 16: return launch_l<T, WT, 16>(a, turns, s);
    case 32: return launch_l<T, WT, 32>(a, turns, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_qk_norm_rope(void* q_out, void* k_out, const void* q, const void* k,
                                const void* wq, const void* wk, int w_is_bf16,
                                const int32_t* positions, int64_t tokens, int64_t hq, int64_t hk,
                                int64_t head_dim, int64_t q_tok_stride, int64_t k_tok_stride,
                                float eps, const RopeTurns& turns, int gemma, int64_t rotary_dim,
                                int interleaved, int mrope, int is_bf16, cudaStream_t stream) {
  const int n = is_bf16 ? 8 : 4;
  const int lanes = static_cast<int>(head_dim / (2 * n));
  QkArgs a;
  a.q_out = q_out;
  a.k_out = k_out;
  a.q = q;
  a.k = k;
  a.wq = wq;
  a.wk = wk;
  a.pos = positions;
  a.tokens = tokens;
  a.q_stride = q_tok_stride;
  a.k_stride = k_tok_stride;
  a.hq = static_cast<int>(hq);
  a.hk = static_cast<int>(hk);
  a.eps = eps;
  a.inv_d = 1.0f / static_cast<float>(head_dim);
  a.w_add = gemma ? 1.0f : 0.0f;
  a.rot_vec = static_cast<int>(rotary_dim / n);
  a.interleaved = interleaved;
  a.mrope = mrope;
  a.pos_row_stride = tokens;
  cudaError_t e = status_word(&a.status);
  if (e != cudaSuccess) return e;

  if (is_bf16) {
    if (w_is_bf16) return launch_w<__nv_bfloat16, __nv_bfloat16>(a, lanes, turns, stream);
    return launch_w<__nv_bfloat16, float>(a, lanes, turns, stream);
  }
  if (w_is_bf16) return launch_w<float, __nv_bfloat16>(a, lanes, turns, stream);
  return launch_w<float, float>(a, lanes, turns, stream);
}

}  // namespace nr
