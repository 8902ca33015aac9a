// Per-head Q/K RMSNorm fused with NeoX rotary embedding, for sm_103a.
//
// Computes what vllm.cpp src/vt/cuda/cuda_ops.cu describes in
// "attn_qk_norm_rope_gate" (RMSNorm over head_dim per (token, head), then the
// rotation, no rounding in between) with the angles of "rope_neox"
// (freq_i = theta^(-2i/D), angle = pos * freq_i, pairs (i, i + D/2)).
//
// Design (not the page's, which runs one 256-thread block per (token, head)
// and reads a precomputed f32 cos/sin table from global memory):
//  * A group of L lanes owns one head row.  Lane l loads one 128-bit vector
//    from each half of the row -- elements [l*N, l*N+N) and the same slots
//    shifted by D/2 -- so both members of every rotated pair sit in the same
//    lane and the rotation needs no data exchange.  The row's sum of squares
//    is a butterfly over the L lanes.
//  * A block handles a tile of tokens (all their Q and K heads).  Each
//    (token, pair) angle is computed once per tile into shared memory and
//    reused by every head of that token: the angle pos*freq_i is reduced
//    modulo one turn exactly, as (pos * turn_i) mod 2^64 with
//    turn_i = frac(freq_i / 2pi) * 2^64 prepared on the host in double, then
//    sincospif evaluates the reduced angle.  No f64 math runs on the device
//    and no cos/sin table is read from HBM.
//  * Head rows are read once and written once (in place allowed).
#include "nr_common.cuh"
#include "nr_internal.h"

namespace nr {
namespace {

constexpr int kQkThreads = 256;
constexpr int kQkIter = 4;  // head rows per group held in registers at once

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
  int tile_tokens;
  float eps;
  float inv_d;
  float w_add;
};

// T: storage dtype of q/k; WT: weight dtype; L: lanes per head row
// (head_dim = 2 * L * N with N = 128-bit vector width in elements).
template <typename T, typename WT, int L>
__global__ void __launch_bounds__(kQkThreads) qk_norm_rope_kernel(const QkArgs a,
                                                                  const RopeTurns turns) {
  constexpr int N = Vec<T>::N;
  constexpr int HALF = L * N;
  constexpr int D = 2 * HALF;
  constexpr int G = kQkThreads / L;  // groups (head rows in flight) per block

  extern __shared__ float2 trig[];        // [tile_tokens][HALF] (cos, sin)
  __shared__ __align__(16) float wsm[2 * D];  // q weights then k weights (+ gemma 1)

  const int tid = threadIdx.x;
  const int lane = tid % L;
  const int group = tid / L;
  const int heads = a.hq + a.hk;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * a.tile_tokens;
  const int64_t left = a.tokens - t0;
  const int tc = left < a.tile_tokens ? static_cast<int>(left) : a.tile_tokens;
  const int rows_in_tile = tc * heads;

  // Issue this group's first head-row loads before the per-tile set-up, so
  // their latency overlaps the angle computation.
  uint4 va[kQkIter], vb[kQkIter];
  auto row_ptrs = [&](int r, const uint4*& src, uint4*& dst) {
    const int tt = r / heads;
    const int h = r - tt * heads;
    const int64_t tok = t0 + tt;
    if (h < a.hq) {
      const int64_t off = tok * a.q_stride + static_cast<int64_t>(h) * D;
      src = reinterpret_cast<const uint4*>(static_cast<const T*>(a.q) + off);
      dst = reinterpret_cast<uint4*>(static_cast<T*>(a.q_out) + off);
    } else {
      const int64_t off = tok * a.k_stride + static_cast<int64_t>(h - a.hq) * D;
      src = reinterpret_cast<const uint4*>(static_cast<const T*>(a.k) + off);
      dst = reinterpret_cast<uint4*>(static_cast<T*>(a.k_out) + off);
    }
  };
  auto issue_loads = [&](int chunk) {
#pragma unroll
    for (int it = 0; it < kQkIter; it++) {
      const int r = chunk + group + it * G;
      if (r < rows_in_tile) {
        const uint4* src;
        uint4* dst;
        row_ptrs(r, src, dst);
        va[it] = ld_stream(src + lane);
        vb[it] = ld_stream(src + L + lane);
      }
    }
  };
  issue_loads(0);

  // Per-tile set-up: weights (with the gemma +1) and the angles.
  const WT* wq = static_cast<const WT*>(a.wq);
  const WT* wk = static_cast<const WT*>(a.wk);
  for (int i = tid; i < 2 * D; i += kQkThreads) {
    float wv = 0.0f;
    if (i < D)
      wv = load_w<WT>(wq, i);
    else if (a.hk > 0)
      wv = load_w<WT>(wk, i - D);
    wsm[i] = wv + a.w_add;
  }
  for (int e = tid; e < tc * HALF; e += kQkThreads) {
    const int tt = e / HALF;
    const int i = e - tt * HALF;
    const int64_t p = a.pos[t0 + tt];
    // (p * turn_i) mod 2^64: the angle as a fraction of a turn, exact for any
    // int32 position (two's complement covers negative positions).
    const unsigned long long prod = static_cast<unsigned long long>(p) * turns.turn[i];
    const int hi = static_cast<int>(prod >> 32);  // signed turn fraction * 2^32
    float s, c;
    sincospif(static_cast<float>(hi) * 0x1p-31f, &s, &c);  // angle = pi * (hi / 2^31)
    trig[e] = make_float2(c, s);
  }
  __syncthreads();

  for (int chunk = 0; chunk < rows_in_tile; chunk += G * kQkIter) {
    if (chunk > 0) issue_loads(chunk);
#pragma unroll
    for (int it = 0; it < kQkIter; it++) {
      const int r = chunk + group + it * G;
      const bool valid = r < rows_in_tile;
      float xa[N], xb[N];
      float ss = 0.0f;
      if (valid) {
        Vec<T>::unpack(va[it], xa);
        Vec<T>::unpack(vb[it], xb);
#pragma unroll
        for (int e = 0; e < N; e++) {
          ss = fmaf(xa[e], xa[e], ss);
          ss = fmaf(xb[e], xb[e], ss);
        }
      }
      // Every lane joins the butterfly (full-warp shuffles), valid or not.
      ss = group_sum<L>(ss);
      if (valid) {
        const uint4* src;
        uint4* dst;
        row_ptrs(r, src, dst);
        const int tt = r / heads;
        const bool is_q = (r - tt * heads) < a.hq;
        const float inv = rsqrtf(ss * a.inv_d + a.eps);
        const float* w = wsm + (is_q ? 0 : D);
        const float2* cs = trig + tt * HALF + lane * N;
        float oa[N], ob[N];
#pragma unroll
        for (int e = 0; e < N; e++) {
          const float na = xa[e] * inv * w[lane * N + e];
          const float nb = xb[e] * inv * w[HALF + lane * N + e];
          const float2 t = cs[e];
          oa[e] = fmaf(na, t.x, -nb * t.y);
          ob[e] = fmaf(na, t.y, nb * t.x);
        }
        st_stream(dst + lane, Vec<T>::pack(oa));
        st_stream(dst + L + lane, Vec<T>::pack(ob));
      }
    }
  }
}

template <typename T, typename WT, int L>
cudaError_t launch_l(const QkArgs& a, const RopeTurns& turns, cudaStream_t s) {
  constexpr int HALF = L * Vec<T>::N;
  const int64_t tiles = (a.tokens + a.tile_tokens - 1) / a.tile_tokens;
  const size_t smem = static_cast<size_t>(a.tile_tokens) * HALF * sizeof(float2);
  qk_norm_rope_kernel<T, WT, L><<<dim3(static_cast<unsigned>(tiles)), kQkThreads, smem, s>>>(
      a, turns);
  return cudaGetLastError();
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

// Shared memory for the angle table is kept at or below this per block.
constexpr int kTrigSmemBytes = 32 * 1024;

cudaError_t launch_qk_norm_rope(void* q_out, void* k_out, const void* q, const void* k,
                                const void* wq, const void* wk, int w_is_bf16,
                                const int32_t* positions, int64_t tokens, int64_t hq, int64_t hk,
                                int64_t head_dim, int64_t q_tok_stride, int64_t k_tok_stride,
                                float eps, const RopeTurns& turns, int gemma, int is_bf16,
                                cudaStream_t stream) {
  const int n = is_bf16 ? 8 : 4;
  const int lanes = static_cast<int>(head_dim / (2 * n));
  const int groups = kQkThreads / lanes;
  const int64_t heads = hq + hk;
  // Tokens per block: enough head rows to fill every group kQkIter times,
  // bounded by the angle table's shared memory and by the token count.
  int64_t tile = (static_cast<int64_t>(groups) * kQkIter) / heads;
  const int64_t tile_max = kTrigSmemBytes / ((head_dim / 2) * static_cast<int64_t>(sizeof(float2)));
  if (tile > tile_max) tile = tile_max;
  if (tile > tokens) tile = tokens;
  if (tile < 1) tile = 1;

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
  a.tile_tokens = static_cast<int>(tile);
  a.eps = eps;
  a.inv_d = 1.0f / static_cast<float>(head_dim);
  a.w_add = gemma ? 1.0f : 0.0f;

  if (is_bf16) {
    if (w_is_bf16) return launch_w<__nv_bfloat16, __nv_bfloat16>(a, lanes, turns, stream);
    return launch_w<__nv_bfloat16, float>(a, lanes, turns, stream);
  }
  if (w_is_bf16) return launch_w<float, __nv_bfloat16>(a, lanes, turns, stream);
  return launch_w<float, float>(a, lanes, turns, stream);
}

}  // namespace nr
