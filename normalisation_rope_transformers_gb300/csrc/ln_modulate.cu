// LayerNorm (no affine) fused with adaLN modulation, for sm_103a.
//
// The fusion is named in the FastVideo PAN2 docs ("Performance switches",
// dit_fused_kernels: LayerNorm + modulation) without its formula; this computes
// the plain adaLN reading:
//   mu = mean(x), var = mean((x - mu)^2)  (biased, f32 statistics)
//   out = round((x - mu) / sqrt(var + eps) * (1 + scale) + shift)
// with shift/scale taken from sample row r / rows_per_sample.
//
// Design.  A row belongs to a group of WPR warps, the fewest that hold it
// with at most 8 128-bit vectors per thread (16 at 8 warps): one warp up to
// hidden 2048 bf16, two for the benchmark's 3072 (384 vectors = 6 per lane);
// a block of 64 threads holds 2 / WPR groups (a row of 2 or more warps is its
// own block).  The row is loaded once into registers, the mean and the centred
// variance are two reductions over the register-resident values (warp
// shuffles, plus one shared-memory step when WPR > 1), and the output is
// written once.  bf16 values enter PTX mixed-precision add/sub (.f32.bf16)
// without being unpacked first (RowMath).  Rows beyond 16 vectors per thread
// at 8 warps use a three-pass kernel that re-reads the (L2-resident) row.
// (Measured slower
// here and not used: a persistent variant streaming rows through a cp.async
// ring, which trades resident warps for ring depth; staging (1 + scale) and
// shift per block in shared memory, which re-reads them from L2 for every
// block instead of hitting L1; one warp x 12 vectors per 3072-wide row.)
#include "nr_common.cuh"
#include "nr_internal.h"

namespace nr {
namespace {

// Block size of a WPR-warp row group kernel: 128 threads, or one row group
// when a row needs more than 4 warps.
template <int WPR>
__host__ __device__ constexpr int ln_threads() {
  return WPR > 4 ? kWarp * WPR : 128;
}

// Block size of the LayerNorm kernel (a build-time knob): 64 threads, i.e. one
// row group of 2 warps per block for hidden 3072.  The same 20 rows are
// resident per SM at 48 registers, but a row that finishes frees its slot
// without waiting for a block-mate: measured 55.3 µs instead of 55.9 µs at
// [26598, 3072] (ncu, 16384 rows: 34.6 instead of 36.3 µs).  The gated kernel
// keeps 128-thread blocks (its register cap is chosen for them).
#ifndef NR_LN_BLOCK
#define NR_LN_BLOCK 64
#endif
template <int WPR>
__host__ __device__ constexpr int ln_row_threads() {
  return kWarp * WPR > NR_LN_BLOCK ? kWarp * WPR : NR_LN_BLOCK;
}

// Sum over the WPR warps of a row group; every thread of the group gets the
// same total.  `scratch` holds one float per warp of the block; the caller
// separates two uses of one scratch array by a barrier (or uses two arrays).
template <int WPR>
__device__ __forceinline__ float row_group_sum(float v, float* scratch) {
  v = group_sum<kWarp>(v);
  if (WPR == 1) return v;
  const int warp = threadIdx.x / kWarp;
  if (threadIdx.x % kWarp == 0) scratch[warp] = v;
  __syncthreads();
  const int first = (warp / WPR) * WPR;
  float total = 0.0f;
#pragma unroll
  for (int i = 0; i < WPR; i++) total += scratch[first + i];
  return total;
}

// 1: the bf16 LayerNorm row kernel widens its bf16 operands inside PTX
// mixed-precision add/sub (.f32.bf16) instead of unpacking them first (a
// build-time knob; the results are the same f32 operations).
#ifndef NR_LN_MIXED
#define NR_LN_MIXED 1
#endif

// Vector offset of row r's modulation sample, r / rows_per_sample * nvec:
// 0 without a division when one sample covers every row (the common case),
// a 32-bit division when both fit, else the 64-bit one.
__device__ __forceinline__ int64_t sample_offset(int64_t r, int64_t rows_per_sample,
                                                 int64_t rows, int nvec) {
  if (rows_per_sample >= rows) return 0;
  if (((r | rows_per_sample) >> 31) == 0)
    return static_cast<int64_t>(static_cast<uint32_t>(r) /
                                static_cast<uint32_t>(rows_per_sample)) * nvec;
  return (r / rows_per_sample) * nvec;
}

// The three per-vector steps of LayerNorm + modulation: add the values to a
// running sum, add their squared deviations from mu, and modulate them.  For
// bf16 with NR_LN_MIXED the bf16 operands enter PTX mixed-precision
// instructions directly (same f32 results, fewer instructions).
template <typename T, bool MIXED = (NR_LN_MIXED && sizeof(T) == 2)>
struct RowMath {
  static constexpr int N = Vec<T>::N;
  __device__ __forceinline__ static float sum(const uint4& u, float acc) {
    float v[N];
    Vec<T>::unpack(u, v);
#pragma unroll
    for (int e = 0; e < N; e++) acc += v[e];
    return acc;
  }
  __device__ __forceinline__ static float dev(const uint4& u, float mu, float acc) {
    float v[N];
    Vec<T>::unpack(u, v);
#pragma unroll
    for (int e = 0; e < N; e++) {
      const float d = v[e] - mu;
      acc = fmaf(d, d, acc);
    }
    return acc;
  }
  __device__ __forceinline__ static uint4 modulate(const uint4& u, float mu, float rstd,
                                                   const uint4& shp, const uint4& scp) {
    float v[N], sh[N], sc[N];
    Vec<T>::unpack(u, v);
    Vec<T>::unpack(shp, sh);
    Vec<T>::unpack(scp, sc);
#pragma unroll
    for (int e = 0; e < N; e++) v[e] = fmaf((v[e] - mu) * rstd, 1.0f + sc[e], sh[e]);
    return Vec<T>::pack(v);
  }
};

template <typename T>
struct RowMath<T, true> {
  static constexpr int N = 8;
  __device__ __forceinline__ static float sum(const uint4& u, float acc) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int q = 0; q < 4; q++) {
      acc = add_bf16<false>(w[q], acc);
      acc = add_bf16<true>(w[q], acc);
    }
    return acc;
  }
  __device__ __forceinline__ static float dev(const uint4& u, float mu, float acc) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int q = 0; q < 4; q++) {
      const float d0 = sub_bf16<false>(w[q], mu);
      acc = fmaf(d0, d0, acc);
      const float d1 = sub_bf16<true>(w[q], mu);
      acc = fmaf(d1, d1, acc);
    }
    return acc;
  }
  __device__ __forceinline__ static uint4 modulate(const uint4& u, float mu, float rstd,
                                                   const uint4& shp, const uint4& scp) {
    const uint32_t x[4] = {u.x, u.y, u.z, u.w};
    const uint32_t h[4] = {shp.x, shp.y, shp.z, shp.w};
    const uint32_t c[4] = {scp.x, scp.y, scp.z, scp.w};
    float v[N];
#pragma unroll
    for (int q = 0; q < 4; q++) {
      v[2 * q] = fmaf(sub_bf16<false>(x[q], mu) * rstd, add_bf16<false>(c[q], 1.0f),
                      bf16_lo(h[q]));
      v[2 * q + 1] = fmaf(sub_bf16<true>(x[q], mu) * rstd, add_bf16<true>(c[q], 1.0f),
                          bf16_hi(h[q]));
    }
    return Vec<__nv_bfloat16>::pack(v);
  }
};

// Rows ahead of its own whose inputs a gated row group asks L2 to prefetch,
// as a multiple of the row groups resident at once (a build-time knob; 0:
// none).  A block launched later for that row then finds it in L2, so HBM
// keeps a resident set's worth of rows more in flight than registers alone
// allow.  Measured at [26598, 3072]: 98.5 -> 97.1 µs with one set ahead (two:
// 114.5 µs); the same prefetch slowed LayerNorm + modulation (53.7 -> 54.7 µs),
// which has none.
#ifndef NR_GATED_L2PF
#define NR_GATED_L2PF 1
#endif

template <typename T, int VPT, int WPR>
__global__ void __launch_bounds__(ln_row_threads<WPR>()) ln_modulate_rows_kernel(
    T* __restrict__ out, const T* __restrict__ x, const T* __restrict__ shift,
    const T* __restrict__ scale, int64_t rows, int nvec, int64_t rows_per_sample, float hidden_f,
    float inv_hidden, float eps) {
  pdl_enter();  // before any global read: the previous kernel may still run
  constexpr int THREADS = ln_row_threads<WPR>();
  constexpr int TPR = kWarp * WPR;       // threads per row
  constexpr int RPB = THREADS / TPR;     // rows per block
  static_assert(RPB >= 1 && RPB * TPR == THREADS, "row groups must tile the block");
  __shared__ float scratch_mean[THREADS / kWarp];
  __shared__ float scratch_var[THREADS / kWarp];
  const int t = threadIdx.x % TPR;
  {
    const int64_t row = static_cast<int64_t>(blockIdx.x) * RPB + threadIdx.x / TPR;
    // Rows past the end still take part in the reductions' barriers (WPR > 1).
    // A block of one row group is never past the end (one block per row).
    const bool active = RPB == 1 || row < rows;
    const int64_t r = active ? row : 0;
    const uint4* xr = reinterpret_cast<const uint4*>(x) + r * nvec;
    uint4* orow = reinterpret_cast<uint4*>(out) + r * nvec;
    const int64_t sample_off = sample_offset(r, rows_per_sample, rows, nvec);
    const uint4* shv = reinterpret_cast<const uint4*>(shift) + sample_off;
    const uint4* scv = reinterpret_cast<const uint4*>(scale) + sample_off;
    auto in_row = [&](int k) { return t + k * TPR < nvec; };

    uint4 xv[VPT];
#pragma unroll
    for (int k = 0; k < VPT; k++)
      if (active && in_row(k)) xv[k] = ld_stream(xr + t + k * TPR);

    float sum = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; k++)
      if (active && in_row(k)) sum = RowMath<T>::sum(xv[k], sum);
    const float mu = row_mean_of(row_group_sum<WPR>(sum, scratch_mean), hidden_f, inv_hidden);

    float dev = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; k++)
      if (active && in_row(k)) dev = RowMath<T>::dev(xv[k], mu, dev);
    const float rstd = row_rstd_of(
        row_mean_of(row_group_sum<WPR>(dev, scratch_var), hidden_f, inv_hidden), eps);
    if (!active) return;

#pragma unroll
    for (int k = 0; k < VPT; k++) {
      const int vi = t + k * TPR;
      if (in_row(k))
        st_stream(orow + vi,
                  RowMath<T>::modulate(xv[k], mu, rstd, ld_param(shv + vi), ld_param(scv + vi)));
    }
  }
}

// ---------------------------------------------------------------------------
// Gated residual + LayerNorm + modulation: residual <- round(residual + gate*y)
// (one rounding of the exact value), then out = LN(residual)*(1+scale)+shift.
// ---------------------------------------------------------------------------
template <typename T>
struct GatedAdd;

template <>
struct GatedAdd<float> {
  // fmaf rounds the exact r + g*y once.
  __device__ __forceinline__ static uint4 apply(const uint4& r, const uint4& g, const uint4& y) {
    float rv[4], gv[4], yv[4];
    Vec<float>::unpack(r, rv);
    Vec<float>::unpack(g, gv);
    Vec<float>::unpack(y, yv);
#pragma unroll
    for (int e = 0; e < 4; e++) rv[e] = fmaf(gv[e], yv[e], rv[e]);
    return Vec<float>::pack(rv);
  }
};

template <>
struct GatedAdd<__nv_bfloat16> {
  // g*y of two bf16 values is exact in f32.  The sum with r is rounded to odd
  // in f32: the sums rounded down and up are equal when the sum is exact (the
  // upward one then carries the sign IEEE gives an exact zero), and otherwise
  // are the two floats around it, of which the one with an odd last bit is
  // taken.  f32 keeps 16 more bits than bf16 (at least two are needed), so
  // rounding that to nearest bf16 rounds the exact r + g*y once (Boldo and
  // Melquiond, "Emulation of FMA and correctly rounded sums: proved
  // algorithms using rounding to odd", IEEE Trans. Computers 57(4), 2008).
  // With NR_LN_MIXED the two directed sums are mixed-precision fmas of the
  // bf16 gate and y (an exact product) and the f32 residual.
  __device__ __forceinline__ static uint4 apply(const uint4& r, const uint4& g, const uint4& y) {
    float odd[8];
    if constexpr (NR_LN_MIXED) {
      const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
      const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
      const uint32_t yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int q = 0; q < 4; q++) {
        float down, up;
        fma_bf16_down_up<false>(gw[q], yw[q], bf16_lo(rw[q]), down, up);
        odd[2 * q] = (down != up && (__float_as_uint(down) & 1u)) ? down : up;
        fma_bf16_down_up<true>(gw[q], yw[q], bf16_hi(rw[q]), down, up);
        odd[2 * q + 1] = (down != up && (__float_as_uint(down) & 1u)) ? down : up;
      }
    } else {
      float rv[8], gv[8], yv[8];
      Vec<__nv_bfloat16>::unpack(r, rv);
      Vec<__nv_bfloat16>::unpack(g, gv);
      Vec<__nv_bfloat16>::unpack(y, yv);
#pragma unroll
      for (int e = 0; e < 8; e++) {
        const float p = gv[e] * yv[e];
        const float down = __fadd_rd(p, rv[e]);
        const float up = __fadd_ru(p, rv[e]);
        odd[e] = (down != up && (__float_as_uint(down) & 1u)) ? down : up;
      }
    }
    return Vec<__nv_bfloat16>::pack(odd);
  }
};

// Resident 128-thread equivalents per SM asked of the compiler for the gated
// kernel with bf16 rows of at most 6 vectors per thread and stream (a
// build-time knob): 7 caps it at 72 registers without spills (70 used), so
// 14 rows of 3072 are in flight per SM instead of 12 with the 85-register
// build of the TwoSum rounding (measured 3% faster at [26598, 3072]); 8 (64
// registers) spills.  Other geometries ask for 4, which leaves them unspilled.
#ifndef NR_GATED_MINB
#define NR_GATED_MINB 7
#endif

// Block size of the gated kernel for rows of 2 or more warps (a build-time
// knob; one-warp rows keep 128-thread blocks): 64 threads, one row per block,
// measured 106.9 µs instead of 108.1 µs (two rows per 128-thread block) at
// [26598, 3072], with the same register cap.
#ifndef NR_GATED_BLOCK
#define NR_GATED_BLOCK 64
#endif
template <int WPR>
__host__ __device__ constexpr int gated_threads() {
  return WPR == 1 ? 128 : (kWarp * WPR > NR_GATED_BLOCK ? kWarp * WPR : NR_GATED_BLOCK);
}

// Minimum blocks per SM, counted so that the register cap is the same for
// any block size (NR_GATED_MINB is per 128 threads).
template <typename T, int VPT, int WPR>
__host__ __device__ constexpr int gated_min_blocks() {
  constexpr int per128 = (sizeof(T) == 2 && VPT <= 6) ? NR_GATED_MINB : 4;
  return per128 * 128 / gated_threads<WPR>() > 0 ? per128 * 128 / gated_threads<WPR>() : 1;
}

template <typename T, int VPT, int WPR>
__global__ void __launch_bounds__(gated_threads<WPR>(), gated_min_blocks<T, VPT, WPR>())
    gated_ln_modulate_kernel(
    T* __restrict__ out, T* __restrict__ residual, const T* __restrict__ y,
    const T* __restrict__ gate, const T* __restrict__ shift, const T* __restrict__ scale,
    int64_t rows, int nvec, int64_t rows_per_sample, float hidden_f, float inv_hidden, float eps,
    int64_t prefetch_rows) {
  pdl_enter();  // before any global read: the previous kernel may still run
  constexpr int THREADS = gated_threads<WPR>();
  constexpr int TPR = kWarp * WPR;
  constexpr int RPB = THREADS / TPR;
  static_assert(RPB >= 1 && RPB * TPR == THREADS, "row groups must tile the block");
  __shared__ float scratch_mean[THREADS / kWarp];
  __shared__ float scratch_var[THREADS / kWarp];
  const int t = threadIdx.x % TPR;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * RPB + threadIdx.x / TPR;
  const bool active = row < rows;
  const int64_t r = active ? row : 0;
  uint4* rr = reinterpret_cast<uint4*>(residual) + r * nvec;
  const uint4* yr = reinterpret_cast<const uint4*>(y) + r * nvec;
  uint4* orow = reinterpret_cast<uint4*>(out) + r * nvec;
  const int64_t sample_off = sample_offset(r, rows_per_sample, rows, nvec);
  const uint4* gv = reinterpret_cast<const uint4*>(gate) + sample_off;
  const uint4* shv = reinterpret_cast<const uint4*>(shift) + sample_off;
  const uint4* scv = reinterpret_cast<const uint4*>(scale) + sample_off;

  uint4 xv[VPT], yv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int vi = t + k * TPR;
    if (active && vi < nvec) {
      xv[k] = ld_stream(rr + vi);
      yv[k] = ld_stream(yr + vi);
    }
  }
  if (prefetch_rows > 0 && t == 0 && active && row + prefetch_rows < rows) {
    bulk_prefetch_l2(rr + prefetch_rows * nvec, static_cast<unsigned>(nvec) * 16u);
    bulk_prefetch_l2(yr + prefetch_rows * nvec, static_cast<unsigned>(nvec) * 16u);
  }
  float sum = 0.0f;
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int vi = t + k * TPR;
    if (active && vi < nvec) {
      xv[k] = GatedAdd<T>::apply(xv[k], ld_param(gv + vi), yv[k]);
      st_stream(rr + vi, xv[k]);
      sum = RowMath<T>::sum(xv[k], sum);
    }
  }
  const float mu = row_mean_of(row_group_sum<WPR>(sum, scratch_mean), hidden_f, inv_hidden);
  float dev = 0.0f;
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int vi = t + k * TPR;
    if (active && vi < nvec) dev = RowMath<T>::dev(xv[k], mu, dev);
  }
  const float rstd = row_rstd_of(
      row_mean_of(row_group_sum<WPR>(dev, scratch_var), hidden_f, inv_hidden), eps);
  if (!active) return;
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int vi = t + k * TPR;
    if (vi < nvec)
      st_stream(orow + vi,
                RowMath<T>::modulate(xv[k], mu, rstd, ld_param(shv + vi), ld_param(scv + vi)));
  }
}

template <typename T>
__global__ void __launch_bounds__(1024) ln_modulate_long_row_kernel(
    T* __restrict__ out, const T* __restrict__ x, const T* __restrict__ shift,
    const T* __restrict__ scale, int64_t nvec, int64_t rows_per_sample, float hidden_f,
    float inv_hidden, float eps) {
  pdl_enter();  // before any global read: the previous kernel may still run
  constexpr int N = Vec<T>::N;
  __shared__ float scratch_mean[32];
  __shared__ float scratch_var[32];
  const int64_t row = blockIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(x) + row * nvec;
  uint4* orow = reinterpret_cast<uint4*>(out) + row * nvec;
  const int64_t sample_off = (row / rows_per_sample) * nvec;
  const uint4* shv = reinterpret_cast<const uint4*>(shift) + sample_off;
  const uint4* scv = reinterpret_cast<const uint4*>(scale) + sample_off;

  float sum = 0.0f;
  for (int64_t vi = threadIdx.x; vi < nvec; vi += blockDim.x) {
    float v[N];
    Vec<T>::unpack(ld_coherent(xr + vi), v);
#pragma unroll
    for (int e = 0; e < N; e++) sum += v[e];
  }
  const float mu = row_mean_of(block_sum(sum, scratch_mean), hidden_f, inv_hidden);
  float dev = 0.0f;
  for (int64_t vi = threadIdx.x; vi < nvec; vi += blockDim.x) {
    float v[N];
    Vec<T>::unpack(ld_coherent(xr + vi), v);
#pragma unroll
    for (int e = 0; e < N; e++) {
      const float d = v[e] - mu;
      dev = fmaf(d, d, dev);
    }
  }
  const float rstd =
      row_rstd_of(row_mean_of(block_sum(dev, scratch_var), hidden_f, inv_hidden), eps);
  // out may alias x: each thread overwrites only vectors it has finished reading.
  for (int64_t vi = threadIdx.x; vi < nvec; vi += blockDim.x) {
    float v[N], sh[N], sc[N];
    Vec<T>::unpack(ld_coherent(xr + vi), v);
    Vec<T>::unpack(ld_param(shv + vi), sh);
    Vec<T>::unpack(ld_param(scv + vi), sc);
#pragma unroll
    for (int e = 0; e < N; e++) v[e] = fmaf((v[e] - mu) * rstd, 1.0f + sc[e], sh[e]);
    st_stream(orow + vi, Vec<T>::pack(v));
  }
}

struct LnArgs {
  void* out;
  const void* x;
  const void* shift;
  const void* scale;
  int64_t rows;
  int nvec;
  int64_t rps;
  float hidden_f;
  float inv_hidden;
  float eps;
};

template <typename T, int VPT, int WPR>
cudaError_t launch_rows(const LnArgs& a, cudaStream_t s) {
  constexpr int THREADS = ln_row_threads<WPR>();
  constexpr int RPB = THREADS / (kWarp * WPR);
  static_assert(RPB >= 1, "row groups must fit the block");
  const int64_t blocks = (a.rows + RPB - 1) / RPB;
  return launch_pdl(ln_modulate_rows_kernel<T, VPT, WPR>, dim3(static_cast<unsigned>(blocks)), dim3(THREADS), 0, s,
      static_cast<T*>(a.out), static_cast<const T*>(a.x), static_cast<const T*>(a.shift),
      static_cast<const T*>(a.scale), a.rows, a.nvec, a.rps, a.hidden_f, a.inv_hidden, a.eps);
}

// Vectors per thread offered for one-warp rows, and for rows spread over
// 2, 4 or 8 warps.  A row takes the fewest warps that hold it with at most 8
// vectors per thread (16 at 8 warps): hidden 3072 bf16 runs on 2 warps x 6
// vectors, measured 4-5% faster than 1 warp x 12 (shorter per-row chain of
// reductions, fewer registers, more rows in flight per SM).
constexpr int kLnVptOneWarp[] = {1, 2, 3, 4, 6, 8};
constexpr int kLnVptMultiWarp[] = {6, 8, 12, 16};

template <typename T>
cudaError_t launch_typed(const LnArgs& a, cudaStream_t s) {
  const int64_t nvec = a.nvec;
  for (int wpr : {1, 2, 4, 8}) {
    const int64_t need = (nvec + kWarp * wpr - 1) / (kWarp * wpr);
    if (need > (wpr == 8 ? 16 : 8)) continue;
    int vpt = 0;
    if (wpr == 1) {
      for (int v : kLnVptOneWarp)
        if (vpt == 0 && v >= need) vpt = v;
    } else {
      for (int v : kLnVptMultiWarp)
        if (vpt == 0 && v >= need) vpt = v;
    }
    switch (wpr * 100 + vpt) {
      case 101: return launch_rows<T, 1, 1>(a, s);
      case 102: return launch_rows<T, 2, 1>(a, s);
      case 103: return launch_rows<T, 3, 1>(a, s);
      case 104: return launch_rows<T, 4, 1>(a, s);
      case 106: return launch_rows<T, 6, 1>(a, s);
      case 108: return launch_rows<T, 8, 1>(a, s);
      case 206: return launch_rows<T, 6, 2>(a, s);
      case 208: return launch_rows<T, 8, 2>(a, s);
      case 406: return launch_rows<T, 6, 4>(a, s);
      case 408: return launch_rows<T, 8, 4>(a, s);
      case 806: return launch_rows<T, 6, 8>(a, s);
      case 808: return launch_rows<T, 8, 8>(a, s);
      case 812: return launch_rows<T, 12, 8>(a, s);
      case 816: return launch_rows<T, 16, 8>(a, s);
      default: break;
    }
  }
  return launch_pdl(ln_modulate_long_row_kernel<T>, dim3(static_cast<unsigned>(a.rows)), dim3(1024),
                    0, s,
      static_cast<T*>(a.out), static_cast<const T*>(a.x), static_cast<const T*>(a.shift),
      static_cast<const T*>(a.scale), nvec, a.rps, a.hidden_f, a.inv_hidden, a.eps);
}

struct GatedArgs {
  void* out;
  void* residual;
  const void* y;
  const void* gate;
  const void* shift;
  const void* scale;
  int64_t rows;
  int nvec;
  int64_t rps;
  float hidden_f;
  float inv_hidden;
  float eps;
};

template <typename T, int VPT, int WPR>
cudaError_t launch_gated_rows(const GatedArgs& a, cudaStream_t s) {
  constexpr int THREADS = gated_threads<WPR>();
  constexpr int RPB = THREADS / (kWarp * WPR);
  const int64_t blocks = (a.rows + RPB - 1) / RPB;
  int64_t prefetch_rows = 0;
  if (NR_GATED_L2PF > 0) {
    static std::atomic<int> cache[64];
    int resident = 0;
    const cudaError_t e =
        resident_blocks(gated_ln_modulate_kernel<T, VPT, WPR>, THREADS, cache, &resident);
    if (e != cudaSuccess) return e;
    prefetch_rows = static_cast<int64_t>(NR_GATED_L2PF) * resident * RPB;
  }
  return launch_pdl(gated_ln_modulate_kernel<T, VPT, WPR>, dim3(static_cast<unsigned>(blocks)),
                    dim3(THREADS), 0, s,
      static_cast<T*>(a.out), static_cast<T*>(a.residual), static_cast<const T*>(a.y),
      static_cast<const T*>(a.gate), static_cast<const T*>(a.shift),
      static_cast<const T*>(a.scale), a.rows, a.nvec, a.rps, a.hidden_f, a.inv_hidden, a.eps,
      prefetch_rows);
}

template <typename T>
cudaError_t launch_gated_typed(const GatedArgs& a, cudaStream_t s) {
  for (int wpr : {1, 2, 4}) {
    const int64_t need = (a.nvec + kWarp * wpr - 1) / (kWarp * wpr);
    const int vpt = need <= 2 ? 2 : need <= 4 ? 4 : need <= 6 ? 6 : need <= 8 ? 8 : 0;
    switch (wpr * 100 + vpt) {
      case 102: return launch_gated_rows<T, 2, 1>(a, s);
      case 104: return launch_gated_rows<T, 4, 1>(a, s);
      case 106: return launch_gated_rows<T, 6, 1>(a, s);
      case 108: return launch_gated_rows<T, 8, 1>(a, s);
      case 206: return launch_gated_rows<T, 6, 2>(a, s);
      case 208: return launch_gated_rows<T, 8, 2>(a, s);
      case 406: return launch_gated_rows<T, 6, 4>(a, s);
      case 408: return launch_gated_rows<T, 8, 4>(a, s);
      default: break;
    }
  }
  return cudaErrorNotSupported;  // rows beyond kGatedMaxVectors (rejected by the ABI first)
}

}  // namespace

cudaError_t launch_gated_ln_modulate(void* out, void* residual, const void* y, const void* gate,
                                     const void* shift, const void* scale, int64_t rows,
                                     int64_t hidden, int64_t rows_per_sample, int is_bf16,
                                     float eps, cudaStream_t stream) {
  GatedArgs a;
  a.out = out;
  a.residual = residual;
  a.y = y;
  a.gate = gate;
  a.shift = shift;
  a.scale = scale;
  a.rows = rows;
  a.nvec = static_cast<int>(hidden / (is_bf16 ? 8 : 4));
  a.rps = rows_per_sample;
  a.hidden_f = static_cast<float>(hidden);
  a.inv_hidden = 1.0f / a.hidden_f;
  a.eps = eps;
  if (is_bf16) return launch_gated_typed<__nv_bfloat16>(a, stream);
  return launch_gated_typed<float>(a, stream);
}

cudaError_t launch_ln_modulate(void* out, const void* x, const void* shift, const void* scale,
                               int64_t rows, int64_t hidden, int64_t rows_per_sample,
                               int is_bf16, float eps, cudaStream_t stream) {
  LnArgs a;
  a.out = out;
  a.x = x;
  a.shift = shift;
  a.scale = scale;
  a.rows = rows;
  a.nvec = static_cast<int>(hidden / (is_bf16 ? 8 : 4));
  a.rps = rows_per_sample;
  a.hidden_f = static_cast<float>(hidden);
  a.inv_hidden = 1.0f / a.hidden_f;
  a.eps = eps;
  if (is_bf16) return launch_typed<__nv_bfloat16>(a, stream);
  return launch_typed<float>(a, stream);
}

}  // namespace nr
