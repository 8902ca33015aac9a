// RMSNorm with the optional fused residual add, for sm_103a.
//
// Computes what the vllm.cpp page src/vt/cuda/cuda_ops.cu gives in its
// row-RMSNorm section and the residual-rounding helper before it:
// v = round(x + residual) (written back in place),
// inv = 1/sqrt(mean(v^2) + eps), out = round(v * inv * (w [+1])).
//
// Design (not the page's): the page's kernel walks a row twice with scalar
// loads and a 256-wide shared-memory tree.  Here each row is held in
// registers: a block owns one row, each thread loads VPT 128-bit vectors of x
// (and of the residual) once, writes the rounded residual back immediately,
// and the row's sum of squares is reduced with warp shuffles plus one
// shared-memory step.  Each row is read from HBM once and written once.
// Rows longer than the register budget use a two-pass kernel that re-reads
// the (L2-resident) row.
#include <type_traits>

#include "nr_common.cuh"
#include "nr_internal.h"

namespace nr {
namespace {

// How a normalised vector leaves the kernel.
struct StoreOut {  // out = round_T(n)
  void* out;
};
struct StoreFp8 {  // e4m3 code of f32(round_bf16(n)) * inv_scale; optionally the bf16 value too
  uint8_t* codes;
  __nv_bfloat16* nb;  // may be null
  float inv_scale;
};

template <typename T>
__device__ __forceinline__ void store_normed(const StoreOut& e, int64_t vec_index,
                                             const float (&v)[Vec<T>::N]) {
  st_stream(reinterpret_cast<uint4*>(e.out) + vec_index, Vec<T>::pack(v));
}

template <typename T>
__device__ __forceinline__ void store_normed(const StoreFp8& e, int64_t vec_index,
                                             const float (&v)[Vec<T>::N]) {
  constexpr int N = Vec<T>::N;
  uint32_t packed[N / 2];
  float code_in[N];
#pragma unroll
  for (int j = 0; j < N / 2; j++) {
    packed[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);  // the bf16-rounded normed values
    code_in[2 * j] = bf16_lo(packed[j]) * e.inv_scale;
    code_in[2 * j + 1] = bf16_hi(packed[j]) * e.inv_scale;
  }
  const int64_t elem = vec_index * N;
  if constexpr (N == 8) {
    const uint2 c = make_uint2(e4m3x2(code_in[0], code_in[1]) | (e4m3x2(code_in[2], code_in[3]) << 16),
                               e4m3x2(code_in[4], code_in[5]) | (e4m3x2(code_in[6], code_in[7]) << 16));
    st_stream8(e.codes + elem, c);
    if (e.nb != nullptr) st_stream(e.nb + elem, make_uint4(packed[0], packed[1], packed[2], packed[3]));
  } else {
    st_stream4(e.codes + elem, e4m3x2(code_in[0], code_in[1]) | (e4m3x2(code_in[2], code_in[3]) << 16));
    if (e.nb != nullptr) st_stream8(e.nb + elem, make_uint2(packed[0], packed[1]));
  }
}

// The residual add and the sum of squares of one 128-bit vector.
template <typename T>
struct RmsMath {
  static constexpr int N = Vec<T>::N;
  // round_T(x + r) elementwise: for bf16 the f32 sum is exact when the
  // exponents differ by at most 15 and otherwise far from a bf16 midpoint, so
  // one rounding of it equals rounding the exact sum.
  __device__ __forceinline__ static uint4 add(const uint4& x, const uint4& r) {
    float v[N], rv[N];
    Vec<T>::unpack(x, v);
    Vec<T>::unpack(r, rv);
#pragma unroll
    for (int e = 0; e < N; e++) v[e] += rv[e];
    return Vec<T>::pack(v);
  }
  __device__ __forceinline__ static float sumsq(const uint4& u, float acc) {
    float v[N];
    Vec<T>::unpack(u, v);
#pragma unroll
    for (int e = 0; e < N; e++) acc = fmaf(v[e], v[e], acc);
    return acc;
  }
};

// One block per row; thread t owns vectors t, t + blockDim, ..., (VPT of them).
// PW: load the weight together with the row (saves a dependent round trip when
// there are few rows, e.g. decode; costs registers when there are many).
// Threads per block of the few-row geometry (at most 2 vectors per thread).
constexpr int kDecodeMaxThreads = 1024;

template <typename T, int VPT, bool RES, bool PW, typename EPI>
__global__ void __launch_bounds__((PW && VPT <= 2) ? kDecodeMaxThreads : kRowMaxThreads)
    rmsnorm_row_kernel(const EPI epi,
                                                           const T* __restrict__ x,
                                                           const T* __restrict__ w,
                                                           T* __restrict__ res, int nvec,
                                                           float hidden_f, float inv_hidden,
                                                           float eps, float w_add, int64_t rows,
                                                           int64_t prefetch_rows) {
  pdl_enter();  // before any global read: the previous kernel may still run
  constexpr int N = Vec<T>::N;
  __shared__ float scratch[32];
  const int64_t row_off = static_cast<int64_t>(blockIdx.x) * nvec;  // in vectors
  const uint4* xr = reinterpret_cast<const uint4*>(x) + row_off;
  uint4* rr = RES ? reinterpret_cast<uint4*>(res) + row_off : nullptr;
  const uint4* wv = reinterpret_cast<const uint4*>(w);

  uint4 xv[VPT];
  uint4 rv[VPT];
  uint4 wpre[PW ? VPT : 1];
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int vi = threadIdx.x + k * blockDim.x;
    if (vi < nvec) {
      xv[k] = ld_stream(xr + vi);
      if (RES) rv[k] = ld_stream(rr + vi);
      if (PW) wpre[PW ? k : 0] = ld_param(wv + vi);
    }
  }
  if (prefetch_rows > 0 && threadIdx.x == 0 && blockIdx.x + prefetch_rows < rows) {
    bulk_prefetch_l2(xr + prefetch_rows * nvec, static_cast<unsigned>(nvec) * 16u);
    if (RES) bulk_prefetch_l2(rr + prefetch_rows * nvec, static_cast<unsigned>(nvec) * 16u);
  }

  float sum_sq = 0.0f;
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int vi = threadIdx.x + k * blockDim.x;
    if (vi < nvec) {
      if (RES) {
        // Rounded to the residual's storage dtype: the rounded value is both
        // written back and squared.
        xv[k] = RmsMath<T>::add(xv[k], rv[k]);
        st_stream(rr + vi, xv[k]);
      }
      sum_sq = RmsMath<T>::sumsq(xv[k], sum_sq);
    }
  }

  const float total = block_sum(sum_sq, scratch);
  const float inv = row_rstd_of(row_mean_of(total, hidden_f, inv_hidden), eps);

#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int vi = threadIdx.x + k * blockDim.x;
    if (vi < nvec) {
      float v[N], wf[N];
      Vec<T>::unpack(xv[k], v);
      Vec<T>::unpack(PW ? wpre[PW ? k : 0] : ld_param(wv + vi), wf);
#pragma unroll
      for (int e = 0; e < N; e++) v[e] = v[e] * inv * (wf[e] + w_add);
      store_normed<T>(epi, row_off + vi, v);
    }
  }
}

// Rows too long for registers: pass 1 adds, writes the residual and reduces;
// pass 2 re-reads the stored values (L2-resident) and normalises.
template <typename T, bool RES>
__global__ void __launch_bounds__(1024) rmsnorm_long_row_kernel(T* __restrict__ out,
                                                                const T* __restrict__ x,
                                                                const T* __restrict__ w,
                                                                T* __restrict__ res, int64_t nvec,
                                                                float hidden_f,
                                                                float inv_hidden, float eps,
                                                                float w_add) {
  pdl_enter();  // before any global read: the previous kernel may still run
  constexpr int N = Vec<T>::N;
  __shared__ float scratch[32];
  const int64_t row_off = static_cast<int64_t>(blockIdx.x) * nvec;
  const uint4* xr = reinterpret_cast<const uint4*>(x) + row_off;
  uint4* rr = RES ? reinterpret_cast<uint4*>(res) + row_off : nullptr;
  uint4* orow = reinterpret_cast<uint4*>(out) + row_off;
  const uint4* wv = reinterpret_cast<const uint4*>(w);

  float sum_sq = 0.0f;
  for (int64_t vi = threadIdx.x; vi < nvec; vi += blockDim.x) {
    float v[N];
    Vec<T>::unpack(ld_coherent(xr + vi), v);
    if (RES) {
      float r[N];
      Vec<T>::unpack(ld_coherent(rr + vi), r);
#pragma unroll
      for (int e = 0; e < N; e++) v[e] += r[e];
      const uint4 packed = Vec<T>::pack(v);
      st_plain(rr + vi, packed);
      Vec<T>::unpack(packed, v);
    }
#pragma unroll
    for (int e = 0; e < N; e++) sum_sq = fmaf(v[e], v[e], sum_sq);
  }
  const float total = block_sum(sum_sq, scratch);
  const float inv = row_rstd_of(row_mean_of(total, hidden_f, inv_hidden), eps);
  // Each thread re-reads only the vectors it wrote itself, so program order
  // makes its own residual stores visible to it.
  for (int64_t vi = threadIdx.x; vi < nvec; vi += blockDim.x) {
    float v[N], wf[N];
    Vec<T>::unpack(RES ? ld_coherent(rr + vi) : ld_coherent(xr + vi), v);
    Vec<T>::unpack(ld_param(wv + vi), wf);
#pragma unroll
    for (int e = 0; e < N; e++) v[e] = v[e] * inv * (wf[e] + w_add);
    st_stream(orow + vi, Vec<T>::pack(v));
  }
}

// Rows ahead of its own whose input a many-row block asks L2 to prefetch, as
// a multiple of the blocks resident at once (build-time knobs; 0: none), for
// the plain output and for the FP8 epilogue.  Measured at [8192, 5120]: the
// FP8 kernel 45.2 -> 43.8 µs with one resident set ahead; add + RMSNorm
// 53.4 -> 54.6 µs, so it prefetches nothing.
#ifndef NR_RMS_L2PF
#define NR_RMS_L2PF 0
#endif
#ifndef NR_FP8_L2PF
#define NR_FP8_L2PF 1
#endif

template <typename T, int VPT, bool RES, bool PW, typename EPI>
cudaError_t launch_rows_res(const RowLaunch& g, const EPI& epi, const void* x, const void* w,
                            void* res, int64_t rows, int nvec, float hidden_f, float eps,
                            float w_add, cudaStream_t s) {
  auto kernel = rmsnorm_row_kernel<T, VPT, RES, PW, EPI>;
  constexpr int PF = std::is_same<EPI, StoreFp8>::value ? NR_FP8_L2PF : NR_RMS_L2PF;
  int64_t prefetch_rows = 0;
  if (PF > 0 && !PW) {
    static std::atomic<int> cache[64];
    int resident = 0;
    const cudaError_t e = resident_blocks(kernel, g.threads, cache, &resident);
    if (e != cudaSuccess) return e;
    prefetch_rows = static_cast<int64_t>(PF) * resident;
  }
  return launch_pdl(kernel, dim3(static_cast<unsigned>(rows)), dim3(g.threads), 0, s, epi,
                    static_cast<const T*>(x), static_cast<const T*>(w), static_cast<T*>(res), nvec,
                    hidden_f, 1.0f / hidden_f, eps, w_add, rows, prefetch_rows);
}

template <typename T, int VPT, bool PW, typename EPI>
cudaError_t launch_rows_pw(const RowLaunch& g, const EPI& epi, const void* x, const void* w,
                           void* res, int64_t rows, int nvec, float hidden_f, float eps,
                           float w_add, cudaStream_t s) {
  if (res != nullptr)
    return launch_rows_res<T, VPT, true, PW>(g, epi, x, w, res, rows, nvec, hidden_f, eps, w_add,
                                             s);
  return launch_rows_res<T, VPT, false, PW>(g, epi, x, w, nullptr, rows, nvec, hidden_f, eps,
                                            w_add, s);
}

// Rows per launch up to which the weight is fetched together with the row.
constexpr int64_t kPrefetchWeightRows = 1024;

template <typename T, int VPT, typename EPI>
cudaError_t launch_rows(const RowLaunch& g, const EPI& epi, const void* x, const void* w,
                        void* res, int64_t rows, int nvec, float hidden_f, float eps, float w_add,
                        cudaStream_t s) {
  if (rows <= kPrefetchWeightRows)
    return launch_rows_pw<T, VPT, true>(g, epi, x, w, res, rows, nvec, hidden_f, eps, w_add, s);
  return launch_rows_pw<T, VPT, false>(g, epi, x, w, res, rows, nvec, hidden_f, eps, w_add, s);
}

// Few rows (decode): at most 2 vectors per thread, up to kDecodeMaxThreads
// threads, so each thread's chain of loads, adds and stores is short (a
// build-time knob: 0 keeps the many-row geometry for every launch).  Used up
// to the largest decode batch measured with it (256 rows).
#ifndef NR_RMS_DECODE_GEOM
#define NR_RMS_DECODE_GEOM 1
#endif
constexpr int64_t kDecodeGeomRows = 256;
// Vectors per thread of the few-row geometry (a build-time knob: 1 or 2).
#ifndef NR_RMS_DECODE_VPT
#define NR_RMS_DECODE_VPT 2
#endif

// Launch the row kernel for the geometry picked for this row length; false
// when the row is too long for it (the caller then needs the multi-pass kernel).
template <typename T, typename EPI>
bool launch_row_kernel(cudaError_t& err, const EPI& epi, const void* x, const void* w, void* res,
                       int64_t rows, int64_t nvec, float hidden_f, float eps, float w_add,
                       cudaStream_t s) {
  constexpr int DV = NR_RMS_DECODE_VPT;
  // Up to 32 rows of at most 512 vectors: one vector per thread (measured
  // [32, 4096] bf16 1.90 / 2.14 µs hot / cold against 2.01 / 2.37 µs with two;
  // from 128 rows, or with longer rows, two per thread are as fast or faster).
  if (NR_RMS_DECODE_GEOM && DV == 2 && rows <= 32 && nvec > kRowMaxThreads && nvec <= 512) {
    const RowLaunch g{1, static_cast<int>((nvec + 31) / 32 * 32)};
    err = launch_rows_pw<T, 1, true>(g, epi, x, w, res, rows, static_cast<int>(nvec), hidden_f,
                                     eps, w_add, s);
    return true;
  }
  // Measured exception: 17-64 rows of at least 1024 vectors keep the
  // many-row geometry ([32, 8192] bf16: 2.22 / 2.65 µs hot / cold against
  // 2.60 / 2.88 µs with 2 vectors per thread; at 8 and at 128 rows the few-row
  // geometry is as fast or faster).
  const bool few_row_loses = rows > 16 && rows <= 64 && nvec >= 1024;
  if (NR_RMS_DECODE_GEOM && rows <= kDecodeGeomRows && nvec > kRowMaxThreads &&
      nvec <= DV * kDecodeMaxThreads && !few_row_loses) {
    const int nv = static_cast<int>(nvec);
    const RowLaunch g{DV, static_cast<int>(((nvec + DV - 1) / DV + 31) / 32 * 32)};
    err = launch_rows_pw<T, DV, true>(g, epi, x, w, res, rows, nv, hidden_f, eps, w_add, s);
    return true;
  }
  const RowLaunch g = pick_row_launch(nvec);
  const int nv = static_cast<int>(nvec);
  switch (g.vpt) {
    case 1: err = launch_rows<T, 1>(g, epi, x, w, res, rows, nv, hidden_f, eps, w_add, s); return true;
    case 2: err = launch_rows<T, 2>(g, epi, x, w, res, rows, nv, hidden_f, eps, w_add, s); return true;
    case 3: err = launch_rows<T, 3>(g, epi, x, w, res, rows, nv, hidden_f, eps, w_add, s); return true;
    case 4: err = launch_rows<T, 4>(g, epi, x, w, res, rows, nv, hidden_f, eps, w_add, s); return true;
    case 5: err = launch_rows<T, 5>(g, epi, x, w, res, rows, nv, hidden_f, eps, w_add, s); return true;
    case 6: err = launch_rows<T, 6>(g, epi, x, w, res, rows, nv, hidden_f, eps, w_add, s); return true;
    case 8: err = launch_rows<T, 8>(g, epi, x, w, res, rows, nv, hidden_f, eps, w_add, s); return true;
    case 12: err = launch_rows<T, 12>(g, epi, x, w, res, rows, nv, hidden_f, eps, w_add, s); return true;
    case 16: err = launch_rows<T, 16>(g, epi, x, w, res, rows, nv, hidden_f, eps, w_add, s); return true;
    default: return false;
  }
}

template <typename T>
cudaError_t launch_typed(void* out, const void* x, const void* w, void* res, int64_t rows,
                         int64_t hidden, float eps, int gemma, cudaStream_t s) {
  const int64_t nvec = hidden / Vec<T>::N;
  const float hidden_f = static_cast<float>(hidden);
  const float w_add = gemma ? 1.0f : 0.0f;
  cudaError_t err = cudaSuccess;
  if (launch_row_kernel<T>(err, StoreOut{out}, x, w, res, rows, nvec, hidden_f, eps, w_add, s))
    return err;
  // Long rows: 1024 threads stride over the row twice.
  const dim3 grid(static_cast<unsigned>(rows));
  if (res != nullptr)
    return launch_pdl(rmsnorm_long_row_kernel<T, true>, grid, dim3(1024), 0, s,
        static_cast<T*>(out), static_cast<const T*>(x), static_cast<const T*>(w),
        static_cast<T*>(res), nvec, hidden_f, 1.0f / hidden_f, eps, w_add);
  else
    return launch_pdl(rmsnorm_long_row_kernel<T, false>, grid, dim3(1024), 0, s,
        static_cast<T*>(out), static_cast<const T*>(x), static_cast<const T*>(w), nullptr, nvec,
        hidden_f, 1.0f / hidden_f, eps, w_add);
}

}  // namespace

cudaError_t launch_rmsnorm(void* out, const void* x, const void* w, void* residual, int64_t rows,
                           int64_t hidden, int is_bf16, float eps, int gemma,
                           cudaStream_t stream) {
  if (is_bf16)
    return launch_typed<__nv_bfloat16>(out, x, w, residual, rows, hidden, eps, gemma, stream);
  return launch_typed<float>(out, x, w, residual, rows, hidden, eps, gemma, stream);
}

cudaError_t launch_rmsnorm_quant_fp8(void* codes, void* out_bf16, const void* x, const void* w,
                                     void* residual, int64_t rows, int64_t hidden, int is_bf16,
                                     float eps, int gemma, float inv_scale, cudaStream_t stream) {
  const StoreFp8 epi{static_cast<uint8_t*>(codes), static_cast<__nv_bfloat16*>(out_bf16),
                     inv_scale};
  const float hidden_f = static_cast<float>(hidden);
  const float w_add = gemma ? 1.0f : 0.0f;
  cudaError_t err = cudaErrorNotSupported;  // rows past the row kernel (rejected by the ABI first)
  if (is_bf16)
    launch_row_kernel<__nv_bfloat16>(err, epi, x, w, residual, rows, hidden / 8, hidden_f, eps,
                                     w_add, stream);
  else
    launch_row_kernel<float>(err, epi, x, w, residual, rows, hidden / 4, hidden_f, eps, w_add,
                             stream);
  return err;
}

}  // namespace nr
