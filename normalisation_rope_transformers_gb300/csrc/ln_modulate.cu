// LayerNorm (no affine) fused with adaLN modulation, for sm_103a.
//
// The fusion is named in the FastVideo PAN2 docs ("Performance switches",
// dit_fused_kernels: LayerNorm + modulation) without its formula; this computes
// the plain adaLN reading:
//   mu = mean(x), var = mean((x - mu)^2)  (biased, f32 statistics)
//   out = round((x - mu) * rsqrt(var + eps) * (1 + scale) + shift)
// with shift/scale taken from sample row r / rows_per_sample.
//
// Design: one block per row with the row held in registers (read once, written
// once).  The mean and the centred variance are two reductions over the
// register-resident values, so the variance does not suffer the cancellation of
// the one-pass E[x^2] - mu^2 form.  Rows longer than the register budget use a
// three-pass kernel that re-reads the (L2-resident) row.
#include "nr_common.cuh"
#include "nr_internal.h"

namespace nr {
namespace {

template <typename T, int VPT>
__global__ void __launch_bounds__(kRowMaxThreads) ln_modulate_row_kernel(
    T* __restrict__ out, const T* __restrict__ x, const T* __restrict__ shift,
    const T* __restrict__ scale, int nvec, int64_t rows_per_sample, float hidden_f, float eps) {
  constexpr int N = Vec<T>::N;
  __shared__ float scratch_mean[32];
  __shared__ float scratch_var[32];
  const int64_t row = blockIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(x) + row * nvec;
  uint4* orow = reinterpret_cast<uint4*>(out) + row * nvec;
  const int64_t sample_off = (row / rows_per_sample) * nvec;
  const uint4* shv = reinterpret_cast<const uint4*>(shift) + sample_off;
  const uint4* scv = reinterpret_cast<const uint4*>(scale) + sample_off;

  uint4 xv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int vi = threadIdx.x + k * blockDim.x;
    if (vi < nvec) xv[k] = ld_stream(xr + vi);
  }

  float sum = 0.0f;
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int vi = threadIdx.x + k * blockDim.x;
    if (vi < nvec) {
      float v[N];
      Vec<T>::unpack(xv[k], v);
#pragma unroll
      for (int e = 0; e < N; e++) sum += v[e];
    }
  }
  const float mu = __fdiv_rn(block_sum(sum, scratch_mean), hidden_f);

  float dev = 0.0f;
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int vi = threadIdx.x + k * blockDim.x;
    if (vi < nvec) {
      float v[N];
      Vec<T>::unpack(xv[k], v);
#pragma unroll
      for (int e = 0; e < N; e++) {
        const float d = v[e] - mu;
        dev = fmaf(d, d, dev);
      }
    }
  }
  const float rstd = 1.0f / sqrtf(__fdiv_rn(block_sum(dev, scratch_var), hidden_f) + eps);

#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int vi = threadIdx.x + k * blockDim.x;
    if (vi < nvec) {
      float v[N], sh[N], sc[N];
      Vec<T>::unpack(xv[k], v);
      Vec<T>::unpack(ld_param(shv + vi), sh);
      Vec<T>::unpack(ld_param(scv + vi), sc);
#pragma unroll
      for (int e = 0; e < N; e++) v[e] = fmaf((v[e] - mu) * rstd, 1.0f + sc[e], sh[e]);
      st_stream(orow + vi, Vec<T>::pack(v));
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(1024) ln_modulate_long_row_kernel(
    T* __restrict__ out, const T* __restrict__ x, const T* __restrict__ shift,
    const T* __restrict__ scale, int64_t nvec, int64_t rows_per_sample, float hidden_f,
    float eps) {
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
  const float mu = __fdiv_rn(block_sum(sum, scratch_mean), hidden_f);
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
  const float rstd = 1.0f / sqrtf(__fdiv_rn(block_sum(dev, scratch_var), hidden_f) + eps);
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

template <typename T, int VPT>
cudaError_t launch_rows(const RowLaunch& g, void* out, const void* x, const void* shift,
                        const void* scale, int64_t rows, int nvec, int64_t rps, float hidden_f,
                        float eps, cudaStream_t s) {
  ln_modulate_row_kernel<T, VPT><<<dim3(static_cast<unsigned>(rows)), dim3(g.threads), 0, s>>>(
      static_cast<T*>(out), static_cast<const T*>(x), static_cast<const T*>(shift),
      static_cast<const T*>(scale), nvec, rps, hidden_f, eps);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(void* out, const void* x, const void* shift, const void* scale,
                         int64_t rows, int64_t hidden, int64_t rps, float eps, cudaStream_t s) {
  const int64_t nvec = hidden / Vec<T>::N;
  const float hidden_f = static_cast<float>(hidden);
  const RowLaunch g = pick_row_launch(nvec);
  const int nv = static_cast<int>(nvec);
  switch (g.vpt) {
    case 1: return launch_rows<T, 1>(g, out, x, shift, scale, rows, nv, rps, hidden_f, eps, s);
    case 2: return launch_rows<T, 2>(g, out, x, shift, scale, rows, nv, rps, hidden_f, eps, s);
    case 3: return launch_rows<T, 3>(g, out, x, shift, scale, rows, nv, rps, hidden_f, eps, s);
    case 4: return launch_rows<T, 4>(g, out, x, shift, scale, rows, nv, rps, hidden_f, eps, s);
    case 5: return launch_rows<T, 5>(g, out, x, shift, scale, rows, nv, rps, hidden_f, eps, s);
    case 6: return launch_rows<T, 6>(g, out, x, shift, scale, rows, nv, rps, hidden_f, eps, s);
    case 8: return launch_rows<T, 8>(g, out, x, shift, scale, rows, nv, rps, hidden_f, eps, s);
    case 12: return launch_rows<T, 12>(g, out, x, shift, scale, rows, nv, rps, hidden_f, eps, s);
    case 16: return launch_rows<T, 16>(g, out, x, shift, scale, rows, nv, rps, hidden_f, eps, s);
    default: break;
  }
  ln_modulate_long_row_kernel<T><<<dim3(static_cast<unsigned>(rows)), 1024, 0, s>>>(
      static_cast<T*>(out), static_cast<const T*>(x), static_cast<const T*>(shift),
      static_cast<const T*>(scale), nvec, rps, hidden_f, eps);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ln_modulate(void* out, const void* x, const void* shift, const void* scale,
                               int64_t rows, int64_t hidden, int64_t rows_per_sample,
                               int is_bf16, float eps, cudaStream_t stream) {
  if (is_bf16)
    return launch_typed<__nv_bfloat16>(out, x, shift, scale, rows, hidden, rows_per_sample, eps,
                                       stream);
  return launch_typed<float>(out, x, shift, scale, rows, hidden, rows_per_sample, eps, stream);
}

}  // namespace nr
