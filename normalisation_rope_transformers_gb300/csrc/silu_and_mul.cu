// silu_and_mul for sm_103a: out[r, j] = silu(x[r, j]) * x[r, inter + j].
//
// Follows vllm.cpp src/vt/cuda/cuda_ops.cu, "silu_and_mul" (gate = first half
// of the row, up = second half, f32 math).  Design: a 2-D grid (vector column
// blocks x rows) so no thread divides a flat index; each thread moves UNROLL
// 128-bit vectors of gate and of up, issuing every load before any math.  The
// exponential and division are the cheap hardware forms for bf16 outputs
// (see silu<T> below), so the kernel stays memory-bound.
#include "nr_common.cuh"
#include "nr_internal.h"

namespace nr {
namespace {

constexpr int kSiluThreads = 128;

// silu(a) = a * sigmoid(a).  For bf16 outputs (8 significant bits) the
// hardware exponential and reciprocal (relative error ~1e-6) are exact to well
// within half an output ulp.  They are used in an overflow-free form:
// t = e^-|a| lies in (0, 1], sigmoid(|a|) = 1 / (1 + t) and
// sigmoid(-|a|) = t / (1 + t), so the divisor stays in [1, 2] and large
// negative gates keep their tiny (possibly subnormal) result.  f32 outputs use
// the accurate expf and an IEEE division.
template <typename T>
__device__ __forceinline__ float silu(float a);
template <>
__device__ __forceinline__ float silu<__nv_bfloat16>(float a) {
  const float t = exp2f(-fabsf(a) * 1.4426950408889634f);  // e^-|a|, subnormals kept
  const float r = __fdividef(1.0f, 1.0f + t);
  return a * (a >= 0.0f ? r : t * r);
}
template <>
__device__ __forceinline__ float silu<float>(float a) {
  return a / (1.0f + expf(-a));
}

constexpr unsigned kMaxGridY = 65535;

template <typename T, int UNROLL>
__global__ void __launch_bounds__(kSiluThreads) silu_and_mul_kernel(T* __restrict__ out,
                                                                    const T* __restrict__ x,
                                                                    int64_t rows, int ivec) {
  constexpr int N = Vec<T>::N;
  const int col0 = blockIdx.x * (kSiluThreads * UNROLL) + threadIdx.x;
  for (int64_t row = blockIdx.y; row < rows; row += gridDim.y) {
    const uint4* gate = reinterpret_cast<const uint4*>(x) + row * 2 * ivec;
    const uint4* up = gate + ivec;
    uint4* o = reinterpret_cast<uint4*>(out) + row * ivec;
    uint4 gv[UNROLL], uv[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; u++) {
      const int c = col0 + u * kSiluThreads;
      if (c < ivec) {
        gv[u] = ld_stream(gate + c);
        uv[u] = ld_stream(up + c);
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; u++) {
      const int c = col0 + u * kSiluThreads;
      if (c < ivec) {
        float a[N], b[N];
        Vec<T>::unpack(gv[u], a);
        Vec<T>::unpack(uv[u], b);
#pragma unroll
        for (int e = 0; e < N; e++) a[e] = silu<T>(a[e]) * b[e];
        st_stream(o + c, Vec<T>::pack(a));
      }
    }
  }
}

template <typename T, int UNROLL>
cudaError_t launch_u(void* out, const void* x, int64_t rows, int ivec, cudaStream_t s) {
  const unsigned gx = static_cast<unsigned>((ivec + kSiluThreads * UNROLL - 1) /
                                            (kSiluThreads * UNROLL));
  const unsigned gy = static_cast<unsigned>(rows < kMaxGridY ? rows : kMaxGridY);
  silu_and_mul_kernel<T, UNROLL><<<dim3(gx, gy), kSiluThreads, 0, s>>>(
      static_cast<T*>(out), static_cast<const T*>(x), rows, ivec);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(void* out, const void* x, int64_t rows, int64_t inter, cudaStream_t s) {
  const int ivec = static_cast<int>(inter / Vec<T>::N);
  // Small problems (decode) spread one vector per thread over as many SMs as
  // possible; large ones give each thread more bytes in flight.
  if (static_cast<int64_t>(ivec) * rows >= int64_t(152) * 4 * kSiluThreads * 4)
    return launch_u<T, 4>(out, x, rows, ivec, s);
  return launch_u<T, 1>(out, x, rows, ivec, s);
}

}  // namespace

cudaError_t launch_silu_and_mul(void* out, const void* x, int64_t rows, int64_t inter,
                                int is_bf16, cudaStream_t stream) {
  if (is_bf16) return launch_typed<__nv_bfloat16>(out, x, rows, inter, stream);
  return launch_typed<float>(out, x, rows, inter, stream);
}

}  // namespace nr
