// Gated activations for sm_103a: out[r, j] = act(x[r, j]) * x[r, inter + j]
// with act = silu (the vllm.cpp page src/vt/cuda/cuda_ops.cu, SiLU
// gated-activation section) or the tanh form of GELU (its GELU
// gated-activation section); gate = first half of the row, up = second half,
// f32 math.  Design: a 2-D grid (vector column blocks x rows) so
// no thread divides a flat index; each thread moves UNROLL 128-bit vectors of
// gate and of up, issuing every load before any math.  Both activations are
// a * sigmoid(s * z(a)) evaluated in an overflow-free form (below); bf16
// outputs use the hardware exponential and reciprocal, so the kernel stays
// memory-bound.
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
// the same form with the accurate expf and IEEE divisions: e^-a is never
// formed, so gates below -88.7 (where e^-a overflows f32) still give a * e^a
// to a few ulps while that value is a normal f32 (gates down to about -92;
// t itself loses bits gradually below -87.3, about 2e-6 relative at -90).
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
  const float t = expf(-fabsf(a));
  return a * (a >= 0.0f ? 1.0f / (1.0f + t) : t / (1.0f + t));
}

// tanh-GELU: 0.5 a (1 + tanh(z)), z = sqrt(2/pi) (a + 0.044715 a^3), computed
// as a * sigmoid(2z) (the same function: (1 + tanh z) / 2 = sigmoid(2z)) with
// the overflow-free sigmoid, which keeps full relative accuracy where
// 1 + tanh(z) would cancel.  bf16 outputs: 2z in plain f32, exp2f and a fast
// reciprocal, whose errors stay far inside one bf16 ulp.
template <typename T>
__device__ __forceinline__ float gelu_tanh(float a) {
  const float two_z = 1.5957691216057308f * fmaf(0.044715f * a, a * a, a);  // 2 sqrt(2/pi) (...)
  const float t = exp2f(-fabsf(two_z) * 1.4426950408889634f);
  const float r = __fdividef(1.0f, 1.0f + t);
  return a * (two_z >= 0.0f ? r : t * r);
}

// f32 outputs.  For a < 0 the result is about a * e^{2z}, so a relative error
// d in 2z becomes |2z| * d in the result: with 2z rounded a few times in f32
// that is ~2e-5 at 2z = -70, too much for a 1e-5 relative tolerance.  So
// 2z = a (kK + kKc a^2), kK = 2 sqrt(2/pi), kKc = 0.044715 kK, is carried as
// an unevaluated sum r + r_lo of two floats: each constant split into two
// floats, products made error-free with fmaf, the sum with Knuth's TwoSum.
// Then e^{-|2z|} = e^{-|r|} (1 -+ r_lo) to first order (|r_lo| <= 5e-6).
// The gate is clamped to +-20 inside the sigmoid only: beyond it sigmoid(2z)
// is 1 or 0 exactly in f32, and a^2 stays finite.
template <>
__device__ __forceinline__ float gelu_tanh<float>(float a_in) {
  constexpr float kKHi = 0x1.988454p+0f, kKLo = -0x1.857936p-25f;
  constexpr float kKcHi = 0x1.2444f2p-4f, kKcLo = 0x1.49b16ap-29f;
  const float a = fminf(fmaxf(a_in, -20.0f), 20.0f);
  const float s = a * a, s_lo = fmaf(a, a, -s);  // a^2 = s + s_lo
  const float p = kKcHi * s;
  const float p_lo = fmaf(kKcHi, s, -p) + fmaf(kKcHi, s_lo, kKcLo * s);  // kKc a^2
  const float q = kKHi + p;  // TwoSum(kKHi, p)
  const float qb = q - kKHi;
  const float q_lo = ((kKHi - (q - qb)) + (p - qb)) + (kKLo + p_lo);
  const float r = a * q;
  const float r_lo = fmaf(a, q, -r) + a * q_lo;  // 2z = r + r_lo
  const float t0 = expf(-fabsf(r));
  const float t = fmaf(t0, r >= 0.0f ? -r_lo : r_lo, t0);
  return a_in * (r >= 0.0f ? 1.0f / (1.0f + t) : t / (1.0f + t));
}

enum class Act { kSilu, kGeluTanh };

template <typename T, Act ACT>
__device__ __forceinline__ float activate(float a) {
  if constexpr (ACT == Act::kSilu)
    return silu<T>(a);
  else
    return gelu_tanh<T>(a);
}

// Vectors of gate and of up per thread for large problems; a build-time knob.
// 2 against 4: silu [128, 2 x 24576] 5.94 -> 4.95 µs and [256, 2 x 12288]
// 5.85 -> 4.91 µs cold (more blocks for the same bytes in flight), gelu
// [8192, 2 x 15360] 106.8 -> 104.9 µs; 8 was slower everywhere.
#ifndef NR_ACT_UNROLL
#define NR_ACT_UNROLL 2
#endif

constexpr unsigned kMaxGridY = 65535;

template <typename T, int UNROLL, Act ACT>
__global__ void __launch_bounds__(kSiluThreads) act_and_mul_kernel(T* __restrict__ out,
                                                                    const T* __restrict__ x,
                                                                    int64_t rows, int ivec) {
  pdl_enter();  // before any global read: the previous kernel may still run
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
        for (int e = 0; e < N; e++) a[e] = activate<T, ACT>(a[e]) * b[e];
        st_stream(o + c, Vec<T>::pack(a));
      }
    }
  }
}

template <typename T, int UNROLL, Act ACT>
cudaError_t launch_u(void* out, const void* x, int64_t rows, int ivec, cudaStream_t s) {
  const unsigned gx = static_cast<unsigned>((ivec + kSiluThreads * UNROLL - 1) /
                                            (kSiluThreads * UNROLL));
  const unsigned gy = static_cast<unsigned>(rows < kMaxGridY ? rows : kMaxGridY);
  return launch_pdl(act_and_mul_kernel<T, UNROLL, ACT>, dim3(gx, gy), dim3(kSiluThreads), 0, s,
      static_cast<T*>(out), static_cast<const T*>(x), rows, ivec);
}

template <typename T, Act ACT>
cudaError_t launch_typed(void* out, const void* x, int64_t rows, int64_t inter, cudaStream_t s) {
  const int ivec = static_cast<int>(inter / Vec<T>::N);
  // Small problems (decode) spread one vector per thread over as many SMs as
  // possible; large ones give each thread more bytes in flight.
  if (static_cast<int64_t>(ivec) * rows >= int64_t(152) * 4 * kSiluThreads * 4)
    return launch_u<T, NR_ACT_UNROLL, ACT>(out, x, rows, ivec, s);
  return launch_u<T, 1, ACT>(out, x, rows, ivec, s);
}

}  // namespace

cudaError_t launch_silu_and_mul(void* out, const void* x, int64_t rows, int64_t inter,
                                int is_bf16, cudaStream_t stream) {
  if (is_bf16) return launch_typed<__nv_bfloat16, Act::kSilu>(out, x, rows, inter, stream);
  return launch_typed<float, Act::kSilu>(out, x, rows, inter, stream);
}

cudaError_t launch_gelu_and_mul(void* out, const void* x, int64_t rows, int64_t inter,
                                int is_bf16, cudaStream_t stream) {
  if (is_bf16) return launch_typed<__nv_bfloat16, Act::kGeluTanh>(out, x, rows, inter, stream);
  return launch_typed<float, Act::kGeluTanh>(out, x, rows, inter, stream);
}

}  // namespace nr
