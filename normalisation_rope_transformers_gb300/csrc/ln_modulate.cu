// LayerNorm (no affine) fused with adaLN modulation, for sm_103a.
//
// The fusion is named in the FastVideo PAN2 docs ("Performance switches",
// dit_fused_kernels: LayerNorm + modulation) without its formula; this computes
// the plain adaLN reading:
//   mu = mean(x), var = mean((x - mu)^2)  (biased, f32 statistics)
//   out = round((x - mu) / sqrt(var + eps) * (1 + scale) + shift)
// with shift/scale taken from sample row r / rows_per_sample.
//
// Design.  Rows of up to 512 vectors (hidden 4096 bf16; the benchmark's 3072
// is 384 vectors = 12 per lane) belong to one warp, persistently: warp w of W
// takes rows w, w + W, ... and streams them through a per-warp shared-memory
// ring with cp.async, so the next RING rows are in flight while one is
// computed.  The row is read once (into the ring, then registers), the mean
// and the centred variance are warp-shuffle reductions over the registers,
// and the output is written once.  Longer rows belong to a group of 2, 4 or 8
// warps (one shared-memory step in each reduction); rows beyond 16 vectors
// per thread at 8 warps use a three-pass kernel that re-reads the
// (L2-resident) row.
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

template <typename T, int VPT, int WPR>
__global__ void __launch_bounds__(ln_threads<WPR>()) ln_modulate_rows_kernel(
    T* __restrict__ out, const T* __restrict__ x, const T* __restrict__ shift,
    const T* __restrict__ scale, int64_t rows, int nvec, int64_t rows_per_sample, float hidden_f,
    float eps) {
  constexpr int N = Vec<T>::N;
  constexpr int THREADS = ln_threads<WPR>();
  constexpr int TPR = kWarp * WPR;       // threads per row
  constexpr int RPB = THREADS / TPR;     // rows per block
  static_assert(RPB >= 1 && RPB * TPR == THREADS, "row groups must tile the block");
  __shared__ float scratch_mean[THREADS / kWarp];
  __shared__ float scratch_var[THREADS / kWarp];
  const int t = threadIdx.x % TPR;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * RPB + threadIdx.x / TPR;
  // Rows past the end still take part in the reductions' barriers (WPR > 1).
  const bool active = row < rows;
  const int64_t r = active ? row : 0;
  const uint4* xr = reinterpret_cast<const uint4*>(x) + r * nvec;
  uint4* orow = reinterpret_cast<uint4*>(out) + r * nvec;
  const int64_t sample_off = (r / rows_per_sample) * nvec;
  const uint4* shv = reinterpret_cast<const uint4*>(shift) + sample_off;
  const uint4* scv = reinterpret_cast<const uint4*>(scale) + sample_off;

  uint4 xv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int vi = t + k * TPR;
    if (active && vi < nvec) xv[k] = ld_stream(xr + vi);
  }

  float sum = 0.0f;
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int vi = t + k * TPR;
    if (active && vi < nvec) {
      float v[N];
      Vec<T>::unpack(xv[k], v);
#pragma unroll
      for (int e = 0; e < N; e++) sum += v[e];
    }
  }
  const float mu = __fdiv_rn(row_group_sum<WPR>(sum, scratch_mean), hidden_f);

  float dev = 0.0f;
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int vi = t + k * TPR;
    if (active && vi < nvec) {
      float v[N];
      Vec<T>::unpack(xv[k], v);
#pragma unroll
      for (int e = 0; e < N; e++) {
        const float d = v[e] - mu;
        dev = fmaf(d, d, dev);
      }
    }
  }
  const float rstd = 1.0f / sqrtf(__fdiv_rn(row_group_sum<WPR>(dev, scratch_var), hidden_f) + eps);
  if (!active) return;

#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int vi = t + k * TPR;
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

// Rows in flight per warp for rows of more than 4 vectors per lane; a
// build-time knob.
#ifndef NR_LN_RING
#define NR_LN_RING 2
#endif

constexpr int kLnRingThreads = 128;
constexpr int kLnRingWarps = kLnRingThreads / kWarp;

// Shared memory of the ring kernel: per warp RING rows of VPT x 32 vectors.
template <int VPT, int RING>
constexpr size_t ln_ring_smem() {
  return static_cast<size_t>(kLnRingWarps) * RING * VPT * kWarp * sizeof(uint4);
}

template <typename T, int VPT, int RING>
__global__ void __launch_bounds__(kLnRingThreads) ln_modulate_ring_kernel(
    T* __restrict__ out, const T* __restrict__ x, const T* __restrict__ shift,
    const T* __restrict__ scale, int64_t rows, int nvec, int64_t rows_per_sample, float hidden_f,
    float eps) {
  constexpr int N = Vec<T>::N;
  extern __shared__ __align__(16) unsigned char smem[];
  const int warp = threadIdx.x / kWarp;
  const int lane = threadIdx.x % kWarp;
  uint4* ring = reinterpret_cast<uint4*>(smem) + warp * RING * VPT * kWarp;  // [RING][VPT][32]
  const int64_t W = static_cast<int64_t>(gridDim.x) * kLnRingWarps;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kLnRingWarps + warp;
  if (first >= rows) return;

  int64_t next = first;  // next row to copy
  auto issue = [&](int slot) {
    if (next < rows) {
      const uint4* xr = reinterpret_cast<const uint4*>(x) + next * nvec;
#pragma unroll
      for (int k = 0; k < VPT; k++) {
        const int vi = lane + k * kWarp;
        if (vi < nvec) cp_async16(smem_addr(ring + (slot * VPT + k) * kWarp + lane), xr + vi);
      }
      next += W;
    }
    cp_async_commit();  // possibly empty: one group per ring slot use
  };
  for (int s = 0; s < RING; s++) issue(s);

  int slot = 0;
  for (int64_t row = first; row < rows; row += W) {
    cp_async_wait<RING - 1>();  // this row's copies have landed
    uint4 xv[VPT];
#pragma unroll
    for (int k = 0; k < VPT; k++)
      if (lane + k * kWarp < nvec) xv[k] = lds128(ring + (slot * VPT + k) * kWarp + lane);
    issue(slot);  // the slot is in registers: refill it RING rows ahead

    float sum = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; k++) {
      if (lane + k * kWarp < nvec) {
        float v[N];
        Vec<T>::unpack(xv[k], v);
#pragma unroll
        for (int e = 0; e < N; e++) sum += v[e];
      }
    }
    const float mu = __fdiv_rn(group_sum<kWarp>(sum), hidden_f);
    float dev = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; k++) {
      if (lane + k * kWarp < nvec) {
        float v[N];
        Vec<T>::unpack(xv[k], v);
#pragma unroll
        for (int e = 0; e < N; e++) {
          const float d = v[e] - mu;
          dev = fmaf(d, d, dev);
        }
      }
    }
    const float rstd = 1.0f / sqrtf(__fdiv_rn(group_sum<kWarp>(dev), hidden_f) + eps);

    const int64_t sample_off = (row / rows_per_sample) * nvec;
    const uint4* shv = reinterpret_cast<const uint4*>(shift) + sample_off;
    const uint4* scv = reinterpret_cast<const uint4*>(scale) + sample_off;
    uint4* orow = reinterpret_cast<uint4*>(out) + row * nvec;
#pragma unroll
    for (int k = 0; k < VPT; k++) {
      const int vi = lane + k * kWarp;
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
    slot = slot + 1 == RING ? 0 : slot + 1;
  }
  cp_async_wait<0>();
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

struct LnArgs {
  void* out;
  const void* x;
  const void* shift;
  const void* scale;
  int64_t rows;
  int nvec;
  int64_t rps;
  float hidden_f;
  float eps;
};

template <typename T, int VPT, int WPR>
cudaError_t launch_rows(const LnArgs& a, cudaStream_t s) {
  constexpr int THREADS = ln_threads<WPR>();
  constexpr int RPB = THREADS / (kWarp * WPR);
  static_assert(RPB >= 1, "row groups must fit the block");
  const int64_t blocks = (a.rows + RPB - 1) / RPB;
  ln_modulate_rows_kernel<T, VPT, WPR><<<dim3(static_cast<unsigned>(blocks)), THREADS, 0, s>>>(
      static_cast<T*>(a.out), static_cast<const T*>(a.x), static_cast<const T*>(a.shift),
      static_cast<const T*>(a.scale), a.rows, a.nvec, a.rps, a.hidden_f, a.eps);
  return cudaGetLastError();
}

int ln_sm_count(int device) {
  static int cached[64] = {0};
  if (device < 0 || device >= 64) return 1;
  if (cached[device] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n < 1)
      n = 1;
    cached[device] = n;
  }
  return cached[device];
}

// Persistent grid for the ring kernel: as many blocks as fit on the GPU (or
// one warp per row when there are fewer rows).
template <typename T, int VPT>
cudaError_t launch_ring(const LnArgs& a, cudaStream_t s) {
  constexpr int RING = VPT <= 4 ? 4 : NR_LN_RING;
  constexpr size_t smem = ln_ring_smem<VPT, RING>();
  static int resident_per_sm[64] = {0};
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  if (device < 0 || device >= 64) device = 0;
  if (resident_per_sm[device] == 0) {
    cudaFuncSetAttribute(ln_modulate_ring_kernel<T, VPT, RING>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, ln_modulate_ring_kernel<T, VPT, RING>,
                                                      kLnRingThreads, smem) != cudaSuccess ||
        n < 1)
      n = 1;
    resident_per_sm[device] = n;
  }
  const int64_t resident = static_cast<int64_t>(ln_sm_count(device)) * resident_per_sm[device];
  const int64_t needed = (a.rows + kLnRingWarps - 1) / kLnRingWarps;
  const int64_t blocks = needed < resident ? needed : resident;
  ln_modulate_ring_kernel<T, VPT, RING><<<dim3(static_cast<unsigned>(blocks)), kLnRingThreads,
                                          smem, s>>>(
      static_cast<T*>(a.out), static_cast<const T*>(a.x), static_cast<const T*>(a.shift),
      static_cast<const T*>(a.scale), a.rows, a.nvec, a.rps, a.hidden_f, a.eps);
  return cudaGetLastError();
}

// Vectors per thread offered for one-warp rows, and for rows spread over
// 2, 4 or 8 warps.
constexpr int kLnVptOneWarp[] = {1, 2, 3, 4, 6, 8, 10, 12, 16};
constexpr int kLnVptMultiWarp[] = {8, 12, 16};

template <typename T>
cudaError_t launch_typed(const LnArgs& a, cudaStream_t s) {
  const int64_t nvec = a.nvec;
  for (int wpr : {1, 2, 4, 8}) {
    const int64_t need = (nvec + kWarp * wpr - 1) / (kWarp * wpr);
    if (need > 16) continue;
    int vpt = 0;
    if (wpr == 1) {
      for (int v : kLnVptOneWarp)
        if (vpt == 0 && v >= need) vpt = v;
    } else {
      for (int v : kLnVptMultiWarp)
        if (vpt == 0 && v >= need) vpt = v;
    }
    switch (wpr * 100 + vpt) {
      case 101: return launch_ring<T, 1>(a, s);
      case 102: return launch_ring<T, 2>(a, s);
      case 103: return launch_ring<T, 3>(a, s);
      case 104: return launch_ring<T, 4>(a, s);
      case 106: return launch_ring<T, 6>(a, s);
      case 108: return launch_ring<T, 8>(a, s);
      case 110: return launch_ring<T, 10>(a, s);
      case 112: return launch_ring<T, 12>(a, s);
      case 116: return launch_ring<T, 16>(a, s);
      case 208: return launch_rows<T, 8, 2>(a, s);
      case 212: return launch_rows<T, 12, 2>(a, s);
      case 216: return launch_rows<T, 16, 2>(a, s);
      case 408: return launch_rows<T, 8, 4>(a, s);
      case 412: return launch_rows<T, 12, 4>(a, s);
      case 416: return launch_rows<T, 16, 4>(a, s);
      case 808: return launch_rows<T, 8, 8>(a, s);
      case 812: return launch_rows<T, 12, 8>(a, s);
      case 816: return launch_rows<T, 16, 8>(a, s);
      default: break;
    }
  }
  ln_modulate_long_row_kernel<T><<<dim3(static_cast<unsigned>(a.rows)), 1024, 0, s>>>(
      static_cast<T*>(a.out), static_cast<const T*>(a.x), static_cast<const T*>(a.shift),
      static_cast<const T*>(a.scale), nvec, a.rps, a.hidden_f, a.eps);
  return cudaGetLastError();
}

}  // namespace

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
  a.eps = eps;
  if (is_bf16) return launch_typed<__nv_bfloat16>(a, stream);
  return launch_typed<float>(a, stream);
}

}  // namespace nr
