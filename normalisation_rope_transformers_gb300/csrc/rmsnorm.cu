// RMSNorm with the optional fused residual add, for sm_103a.
//
// Computes what vllm.cpp src/vt/cuda/cuda_ops.cu describes in "rmsnorm: one
// block per row" and "ResRound": v = round(x + residual) (written back in
// place), inv = 1/sqrt(mean(v^2) + eps), out = round(v * inv * (w [+1])).
//
// Design (not the page's): the page's kernel walks a row twice with scalar
// loads and a 256-wide shared-memory tree.  Here each row is held in
// registers: a block owns one row, each thread loads VPT 128-bit vectors of x
// (and of the residual) once, writes the rounded residual back immediately,
// and the row's sum of squares is reduced with warp shuffles plus one
// shared-memory step.  Each row is read from HBM once and written once.
// Rows longer than the register budget use a two-pass kernel that re-reads
// the (L2-resident) row.
#include "nr_common.cuh"
#include "nr_internal.h"

namespace nr {
namespace {

// One block per row; thread t owns vectors t, t + blockDim, ..., (VPT of them).
// PW: load the weight together with the row (saves a dependent round trip when
// there are few rows, e.g. decode; costs registers when there are many).
template <typename T, int VPT, bool RES, bool PW>
__global__ void __launch_bounds__(kRowMaxThreads) rmsnorm_row_kernel(T* __restrict__ out,
                                                           const T* __restrict__ x,
                                                           const T* __restrict__ w,
                                                           T* __restrict__ res, int nvec,
                                                           float hidden_f, float eps,
                                                           float w_add) {
  constexpr int N = Vec<T>::N;
  __shared__ float scratch[32];
  const int64_t row_off = static_cast<int64_t>(blockIdx.x) * nvec;  // in vectors
  const uint4* xr = reinterpret_cast<const uint4*>(x) + row_off;
  uint4* rr = RES ? reinterpret_cast<uint4*>(res) + row_off : nullptr;
  uint4* orow = reinterpret_cast<uint4*>(out) + row_off;
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

  float sum_sq = 0.0f;
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int vi = threadIdx.x + k * blockDim.x;
    if (vi < nvec) {
      float v[N];
      Vec<T>::unpack(xv[k], v);
      if (RES) {
        float r[N];
        Vec<T>::unpack(rv[k], r);
#pragma unroll
        for (int e = 0; e < N; e++) v[e] += r[e];
        // Round to the residual's storage dtype; the rounded value is both
        // written back and squared.  (For bf16, f32 add then one rounding
        // equals rounding the exact sum: f32 holds >= 2*8+2 bits.)
        xv[k] = Vec<T>::pack(v);
        st_stream(rr + vi, xv[k]);
        Vec<T>::unpack(xv[k], v);
      }
#pragma unroll
      for (int e = 0; e < N; e++) sum_sq = fmaf(v[e], v[e], sum_sq);
    }
  }

  const float total = block_sum(sum_sq, scratch);
  const float inv = 1.0f / sqrtf(__fdiv_rn(total, hidden_f) + eps);

#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int vi = threadIdx.x + k * blockDim.x;
    if (vi < nvec) {
      float v[N], wf[N];
      Vec<T>::unpack(xv[k], v);
      Vec<T>::unpack(PW ? wpre[PW ? k : 0] : ld_param(wv + vi), wf);
#pragma unroll
      for (int e = 0; e < N; e++) v[e] = v[e] * inv * (wf[e] + w_add);
      st_stream(orow + vi, Vec<T>::pack(v));
    }
  }
}

// Rows in flight per block for the persistent ring kernel; a build-time knob.
#ifndef NR_RMS_RING
#define NR_RMS_RING 2
#endif

// Persistent variant for many rows: block b takes rows b, b + G, ...  Each
// thread streams its own vectors of x (and of the residual) through a
// RING-deep shared-memory ring with cp.async, so the next rows are in flight
// while one is reduced; the weight stays in registers for all rows.  One
// barrier per row: the cross-warp partial sums alternate between two buffers.
template <typename T, int VPT, bool RES, int RING>
__global__ void __launch_bounds__(kRowMaxThreads) rmsnorm_ring_kernel(
    T* __restrict__ out, const T* __restrict__ x, const T* __restrict__ w, T* __restrict__ res,
    int64_t rows, int nvec, float hidden_f, float eps, float w_add) {
  constexpr int N = Vec<T>::N;
  constexpr int NBUF = RES ? 2 : 1;
  extern __shared__ __align__(16) unsigned char smem[];
  uint4* ring = reinterpret_cast<uint4*>(smem);  // [RING][NBUF][VPT][blockDim]
  __shared__ float partial[2][kRowMaxThreads / kWarp];
  const int tid = threadIdx.x;
  const int nthreads = blockDim.x;
  const int nwarps = (nthreads + kWarp - 1) / kWarp;
  const int64_t G = gridDim.x;
  auto slot_ptr = [&](int slot, int buf, int k) {
    return ring + ((slot * NBUF + buf) * VPT + k) * nthreads + tid;
  };

  uint4 wpk[VPT];  // the weight, packed, for all of this block's rows
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int vi = tid + k * nthreads;
    if (vi < nvec) wpk[k] = ld_param(reinterpret_cast<const uint4*>(w) + vi);
  }

  int64_t next = blockIdx.x;
  auto issue = [&](int slot) {
    if (next < rows) {
      const uint4* xr = reinterpret_cast<const uint4*>(x) + next * nvec;
      const uint4* rr = RES ? reinterpret_cast<const uint4*>(res) + next * nvec : nullptr;
#pragma unroll
      for (int k = 0; k < VPT; k++) {
        const int vi = tid + k * nthreads;
        if (vi < nvec) {
          cp_async16(smem_addr(slot_ptr(slot, 0, k)), xr + vi);
          if (RES) cp_async16(smem_addr(slot_ptr(slot, NBUF - 1, k)), rr + vi);
        }
      }
      next += G;
    }
    cp_async_commit();
  };
  for (int s = 0; s < RING; s++) issue(s);

  int slot = 0, parity = 0;
  for (int64_t row = blockIdx.x; row < rows; row += G) {
    cp_async_wait<RING - 1>();
    uint4 xv[VPT], rv[VPT];
#pragma unroll
    for (int k = 0; k < VPT; k++) {
      if (tid + k * nthreads < nvec) {
        xv[k] = lds128(slot_ptr(slot, 0, k));
        if (RES) rv[k] = lds128(slot_ptr(slot, NBUF - 1, k));
      }
    }
    issue(slot);  // the slot is in registers: refill it RING rows ahead

    uint4* rrow = RES ? reinterpret_cast<uint4*>(res) + row * nvec : nullptr;
    float sum_sq = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; k++) {
      const int vi = tid + k * nthreads;
      if (vi < nvec) {
        float v[N];
        Vec<T>::unpack(xv[k], v);
        if (RES) {
          float r[N];
          Vec<T>::unpack(rv[k], r);
#pragma unroll
          for (int e = 0; e < N; e++) v[e] += r[e];
          xv[k] = Vec<T>::pack(v);  // rounded once to the residual's dtype
          st_stream(rrow + vi, xv[k]);
          Vec<T>::unpack(xv[k], v);
        }
#pragma unroll
        for (int e = 0; e < N; e++) sum_sq = fmaf(v[e], v[e], sum_sq);
      }
    }
    sum_sq = group_sum<kWarp>(sum_sq);
    if (tid % kWarp == 0) partial[parity][tid / kWarp] = sum_sq;
    __syncthreads();
    float total = 0.0f;
    for (int i = 0; i < nwarps; i++) total += partial[parity][i];
    const float inv = 1.0f / sqrtf(__fdiv_rn(total, hidden_f) + eps);

    uint4* orow = reinterpret_cast<uint4*>(out) + row * nvec;
#pragma unroll
    for (int k = 0; k < VPT; k++) {
      const int vi = tid + k * nthreads;
      if (vi < nvec) {
        float v[N], wf[N];
        Vec<T>::unpack(xv[k], v);
        Vec<T>::unpack(wpk[k], wf);
#pragma unroll
        for (int e = 0; e < N; e++) v[e] = v[e] * inv * (wf[e] + w_add);
        st_stream(orow + vi, Vec<T>::pack(v));
      }
    }
    slot = slot + 1 == RING ? 0 : slot + 1;
    parity ^= 1;
  }
  cp_async_wait<0>();
}

// Rows too long for registers: pass 1 adds, writes the residual and reduces;
// pass 2 re-reads the stored values (L2-resident) and normalises.
template <typename T, bool RES>
__global__ void __launch_bounds__(1024) rmsnorm_long_row_kernel(T* __restrict__ out,
                                                                const T* __restrict__ x,
                                                                const T* __restrict__ w,
                                                                T* __restrict__ res, int64_t nvec,
                                                                float hidden_f, float eps,
                                                                float w_add) {
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
  const float inv = 1.0f / sqrtf(__fdiv_rn(total, hidden_f) + eps);
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

template <typename T, int VPT, bool PW>
cudaError_t launch_rows_pw(const RowLaunch& g, void* out, const void* x, const void* w, void* res,
                           int64_t rows, int nvec, float hidden_f, float eps, float w_add,
                           cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(rows));
  const dim3 block(g.threads);
  if (res != nullptr)
    rmsnorm_row_kernel<T, VPT, true, PW><<<grid, block, 0, s>>>(
        static_cast<T*>(out), static_cast<const T*>(x), static_cast<const T*>(w),
        static_cast<T*>(res), nvec, hidden_f, eps, w_add);
  else
    rmsnorm_row_kernel<T, VPT, false, PW><<<grid, block, 0, s>>>(
        static_cast<T*>(out), static_cast<const T*>(x), static_cast<const T*>(w), nullptr, nvec,
        hidden_f, eps, w_add);
  return cudaGetLastError();
}

int rms_sm_count(int device) {
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

template <typename T, int VPT, bool RES>
cudaError_t launch_ring(const RowLaunch& g, void* out, const void* x, const void* w, void* res,
                        int64_t rows, int nvec, float hidden_f, float eps, float w_add,
                        cudaStream_t s) {
  constexpr int RING = NR_RMS_RING;
  const size_t smem = static_cast<size_t>(RING) * (RES ? 2 : 1) * VPT * g.threads * sizeof(uint4);
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  if (device < 0 || device >= 64) device = 0;
  // Occupancy depends on the block size, so it is cached per (device, threads/32).
  static int resident_per_sm[64][kRowMaxThreads / kWarp + 1] = {{0}};
  int& cached = resident_per_sm[device][g.threads / kWarp];
  if (cached == 0) {
    cudaFuncSetAttribute(rmsnorm_ring_kernel<T, VPT, RES, RING>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, rmsnorm_ring_kernel<T, VPT, RES, RING>,
                                                      g.threads, smem) != cudaSuccess ||
        n < 1)
      n = 1;
    cached = n;
  }
  const int64_t resident = static_cast<int64_t>(rms_sm_count(device)) * cached;
  const int64_t blocks = rows < resident ? rows : resident;
  rmsnorm_ring_kernel<T, VPT, RES, RING><<<dim3(static_cast<unsigned>(blocks)), g.threads, smem,
                                           s>>>(
      static_cast<T*>(out), static_cast<const T*>(x), static_cast<const T*>(w),
      static_cast<T*>(res), rows, nvec, hidden_f, eps, w_add);
  return cudaGetLastError();
}

// Rows per launch up to which the weight is fetched together with the row;
// beyond this the persistent ring kernel runs.
constexpr int64_t kPrefetchWeightRows = 1024;
// Ring slots above this many bytes per block fall back to the row kernel.
constexpr size_t kRingMaxSmem = 96 * 1024;

template <typename T, int VPT>
cudaError_t launch_rows(const RowLaunch& g, void* out, const void* x, const void* w, void* res,
                        int64_t rows, int nvec, float hidden_f, float eps, float w_add,
                        cudaStream_t s) {
  if (rows <= kPrefetchWeightRows)
    return launch_rows_pw<T, VPT, true>(g, out, x, w, res, rows, nvec, hidden_f, eps, w_add, s);
  if constexpr (VPT <= 8) {
    const size_t ring_smem =
        static_cast<size_t>(NR_RMS_RING) * (res ? 2 : 1) * VPT * g.threads * sizeof(uint4);
    if (ring_smem <= kRingMaxSmem) {
      if (res != nullptr)
        return launch_ring<T, VPT, true>(g, out, x, w, res, rows, nvec, hidden_f, eps, w_add, s);
      return launch_ring<T, VPT, false>(g, out, x, w, res, rows, nvec, hidden_f, eps, w_add, s);
    }
  }
  return launch_rows_pw<T, VPT, false>(g, out, x, w, res, rows, nvec, hidden_f, eps, w_add, s);
}

template <typename T>
cudaError_t launch_typed(void* out, const void* x, const void* w, void* res, int64_t rows,
                         int64_t hidden, float eps, int gemma, cudaStream_t s) {
  const int64_t nvec = hidden / Vec<T>::N;
  const float hidden_f = static_cast<float>(hidden);
  const float w_add = gemma ? 1.0f : 0.0f;
  const RowLaunch g = pick_row_launch(nvec);
  switch (g.vpt) {
    case 1: return launch_rows<T, 1>(g, out, x, w, res, rows, (int)nvec, hidden_f, eps, w_add, s);
    case 2: return launch_rows<T, 2>(g, out, x, w, res, rows, (int)nvec, hidden_f, eps, w_add, s);
    case 3: return launch_rows<T, 3>(g, out, x, w, res, rows, (int)nvec, hidden_f, eps, w_add, s);
    case 4: return launch_rows<T, 4>(g, out, x, w, res, rows, (int)nvec, hidden_f, eps, w_add, s);
    case 5: return launch_rows<T, 5>(g, out, x, w, res, rows, (int)nvec, hidden_f, eps, w_add, s);
    case 6: return launch_rows<T, 6>(g, out, x, w, res, rows, (int)nvec, hidden_f, eps, w_add, s);
    case 8: return launch_rows<T, 8>(g, out, x, w, res, rows, (int)nvec, hidden_f, eps, w_add, s);
    case 12: return launch_rows<T, 12>(g, out, x, w, res, rows, (int)nvec, hidden_f, eps, w_add, s);
    case 16: return launch_rows<T, 16>(g, out, x, w, res, rows, (int)nvec, hidden_f, eps, w_add, s);
    default: break;
  }
  // Long rows: 1024 threads stride over the row twice.
  const dim3 grid(static_cast<unsigned>(rows));
  if (res != nullptr)
    rmsnorm_long_row_kernel<T, true><<<grid, 1024, 0, s>>>(
        static_cast<T*>(out), static_cast<const T*>(x), static_cast<const T*>(w),
        static_cast<T*>(res), nvec, hidden_f, eps, w_add);
  else
    rmsnorm_long_row_kernel<T, false><<<grid, 1024, 0, s>>>(
        static_cast<T*>(out), static_cast<const T*>(x), static_cast<const T*>(w), nullptr, nvec,
        hidden_f, eps, w_add);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rmsnorm(void* out, const void* x, const void* w, void* residual, int64_t rows,
                           int64_t hidden, int is_bf16, float eps, int gemma,
                           cudaStream_t stream) {
  if (is_bf16)
    return launch_typed<__nv_bfloat16>(out, x, w, residual, rows, hidden, eps, gemma, stream);
  return launch_typed<float>(out, x, w, residual, rows, hidden, eps, gemma, stream);
}

}  // namespace nr
