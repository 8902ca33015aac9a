// Internal launcher interface between the C ABI (nr_api.cu) and the kernels.
// Arguments reaching these functions have been validated by the ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

namespace nr {

// 1: launch every kernel with programmatic stream serialisation (the kernels
// wait for their predecessor on the device; see pdl_enter); 0: plain
// stream-ordered launches.  A build-time knob.
#ifndef NR_PDL
#define NR_PDL 1
#endif

// Launch `kernel` on `stream` with programmatic stream serialisation.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = NR_PDL ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Blocks of `kernel` (with `threads` threads, no dynamic shared memory)
// resident at once over the current device's SMs, cached per device in
// `cache` (64 entries; a racing thread at worst repeats the queries).
template <typename Kernel>
cudaError_t resident_blocks(Kernel kernel, int threads, std::atomic<int>* cache, int* blocks) {
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  int n = cache[device].load(std::memory_order_relaxed);
  if (n == 0) {
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0);
    if (e != cudaSuccess) return e;
    n = sms * (per_sm > 0 ? per_sm : 1);
    cache[device].store(n, std::memory_order_relaxed);
  }
  *blocks = n;
  return cudaSuccess;
}

// Geometry of the row-resident kernels: one block per row, `threads` threads,
// each owning up to `vpt` 128-bit vectors.  vpt == 0 selects the multi-pass
// kernel for rows longer than the register budget.
struct RowLaunch {
  int vpt;
  int threads;
};

constexpr int kRowMaxThreads = 256;
constexpr int kRowVpts[] = {1, 2, 3, 4, 5, 6, 8, 12, 16};

// Pick the vectors-per-thread count that covers the row with at most
// kRowMaxThreads threads and the fewest idle vector slots (ties: fewer vectors
// per thread, i.e. more threads).
inline RowLaunch pick_row_launch(int64_t nvec) {
  RowLaunch best{0, 1024};
  int64_t best_waste = -1;
  for (int v : kRowVpts) {
    const int64_t need = (nvec + v - 1) / v;
    const int64_t threads = ((need + 31) / 32) * 32;
    if (threads > kRowMaxThreads) continue;
    const int64_t waste = threads * v - nvec;
    if (best_waste < 0 || waste < best_waste) {
      best_waste = waste;
      best = RowLaunch{v, static_cast<int>(threads)};
    }
  }
  return best;
}

cudaError_t launch_rmsnorm(void* out, const void* x, const void* w, void* residual, int64_t rows,
                           int64_t hidden, int is_bf16, float eps, int gemma,
                           cudaStream_t stream);

// RMSNorm + e4m3 quantisation: rows of at most kRowMaxThreads * 16 vectors.
constexpr int64_t kQuantMaxVectors = kRowMaxThreads * 16;

cudaError_t launch_rmsnorm_quant_fp8(void* codes, void* out_bf16, const void* x, const void* w,
                                     void* residual, int64_t rows, int64_t hidden, int is_bf16,
                                     float eps, int gemma, float inv_scale, cudaStream_t stream);

cudaError_t launch_ln_modulate(void* out, const void* x, const void* shift, const void* scale,
                               int64_t rows, int64_t hidden, int64_t rows_per_sample,
                               int is_bf16, float eps, cudaStream_t stream);

// Rows of the gated kernel hold at most this many 128-bit vectors
// (4 warps x 32 lanes x 8 vectors).
constexpr int64_t kGatedMaxVectors = 4 * 32 * 8;

cudaError_t launch_gated_ln_modulate(void* out, void* residual, const void* y, const void* gate,
                                     const void* shift, const void* scale, int64_t rows,
                                     int64_t hidden, int64_t rows_per_sample, int is_bf16,
                                     float eps, cudaStream_t stream);

cudaError_t launch_silu_and_mul(void* out, const void* x, int64_t rows, int64_t inter,
                                int is_bf16, cudaStream_t stream);

cudaError_t launch_gelu_and_mul(void* out, const void* x, int64_t rows, int64_t inter,
                                int is_bf16, cudaStream_t stream);

// Per-call rotary constants: turn[i] = frac(freq_i / (2*pi)) * 2^64 for pair i
// (freq_i = theta^(-2i/rotary_dim), Llama-3 rescaled when asked), so that
// (pos * turn[i]) mod 2^64 is the angle pos*freq_i as a fraction of a full
// turn; axis[i] is the M-RoPE position row of pair i (0 without M-RoPE).
constexpr int kMaxHalfDim = 256;
struct RopeTurns {
  unsigned long long turn[kMaxHalfDim];
  unsigned char axis[kMaxHalfDim];
};

cudaError_t launch_qk_norm_rope(void* q_out, void* k_out, const void* q, const void* k,
                                const void* wq, const void* wk, int w_is_bf16,
                                const int32_t* positions, int64_t tokens, int64_t hq, int64_t hk,
                                int64_t head_dim, int64_t q_tok_stride, int64_t k_tok_stride,
                                float eps, const RopeTurns& turns, int gemma, int64_t rotary_dim,
                                int interleaved, int mrope, int is_bf16, cudaStream_t stream);

// Device status word: bits set by kernels whose bounded waits ran out.
constexpr unsigned kStatusBitQkBulkWait = 1u;
constexpr unsigned kStatusBitProbeWait = 2u;

// Device address of the current device's status word (status.cu), looked up
// once per device.  Kernels that bound a wait take it as an argument.
cudaError_t status_word(unsigned** word);

// On the device of `stream`: waits for `stream`, reads the status word and
// clears the bits it read (bits set after the read stay set).
cudaError_t take_device_status(cudaStream_t stream, unsigned* bits);

// One block whose single wait nothing completes, given up after
// `limit_cycles` SM clock cycles (it sets kStatusBitProbeWait).
cudaError_t launch_wait_probe(long long limit_cycles, cudaStream_t stream);

}  // namespace nr
