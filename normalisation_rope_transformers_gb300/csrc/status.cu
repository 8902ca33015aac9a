// Device status word of the library: one 32-bit word per device, kept in this
// translation unit only.  A kernel whose bounded wait runs out ORs its bit
// into the word through the pointer it was launched with (status_word()), so
// any kernel in any file can report.  nr_device_status reads the word and
// clears exactly the bits it read (an atomic AND on the device), so a bit set
// by a kernel on another stream after the read stays set for the next read.
#include <atomic>

#include "nr_common.cuh"
#include "nr_internal.h"

namespace nr {
namespace {

__device__ unsigned int g_status_word;

__global__ void clear_status_bits_kernel(unsigned* word, unsigned bits) {
  atomicAnd(word, ~bits);
}

// A wait that nothing completes: one mbarrier with no arrivals, waited on for
// `limit` cycles.  Exercises the expiry path that the real kernels take.
__global__ void wait_probe_kernel(unsigned* status, long long limit) {
  __shared__ __align__(8) unsigned long long bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (!mbar_wait_bounded(smem_addr(&bar), 0, limit) && threadIdx.x == 0)
    atomicOr(status, kStatusBitProbeWait);
}

constexpr int kMaxDevices = 64;

}  // namespace

cudaError_t status_word(unsigned** word) {
  static std::atomic<unsigned*> cached[kMaxDevices];
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned* p = cached[device].load(std::memory_order_acquire);
  if (p == nullptr) {
    // The symbol's device address on the current device (a racing thread at
    // worst repeats the query and stores the same address).
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_status_word);
    if (e != cudaSuccess) return e;
    cached[device].store(p, std::memory_order_release);
  }
  *word = p;
  return cudaSuccess;
}

cudaError_t take_device_status(cudaStream_t stream, unsigned* bits) {
  // The word of the stream's device: make that device current for the call.
  int prev = 0, device = 0;
  cudaError_t e = cudaGetDevice(&prev);
  if (e != cudaSuccess) return e;
  e = cudaStreamGetDevice(stream, &device);
  if (e != cudaSuccess) return e;
  if (device != prev && (e = cudaSetDevice(device)) != cudaSuccess) return e;
  unsigned* word = nullptr;
  unsigned v = 0;
  // The read is ordered after the stream's work and waits for nothing else.
  e = status_word(&word);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&v, word, sizeof(v), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess && v != 0) {
    clear_status_bits_kernel<<<1, 1, 0, stream>>>(word, v);
    e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  }
  if (device != prev) {
    const cudaError_t e2 = cudaSetDevice(prev);
    if (e == cudaSuccess) e = e2;
  }
  if (e == cudaSuccess) *bits = v;
  return e;
}

cudaError_t launch_wait_probe(long long limit_cycles, cudaStream_t stream) {
  unsigned* word = nullptr;
  cudaError_t e = status_word(&word);
  if (e != cudaSuccess) return e;
  wait_probe_kernel<<<1, 32, 0, stream>>>(word, limit_cycles);
  return cudaGetLastError();
}

}  // namespace nr
