// Shared device helpers for the row-normalisation kernels (sm_103a).
//
// Every kernel moves data as 128-bit vectors (8 bf16 or 4 f32 values per
// thread per access), so a warp covers 512 contiguous bytes per instruction.
// Streaming data is read with L1::no_allocate (it is touched once) and written
// with the .cs (evict-first) hint; parameters reused by every row (weights,
// shift, scale) use the default caching path so they stay L1/L2 resident.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nr {

constexpr int kWarp = 32;

// ---------------------------------------------------------------------------
// 128-bit global memory access
// ---------------------------------------------------------------------------
// Read-once data (x, residual, q, k): no L1 allocation, and ask L2 to fetch the
// whole 256-byte sector group.  Only used on data that no thread of the same
// launch writes before reading it (each thread reads its own elements before it
// overwrites them in place).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Data shared by all rows (weights, shift, scale): normal cached read-only path.
__device__ __forceinline__ uint4 ld_param(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Coherent read (for data this launch may already have written, e.g. the
// residual re-read by the multi-pass kernels for very long rows).
__device__ __forceinline__ uint4 ld_coherent(const void* p) {
  uint4 v;
  asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// Streaming store: evict-first, the result is not re-read by this launch.
__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// Streaming stores of 8 and 4 bytes (FP8 codes, bf16 halves of f32 rows).
__device__ __forceinline__ void st_stream8(void* p, uint2 v) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ void st_stream4(void* p, uint32_t v) {
  asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Plain store (for data a later pass of the same launch reads back).
__device__ __forceinline__ void st_plain(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialisation, so it may be scheduled while the kernel
// before it in the stream is still finishing.  pdl_enter, the first statement
// of every kernel, lets the next kernel in the stream be scheduled early
// (griddepcontrol.launch_dependents) and then waits until the previous kernel
// has completed and its writes are visible (griddepcontrol.wait) -- so no
// global memory is read before that, whoever launched the previous kernel.
// Without a programmatic predecessor the wait returns at once.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Asynchronous global -> shared copies (cp.async).  Each thread copies its own
// vectors and waits for its own copy groups; the data is then visible to that
// thread (no other thread reads it), so no barrier is involved.  The wait is
// a hardware wait on the thread's outstanding groups, not a spin loop.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned smem_addr(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

// 16 bytes, L1 bypassed, ask L2 for the whole 256-byte sector group.
__device__ __forceinline__ void cp_async16(unsigned dst, const void* src) {
  asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16;" ::"r"(dst), "l"(src)
               : "memory");
}

// 4 bytes (through L1: small, shared by many threads).
__device__ __forceinline__ void cp_async4(unsigned dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait until at most `pending` of this thread's committed groups are still in flight.
template <int pending>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(pending) : "memory");
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// ---------------------------------------------------------------------------
// Bulk copies by the TMA engine (cp.async.bulk, no tensor map) and the
// shared-memory mbarriers that count their bytes.  Sizes and both addresses
// must be multiples of 16 bytes.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(unsigned bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes initialised mbarriers visible to the async proxy (the TMA engine).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// One arrival that also announces `bytes` of copies to be counted.
__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

// True if the phase with the given parity has completed.  Never blocks
// (test_wait, not try_wait: a try_wait on a phase that nothing completes may
// keep the thread suspended, so no clock check after it would ever run).
__device__ __forceinline__ bool mbar_test_wait(unsigned bar, unsigned parity) {
  unsigned done;
  asm volatile(
      "{\n"
      "  .reg .pred p;\n"
      "  mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      "  selp.u32 %0, 1, 0, p;\n"
      "}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Nanoseconds a waiting thread sleeps between two polls (a build-time knob).
// Measured on the Q/K bulk kernel at [26598, 24+24, 128]: 8 ns ties 32 ns,
// 128 ns is 0.5-1 us slower (the wake-up comes late).
#ifndef NR_MBAR_SLEEP_NS
#define NR_MBAR_SLEEP_NS 32
#endif

// Polls the phase (with a short sleep between polls) for at most `limit` SM
// clock cycles; false if it gave up (the caller records the failure and winds
// down).  Every poll returns at once, so the bound always holds.
__device__ __forceinline__ bool mbar_wait_bounded(unsigned bar, unsigned parity, long long limit) {
  if (mbar_test_wait(bar, parity)) return true;
  const long long t0 = clock64();
  do {
    __nanosleep(NR_MBAR_SLEEP_NS);
    if (mbar_test_wait(bar, parity)) return true;
  } while (clock64() - t0 <= limit);
  return false;
}

// Global -> shared bulk copy; its bytes complete a transaction count on `bar`.
__device__ __forceinline__ void bulk_load(unsigned dst, const void* src, unsigned bytes,
                                          unsigned bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// An L2 policy that evicts first the lines it covers (for data touched once).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
  return policy;
}

// bulk_load / bulk_store with an L2 cache policy.
__device__ __forceinline__ void bulk_load_hint(unsigned dst, const void* src, unsigned bytes,
                                               unsigned bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_store_hint(void* dst, unsigned src, unsigned bytes,
                                                uint64_t policy) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(
                   dst),
               "r"(src), "r"(bytes), "l"(policy)
               : "memory");
}

// Asks L2 to fetch `bytes` from global memory (no completion to wait for).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, unsigned bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Shared -> global bulk copy, tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void bulk_store(void* dst, unsigned src, unsigned bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Until at most `pending` of this thread's bulk groups still read shared memory.
template <int pending>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(pending) : "memory");
}

// Until at most `pending` of this thread's bulk groups are incomplete.
template <int pending>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(pending) : "memory");
}

// Orders this thread's ordinary shared-memory writes before later bulk copies
// (async proxy) that read them.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Element types: a 128-bit vector holds VEC values of T.
// ---------------------------------------------------------------------------
template <typename T>
struct Vec;

template <>
struct Vec<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ __forceinline__ static uint4 pack(const float (&f)[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

// bf16 pair in one 32-bit word: element 2k in the low half, 2k+1 in the high
// half.  Widening is exact (bf16 is the top half of an f32).
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Round two f32 values to bf16 (round to nearest even) and pack them.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Mixed-precision f32 arithmetic on one bf16 half of a packed pair (PTX
// add/sub/fma with .f32.bf16 types): the bf16 operand is widened exactly, so
// each result equals the same f32 operation on the unpacked value.
// HI selects the high half (element 2k + 1).
template <bool HI>
__device__ __forceinline__ float add_bf16(uint32_t u, float c) {  // bf16 + c
  float d;
  if (HI)
    asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n add.rn.f32.bf16 %0, hi, %2;\n}"
        : "=f"(d) : "r"(u), "f"(c));
  else
    asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n add.rn.f32.bf16 %0, lo, %2;\n}"
        : "=f"(d) : "r"(u), "f"(c));
  return d;
}
template <bool HI>
__device__ __forceinline__ float sub_bf16(uint32_t u, float c) {  // bf16 - c
  float d;
  if (HI)
    asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n sub.rn.f32.bf16 %0, hi, %2;\n}"
        : "=f"(d) : "r"(u), "f"(c));
  else
    asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n sub.rn.f32.bf16 %0, lo, %2;\n}"
        : "=f"(d) : "r"(u), "f"(c));
  return d;
}

// a*b + c for the same half of two packed pairs, rounded down (RM) and up
// (RP): the product of two bf16 values is exact, so each is the exact
// a*b + c rounded once in that direction.
template <bool HI>
__device__ __forceinline__ void fma_bf16_down_up(uint32_t a, uint32_t b, float c, float& down,
                                                 float& up) {
  if (HI)
    asm("{\n .reg .b16 alo, ahi, blo, bhi;\n mov.b32 {alo, ahi}, %2;\n mov.b32 {blo, bhi}, %3;\n"
        " fma.rm.f32.bf16 %0, ahi, bhi, %4;\n fma.rp.f32.bf16 %1, ahi, bhi, %4;\n}"
        : "=f"(down), "=f"(up) : "r"(a), "r"(b), "f"(c));
  else
    asm("{\n .reg .b16 alo, ahi, blo, bhi;\n mov.b32 {alo, ahi}, %2;\n mov.b32 {blo, bhi}, %3;\n"
        " fma.rm.f32.bf16 %0, alo, blo, %4;\n fma.rp.f32.bf16 %1, alo, blo, %4;\n}"
        : "=f"(down), "=f"(up) : "r"(a), "r"(b), "f"(c));
}

template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[8]) {
    f[0] = bf16_lo(v.x);
    f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y);
    f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z);
    f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w);
    f[7] = bf16_hi(v.w);
  }
  __device__ __forceinline__ static uint4 pack(const float (&f)[8]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
  }
};

// ---------------------------------------------------------------------------
// FP8 e4m3 codes: round to nearest even, finite values beyond +-448 saturate
// (CUDA's conversion, two values per call).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  return static_cast<uint32_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// ---------------------------------------------------------------------------
// Reductions
// ---------------------------------------------------------------------------
// Butterfly sum over groups of `width` consecutive lanes (width a power of two
// <= 32); every lane of the group ends with the same value.
template <int width>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int m = width / 2; m > 0; m >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, m);
  return v;
}

// Sum over the whole thread block.  `scratch` holds one float per warp; every
// thread returns the same total, summed in warp order.  Contains one barrier;
// callers that reuse `scratch` must separate the uses with another barrier or
// use distinct arrays.
__device__ __forceinline__ float block_sum(float v, float* scratch) {
  v = group_sum<kWarp>(v);
  const int warp = threadIdx.x / kWarp;
  const int lane = threadIdx.x % kWarp;
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  const int nwarps = (blockDim.x + kWarp - 1) / kWarp;
  float total = 0.0f;
  for (int i = 0; i < nwarps; i++) total += scratch[i];
  return total;
}

// ---------------------------------------------------------------------------
// Row statistics from a row's totals (the LayerNorm mean and variance, the
// RMSNorm mean square).  With NR_FAST_STATS (a build-time knob) a mean is
// total * (1/n) refined by one fma step -- the remainder total - q*n is exact,
// so a quotient that is a float comes out exactly -- and the reciprocal
// square root is the hardware approximation; otherwise an IEEE division and
// 1 / sqrtf.
// ---------------------------------------------------------------------------
#ifndef NR_FAST_STATS
#define NR_FAST_STATS 1
#endif
__device__ __forceinline__ float row_mean_of(float total, float n, float inv_n) {
#if NR_FAST_STATS
  const float q = total * inv_n;
  return fmaf(fmaf(-q, n, total), inv_n, q);
#else
  (void)inv_n;
  return __fdiv_rn(total, n);
#endif
}
__device__ __forceinline__ float row_rstd_of(float mean_square, float eps) {
#if NR_FAST_STATS
  return rsqrtf(mean_square + eps);
#else
  return 1.0f / sqrtf(mean_square + eps);
#endif
}

}  // namespace nr
