// C ABI of the fused row-normalisation library: argument validation, the
// per-call rotary constants, and status reporting.  Every check runs on the
// host before any launch; a rejected call touches no device memory.
#include <math.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include <nvtx3/nvToolsExt.h>

#include "../../include/nr.h"
#include "nr_internal.h"

namespace {

// One NVTX range per entry-point call, named after the entry point, so that
// profilers (nsys, ncu --nvtx) can attribute kernels to the call that
// launched them.  Without a tool attached the push and pop cost a few
// nanoseconds.
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};

thread_local char g_message[512];

nr_status fail(nr_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_message, sizeof g_message, fmt, ap);
  va_end(ap);
  return s;
}

nr_status ok() {
  g_message[0] = '\0';
  return NR_OK;
}

nr_status from_cuda(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ok();
  return fail(NR_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_size(nr_dtype d) { return d == NR_BF16 ? 2 : 4; }
int vec_elems(nr_dtype d) { return d == NR_BF16 ? 8 : 4; }
bool valid_dtype(int d) { return d == NR_F32 || d == NR_BF16; }

// `count` rows of `span` bytes, `stride` bytes apart, starting at `base`.
struct Region {
  uintptr_t base;
  int64_t stride;
  int64_t span;
  int64_t count;
};

Region dense(const void* p, int64_t bytes) {
  return Region{reinterpret_cast<uintptr_t>(p), bytes, bytes, 1};
}

// Conservative overlap test: false only when the two regions are provably
// disjoint (disjoint address ranges, or equal strides with rows that interleave
// without touching -- e.g. Q and K heads inside one fused QKV row).
bool overlap(const Region& a, const Region& b) {
  if (a.count <= 0 || b.count <= 0 || a.span <= 0 || b.span <= 0) return false;
  const uintptr_t a_end = a.base + static_cast<uintptr_t>((a.count - 1) * a.stride + a.span);
  const uintptr_t b_end = b.base + static_cast<uintptr_t>((b.count - 1) * b.stride + b.span);
  if (a_end <= b.base || b_end <= a.base) return false;
  if (a.stride == b.stride && a.stride >= a.span && a.stride >= b.span) {
    const int64_t s = a.stride;
    const int64_t diff = static_cast<int64_t>(b.base - a.base);  // two's complement
    const int64_t delta = ((diff % s) + s) % s;                   // b's row start inside a's period
    if (a.span <= delta && delta + b.span <= s) return false;
  }
  return true;
}

bool eps_ok(float eps) { return isfinite(eps) && eps >= 0.0f; }

}  // namespace

extern "C" {

int nr_version(void) { return 100; }

const char* nr_last_error_message(void) { return g_message; }

const char* nr_status_string(nr_status s) {
  switch (s) {
    case NR_OK: return "NR_OK";
    case NR_ERR_NULL: return "NR_ERR_NULL";
    case NR_ERR_SHAPE: return "NR_ERR_SHAPE";
    case NR_ERR_DTYPE: return "NR_ERR_DTYPE";
    case NR_ERR_ALIGN: return "NR_ERR_ALIGN";
    case NR_ERR_ALIAS: return "NR_ERR_ALIAS";
    case NR_ERR_UNSUPPORTED: return "NR_ERR_UNSUPPORTED";
    case NR_ERR_CUDA: return "NR_ERR_CUDA";
    case NR_ERR_VALUE: return "NR_ERR_VALUE";
    case NR_ERR_TIMEOUT: return "NR_ERR_TIMEOUT";
  }
  return "NR_ERR_UNKNOWN";
}

nr_status nr_rmsnorm(void* out, const void* x, const void* w, void* residual, int64_t rows,
                     int64_t hidden, nr_dtype dtype, float eps, int gemma, cudaStream_t stream) {
  CallRange range("nr_rmsnorm");
  if (!valid_dtype(dtype)) return fail(NR_ERR_DTYPE, "nr_rmsnorm: unknown dtype %d", (int)dtype);
  if (rows < 0) return fail(NR_ERR_SHAPE, "nr_rmsnorm: rows = %lld < 0", (long long)rows);
  if (hidden <= 0) return fail(NR_ERR_SHAPE, "nr_rmsnorm: hidden = %lld <= 0", (long long)hidden);
  if (!eps_ok(eps)) return fail(NR_ERR_VALUE, "nr_rmsnorm: eps must be finite and >= 0");
  if (gemma != 0 && gemma != 1) return fail(NR_ERR_VALUE, "nr_rmsnorm: gemma must be 0 or 1");
  if (rows == 0) return ok();
  if (!out || !x || !w) return fail(NR_ERR_NULL, "nr_rmsnorm: out, x and w must be non-NULL");
  const int vec = vec_elems(dtype);
  if (hidden % vec != 0)
    return fail(NR_ERR_UNSUPPORTED, "nr_rmsnorm: hidden = %lld is not a multiple of %d",
                (long long)hidden, vec);
  if (rows > INT32_MAX || hidden / vec > INT32_MAX)
    return fail(NR_ERR_SHAPE, "nr_rmsnorm: rows or hidden too large");
  if (!aligned16(out) || !aligned16(x) || !aligned16(w) || (residual && !aligned16(residual)))
    return fail(NR_ERR_ALIGN, "nr_rmsnorm: pointers must be 16-byte aligned");
  const int64_t row_bytes = hidden * elem_size(dtype);
  const Region ro = dense(out, rows * row_bytes), rx = dense(x, rows * row_bytes);
  const Region rw = dense(w, row_bytes);
  if (out != x && overlap(ro, rx))
    return fail(NR_ERR_ALIAS, "nr_rmsnorm: out partially overlaps x (only out == x is allowed)");
  if (overlap(ro, rw)) return fail(NR_ERR_ALIAS, "nr_rmsnorm: out overlaps w");
  if (residual) {
    const Region rr = dense(residual, rows * row_bytes);
    if (overlap(rr, rx) || overlap(rr, ro) || overlap(rr, rw))
      return fail(NR_ERR_ALIAS, "nr_rmsnorm: residual overlaps x, out or w");
  }
  return from_cuda(nr::launch_rmsnorm(out, x, w, residual, rows, hidden, dtype == NR_BF16, eps,
                                      gemma, stream),
                   "nr_rmsnorm launch");
}

nr_status nr_rmsnorm_quant_fp8(void* codes, void* out_bf16, const void* x, const void* w,
                               void* residual, int64_t rows, int64_t hidden, nr_dtype dtype,
                               float eps, int gemma, float scale, cudaStream_t stream) {
  CallRange range("nr_rmsnorm_quant_fp8");
  const char* fn = "nr_rmsnorm_quant_fp8";
  if (!valid_dtype(dtype)) return fail(NR_ERR_DTYPE, "%s: unknown dtype %d", fn, (int)dtype);
  if (rows < 0 || hidden <= 0)
    return fail(NR_ERR_SHAPE, "%s: need rows >= 0 and hidden > 0", fn);
  if (!eps_ok(eps)) return fail(NR_ERR_VALUE, "%s: eps must be finite and >= 0", fn);
  if (gemma != 0 && gemma != 1) return fail(NR_ERR_VALUE, "%s: gemma must be 0 or 1", fn);
  const float inv_scale = 1.0f / scale;
  if (!(isfinite(scale) && scale > 0.0f && isfinite(inv_scale)))
    return fail(NR_ERR_VALUE, "%s: scale must be finite and > 0 with a finite reciprocal", fn);
  if (rows == 0) return ok();
  if (!codes || !x || !w) return fail(NR_ERR_NULL, "%s: codes, x and w must be non-NULL", fn);
  const int vec = vec_elems(dtype);
  if (hidden % vec != 0)
    return fail(NR_ERR_UNSUPPORTED, "%s: hidden = %lld is not a multiple of %d", fn,
                (long long)hidden, vec);
  if (hidden / vec > nr::kQuantMaxVectors)
    return fail(NR_ERR_UNSUPPORTED, "%s: hidden = %lld is above %lld for this dtype", fn,
                (long long)hidden, (long long)(nr::kQuantMaxVectors * vec));
  if (rows > INT32_MAX) return fail(NR_ERR_SHAPE, "%s: rows too large", fn);
  if (!aligned16(codes) || !aligned16(x) || !aligned16(w) || (residual && !aligned16(residual)) ||
      (out_bf16 && !aligned16(out_bf16)))
    return fail(NR_ERR_ALIGN, "%s: pointers must be 16-byte aligned", fn);
  const int64_t row_bytes = hidden * elem_size(dtype);
  const Region rc = dense(codes, rows * hidden), rb = dense(out_bf16, out_bf16 ? rows * hidden * 2 : 0);
  const Region rx = dense(x, rows * row_bytes), rw = dense(w, row_bytes);
  const Region rr = dense(residual, residual ? rows * row_bytes : 0);
  if (overlap(rc, rx) || overlap(rc, rw) || overlap(rc, rr) || overlap(rc, rb) || overlap(rb, rx) ||
      overlap(rb, rw) || overlap(rb, rr))
    return fail(NR_ERR_ALIAS, "%s: an output overlaps an input or the other output", fn);
  if (overlap(rr, rx) || overlap(rr, rw))
    return fail(NR_ERR_ALIAS, "%s: residual overlaps x or w", fn);
  return from_cuda(nr::launch_rmsnorm_quant_fp8(codes, out_bf16, x, w, residual, rows, hidden,
                                                dtype == NR_BF16, eps, gemma, inv_scale, stream),
                   "nr_rmsnorm_quant_fp8 launch");
}

}  // extern "C"

namespace {

// Llama-3 rescale of one rotary frequency: keep short wavelengths, divide long
// ones by `factor`, and blend linearly (in 1/wavelength) between the two bands.
double llama3_rescale(double freq, const nr_rope_config& c) {
  if (!(c.llama3_factor > 0.0)) return freq;
  const double wavelength = 2.0 * M_PI / freq;
  const double short_band = c.llama3_original_max_position / c.llama3_high_freq_factor;
  const double long_band = c.llama3_original_max_position / c.llama3_low_freq_factor;
  if (wavelength < short_band) return freq;
  if (wavelength > long_band) return freq / c.llama3_factor;
  const double blend =
      c.llama3_high_freq_factor == c.llama3_low_freq_factor
          ? 0.0
          : (c.llama3_original_max_position / wavelength - c.llama3_low_freq_factor) /
                (c.llama3_high_freq_factor - c.llama3_low_freq_factor);
  return blend * freq + (1.0 - blend) * freq / c.llama3_factor;
}

// M-RoPE position row (0 = t, 1 = h, 2 = w) of rotary pair i.
unsigned char mrope_row(int64_t i, const nr_rope_config& c) {
  const int32_t* sec = c.mrope_section;
  if (c.mrope_interleaved) {
    const int64_t cycle = i / 3;
    if (i % 3 == 1 && cycle < sec[1]) return 1;
    if (i % 3 == 2 && cycle < sec[2]) return 2;
    return 0;
  }
  if (i < sec[0]) return 0;
  return i < sec[0] + sec[1] ? 1 : 2;
}

nr_status qk_norm_rope_impl(const char* fn, void* q_out, void* k_out, const void* q, const void* k,
                            const void* wq, const void* wk, nr_dtype w_dtype,
                            const int32_t* positions, int64_t tokens, int64_t hq, int64_t hk,
                            int64_t head_dim, int64_t q_tok_stride, int64_t k_tok_stride,
                            float eps, int gemma, const nr_rope_config& rope, nr_dtype dtype,
                            cudaStream_t stream) {
  if (!valid_dtype(dtype) || !valid_dtype(w_dtype))
    return fail(NR_ERR_DTYPE, "%s: unknown dtype (%d, weights %d)", fn, (int)dtype, (int)w_dtype);
  if (tokens < 0 || hq < 1 || hk < 0 || head_dim <= 0)
    return fail(NR_ERR_SHAPE, "%s: need tokens >= 0, hq >= 1, hk >= 0, head_dim > 0", fn);
  if (head_dim % 2 != 0) return fail(NR_ERR_SHAPE, "%s: head_dim must be even", fn);
  const int vec = vec_elems(dtype);
  const int64_t lanes = head_dim / (2 * vec);
  if (head_dim % (2 * vec) != 0 || lanes > 32 || (lanes & (lanes - 1)) != 0)
    return fail(NR_ERR_UNSUPPORTED,
                "%s: head_dim %lld not supported for this dtype (bf16: 16..512, f32: 8..256, "
                "powers of two)",
                fn, (long long)head_dim);
  const int64_t rot = rope.rotary_dim == 0 ? head_dim : rope.rotary_dim;
  if (rot <= 0 || rot > head_dim || rot % 2 != 0)
    return fail(NR_ERR_SHAPE, "%s: rotary_dim %lld must be even and in (0, head_dim]", fn,
                (long long)rot);
  if ((rope.interleaved != 0 && rope.interleaved != 1) ||
      (rope.mrope_interleaved != 0 && rope.mrope_interleaved != 1))
    return fail(NR_ERR_VALUE, "%s: interleaved flags must be 0 or 1", fn);
  if (rot % (rope.interleaved ? vec : 2 * vec) != 0)
    return fail(NR_ERR_UNSUPPORTED, "%s: rotary_dim %lld must be a multiple of %d", fn,
                (long long)rot, rope.interleaved ? vec : 2 * vec);
  if (!eps_ok(eps)) return fail(NR_ERR_VALUE, "%s: eps must be finite and >= 0", fn);
  if (!(isfinite(rope.theta) && rope.theta > 0.0))
    return fail(NR_ERR_VALUE, "%s: theta must be finite and > 0", fn);
  if (!isfinite(rope.llama3_factor) ||
      (rope.llama3_factor > 0.0 &&
       !(rope.llama3_low_freq_factor > 0.0 &&
         rope.llama3_high_freq_factor >= rope.llama3_low_freq_factor &&
         rope.llama3_original_max_position > 0.0 && isfinite(rope.llama3_high_freq_factor) &&
         isfinite(rope.llama3_original_max_position))))
    return fail(NR_ERR_VALUE, "%s: Llama-3 factors must be positive and finite, high >= low", fn);
  const int32_t* sec = rope.mrope_section;
  const bool mrope = sec[0] != 0 || sec[1] != 0 || sec[2] != 0;
  if (sec[0] < 0 || sec[1] < 0 || sec[2] < 0 ||
      (mrope && static_cast<int64_t>(sec[0]) + sec[1] + sec[2] != rot / 2))
    return fail(NR_ERR_SHAPE, "%s: M-RoPE sections must be >= 0 and sum to rotary_dim / 2", fn);
  if (gemma != 0 && gemma != 1) return fail(NR_ERR_VALUE, "%s: gemma must be 0 or 1", fn);
  if (q_tok_stride < hq * head_dim || (hk > 0 && k_tok_stride < hk * head_dim))
    return fail(NR_ERR_SHAPE, "%s: token stride smaller than heads * head_dim", fn);
  if (tokens > INT32_MAX || hq + hk > 65536)
    return fail(NR_ERR_SHAPE, "%s: tokens or head count too large", fn);
  if (tokens == 0) return ok();
  if (!q_out || !q || !wq || !positions)
    return fail(NR_ERR_NULL, "%s: q_out, q, wq and positions must be non-NULL", fn);
  if (hk > 0 && (!k_out || !k || !wk))
    return fail(NR_ERR_NULL, "%s: k_out, k and wk must be non-NULL when hk > 0", fn);
  const int es = elem_size(dtype);
  if ((q_tok_stride * es) % 16 != 0 || (hk > 0 && (k_tok_stride * es) % 16 != 0))
    return fail(NR_ERR_ALIGN, "%s: token strides must be multiples of 16 bytes", fn);
  if (!aligned16(q_out) || !aligned16(q) || !aligned16(wq) ||
      (hk > 0 && (!aligned16(k_out) || !aligned16(k) || !aligned16(wk))) ||
      (reinterpret_cast<uintptr_t>(positions) & 3u))
    return fail(NR_ERR_ALIGN,
                "%s: q/k/weights must be 16-byte aligned, positions 4-byte aligned", fn);

  const Region rq{reinterpret_cast<uintptr_t>(q), q_tok_stride * es, hq * head_dim * es, tokens};
  const Region rqo{reinterpret_cast<uintptr_t>(q_out), q_tok_stride * es, hq * head_dim * es,
                   tokens};
  const Region rk{reinterpret_cast<uintptr_t>(k), k_tok_stride * es, hk * head_dim * es,
                  hk > 0 ? tokens : 0};
  const Region rko{reinterpret_cast<uintptr_t>(k_out), k_tok_stride * es, hk * head_dim * es,
                   hk > 0 ? tokens : 0};
  const int ws = elem_size(w_dtype);
  const Region rwq = dense(wq, head_dim * ws);
  const Region rwk = dense(wk, hk > 0 ? head_dim * ws : 0);
  const Region rpos = dense(positions, (mrope ? 3 : 1) * tokens * 4);
  if ((q_out != q && overlap(rqo, rq)) || overlap(rqo, rk) || overlap(rqo, rwq) ||
      overlap(rqo, rwk) || overlap(rqo, rpos) || overlap(rqo, rko))
    return fail(NR_ERR_ALIAS, "%s: q_out overlaps an input or k_out", fn);
  if ((k_out != k && overlap(rko, rk)) || overlap(rko, rq) || overlap(rko, rwq) ||
      overlap(rko, rwk) || overlap(rko, rpos))
    return fail(NR_ERR_ALIAS, "%s: k_out overlaps an input", fn);

  // turn_i = frac(freq_i / 2pi) * 2^64, freq_i = theta^(-2i/rot) (Llama-3
  // rescaled when asked), in double.  Positions are integers, so
  // pos * freq_i mod 2pi = pos * (freq_i mod 2pi) mod 2pi.
  nr::RopeTurns turns;
  for (int64_t i = 0; i < nr::kMaxHalfDim; i++) {
    turns.turn[i] = 0;
    turns.axis[i] = 0;
  }
  for (int64_t i = 0; i < rot / 2; i++) {
    const double freq = llama3_rescale(
        pow(rope.theta, -2.0 * static_cast<double>(i) / static_cast<double>(rot)), rope);
    const double turns_per_step = freq / (2.0 * M_PI);
    const double frac = turns_per_step - floor(turns_per_step);
    const double scaled = ldexp(frac, 64);
    turns.turn[i] =
        scaled >= 18446744073709551616.0 ? 0ull : static_cast<unsigned long long>(scaled);
    turns.axis[i] = mrope ? mrope_row(i, rope) : 0;
  }
  return from_cuda(nr::launch_qk_norm_rope(q_out, k_out, q, k, wq, wk, w_dtype == NR_BF16,
                                           positions, tokens, hq, hk, head_dim, q_tok_stride,
                                           k_tok_stride, eps, turns, gemma, rot, rope.interleaved,
                                           mrope ? 1 : 0, dtype == NR_BF16, stream),
                   fn);
}

}  // namespace

extern "C" {

nr_status nr_qk_norm_rope(void* q_out, void* k_out, const void* q, const void* k, const void* wq,
                          const void* wk, nr_dtype w_dtype, const int32_t* positions,
                          int64_t tokens, int64_t hq, int64_t hk, int64_t head_dim,
                          int64_t q_tok_stride, int64_t k_tok_stride, float eps, double theta,
                          int gemma, nr_dtype dtype, cudaStream_t stream) {
  CallRange range("nr_qk_norm_rope");
  nr_rope_config rope = {};
  rope.theta = theta;
  return qk_norm_rope_impl("nr_qk_norm_rope", q_out, k_out, q, k, wq, wk, w_dtype, positions,
                           tokens, hq, hk, head_dim, q_tok_stride, k_tok_stride, eps, gemma, rope,
                           dtype, stream);
}

nr_status nr_qk_norm_rope_ex(void* q_out, void* k_out, const void* q, const void* k,
                             const void* wq, const void* wk, nr_dtype w_dtype,
                             const int32_t* positions, int64_t tokens, int64_t hq, int64_t hk,
                             int64_t head_dim, int64_t q_tok_stride, int64_t k_tok_stride,
                             float eps, int gemma, const nr_rope_config* rope, nr_dtype dtype,
                             cudaStream_t stream) {
  CallRange range("nr_qk_norm_rope_ex");
  if (rope == nullptr) return fail(NR_ERR_NULL, "nr_qk_norm_rope_ex: rope config is NULL");
  return qk_norm_rope_impl("nr_qk_norm_rope_ex", q_out, k_out, q, k, wq, wk, w_dtype, positions,
                           tokens, hq, hk, head_dim, q_tok_stride, k_tok_stride, eps, gemma, *rope,
                           dtype, stream);
}

nr_status nr_ln_modulate(void* out, const void* x, const void* shift, const void* scale,
                         int64_t rows, int64_t hidden, int64_t rows_per_sample, float eps,
                         nr_dtype dtype, cudaStream_t stream) {
  CallRange range("nr_ln_modulate");
  if (!valid_dtype(dtype)) return fail(NR_ERR_DTYPE, "nr_ln_modulate: unknown dtype %d", (int)dtype);
  if (rows < 0 || hidden <= 0 || rows_per_sample < 1)
    return fail(NR_ERR_SHAPE, "nr_ln_modulate: need rows >= 0, hidden > 0, rows_per_sample >= 1");
  if (!eps_ok(eps)) return fail(NR_ERR_VALUE, "nr_ln_modulate: eps must be finite and >= 0");
  if (rows == 0) return ok();
  if (!out || !x || !shift || !scale)
    return fail(NR_ERR_NULL, "nr_ln_modulate: out, x, shift and scale must be non-NULL");
  const int vec = vec_elems(dtype);
  if (hidden % vec != 0)
    return fail(NR_ERR_UNSUPPORTED, "nr_ln_modulate: hidden = %lld is not a multiple of %d",
                (long long)hidden, vec);
  if (rows > INT32_MAX || hidden / vec > INT32_MAX)
    return fail(NR_ERR_SHAPE, "nr_ln_modulate: rows or hidden too large");
  if (!aligned16(out) || !aligned16(x) || !aligned16(shift) || !aligned16(scale))
    return fail(NR_ERR_ALIGN, "nr_ln_modulate: pointers must be 16-byte aligned");
  const int64_t row_bytes = hidden * elem_size(dtype);
  const int64_t samples = (rows + rows_per_sample - 1) / rows_per_sample;
  const Region ro = dense(out, rows * row_bytes), rx = dense(x, rows * row_bytes);
  if (out != x && overlap(ro, rx))
    return fail(NR_ERR_ALIAS, "nr_ln_modulate: out partially overlaps x (only out == x is allowed)");
  if (overlap(ro, dense(shift, samples * row_bytes)) || overlap(ro, dense(scale, samples * row_bytes)))
    return fail(NR_ERR_ALIAS, "nr_ln_modulate: out overlaps shift or scale");
  return from_cuda(nr::launch_ln_modulate(out, x, shift, scale, rows, hidden, rows_per_sample,
                                          dtype == NR_BF16, eps, stream),
                   "nr_ln_modulate launch");
}

nr_status nr_gated_residual_ln_modulate(void* out, void* residual, const void* y,
                                        const void* gate, const void* shift, const void* scale,
                                        int64_t rows, int64_t hidden, int64_t rows_per_sample,
                                        float eps, nr_dtype dtype, cudaStream_t stream) {
  CallRange range("nr_gated_residual_ln_modulate");
  const char* fn = "nr_gated_residual_ln_modulate";
  if (!valid_dtype(dtype)) return fail(NR_ERR_DTYPE, "%s: unknown dtype %d", fn, (int)dtype);
  if (rows < 0 || hidden <= 0 || rows_per_sample < 1)
    return fail(NR_ERR_SHAPE, "%s: need rows >= 0, hidden > 0, rows_per_sample >= 1", fn);
  if (!eps_ok(eps)) return fail(NR_ERR_VALUE, "%s: eps must be finite and >= 0", fn);
  if (rows == 0) return ok();
  if (!out || !residual || !y || !gate || !shift || !scale)
    return fail(NR_ERR_NULL, "%s: every pointer must be non-NULL", fn);
  const int vec = vec_elems(dtype);
  if (hidden % vec != 0)
    return fail(NR_ERR_UNSUPPORTED, "%s: hidden = %lld is not a multiple of %d", fn,
                (long long)hidden, vec);
  if (hidden / vec > nr::kGatedMaxVectors)
    return fail(NR_ERR_UNSUPPORTED, "%s: hidden = %lld is above %lld for this dtype", fn,
                (long long)hidden, (long long)(nr::kGatedMaxVectors * vec));
  if (rows > INT32_MAX) return fail(NR_ERR_SHAPE, "%s: rows too large", fn);
  if (!aligned16(out) || !aligned16(residual) || !aligned16(y) || !aligned16(gate) ||
      !aligned16(shift) || !aligned16(scale))
    return fail(NR_ERR_ALIGN, "%s: pointers must be 16-byte aligned", fn);
  const int64_t row_bytes = hidden * elem_size(dtype);
  const int64_t samples = (rows + rows_per_sample - 1) / rows_per_sample;
  const Region ro = dense(out, rows * row_bytes), rr = dense(residual, rows * row_bytes);
  const Region ins[] = {dense(y, rows * row_bytes), dense(gate, samples * row_bytes),
                        dense(shift, samples * row_bytes), dense(scale, samples * row_bytes)};
  if (overlap(ro, rr)) return fail(NR_ERR_ALIAS, "%s: out overlaps residual", fn);
  for (const Region& in : ins)
    if (overlap(ro, in) || overlap(rr, in))
      return fail(NR_ERR_ALIAS, "%s: out or residual overlaps an input", fn);
  return from_cuda(nr::launch_gated_ln_modulate(out, residual, y, gate, shift, scale, rows, hidden,
                                                rows_per_sample, dtype == NR_BF16, eps, stream),
                   "nr_gated_residual_ln_modulate launch");
}

}  // extern "C"

namespace {

nr_status act_and_mul(const char* fn, int gelu, void* out, const void* x, int64_t rows,
                      int64_t inter, nr_dtype dtype, cudaStream_t stream) {
  if (!valid_dtype(dtype)) return fail(NR_ERR_DTYPE, "%s: unknown dtype %d", fn, (int)dtype);
  if (rows < 0 || inter <= 0) return fail(NR_ERR_SHAPE, "%s: need rows >= 0 and inter > 0", fn);
  if (rows == 0) return ok();
  if (!out || !x) return fail(NR_ERR_NULL, "%s: out and x must be non-NULL", fn);
  const int vec = vec_elems(dtype);
  if (inter % vec != 0)
    return fail(NR_ERR_UNSUPPORTED, "%s: inter = %lld is not a multiple of %d", fn,
                (long long)inter, vec);
  if (inter / vec > INT32_MAX / 2) return fail(NR_ERR_SHAPE, "%s: inter too large", fn);
  if (!aligned16(out) || !aligned16(x))
    return fail(NR_ERR_ALIGN, "%s: pointers must be 16-byte aligned", fn);
  const int64_t es = elem_size(dtype);
  if (overlap(dense(out, rows * inter * es), dense(x, rows * 2 * inter * es)))
    return fail(NR_ERR_ALIAS, "%s: out overlaps x", fn);
  const cudaError_t e = gelu ? nr::launch_gelu_and_mul(out, x, rows, inter, dtype == NR_BF16, stream)
                             : nr::launch_silu_and_mul(out, x, rows, inter, dtype == NR_BF16, stream);
  return from_cuda(e, fn);
}

}  // namespace

extern "C" {

nr_status nr_device_status(cudaStream_t stream) {
  CallRange range("nr_device_status");
  unsigned bits = 0;
  const cudaError_t e = nr::take_device_status(stream, &bits);
  if (e != cudaSuccess) return from_cuda(e, "nr_device_status");
  if (bits & nr::kStatusBitQkBulkWait)
    return fail(NR_ERR_TIMEOUT, "nr_device_status: a bounded wait for a bulk copy ran out in the "
                                "Q/K norm + RoPE kernel (status bits 0x%x)", bits);
  if (bits != 0)
    return fail(NR_ERR_TIMEOUT, "nr_device_status: the wait probe's wait ran out (status bits "
                                "0x%x)", bits);
  return ok();
}

nr_status nr_test_wait_probe(int64_t limit_cycles, cudaStream_t stream) {
  CallRange range("nr_test_wait_probe");
  if (limit_cycles < 1 || limit_cycles > (int64_t(1) << 32))
    return fail(NR_ERR_VALUE, "nr_test_wait_probe: limit_cycles must be in [1, 2^32]");
  return from_cuda(nr::launch_wait_probe(limit_cycles, stream), "nr_test_wait_probe");
}

nr_status nr_silu_and_mul(void* out, const void* x, int64_t rows, int64_t inter, nr_dtype dtype,
                          cudaStream_t stream) {
  CallRange range("nr_silu_and_mul");
  return act_and_mul("nr_silu_and_mul", 0, out, x, rows, inter, dtype, stream);
}

nr_status nr_gelu_and_mul(void* out, const void* x, int64_t rows, int64_t inter, nr_dtype dtype,
                          cudaStream_t stream) {
  CallRange range("nr_gelu_and_mul");
  return act_and_mul("nr_gelu_and_mul", 1, out, x, rows, inter, dtype, stream);
}

}  // extern "C"
