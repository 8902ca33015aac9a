/*
 * nr.h -- C ABI of the fused row-normalisation library (libnormrope.so).
 *
 * Ops that sit between a transformer's GEMMs, as hand-written CUDA kernels
 * for sm_103a:
 *   nr_rmsnorm                      RMSNorm, optionally with the fused residual
 *                                   add (gemma w+1)
 *   nr_rmsnorm_quant_fp8            the same, writing static-scale FP8 e4m3 codes
 *   nr_qk_norm_rope                 per-head Q/K RMSNorm fused with NeoX rotary
 *                                   embedding
 *   nr_qk_norm_rope_ex              the same with RoPE variants (partial rotary,
 *                                   GPT-J pairs, Llama-3 rescale, M-RoPE)
 *   nr_ln_modulate                  LayerNorm (no affine) fused with DiT adaLN
 *                                   modulation
 *   nr_gated_residual_ln_modulate   residual += gate * y, then LayerNorm +
 *                                   modulation of the new residual
 *   nr_silu_and_mul                 silu(gate) * up
 *   nr_gelu_and_mul                 gelu_tanh(gate) * up
 *
 * Conventions shared by every entry point
 *   - Pointers are DEVICE pointers (CUDA global memory) owned by the caller; the
 *     library allocates nothing and frees nothing.  Its only state is one
 *     status word per device that kernels set when a bounded wait runs out
 *     (nr_device_status reads and clears it).
 *   - Each call opens one NVTX range named after the entry point for the
 *     time of the host call (validation and launch), so profilers can tell
 *     which call launched which kernel.
 *   - Every pointer must be 16-byte aligned, and every row start (row stride in
 *     bytes) a multiple of 16, so that each thread moves 128-bit vectors.
 *   - Work is enqueued asynchronously on `stream` (0 = the legacy default
 *     stream); the call returns once the kernel is launched.
 *   - All arithmetic is f32 (bf16 values are widened exactly); each stored
 *     output is rounded once, to nearest even, to its storage dtype.
 *   - Arguments are validated on the host before anything is launched.  A
 *     rejected call launches nothing and returns a non-zero nr_status; the
 *     reason is available from nr_last_error_message() on the same thread.
 *     A call with zero rows (tokens) returns NR_OK without launching and
 *     without looking at its pointers.  No C++ exception crosses this ABI.
 *   - NR_ERR_CUDA reports a failed launch (cudaGetLastError after it); like
 *     any CUDA error it can also surface a fault left by earlier work.
 *
 * Citations name the page and the section each operation follows.
 */
#ifndef NR_H
#define NR_H

#include <stdint.h>

#include <cuda_runtime_api.h> /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nr_status {
  NR_OK = 0,
  NR_ERR_NULL = 1,        /* a required pointer is NULL */
  NR_ERR_SHAPE = 2,       /* a size is negative or zero where it must be positive, or too large */
  NR_ERR_DTYPE = 3,       /* unknown dtype code, or a dtype combination that is not offered */
  NR_ERR_ALIGN = 4,       /* a pointer or row stride is not a multiple of 16 bytes */
  NR_ERR_ALIAS = 5,       /* an output overlaps an input (or another output) it may not overlap */
  NR_ERR_UNSUPPORTED = 6, /* a valid size the kernels do not cover (e.g. hidden % 8 for bf16) */
  NR_ERR_CUDA = 7,        /* the launch failed; see nr_last_error_message() */
  NR_ERR_VALUE = 8,       /* a scalar is out of range (eps < 0 or not finite, theta <= 0) */
  NR_ERR_TIMEOUT = 9      /* a kernel gave up a bounded wait (see nr_device_status) */
} nr_status;

typedef enum nr_dtype {
  NR_F32 = 0, /* IEEE binary32 */
  NR_BF16 = 1 /* bfloat16: 1 sign, 8 exponent, 7 fraction bits */
} nr_dtype;

/*
 * RMSNorm of each row, with the optional fused residual add.
 *
 * Follows the vllm.cpp page src/vt/cuda/cuda_ops.cu, its row-RMSNorm section
 * and the residual-rounding helper before it (the residual is rounded to its
 * storage dtype before it is squared, and that rounded value is what is
 * written back).
 * For row r of x [rows, hidden] (row-major, contiguous):
 *     with a residual:  v_j = round(x_j + residual_j);  residual_j <- v_j   (in place)
 *     without one:      v_j = x_j
 *     inv   = 1 / sqrt(mean_j v_j^2 + eps)
 *     out_j = round(v_j * inv * (gemma ? w_j + 1 : w_j))
 *
 * out       [rows, hidden], dtype `dtype`; may be x itself (then x is overwritten).
 * x         [rows, hidden], dtype `dtype`.
 * w         [hidden], dtype `dtype` (the weight dtype equals x's, as on the page).
 * residual  [rows, hidden], dtype `dtype`, read and written in place; NULL for
 *           plain RMSNorm.  It may not overlap x, w or out.
 * hidden    > 0; a multiple of 8 (bf16) or 4 (f32).
 * eps       finite, >= 0.
 * gemma     0 or 1.
 * Errors: NR_ERR_NULL, NR_ERR_SHAPE, NR_ERR_DTYPE, NR_ERR_ALIGN, NR_ERR_ALIAS,
 *         NR_ERR_UNSUPPORTED, NR_ERR_VALUE, NR_ERR_CUDA.
 */
nr_status nr_rmsnorm(void* out, const void* x, const void* w, void* residual, int64_t rows,
                     int64_t hidden, nr_dtype dtype, float eps, int gemma, cudaStream_t stream);

/*
 * RMSNorm (optionally with the fused residual add) followed by static FP8
 * quantisation of its output.
 *
 * Follows vllm.cpp src/vt/cuda/cuda_ops.cu, fused RMSNorm + static FP8
 * section: the normalised value n_j of nr_rmsnorm is rounded to bf16 (nb_j,
 * whatever the input dtype), and
 *     code_j = e4m3_satfinite(f32(nb_j) * inv_scale),   inv_scale = 1.0f / scale
 * with the product in f32: FP8 E4M3 (bias 7, largest finite 448, no
 * infinities), round to nearest even, finite values beyond +-448 saturating.
 *
 * codes     [rows, hidden] bytes (e4m3 codes).
 * out_bf16  [rows, hidden] bf16 copy of nb, or NULL.
 * x, w, residual, rows, hidden, dtype, eps, gemma: as nr_rmsnorm; hidden is at
 *           most 32768 (bf16) / 16384 (f32) here.
 * scale     finite, > 0, with 1/scale finite.
 * No output may overlap an input or the other output.
 * Errors: as nr_rmsnorm.
 */
nr_status nr_rmsnorm_quant_fp8(void* codes, void* out_bf16, const void* x, const void* w,
                               void* residual, int64_t rows, int64_t hidden, nr_dtype dtype,
                               float eps, int gemma, float scale, cudaStream_t stream);

/*
 * Per-head RMSNorm of Q and K followed by NeoX rotary embedding, in one pass.
 *
 * Follows vllm.cpp src/vt/cuda/cuda_ops.cu, the fused attention-preamble
 * section (RMSNorm over head_dim per (token, head), then the rotation, with no
 * rounding between them) and the NeoX RoPE section
 * (freq_i = theta^(-2i/head_dim), angle = pos * freq_i,
 * rotate-half pairing (i, i + head_dim/2)).  For token t, head h of Q (and of K
 * with wk):
 *     inv  = 1 / sqrt(mean_j v_j^2 + eps);   n_j = v_j * inv * (gemma ? w_j + 1 : w_j)
 *     out_i        = round(n_i cos(a_i) - n_{i+D/2} sin(a_i))
 *     out_{i+D/2}  = round(n_i sin(a_i) + n_{i+D/2} cos(a_i)),   a_i = pos_t * freq_i
 * The rotary dimension is the whole head_dim.  The angle p * freq_i is reduced
 * modulo 2*pi exactly in 64-bit fixed point before sin/cos, so large positions
 * keep full accuracy.
 *
 * Layout: element (t, h, d) of q lives at q + t*q_tok_stride + h*head_dim + d
 * (elements, not bytes), heads contiguous within a token; k likewise with
 * k_tok_stride.  q_out/k_out use the same strides as q/k.  q_out may be q and
 * k_out may be k (in place); otherwise outputs may not overlap any input or
 * each other (Q and K may be interleaved views of one fused buffer).
 *
 * q_out, q   [tokens, hq, head_dim] strided as above, dtype `dtype`.
 * k_out, k   [tokens, hk, head_dim], dtype `dtype`; may be NULL when hk == 0.
 * wq, wk     [head_dim], dtype `w_dtype` (NR_F32 or NR_BF16), one vector per
 *            tensor shared by all its heads; wk may be NULL when hk == 0.
 * positions  [tokens] int32, device memory; any value (negative too).
 * tokens >= 0, hq >= 1, hk >= 0.
 * head_dim   bf16: 16, 32, 64, 128, 256 or 512;  f32: 8, 16, 32, 64, 128 or 256.
 * q_tok_stride >= hq*head_dim and k_tok_stride >= hk*head_dim, each a multiple
 *            of 16 bytes.
 * eps finite >= 0;  theta > 0 and finite;  gemma 0 or 1.
 * Errors: as nr_rmsnorm.
 */
nr_status nr_qk_norm_rope(void* q_out, void* k_out, const void* q, const void* k, const void* wq,
                          const void* wk, nr_dtype w_dtype, const int32_t* positions,
                          int64_t tokens, int64_t hq, int64_t hk, int64_t head_dim,
                          int64_t q_tok_stride, int64_t k_tok_stride, float eps, double theta,
                          int gemma, nr_dtype dtype, cudaStream_t stream);

/*
 * RoPE variants for nr_qk_norm_rope_ex.  Zero-initialise, then set theta.
 *   rotary_dim           0 or head_dim: rotate the whole head; else the first
 *                        rotary_dim elements rotate and the rest keep their
 *                        normed value (vllm.cpp cuda_ops.cu, fused
 *                        attention-preamble section); freq_i = theta^(-2i/rotary_dim).
 *   interleaved          0: rotate-half pairs (i, i + rotary_dim/2) (NeoX);
 *                        1: GPT-J pairs (2i, 2i + 1) (cache-driven RoPE section).
 *   llama3_factor > 0    Llama-3 frequency rescale (NeoX RoPE section, Llama-3
 *                        rescale): with wavelength L = 2pi / freq, L below
 *                        original_max_position / high_freq_factor keeps freq,
 *                        L above original_max_position / low_freq_factor
 *                        divides it by llama3_factor, and in between it is
 *                        interpolated.
 *   mrope_section        all zero: positions are [tokens]; else M-RoPE with
 *                        positions [3, tokens] (rows t, h, w) and sections
 *                        (t, h, w) summing to rotary_dim / 2: contiguous, or
 *                        with mrope_interleaved = 1 the t/h/w rows cycle over
 *                        pairs i % 3 = 0/1/2 while each of h and w has pairs
 *                        left (cache-driven RoPE section, M-RoPE axis selection).
 */
typedef struct nr_rope_config {
  int64_t rotary_dim;
  int32_t interleaved;
  int32_t mrope_interleaved;
  double theta;
  double llama3_factor;
  double llama3_low_freq_factor;
  double llama3_high_freq_factor;
  double llama3_original_max_position;
  int32_t mrope_section[3];
} nr_rope_config;

/*
 * nr_qk_norm_rope with the RoPE variants of nr_rope_config.  Arguments as for
 * nr_qk_norm_rope (theta comes from the config); `positions` is [3, tokens]
 * when M-RoPE is on.  Additional requirements: 0 < rotary_dim <= head_dim,
 * rotary_dim a multiple of 16 (bf16) or 8 (f32) for rotate-half pairs and of 8
 * (bf16) or 4 (f32) for interleaved pairs; Llama-3 factors positive with
 * high_freq_factor >= low_freq_factor; M-RoPE sections >= 0.
 * Errors: as nr_qk_norm_rope; a NULL config is NR_ERR_NULL.
 */
nr_status nr_qk_norm_rope_ex(void* q_out, void* k_out, const void* q, const void* k,
                             const void* wq, const void* wk, nr_dtype w_dtype,
                             const int32_t* positions, int64_t tokens, int64_t hq, int64_t hk,
                             int64_t head_dim, int64_t q_tok_stride, int64_t k_tok_stride,
                             float eps, int gemma, const nr_rope_config* rope, nr_dtype dtype,
                             cudaStream_t stream);

/*
 * LayerNorm (no affine) fused with adaLN modulation.
 *
 * The pages name this fusion (FastVideo compare view
 * feat/pan2-inference-optimizations, PAN2 docs, "Performance switches",
 * dit_fused_kernels) without printing it; this is the plain adaLN reading:
 *     mu = mean_j x_j;  var = mean_j (x_j - mu)^2   (biased)
 *     out_j = round((x_j - mu) / sqrt(var + eps) * (1 + scale_j) + shift_j)
 * with f32 statistics.
 *
 * out, x        [rows, hidden], dtype `dtype`; out may be x.
 * shift, scale  [samples, hidden], dtype `dtype`; row r uses sample
 *               r / rows_per_sample (rows_per_sample >= rows: one sample for all rows;
 *               1: per-row modulation).
 * hidden > 0, a multiple of 8 (bf16) or 4 (f32);  eps finite >= 0.
 * Errors: as nr_rmsnorm.
 */
nr_status nr_ln_modulate(void* out, const void* x, const void* shift, const void* scale,
                         int64_t rows, int64_t hidden, int64_t rows_per_sample, float eps,
                         nr_dtype dtype, cudaStream_t stream);

/*
 * Gated residual add fused with LayerNorm + adaLN modulation -- the DiT step
 * around the fusion that nr_ln_modulate covers:
 *     residual_j <- round(residual_j + gate_j * y_j)    (in place; the exact value
 *                                                         rounded once)
 *     out_j = round((v_j - mu) / sqrt(var + eps) * (1 + scale_j) + shift_j)
 * with mu, var the mean and biased variance of the updated residual row v
 * (f32 statistics).  The pages name the LayerNorm + modulation fusion
 * (FastVideo compare view feat/pan2-inference-optimizations, PAN2 docs,
 * "Performance switches", dit_fused_kernels) but not the gate; this is the
 * plain DiT reading of the residual update next to it.
 *
 * out                    [rows, hidden], dtype `dtype`.
 * residual               [rows, hidden], read and written in place.
 * y                      [rows, hidden] (the branch output the gate scales).
 * gate, shift, scale     [samples, hidden]; row r uses sample r / rows_per_sample.
 * No operand may overlap out or residual.
 * hidden > 0, a multiple of 8 (bf16) or 4 (f32), at most 8192 (bf16) / 4096 (f32);
 * eps finite >= 0; rows_per_sample >= 1.
 * Errors: as nr_rmsnorm.
 */
nr_status nr_gated_residual_ln_modulate(void* out, void* residual, const void* y,
                                        const void* gate, const void* shift, const void* scale,
                                        int64_t rows, int64_t hidden, int64_t rows_per_sample,
                                        float eps, nr_dtype dtype, cudaStream_t stream);

/*
 * silu_and_mul: out[r, j] = silu(x[r, j]) * x[r, inter + j],  silu(a) = a / (1 + e^-a).
 *
 * Follows vllm.cpp src/vt/cuda/cuda_ops.cu, SiLU gated-activation section
 * (gate is the first half of each row, up the second; math in f32).  The
 * sigmoid is evaluated without forming e^-a, so f32 outputs keep their 1e-5
 * relative accuracy for every gate whose silu is a normal f32 (down to about
 * -92); below that silu(a) itself is an f32 subnormal and loses bits.
 *
 * out  [rows, inter], dtype `dtype`; may not overlap x.
 * x    [rows, 2*inter], dtype `dtype`.
 * inter > 0, a multiple of 8 (bf16) or 4 (f32).
 * Errors: as nr_rmsnorm.
 */
nr_status nr_silu_and_mul(void* out, const void* x, int64_t rows, int64_t inter, nr_dtype dtype,
                          cudaStream_t stream);

/*
 * gelu_and_mul: out[r, j] = gelu_tanh(x[r, j]) * x[r, inter + j], with the
 * tanh form of GELU
 *     gelu_tanh(a) = a/2 * (1 + tanh(sqrt(2/pi) * (a + 0.044715 a^3))).
 *
 * Follows vllm.cpp src/vt/cuda/cuda_ops.cu, GELU gated-activation section
 * (the gated MLP of Gemma-family models; same layout as silu_and_mul).
 * Evaluated as
 * a * sigmoid(2z), which equals the formula above and keeps its relative
 * accuracy for negative gates.
 *
 * Arguments, layout and errors: as nr_silu_and_mul.
 */
nr_status nr_gelu_and_mul(void* out, const void* x, int64_t rows, int64_t inter, nr_dtype dtype,
                          cudaStream_t stream);

/*
 * Device-side failure report.  Kernels that wait on hardware events (the
 * bulk-copy path of nr_qk_norm_rope waits for its copies on shared-memory
 * barriers) bound every wait (about one second of SM clock); a wait that runs
 * out sets a bit in a status word the library keeps on each device, the
 * kernel lets its copies in flight finish and returns, and the outputs of
 * that call are not valid.  nr_device_status works on the device that owns
 * `stream` (whatever device is current; the current device is restored): it
 * synchronises `stream`, reads that device's word and clears exactly the bits
 * it read, so a bit set meanwhile by a kernel on another stream is kept for
 * the next read.  The word is shared by every stream and thread of the
 * process on that device, so a report may concern a call made on another
 * stream.  Returns NR_OK if no wait ran out since the last read, else
 * NR_ERR_TIMEOUT (the message names the kernel).  A CUDA error while
 * synchronising is NR_ERR_CUDA.
 */
nr_status nr_device_status(cudaStream_t stream);

/*
 * Test hook for the failure path above: launches one block whose only wait
 * is on a barrier nothing completes, given up after `limit_cycles` SM clock
 * cycles (1 .. 2^32).  nr_device_status then reports NR_ERR_TIMEOUT.  Faults
 * and hangs nothing: the wait is bounded and the context stays usable.
 */
nr_status nr_test_wait_probe(int64_t limit_cycles, cudaStream_t stream);

/* Static, human-readable name of a status code. */
const char* nr_status_string(nr_status s);

/* Detail of the last non-OK status returned on the calling thread ("" if none).
 * The pointer stays valid until the next library call on this thread. */
const char* nr_last_error_message(void);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int nr_version(void);

#ifdef __cplusplus
}
#endif

#endif /* NR_H */
