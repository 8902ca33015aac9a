/*
 * Oracle for the fused row-normalisation family -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU definition of what each op computes, in
 * double precision, with rounding to the storage dtype (bf16 or f32) only where
 * the method stores a value.  Nothing here is blocked, fused or reordered beyond
 * what the definitions state, so each function can be checked by eye against the
 * passage it cites.  It shares no code with the CUDA library and includes none
 * of its headers; only tests/, __graft_entry__.smoke() and bench.py's CPU
 * baseline leg may load it.
 *
 * Sources (page title, then the section on that page):
 *   [VT]  vllm.cpp, src/vt/cuda/cuda_ops.cu, sections named here by what they
 *         hold:
 *           - the bf16 load/store helpers (bf16 stores round to nearest even)
 *           - the residual-rounding helper (the residual is rounded to its
 *             storage dtype before it is squared)
 *           - the row-RMSNorm section (eps inside the sqrt, mean over h, gemma
 *             uses w+1)
 *           - the NeoX RoPE section (freq = base^(-2*pair/rot) in double,
 *             angle = pos*freq, rotate-half pairing (i, i+rot/2))
 *           - the fused attention-preamble section (per-(token, head) RMSNorm
 *             over head_dim, then the rotation, with no bf16 rounding between)
 *           - the SiLU and GELU gated-activation sections (gate = first half,
 *             up = second half)
 *           - the cache-driven RoPE section (GPT-J pairing, M-RoPE axes)
 *           - the fused RMSNorm + static FP8 section
 *   [PAN2] FastVideo compare view feat/pan2-inference-optimizations, PAN2 docs,
 *          "Performance switches" table, row dit_fused_kernels: names the fused
 *          LayerNorm + modulation without printing its formula.  The oracle uses
 *          the plain adaLN reading out = LN(x)*(1+scale)+shift with the biased
 *          (1/N) variance, eps inside the sqrt and no affine weight or bias.
 *
 * Storage dtype codes: 0 = f32, 1 = bf16 (bf16 values travel as uint16 bits).
 *
 * Besides the stored result every op can return y, the exact (double)
 * pre-rounding value of each output.  The two ops whose last step adds terms
 * that can cancel (the RoPE rotation and the LayerNorm modulation) can also
 * return mag, the sum of magnitudes of the quantities combined into that output;
 * comparisons use it to size the f32 evaluation error a GPU makes there.
 */
#include <fenv.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#define NRO_F32 0
#define NRO_BF16 1

/* ------------------------------------------------------------------------ */
/* bf16 storage                                                              */
/* ------------------------------------------------------------------------ */

/* Exact value of a bf16 bit pattern: bf16 is the top half of an f32. */
double nro_bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round a double straight to bf16, round-to-nearest, ties-to-even ([VT]
 * bf16 load/store helpers).  Rounds once, from the double, never via f32.
 * bf16 keeps 8 significant bits; its normal exponents reach down to 2^-126 and
 * below that the grid is the fixed subnormal step 2^-133. */
uint16_t nro_bf16_round(double d) {
  if (isnan(d)) return (uint16_t)0x7FC0;
  const uint16_t sign = signbit(d) ? (uint16_t)0x8000 : (uint16_t)0;
  const double a = fabs(d);
  if (isinf(a)) return (uint16_t)(sign | 0x7F80);
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);               /* a = m * 2^e, 0.5 <= m < 1, so a in [2^(e-1), 2^e) */
  int quantum_exp = (e - 1) - 7;  /* spacing of 8-significant-bit numbers there */
  if (quantum_exp < -133) quantum_exp = -133;
  const double scaled = ldexp(a, -quantum_exp);  /* exact: power-of-two scaling */
  const double n = nearbyint(scaled);            /* default mode: ties to even */
  const double r = ldexp(n, quantum_exp);
  if (r >= 0x1p128) return (uint16_t)(sign | 0x7F80); /* overflow to infinity */
  const float rf = (float)r; /* exact: every bf16 value is an f32 value */
  uint32_t u;
  memcpy(&u, &rf, sizeof u);
  return (uint16_t)(sign | (uint16_t)(u >> 16));
}

/* nro_bf16_round over an array (for exhaustive checks of the rounding). */
void nro_bf16_round_array(const double* d, uint16_t* bits, int64_t n) {
  for (int64_t i = 0; i < n; i++) bits[i] = nro_bf16_round(d[i]);
}

/* Value of element i of a stored array of the given dtype, as a double. */
static double load(int dtype, const void* p, int64_t i) {
  if (dtype == NRO_BF16) return nro_bf16_value(((const uint16_t*)p)[i]);
  return (double)((const float*)p)[i];
}

/* Round v to the storage dtype and return the stored value as a double. */
static double round_to(int dtype, double v) {
  if (dtype == NRO_BF16) return nro_bf16_value(nro_bf16_round(v));
  return (double)(float)v; /* C conversion: round to nearest even */
}

/* Store v (rounded to the dtype) at element i. */
static void store(int dtype, void* p, int64_t i, double v) {
  if (dtype == NRO_BF16)
    ((uint16_t*)p)[i] = nro_bf16_round(v);
  else
    ((float*)p)[i] = (float)v;
}

/* ------------------------------------------------------------------------ */
/* RMSNorm, optionally with the fused residual add ([VT] row-RMSNorm         */
/* section and its residual-rounding helper).                                */
/*                                                                            */
/*   with a residual: v_j = round_dtype(x_j + res_j), and res_j <- v_j        */
/*   without one:     v_j = x_j                                               */
/*   ms  = (sum_j v_j^2) / hidden                                             */
/*   inv = 1 / sqrt(ms + eps)                                                 */
/*   y_j = v_j * inv * (w_j + 1 if gemma else w_j);  out_j = round_dtype(y_j) */
/* ------------------------------------------------------------------------ */
void nro_rmsnorm(int dtype, int64_t rows, int64_t hidden, const void* x, const void* w,
                 const void* res_in, double eps, int gemma, void* out, void* res_out,
                 double* y) {
  for (int64_t r = 0; r < rows; r++) {
    const int64_t base = r * hidden;
    double sum_sq = 0.0;
    for (int64_t j = 0; j < hidden; j++) {
      double v = load(dtype, x, base + j);
      if (res_in != NULL) {
        /* The exact sum of two stored values, rounded once to the residual's
         * storage dtype: the value written back and the value squared. */
        v = round_to(dtype, v + load(dtype, res_in, base + j));
        store(dtype, res_out, base + j, v);
      }
      sum_sq += v * v;
    }
    const double ms = sum_sq / (double)hidden;
    const double inv = 1.0 / sqrt(ms + eps);
    for (int64_t j = 0; j < hidden; j++) {
      const double v = (res_in != NULL) ? load(dtype, res_out, base + j) : load(dtype, x, base + j);
      double wj = load(dtype, w, j);
      if (gemma) wj += 1.0;
      const double yj = v * inv * wj;
      store(dtype, out, base + j, yj);
      if (y != NULL) y[base + j] = yj;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* RMSNorm + static FP8 (e4m3) quantisation ([VT] fused RMSNorm + static FP8  */
/* section): the RMSNorm above, its output rounded to bf16 (nb), and the code */
/*   code_j = e4m3_satfinite( f32(nb_j) * inv_scale ),  inv_scale = 1 / scale  */
/* where inv_scale and the product are f32 operations (the page computes the  */
/* code in f32 from the bf16-rounded value), so the code is decided in f32 on */
/* both sides.                                                                */
/*                                                                            */
/* e4m3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, subnormal     */
/* step 2^-9, no infinities (0x7f/0xff are NaN), largest finite 448.  Values  */
/* round to nearest, ties to even; finite values beyond +-448 saturate to     */
/* +-448.                                                                     */
/* ------------------------------------------------------------------------ */
uint8_t nro_e4m3_satfinite(float f) {
  if (isnan(f)) return (uint8_t)0x7F;
  const uint8_t sign = signbit(f) ? (uint8_t)0x80 : (uint8_t)0;
  const double a = fabs((double)f);
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e); /* a in [2^(e-1), 2^e) */
  int quantum_exp = (e - 1) - 3;
  if (quantum_exp < -9) quantum_exp = -9;
  double r = ldexp(nearbyint(ldexp(a, -quantum_exp)), quantum_exp);
  if (r > 448.0) r = 448.0;
  if (r < 0x1p-6) return (uint8_t)(sign | (uint8_t)ldexp(r, 9)); /* subnormal: r / 2^-9 */
  frexp(r, &e);
  const int exp_field = (e - 1) + 7;
  const int mant = (int)(ldexp(r, -(e - 1)) * 8.0) - 8; /* (r / 2^(e-1) - 1) * 8 */
  return (uint8_t)(sign | (uint8_t)(exp_field << 3) | (uint8_t)mant);
}

void nro_e4m3_array(const float* f, uint8_t* codes, int64_t n) {
  for (int64_t i = 0; i < n; i++) codes[i] = nro_e4m3_satfinite(f[i]);
}

void nro_rmsnorm_quant_fp8(int dtype, int64_t rows, int64_t hidden, const void* x, const void* w,
                           const void* res_in, double eps, int gemma, float scale,
                           uint8_t* out_fp8, uint16_t* out_bf16, void* res_out, double* y) {
  const float inv_scale = 1.0f / scale;
  for (int64_t r = 0; r < rows; r++) {
    const int64_t base = r * hidden;
    double sum_sq = 0.0;
    for (int64_t j = 0; j < hidden; j++) {
      double v = load(dtype, x, base + j);
      if (res_in != NULL) {
        v = round_to(dtype, v + load(dtype, res_in, base + j));
        store(dtype, res_out, base + j, v);
      }
      sum_sq += v * v;
    }
    const double inv = 1.0 / sqrt(sum_sq / (double)hidden + eps);
    for (int64_t j = 0; j < hidden; j++) {
      const double v = (res_in != NULL) ? load(dtype, res_out, base + j) : load(dtype, x, base + j);
      double wj = load(dtype, w, j);
      if (gemma) wj += 1.0;
      const double yj = v * inv * wj;
      const uint16_t nb = nro_bf16_round(yj);
      const float t = (float)nro_bf16_value(nb) * inv_scale; /* f32 multiply */
      out_fp8[base + j] = nro_e4m3_satfinite(t);
      if (out_bf16 != NULL) out_bf16[base + j] = nb;
      if (y != NULL) y[base + j] = yj;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Per-head Q/K RMSNorm followed by NeoX RoPE ([VT] fused attention-preamble */
/* and NeoX RoPE sections).  For token t and head h of a tensor with its own  */
/* norm weight w (one vector of length D, shared by all heads):               */
/*                                                                            */
/*   inv = 1 / sqrt(mean_j v_j^2 + eps),   n_j = v_j * inv * w_j (w_j+1 gemma)  */
/*   for i < D/2:  f_i = theta^(-2i/D)   (double)                             */
/*                 a   = pos_t * f_i     (double);  c = cos a, s = sin a      */
/*                 y_i       = n_i c - n_{i+D/2} s                            */
/*                 y_{i+D/2} = n_i s + n_{i+D/2} c                            */
/*   out = round_dtype(y)  (one rounding: the normed values are not stored)   */
/*                                                                            */
/* The rotary dimension is the whole head_dim.  Element (t, h, j) of an input */
/* or output lives at t*tok_stride + h*D + j; outputs share the input strides. */
/* mag_i = mag_{i+D/2} = |n_i| + |n_{i+D/2}| bounds every term of the rotation. */
/* ------------------------------------------------------------------------ */
static void norm_rope_one(int dtype, int w_dtype, int64_t tokens, int64_t heads, int64_t D,
                          const void* src, int64_t tok_stride, const void* w,
                          const int32_t* pos, double eps, double theta, int gemma, void* dst,
                          double* y, double* mag) {
  const int64_t half = D / 2;
  double n[1024];
  for (int64_t t = 0; t < tokens; t++) {
    for (int64_t h = 0; h < heads; h++) {
      const int64_t base = t * tok_stride + h * D;
      double sum_sq = 0.0;
      for (int64_t j = 0; j < D; j++) {
        const double v = load(dtype, src, base + j);
        sum_sq += v * v;
      }
      const double inv = 1.0 / sqrt(sum_sq / (double)D + eps);
      for (int64_t j = 0; j < D; j++) {
        double wj = load(w_dtype, w, j);
        if (gemma) wj += 1.0;
        n[j] = load(dtype, src, base + j) * inv * wj;
      }
      for (int64_t i = 0; i < half; i++) {
        const double freq = pow(theta, -2.0 * (double)i / (double)D);
        const double angle = (double)pos[t] * freq;
        const double c = cos(angle);
        const double s = sin(angle);
        const double first = n[i] * c - n[i + half] * s;
        const double second = n[i] * s + n[i + half] * c;
        store(dtype, dst, base + i, first);
        store(dtype, dst, base + i + half, second);
        if (y != NULL) {
          y[base + i] = first;
          y[base + i + half] = second;
        }
        if (mag != NULL) {
          mag[base + i] = fabs(n[i]) + fabs(n[i + half]);
          mag[base + i + half] = fabs(n[i]) + fabs(n[i + half]);
        }
      }
    }
  }
}

/* Returns 0 on success, -1 when head_dim is odd or above the oracle's bound. */
int nro_qk_norm_rope(int dtype, int w_dtype, int64_t tokens, int64_t hq, int64_t hk,
                     int64_t head_dim, const void* q, int64_t q_tok_stride, const void* k,
                     int64_t k_tok_stride, const void* wq, const void* wk, const int32_t* pos,
                     double eps, double theta, int gemma, void* q_out, void* k_out, double* q_y,
                     double* k_y, double* q_mag, double* k_mag) {
  if (head_dim <= 0 || head_dim % 2 != 0 || head_dim > 1024) return -1;
  norm_rope_one(dtype, w_dtype, tokens, hq, head_dim, q, q_tok_stride, wq, pos, eps, theta, gemma,
                q_out, q_y, q_mag);
  norm_rope_one(dtype, w_dtype, tokens, hk, head_dim, k, k_tok_stride, wk, pos, eps, theta, gemma,
                k_out, k_y, k_mag);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* RoPE variants on top of the per-head RMSNorm ([VT] NeoX RoPE, cache-driven */
/* RoPE and fused attention-preamble sections):                              */
/*  - rotary dim rot <= D: pairs i < rot/2 rotate; elements [rot, D) keep the */
/*    normed value;  f_i = theta^(-2i/rot)                                     */
/*  - pairing: rotate-half (i, i + rot/2) or interleaved GPT-J (2i, 2i + 1)    */
/*  - Llama-3 frequency rescale (factor > 0): with wavelength L = 2pi / f,     */
/*    L < orig/high keeps f, L > orig/low gives f / factor, and in between    */
/*    f is interpolated with weight s = (orig/L - low) / (high - low) on the  */
/*    unscaled frequency: (1 - s) f / factor + s f                            */
/*  - M-RoPE: positions are [3, tokens] (axis t, h, w); pair i takes the       */
/*    position of axis(i): contiguous sections (t: i < sec_t, h: next sec_h,  */
/*    w: the rest) or interleaved (i % 3 == 1 within the first sec_h such     */
/*    pairs: h; i % 3 == 2 within the first sec_w: w; otherwise t).           */
/* ------------------------------------------------------------------------ */
static double llama3_frequency(double f, double factor, double low, double high, double orig) {
  if (!(factor > 0.0)) return f;
  const double two_pi = 6.283185307179586476925286766559;
  const double wavelength = two_pi / f;
  if (wavelength < orig / high) return f;
  if (wavelength > orig / low) return f / factor;
  const double s = (low != high) ? (orig / wavelength - low) / (high - low) : 0.0;
  return (1.0 - s) * f / factor + s * f;
}

static int mrope_axis(int64_t i, const int* sections, int interleaved) {
  if (sections == NULL) return 0;
  if (interleaved) {
    if (i % 3 == 1 && i / 3 < sections[1]) return 1;
    if (i % 3 == 2 && i / 3 < sections[2]) return 2;
    return 0;
  }
  if (i < sections[0]) return 0;
  if (i < sections[0] + sections[1]) return 1;
  return 2;
}

static void norm_rope_ex_one(int dtype, int w_dtype, int64_t tokens, int64_t heads, int64_t D,
                             const void* src, int64_t tok_stride, const void* w,
                             const int32_t* pos, double eps, int gemma, int64_t rot,
                             int interleaved, double theta, double l3_factor, double l3_low,
                             double l3_high, double l3_orig, const int* sections,
                             int mrope_interleaved, void* dst, double* y, double* mag) {
  double n[1024];
  for (int64_t t = 0; t < tokens; t++) {
    for (int64_t h = 0; h < heads; h++) {
      const int64_t row0 = t * tok_stride + h * D;
      double sum_sq = 0.0;
      for (int64_t j = 0; j < D; j++) {
        const double v = load(dtype, src, row0 + j);
        sum_sq += v * v;
      }
      const double inv = 1.0 / sqrt(sum_sq / (double)D + eps);
      for (int64_t j = 0; j < D; j++) {
        double wj = load(w_dtype, w, j);
        if (gemma) wj += 1.0;
        n[j] = load(dtype, src, row0 + j) * inv * wj;
      }
      for (int64_t j = rot; j < D; j++) { /* not rotated: the normed value */
        store(dtype, dst, row0 + j, n[j]);
        if (y != NULL) y[row0 + j] = n[j];
        if (mag != NULL) mag[row0 + j] = fabs(n[j]);
      }
      for (int64_t i = 0; i < rot / 2; i++) {
        const double f = llama3_frequency(pow(theta, -2.0 * (double)i / (double)rot), l3_factor,
                                          l3_low, l3_high, l3_orig);
        const int axis = mrope_axis(i, sections, mrope_interleaved);
        const double angle = (double)pos[axis * tokens + t] * f;
        const double c = cos(angle), s = sin(angle);
        const int64_t a = interleaved ? 2 * i : i;
        const int64_t b = interleaved ? 2 * i + 1 : i + rot / 2;
        const double ya = n[a] * c - n[b] * s;
        const double yb = n[a] * s + n[b] * c;
        store(dtype, dst, row0 + a, ya);
        store(dtype, dst, row0 + b, yb);
        if (y != NULL) {
          y[row0 + a] = ya;
          y[row0 + b] = yb;
        }
        if (mag != NULL) mag[row0 + a] = mag[row0 + b] = fabs(n[a]) + fabs(n[b]);
      }
    }
  }
}

/* Returns 0, or -1 for a shape the definition does not cover. */
int nro_qk_norm_rope_ex(int dtype, int w_dtype, int64_t tokens, int64_t hq, int64_t hk,
                        int64_t head_dim, const void* q, int64_t q_tok_stride, const void* k,
                        int64_t k_tok_stride, const void* wq, const void* wk, const int32_t* pos,
                        double eps, int gemma, int64_t rot, int interleaved, double theta,
                        double l3_factor, double l3_low, double l3_high, double l3_orig,
                        const int* sections, int mrope_interleaved, void* q_out, void* k_out,
                        double* q_y, double* k_y, double* q_mag, double* k_mag) {
  if (head_dim <= 0 || head_dim > 1024 || rot <= 0 || rot > head_dim || rot % 2 != 0) return -1;
  norm_rope_ex_one(dtype, w_dtype, tokens, hq, head_dim, q, q_tok_stride, wq, pos, eps, gemma,
                   rot, interleaved, theta, l3_factor, l3_low, l3_high, l3_orig, sections,
                   mrope_interleaved, q_out, q_y, q_mag);
  norm_rope_ex_one(dtype, w_dtype, tokens, hk, head_dim, k, k_tok_stride, wk, pos, eps, gemma,
                   rot, interleaved, theta, l3_factor, l3_low, l3_high, l3_orig, sections,
                   mrope_interleaved, k_out, k_y, k_mag);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* LayerNorm (no affine) + adaLN modulation ([PAN2]; formula as read above).   */
/*                                                                            */
/*   mu = mean_j x_j;  var = mean_j (x_j - mu)^2   (two passes, biased)       */
/*   xhat_j = (x_j - mu) / sqrt(var + eps)                                    */
/*   y_j = xhat_j * (1 + scale_j) + shift_j;  out_j = round_dtype(y_j)        */
/*                                                                            */
/* shift and scale hold one row per sample; row r uses sample r / rows_per_sample. */
/* mag_j = (|x_j - mu| + mean_k |x_k|) / sqrt(var + eps) * |1 + scale_j| + |shift_j| */
/* bounds the terms of the last step, including the error a rounded mean      */
/* carries into x_j - mu.                                                     */
/* ------------------------------------------------------------------------ */
void nro_ln_modulate(int dtype, int64_t rows, int64_t hidden, int64_t rows_per_sample,
                     const void* x, const void* shift, const void* scale, double eps, void* out,
                     double* y, double* mag) {
  for (int64_t r = 0; r < rows; r++) {
    const int64_t base = r * hidden;
    const int64_t sample = (r / rows_per_sample) * hidden;
    double sum = 0.0, sum_abs = 0.0;
    for (int64_t j = 0; j < hidden; j++) {
      sum += load(dtype, x, base + j);
      sum_abs += fabs(load(dtype, x, base + j));
    }
    const double mu = sum / (double)hidden;
    double sum_dev = 0.0;
    for (int64_t j = 0; j < hidden; j++) {
      const double d = load(dtype, x, base + j) - mu;
      sum_dev += d * d;
    }
    const double var = sum_dev / (double)hidden;
    const double rstd = 1.0 / sqrt(var + eps);
    for (int64_t j = 0; j < hidden; j++) {
      const double d = load(dtype, x, base + j) - mu;
      const double xhat = d * rstd;
      const double g = 1.0 + load(dtype, scale, sample + j);
      const double sh = load(dtype, shift, sample + j);
      const double yj = xhat * g + sh;
      store(dtype, out, base + j, yj);
      if (y != NULL) y[base + j] = yj;
      if (mag != NULL)
        mag[base + j] = (fabs(d) + sum_abs / (double)hidden) * rstd * fabs(g) + fabs(sh);
    }
  }
}

/* ------------------------------------------------------------------------ */
/* a + b rounded to odd in double: the exact sum when it is a double, else    */
/* whichever of the two doubles around it has an odd last significand bit.   */
/* Rounding to odd in a format with at least two more significand bits than  */
/* the target, then to nearest in the target, rounds the exact value once     */
/* (Boldo and Melquiond, "Emulation of FMA and correctly rounded sums: proved */
/* algorithms using rounding to odd", IEEE Trans. Computers 57(4), 2008).     */
/* The error of the nearest sum comes from Knuth's TwoSum (TAOCP vol. 2,      */
/* 4.2.2), exact in the default rounding mode.                                */
/* ------------------------------------------------------------------------ */
static double sum_round_to_odd(double a, double b) {
  const double s = a + b;
  const double bb = s - a;
  const double err = (a - (s - bb)) + (b - bb); /* a + b = s + err exactly */
  if (err == 0.0) return s;
  /* the exact sum lies strictly between s and its neighbour toward err */
  const double other = nextafter(s, err > 0.0 ? INFINITY : -INFINITY);
  uint64_t bits;
  memcpy(&bits, &s, sizeof bits);
  return (bits & 1u) ? s : other;
}

/* ------------------------------------------------------------------------ */
/* Gated residual add + LayerNorm + adaLN modulation: the DiT step around the */
/* fused LayerNorm + modulation ([PAN2], as read above):                      */
/*   v_j = round_dtype(residual_j + gate_j * y_j)   (the exact value, rounded */
/*         once; written back to the residual)                                */
/*   out = LN(v) * (1 + scale) + shift              (nro_ln_modulate on v)    */
/* gate, shift and scale hold one row per sample (row r: r / rows_per_sample). */
/* ------------------------------------------------------------------------ */
void nro_gated_ln_modulate(int dtype, int64_t rows, int64_t hidden, int64_t rows_per_sample,
                           const void* residual, const void* y, const void* gate,
                           const void* shift, const void* scale, double eps, void* res_out,
                           void* out, double* y_out, double* mag) {
  for (int64_t r = 0; r < rows; r++) {
    const int64_t sample = (r / rows_per_sample) * hidden;
    for (int64_t j = 0; j < hidden; j++) {
      /* gate*y is exact in double (at most 2*24 = 48 significant bits).  The
       * sum with the residual is rounded to odd in double (53 >= 24 + 2
       * bits), so the store's rounding to nearest rounds the exact
       * residual + gate*y once. */
      const double gy = load(dtype, gate, sample + j) * load(dtype, y, r * hidden + j);
      const double v = sum_round_to_odd(load(dtype, residual, r * hidden + j), gy);
      store(dtype, res_out, r * hidden + j, v);
    }
  }
  nro_ln_modulate(dtype, rows, hidden, rows_per_sample, res_out, shift, scale, eps, out, y_out,
                  mag);
}

/* ------------------------------------------------------------------------ */
/* silu_and_mul ([VT] SiLU gated-activation section).  x is [rows, 2*inter]: */
/*   a = x[r, j] (gate, first half), b = x[r, inter + j] (up, second half)    */
/*   y = a / (1 + exp(-a)) * b;  out[r, j] = round_dtype(y)                   */
/* ------------------------------------------------------------------------ */
void nro_silu_and_mul(int dtype, int64_t rows, int64_t inter, const void* x, void* out,
                      double* y) {
  for (int64_t r = 0; r < rows; r++) {
    for (int64_t j = 0; j < inter; j++) {
      const double a = load(dtype, x, r * 2 * inter + j);
      const double b = load(dtype, x, r * 2 * inter + inter + j);
      const double yj = a / (1.0 + exp(-a)) * b;
      store(dtype, out, r * inter + j, yj);
      if (y != NULL) y[r * inter + j] = yj;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* gelu_and_mul ([VT] GELU gated-activation section): tanh GELU of the gate   */
/* (first half) times up (second half):                                      */
/*   gelu(a) = 0.5 a (1 + tanh(z)),  z = sqrt(2/pi) (a + 0.044715 a^3)        */
/*   y = gelu(a) * b;  out[r, j] = round_dtype(y)                             */
/* For z < 0 the sum 1 + tanh(z) is taken from tanh z = (e^2z - 1)/(e^2z + 1) */
/* as 2 e^2z / (1 + e^2z): the same number, without the cancellation that    */
/* leaves 1 + tanh(z) = 0 in double once z < -19 or so.                      */
/* ------------------------------------------------------------------------ */
void nro_gelu_and_mul(int dtype, int64_t rows, int64_t inter, const void* x, void* out,
                      double* y) {
  const double k = sqrt(2.0 / 3.14159265358979323846264338327950288);
  for (int64_t r = 0; r < rows; r++) {
    for (int64_t j = 0; j < inter; j++) {
      const double a = load(dtype, x, r * 2 * inter + j);
      const double b = load(dtype, x, r * 2 * inter + inter + j);
      const double z = k * (a + 0.044715 * a * a * a);
      const double one_plus_tanh = z >= 0 ? 1.0 + tanh(z) : 2.0 * exp(2 * z) / (1.0 + exp(2 * z));
      const double yj = 0.5 * a * one_plus_tanh * b;
      store(dtype, out, r * inter + j, yj);
      if (y != NULL) y[r * inter + j] = yj;
    }
  }
}

/* Rounding mode guard: the oracle's nearbyint and conversions assume the
 * default round-to-nearest mode; callers can check it. */
int nro_rounding_mode_is_nearest(void) { return fegetround() == FE_TONEAREST; }
