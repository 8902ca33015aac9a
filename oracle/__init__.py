"""CPU oracle for the fused row-normalisation family -- TEST INFRASTRUCTURE ONLY.

The arithmetic lives in ``oracle.c`` (plain C, double precision, storage-dtype
rounding only where the method stores).  This module compiles it with gcc and
wraps it with ctypes over numpy arrays.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
it; the CUDA library never does, and the oracle imports nothing from it.

Storage conventions: bf16 arrays are numpy ``uint16`` bit patterns, f32 arrays
are numpy ``float32``.  Every function returns the stored outputs and, on
request, ``y`` (the exact double value before the final rounding) and ``mag``
(for the two ops whose last step can cancel: the sum of magnitudes of the terms
combined into each output).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32 = 0
BF16 = 1

# -ffp-contract=off: no fused multiply-adds, so x86 and aarch64 builds evaluate
# the same roundings in the same order.
_CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (skipped when up to date)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    return compile_source(_SRC, _LIB)


_lib = None


def configure(lib):
    """Declare the C signatures on a loaded oracle library and check the FPU mode."""
    vp, i64, dbl, cint = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double, ctypes.c_int
    lib.nro_bf16_round.argtypes = [dbl]
    lib.nro_bf16_round.restype = ctypes.c_uint16
    lib.nro_bf16_value.argtypes = [ctypes.c_uint16]
    lib.nro_bf16_value.restype = dbl
    lib.nro_bf16_round_array.argtypes = [vp, vp, i64]
    lib.nro_bf16_round_array.restype = None
    lib.nro_e4m3_satfinite.argtypes = [ctypes.c_float]
    lib.nro_e4m3_satfinite.restype = ctypes.c_uint8
    lib.nro_e4m3_array.argtypes = [vp, vp, i64]
    lib.nro_e4m3_array.restype = None
    lib.nro_rmsnorm_quant_fp8.argtypes = [cint, i64, i64, vp, vp, vp, dbl, cint, ctypes.c_float,
                                          vp, vp, vp, vp]
    lib.nro_rmsnorm_quant_fp8.restype = None
    lib.nro_rmsnorm.argtypes = [cint, i64, i64, vp, vp, vp, dbl, cint, vp, vp, vp]
    lib.nro_rmsnorm.restype = None
    lib.nro_qk_norm_rope.argtypes = [cint, cint, i64, i64, i64, i64, vp, i64, vp, i64, vp, vp,
                                     vp, dbl, dbl, cint, vp, vp, vp, vp, vp, vp]
    lib.nro_qk_norm_rope.restype = cint
    lib.nro_qk_norm_rope_ex.argtypes = [cint, cint, i64, i64, i64, i64, vp, i64, vp, i64, vp, vp,
                                        vp, dbl, cint, i64, cint, dbl, dbl, dbl, dbl, dbl, vp,
                                        cint, vp, vp, vp, vp, vp, vp]
    lib.nro_qk_norm_rope_ex.restype = cint
    lib.nro_ln_modulate.argtypes = [cint, i64, i64, i64, vp, vp, vp, dbl, vp, vp, vp]
    lib.nro_ln_modulate.restype = None
    lib.nro_gated_ln_modulate.argtypes = [cint, i64, i64, i64, vp, vp, vp, vp, vp, dbl, vp, vp,
                                          vp, vp]
    lib.nro_gated_ln_modulate.restype = None
    lib.nro_gelu_and_mul.argtypes = [cint, i64, i64, vp, vp, vp]
    lib.nro_gelu_and_mul.restype = None
    lib.nro_silu_and_mul.argtypes = [cint, i64, i64, vp, vp, vp]
    lib.nro_silu_and_mul.restype = None
    lib.nro_rounding_mode_is_nearest.argtypes = []
    lib.nro_rounding_mode_is_nearest.restype = cint
    if not lib.nro_rounding_mode_is_nearest():
        raise RuntimeError("oracle: FPU rounding mode is not round-to-nearest")
    return lib


def compile_source(src_path: str, lib_path: str) -> str:
    """Compile an oracle source file with the oracle's flags (used by build())."""
    tmp = lib_path + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", *_CFLAGS, "-o", tmp, src_path, "-lm"])
    os.replace(tmp, lib_path)
    return lib_path


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = configure(ctypes.CDLL(_LIB))
    return _lib


def _dtype_code(arr: np.ndarray) -> int:
    if arr.dtype == np.uint16:
        return BF16
    if arr.dtype == np.float32:
        return F32
    raise TypeError("oracle inputs are uint16 (bf16 bits) or float32, got %s" % arr.dtype)


def _ptr(arr):
    return None if arr is None else arr.ctypes.data_as(ctypes.c_void_p)


def _c(arr):
    return None if arr is None else np.ascontiguousarray(arr)


def bf16_round(d: float) -> int:
    """bf16 bits of double d rounded once, to nearest, ties to even."""
    return int(_load().nro_bf16_round(float(d)))


def bf16_round_array(d: np.ndarray) -> np.ndarray:
    """bf16 bits (uint16) of each double in d, rounded once to nearest even."""
    d = np.ascontiguousarray(d, dtype=np.float64)
    bits = np.empty(d.shape, np.uint16)
    _load().nro_bf16_round_array(_ptr(d), _ptr(bits), d.size)
    return bits


def bf16_value(bits: int) -> float:
    """Exact value of bf16 bits as a Python float."""
    return float(_load().nro_bf16_value(int(bits)))


def bf16_bits_to_float64(bits: np.ndarray) -> np.ndarray:
    """Exact values of an array of bf16 bit patterns (a widening, not arithmetic)."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rmsnorm(x, w, residual=None, eps=1e-6, gemma=False, want_y=False):
    """RMSNorm of each row of x ([rows, hidden]), with the optional residual add.

    Returns (out, residual_out or None, y or None)."""
    lib = _load()
    x, w, residual = _c(x), _c(w), _c(residual)
    dt = _dtype_code(x)
    if w.dtype != x.dtype or (residual is not None and residual.dtype != x.dtype):
        raise TypeError("x, w and residual share one dtype")
    rows, hidden = x.shape
    out = np.empty_like(x)
    res_out = None if residual is None else np.empty_like(residual)
    y = np.empty(x.shape, np.float64) if want_y else None
    lib.nro_rmsnorm(dt, rows, hidden, _ptr(x), _ptr(w), _ptr(residual), float(eps), int(gemma),
                    _ptr(out), _ptr(res_out), _ptr(y))
    return out, res_out, y


def e4m3_array(f: np.ndarray) -> np.ndarray:
    """e4m3 codes (uint8) of f32 values: nearest, ties to even, saturating at +-448."""
    f = np.ascontiguousarray(f, dtype=np.float32)
    codes = np.empty(f.shape, np.uint8)
    _load().nro_e4m3_array(_ptr(f), _ptr(codes), f.size)
    return codes


def rmsnorm_quant_fp8(x, w, scale, residual=None, eps=1e-6, gemma=False, want_y=False):
    """RMSNorm (optionally with the residual add), its bf16 rounding nb and the
    e4m3 code of f32(nb) * (1/scale).  Returns (codes, nb, residual_out, y)."""
    lib = _load()
    x, w, residual = _c(x), _c(w), _c(residual)
    dt = _dtype_code(x)
    rows, hidden = x.shape
    codes = np.empty(x.shape, np.uint8)
    nb = np.empty(x.shape, np.uint16)
    res_out = None if residual is None else np.empty_like(residual)
    y = np.empty(x.shape, np.float64) if want_y else None
    lib.nro_rmsnorm_quant_fp8(dt, rows, hidden, _ptr(x), _ptr(w), _ptr(residual), float(eps),
                              int(gemma), float(scale), _ptr(codes), _ptr(nb), _ptr(res_out),
                              _ptr(y))
    return codes, nb, res_out, y


def qk_norm_rope(q, k, wq, wk, positions, eps=1e-6, theta=10000.0, gemma=False, want_y=False):
    """Per-head RMSNorm + NeoX RoPE of q [tokens, hq, D] and k [tokens, hk, D].

    q and k may be views with a token stride larger than heads*D (the last two
    axes contiguous).  Returns (q_out, k_out, q_y, k_y, q_mag, k_mag); outputs are
    dense [tokens, heads, D] arrays (the oracle reads strided, writes dense)."""
    lib = _load()
    dt = _dtype_code(q)
    if k.dtype != q.dtype:
        raise TypeError("q and k share one dtype")
    wq, wk = _c(wq), _c(wk)
    wdt = _dtype_code(wq)
    if wk.dtype != wq.dtype:
        raise TypeError("wq and wk share one dtype")
    tokens, hq, D = q.shape
    _, hk, _ = k.shape
    q_d, k_d = np.ascontiguousarray(q), np.ascontiguousarray(k)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    if pos.shape != (tokens,):
        raise ValueError("positions must be [tokens]")
    q_out, k_out = np.empty_like(q_d), np.empty_like(k_d)
    q_y = np.empty(q_d.shape, np.float64) if want_y else None
    k_y = np.empty(k_d.shape, np.float64) if want_y else None
    q_mag = np.empty(q_d.shape, np.float64) if want_y else None
    k_mag = np.empty(k_d.shape, np.float64) if want_y else None
    rc = lib.nro_qk_norm_rope(dt, wdt, tokens, hq, hk, D, _ptr(q_d), hq * D, _ptr(k_d), hk * D,
                              _ptr(wq), _ptr(wk), _ptr(pos), float(eps), float(theta), int(gemma),
                              _ptr(q_out), _ptr(k_out), _ptr(q_y), _ptr(k_y), _ptr(q_mag),
                              _ptr(k_mag))
    if rc != 0:
        raise ValueError("oracle qk_norm_rope: head_dim must be even and <= 1024")
    return q_out, k_out, q_y, k_y, q_mag, k_mag


def qk_norm_rope_ex(q, k, wq, wk, positions, eps=1e-6, gemma=False, rotary_dim=None,
                    interleaved=False, theta=10000.0, llama3=None, mrope_sections=None,
                    mrope_interleaved=False, want_y=False):
    """The RoPE variants on top of the per-head RMSNorm: rotary_dim (default
    head_dim), GPT-J interleaved pairing, Llama-3 frequency rescale
    (llama3 = (factor, low_freq_factor, high_freq_factor, original_max_position)),
    M-RoPE (positions [3, tokens], mrope_sections = (t, h, w), contiguous or
    interleaved).  Returns (q_out, k_out, q_y, k_y, q_mag, k_mag), dense."""
    lib = _load()
    dt = _dtype_code(q)
    wq, wk = _c(wq), _c(wk)
    wdt = _dtype_code(wq)
    tokens, hq, D = q.shape
    _, hk, _ = k.shape
    rot = D if rotary_dim is None else int(rotary_dim)
    q_d, k_d = np.ascontiguousarray(q), np.ascontiguousarray(k)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    want_shape = (3, tokens) if mrope_sections is not None else (tokens,)
    if pos.shape != want_shape:
        raise ValueError("positions must be %s" % (want_shape,))
    l3 = (0.0, 1.0, 4.0, 8192.0) if llama3 is None else tuple(float(v) for v in llama3)
    sec = None if mrope_sections is None else np.ascontiguousarray(mrope_sections, dtype=np.int32)
    q_out, k_out = np.empty_like(q_d), np.empty_like(k_d)
    arrs = [np.empty(a.shape, np.float64) if want_y else None for a in (q_d, k_d, q_d, k_d)]
    rc = lib.nro_qk_norm_rope_ex(dt, wdt, tokens, hq, hk, D, _ptr(q_d), hq * D, _ptr(k_d), hk * D,
                                 _ptr(wq), _ptr(wk), _ptr(pos), float(eps), int(gemma), rot,
                                 int(bool(interleaved)), float(theta), *l3, _ptr(sec),
                                 int(bool(mrope_interleaved)), _ptr(q_out), _ptr(k_out),
                                 *(_ptr(a) for a in arrs))
    if rc != 0:
        raise ValueError("oracle qk_norm_rope_ex: unsupported shape")
    return (q_out, k_out, *arrs)


def ln_modulate(x, shift, scale, eps=1e-6, rows_per_sample=None, want_y=False):
    """LayerNorm (no affine) + adaLN modulation of x [rows, hidden].

    shift/scale are [samples, hidden] (or [hidden] for one sample); row r uses
    sample r // rows_per_sample.  Returns (out, y or None, mag or None)."""
    lib = _load()
    x = _c(x)
    dt = _dtype_code(x)
    shift = _c(np.atleast_2d(shift))
    scale = _c(np.atleast_2d(scale))
    if shift.dtype != x.dtype or scale.dtype != x.dtype:
        raise TypeError("x, shift and scale share one dtype")
    rows, hidden = x.shape
    if rows_per_sample is None:
        rows_per_sample = max(rows, 1)
    out = np.empty_like(x)
    y = np.empty(x.shape, np.float64) if want_y else None
    mag = np.empty(x.shape, np.float64) if want_y else None
    lib.nro_ln_modulate(dt, rows, hidden, int(rows_per_sample), _ptr(x), _ptr(shift), _ptr(scale),
                        float(eps), _ptr(out), _ptr(y), _ptr(mag))
    return out, y, mag


def gated_ln_modulate(residual, y, gate, shift, scale, eps=1e-6, rows_per_sample=None,
                      want_y=False):
    """residual <- round(residual + gate * y) (one rounding of the exact value),
    then LayerNorm + modulation of it.  gate/shift/scale are [samples, hidden].
    Returns (out, residual_out, y or None, mag or None)."""
    lib = _load()
    residual, y = _c(residual), _c(y)
    dt = _dtype_code(residual)
    gate, shift, scale = (_c(np.atleast_2d(a)) for a in (gate, shift, scale))
    for a in (y, gate, shift, scale):
        if a.dtype != residual.dtype:
            raise TypeError("all operands share one dtype")
    rows, hidden = residual.shape
    if rows_per_sample is None:
        rows_per_sample = max(rows, 1)
    out, res_out = np.empty_like(residual), np.empty_like(residual)
    yv = np.empty(residual.shape, np.float64) if want_y else None
    mag = np.empty(residual.shape, np.float64) if want_y else None
    lib.nro_gated_ln_modulate(dt, rows, hidden, int(rows_per_sample), _ptr(residual), _ptr(y),
                              _ptr(gate), _ptr(shift), _ptr(scale), float(eps), _ptr(res_out),
                              _ptr(out), _ptr(yv), _ptr(mag))
    return out, res_out, yv, mag


def silu_and_mul(x, want_y=False):
    """silu(x[:, :I]) * x[:, I:] for x [rows, 2I].  Returns (out, y or None)."""
    lib = _load()
    x = _c(x)
    dt = _dtype_code(x)
    rows, two_i = x.shape
    if two_i % 2:
        raise ValueError("x's last axis must be even")
    inter = two_i // 2
    out = np.empty((rows, inter), x.dtype)
    y = np.empty((rows, inter), np.float64) if want_y else None
    lib.nro_silu_and_mul(dt, rows, inter, _ptr(x), _ptr(out), _ptr(y))
    return out, y


def gelu_and_mul(x, want_y=False):
    """gelu_tanh(x[:, :I]) * x[:, I:] for x [rows, 2I].  Returns (out, y or None)."""
    lib = _load()
    x = _c(x)
    dt = _dtype_code(x)
    rows, two_i = x.shape
    if two_i % 2:
        raise ValueError("x's last axis must be even")
    inter = two_i // 2
    out = np.empty((rows, inter), x.dtype)
    y = np.empty((rows, inter), np.float64) if want_y else None
    lib.nro_gelu_and_mul(dt, rows, inter, _ptr(x), _ptr(out), _ptr(y))
    return out, y
