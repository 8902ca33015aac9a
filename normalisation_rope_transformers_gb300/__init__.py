"""Fused row-normalisation kernels for GB300 (sm_103a): Python binding.

Thin ctypes binding over the C ABI in ``include/nr.h`` (``libnormrope.so``).
Each function marshals torch CUDA tensors into device pointers, sizes and the
current CUDA stream, calls the entry point of the same name, and raises on a
non-OK status.  Every step of the computation runs in the library's kernels;
there is no CPU or PyTorch fallback.  Importing fails loudly when the library
has not been built (``python normalisation_rope_transformers_gb300/build.py``
or ``__graft_entry__.build()``).

    rmsnorm(x, w, residual=None, eps=1e-6, gemma=False, out=None)
    rmsnorm_quant_fp8(x, w, scale, residual=None, eps=1e-6, gemma=False, out_bf16=False)
    qk_norm_rope(q, k, wq, wk, positions, eps=1e-6, theta=10000.0, gemma=False,
                 q_out=None, k_out=None)
    qk_norm_rope_ex(q, k, wq, wk, positions, ..., rotary_dim=None, interleaved=False,
                    llama3=None, mrope_sections=None, mrope_interleaved=False)
    ln_modulate(x, shift, scale, eps=1e-6, rows_per_sample=None, out=None)
    silu_and_mul(x, out=None)
    gelu_and_mul(x, out=None)
    gated_residual_ln_modulate(residual, y, gate, shift, scale, eps=1e-6,
                               rows_per_sample=None, out=None)
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libnormrope.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("%s is missing: build the CUDA library first "
                      "(python normalisation_rope_transformers_gb300/build.py)" % LIB_PATH)

lib = ctypes.CDLL(LIB_PATH)

_vp, _i64, _f32, _f64, _int = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_double,
                                ctypes.c_int)
lib.nr_rmsnorm.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _int, _f32, _int, _vp]
lib.nr_rmsnorm.restype = _int
lib.nr_rmsnorm_quant_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _f32, _int, _f32,
                                     _vp]
lib.nr_rmsnorm_quant_fp8.restype = _int
lib.nr_qk_norm_rope.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _int, _vp, _i64, _i64, _i64, _i64,
                                _i64, _i64, _f32, _f64, _int, _int, _vp]
lib.nr_qk_norm_rope.restype = _int


class RopeConfig(ctypes.Structure):
    """Mirror of nr_rope_config (include/nr.h)."""
    _fields_ = [("rotary_dim", ctypes.c_int64), ("interleaved", ctypes.c_int32),
                ("mrope_interleaved", ctypes.c_int32), ("theta", ctypes.c_double),
                ("llama3_factor", ctypes.c_double), ("llama3_low_freq_factor", ctypes.c_double),
                ("llama3_high_freq_factor", ctypes.c_double),
                ("llama3_original_max_position", ctypes.c_double),
                ("mrope_section", ctypes.c_int32 * 3)]


lib.nr_qk_norm_rope_ex.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _int, _vp, _i64, _i64, _i64,
                                   _i64, _i64, _i64, _f32, _int, ctypes.POINTER(RopeConfig), _int,
                                   _vp]
lib.nr_qk_norm_rope_ex.restype = _int
lib.nr_ln_modulate.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _f32, _int, _vp]
lib.nr_ln_modulate.restype = _int
lib.nr_gated_residual_ln_modulate.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64,
                                              _f32, _int, _vp]
lib.nr_gated_residual_ln_modulate.restype = _int
lib.nr_silu_and_mul.argtypes = [_vp, _vp, _i64, _i64, _int, _vp]
lib.nr_silu_and_mul.restype = _int
lib.nr_gelu_and_mul.argtypes = [_vp, _vp, _i64, _i64, _int, _vp]
lib.nr_gelu_and_mul.restype = _int
lib.nr_device_status.argtypes = [_vp]
lib.nr_device_status.restype = _int
lib.nr_test_wait_probe.argtypes = [_i64, _vp]
lib.nr_test_wait_probe.restype = _int
lib.nr_status_string.argtypes = [_int]
lib.nr_status_string.restype = ctypes.c_char_p
lib.nr_last_error_message.argtypes = []
lib.nr_last_error_message.restype = ctypes.c_char_p
lib.nr_version.argtypes = []
lib.nr_version.restype = _int

NR_F32 = 0
NR_BF16 = 1
ENTRY_POINTS = ("nr_rmsnorm", "nr_rmsnorm_quant_fp8", "nr_qk_norm_rope", "nr_qk_norm_rope_ex", "nr_ln_modulate",
                "nr_silu_and_mul", "nr_gelu_and_mul", "nr_gated_residual_ln_modulate",
                "nr_device_status", "nr_test_wait_probe",
                "nr_status_string", "nr_last_error_message", "nr_version")


class NrError(RuntimeError):
    """A non-OK nr_status from the library."""

    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (lib.nr_status_string(status).decode(), message))
        self.status = status


def _check(status: int):
    if status != 0:
        raise NrError(status, lib.nr_last_error_message().decode())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return NR_BF16
    if t.dtype == torch.float32:
        return NR_F32
    raise TypeError("tensors are bfloat16 or float32, got %s" % t.dtype)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _cuda(*ts):
    """Every tensor on one CUDA device (checked after the shapes, so that a
    shape error is reported as such whatever the device)."""
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError("tensors must all be on one CUDA device (%s and %s)" % (dev, t.device))


def _expect(t, name, dtype, shape, contiguous=True):
    """Raise unless `t` is a tensor of `dtype` and `shape` (and contiguous).
    The C ABI sees only pointers, so a short or mistyped operand would be read
    or written past its end; this is where the sizes are checked."""
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    if contiguous and not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def _rows_2d(t, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch tensor" % name)
    if t.dim() != 2 or not t.is_contiguous():
        raise ValueError("%s must be a contiguous [rows, hidden] tensor" % name)
    _dtype_code(t)


def _heads_3d(t, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch tensor" % name)
    if t.dim() != 3 or t.stride(2) != 1 or (t.shape[1] > 1 and t.stride(1) != t.shape[2]):
        raise ValueError("%s must be [tokens, heads, head_dim] with contiguous heads" % name)
    _dtype_code(t)


def _samples(t, name, dtype, rows, hidden, rows_per_sample):
    """A modulation operand: [hidden] (one sample) or [samples, hidden], with
    at least one sample per started group of rows_per_sample rows."""
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if t.dim() not in (1, 2) or t.shape[-1] != hidden or not t.is_contiguous():
        raise ValueError("%s must be a contiguous [samples, %d] tensor, got %s"
                         % (name, hidden, tuple(t.shape)))
    need = -(-rows // rows_per_sample) if rows > 0 else 0
    have = 1 if t.dim() == 1 else t.shape[0]
    if have < need:
        raise ValueError("%s has %d sample rows; %d rows at %d rows per sample need %d"
                         % (name, have, rows, rows_per_sample, need))


def _rows_per_sample(rows_per_sample, rows):
    if rows_per_sample is None:
        return max(rows, 1)
    rps = int(rows_per_sample)
    if rps < 1:
        raise ValueError("rows_per_sample must be >= 1")
    return rps


def rmsnorm(x, w, residual=None, eps=1e-6, gemma=False, out=None):
    """RMSNorm of each row of x [rows, hidden]; with `residual`, first
    residual <- round(x + residual) in place.  Returns out."""
    _rows_2d(x, "x")
    _expect(w, "w", x.dtype, (x.shape[1],))
    if residual is not None:
        _expect(residual, "residual", x.dtype, x.shape)
    if out is not None:
        _expect(out, "out", x.dtype, x.shape)
    _cuda(x, w, residual, out)
    if out is None:
        out = torch.empty_like(x)
    _check(lib.nr_rmsnorm(_ptr(out), _ptr(x), _ptr(w), _ptr(residual), x.shape[0], x.shape[1],
                          _dtype_code(x), float(eps), int(bool(gemma)), _stream(x)))
    return out


def rmsnorm_quant_fp8(x, w, scale, residual=None, eps=1e-6, gemma=False, codes=None,
                      out_bf16=False):
    """RMSNorm of x [rows, hidden] (with the optional residual add), rounded to
    bf16, then e4m3 codes of that value * (1/scale).  Returns codes (uint8),
    or (codes, the bf16 values) when out_bf16 is True (or a tensor to fill)."""
    _rows_2d(x, "x")
    _expect(w, "w", x.dtype, (x.shape[1],))
    if residual is not None:
        _expect(residual, "residual", x.dtype, x.shape)
    if codes is not None:
        _expect(codes, "codes", torch.uint8, x.shape)
    nb = None
    if out_bf16 is not True and out_bf16 is not False and out_bf16 is not None:
        nb = out_bf16
        _expect(nb, "out_bf16", torch.bfloat16, x.shape)
    _cuda(x, w, residual, codes, nb)
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if out_bf16 is True:
        nb = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
    _check(lib.nr_rmsnorm_quant_fp8(_ptr(codes), _ptr(nb), _ptr(x), _ptr(w), _ptr(residual),
                                    x.shape[0], x.shape[1], _dtype_code(x), float(eps),
                                    int(bool(gemma)), float(scale), _stream(x)))
    return codes if nb is None else (codes, nb)


def _check_qk(q, k, wq, wk, q_out, k_out):
    """q, k [tokens, heads, head_dim] of one dtype and token count; wq, wk
    [head_dim] of one dtype; outputs with the shapes, dtype and strides of
    their inputs."""
    _heads_3d(q, "q")
    _heads_3d(k, "k")
    if k.dtype != q.dtype:
        raise TypeError("q and k share one dtype")
    if k.shape[0] != q.shape[0] or k.shape[2] != q.shape[2]:
        raise ValueError("q %s and k %s must have the same tokens and head_dim"
                         % (tuple(q.shape), tuple(k.shape)))
    if not isinstance(wq, torch.Tensor) or wq.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("wq must be a float32 or bfloat16 tensor")
    _expect(wq, "wq", wq.dtype, (q.shape[2],))
    if wk is not None or k.shape[1] > 0:  # wk may be None when k has no heads
        _expect(wk, "wk", wq.dtype, (q.shape[2],))
    for o, i, name in ((q_out, q, "q_out"), (k_out, k, "k_out")):
        if o is None:
            continue
        _expect(o, name, i.dtype, i.shape, contiguous=False)
        if o.stride() != i.stride():
            raise ValueError("%s must have the strides of its input" % name)


def qk_norm_rope(q, k, wq, wk, positions, eps=1e-6, theta=10000.0, gemma=False, q_out=None,
                 k_out=None):
    """Per-head RMSNorm + NeoX RoPE of q [tokens, hq, D] and k [tokens, hk, D].
    q and k may be token-strided views (last two axes contiguous); outputs share
    their strides (q_out=q / k_out=k for in place).  Returns (q_out, k_out)."""
    _check_qk(q, k, wq, wk, q_out, k_out)
    _expect(positions, "positions", torch.int32, (q.shape[0],))
    _cuda(q, k, wq, wk, positions, q_out, k_out)
    if q_out is None:
        q_out = torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device)
    if k_out is None:
        k_out = torch.empty_strided(k.shape, k.stride(), dtype=k.dtype, device=k.device)
    _check(lib.nr_qk_norm_rope(_ptr(q_out), _ptr(k_out), _ptr(q), _ptr(k), _ptr(wq), _ptr(wk),
                               _dtype_code(wq), _ptr(positions), q.shape[0], q.shape[1],
                               k.shape[1], q.shape[2], q.stride(0), k.stride(0), float(eps),
                               float(theta), int(bool(gemma)), _dtype_code(q), _stream(q)))
    return q_out, k_out


def qk_norm_rope_ex(q, k, wq, wk, positions, eps=1e-6, gemma=False, rotary_dim=None,
                    interleaved=False, theta=10000.0, llama3=None, mrope_sections=None,
                    mrope_interleaved=False, q_out=None, k_out=None):
    """qk_norm_rope with the RoPE variants: rotary_dim (default head_dim), GPT-J
    interleaved pairs, Llama-3 rescale (llama3 = (factor, low_freq_factor,
    high_freq_factor, original_max_position)) and M-RoPE (positions [3, tokens],
    mrope_sections = (t, h, w)).  Returns (q_out, k_out)."""
    _check_qk(q, k, wq, wk, q_out, k_out)
    _expect(positions, "positions", torch.int32,
            (3, q.shape[0]) if mrope_sections is not None else (q.shape[0],))
    _cuda(q, k, wq, wk, positions, q_out, k_out)
    if q_out is None:
        q_out = torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device)
    if k_out is None:
        k_out = torch.empty_strided(k.shape, k.stride(), dtype=k.dtype, device=k.device)
    cfg = RopeConfig()
    cfg.rotary_dim = 0 if rotary_dim is None else int(rotary_dim)
    cfg.interleaved = int(bool(interleaved))
    cfg.mrope_interleaved = int(bool(mrope_interleaved))
    cfg.theta = float(theta)
    if llama3 is not None:
        (cfg.llama3_factor, cfg.llama3_low_freq_factor, cfg.llama3_high_freq_factor,
         cfg.llama3_original_max_position) = (float(v) for v in llama3)
    if mrope_sections is not None:
        for i, v in enumerate(mrope_sections):
            cfg.mrope_section[i] = int(v)
    _check(lib.nr_qk_norm_rope_ex(_ptr(q_out), _ptr(k_out), _ptr(q), _ptr(k), _ptr(wq), _ptr(wk),
                                  _dtype_code(wq), _ptr(positions), q.shape[0], q.shape[1],
                                  k.shape[1], q.shape[2], q.stride(0), k.stride(0), float(eps),
                                  int(bool(gemma)), ctypes.byref(cfg), _dtype_code(q), _stream(q)))
    return q_out, k_out


def ln_modulate(x, shift, scale, eps=1e-6, rows_per_sample=None, out=None):
    """LayerNorm (no affine) of x [rows, hidden] then * (1 + scale) + shift,
    with shift/scale [samples, hidden] (row r uses sample r // rows_per_sample).
    Returns out."""
    _rows_2d(x, "x")
    rows_per_sample = _rows_per_sample(rows_per_sample, x.shape[0])
    for t, name in ((shift, "shift"), (scale, "scale")):
        _samples(t, name, x.dtype, x.shape[0], x.shape[1], rows_per_sample)
    if out is not None:
        _expect(out, "out", x.dtype, x.shape)
    _cuda(x, shift, scale, out)
    if out is None:
        out = torch.empty_like(x)
    _check(lib.nr_ln_modulate(_ptr(out), _ptr(x), _ptr(shift), _ptr(scale), x.shape[0],
                              x.shape[1], int(rows_per_sample), float(eps), _dtype_code(x),
                              _stream(x)))
    return out


def gated_residual_ln_modulate(residual, y, gate, shift, scale, eps=1e-6, rows_per_sample=None,
                               out=None):
    """residual <- round(residual + gate * y) in place, then LayerNorm (no affine)
    of it * (1 + scale) + shift.  gate/shift/scale are [samples, hidden]; row r
    uses sample r // rows_per_sample.  Returns out."""
    _rows_2d(residual, "residual")
    _expect(y, "y", residual.dtype, residual.shape)
    rows, hidden = residual.shape
    rows_per_sample = _rows_per_sample(rows_per_sample, rows)
    for t, name in ((gate, "gate"), (shift, "shift"), (scale, "scale")):
        _samples(t, name, residual.dtype, rows, hidden, rows_per_sample)
    if out is not None:
        _expect(out, "out", residual.dtype, residual.shape)
    _cuda(residual, y, gate, shift, scale, out)
    if out is None:
        out = torch.empty_like(residual)
    _check(lib.nr_gated_residual_ln_modulate(
        _ptr(out), _ptr(residual), _ptr(y), _ptr(gate), _ptr(shift), _ptr(scale),
        residual.shape[0], residual.shape[1], int(rows_per_sample), float(eps),
        _dtype_code(residual), _stream(residual)))
    return out


def _act_and_mul(fn, x, out):
    _rows_2d(x, "x")
    if x.shape[1] % 2:
        raise ValueError("x must be a contiguous [rows, 2*inter] tensor")
    inter = x.shape[1] // 2
    if out is not None:
        _expect(out, "out", x.dtype, (x.shape[0], inter))
    _cuda(x, out)
    if out is None:
        out = torch.empty((x.shape[0], inter), dtype=x.dtype, device=x.device)
    _check(fn(_ptr(out), _ptr(x), x.shape[0], inter, _dtype_code(x), _stream(x)))
    return out


def device_status(device=None):
    """Wait for the current stream of `device` and raise NrError
    (NR_ERR_TIMEOUT) if a kernel gave up a bounded wait since the last check."""
    _check(lib.nr_device_status(torch.cuda.current_stream(device).cuda_stream))


def wait_probe(limit_cycles=100000, device=None):
    """Launch the library's wait probe: one wait that nothing completes, given
    up after `limit_cycles` SM clock cycles (the next device_status() raises)."""
    _check(lib.nr_test_wait_probe(int(limit_cycles), torch.cuda.current_stream(device).cuda_stream))


def silu_and_mul(x, out=None):
    """silu(x[:, :I]) * x[:, I:] for x [rows, 2I].  Returns out [rows, I]."""
    return _act_and_mul(lib.nr_silu_and_mul, x, out)


def gelu_and_mul(x, out=None):
    """gelu_tanh(x[:, :I]) * x[:, I:] for x [rows, 2I].  Returns out [rows, I]."""
    return _act_and_mul(lib.nr_gelu_and_mul, x, out)


__all__ = ["rmsnorm", "rmsnorm_quant_fp8", "qk_norm_rope", "qk_norm_rope_ex", "RopeConfig", "ln_modulate",
           "silu_and_mul", "gelu_and_mul", "device_status", "wait_probe",
           "gated_residual_ln_modulate", "NrError", "lib",
           "LIB_PATH", "ENTRY_POINTS", "NR_F32", "NR_BF16"]
