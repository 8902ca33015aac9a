"""Host-side checks of the C ABI, no GPU needed: the library loads, exports
every entry point include/nr.h declares, and rejects bad arguments with the
documented status before anything is launched.  Pointers below are fake
addresses: every call here fails validation (or has zero rows) and returns
before any CUDA call, so none is ever dereferenced."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nr.h")

OK, NULL, SHAPE, DTYPE, ALIGN, ALIAS, UNSUP, CUDA, VALUE, TIMEOUT = range(10)
F32, BF16 = 0, 1
A = 0x7F0000000000  # fake, 16-byte aligned "device" addresses
MB = 1 << 20


class RopeConfig(ctypes.Structure):
    _fields_ = [("rotary_dim", ctypes.c_int64), ("interleaved", ctypes.c_int32),
                ("mrope_interleaved", ctypes.c_int32), ("theta", ctypes.c_double),
                ("llama3_factor", ctypes.c_double), ("llama3_low_freq_factor", ctypes.c_double),
                ("llama3_high_freq_factor", ctypes.c_double),
                ("llama3_original_max_position", ctypes.c_double),
                ("mrope_section", ctypes.c_int32 * 3)]


@pytest.fixture(scope="module")
def lib(lib_path):
    L = ctypes.CDLL(lib_path)
    vp, i64, f32, f64, cint = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_double,
                               ctypes.c_int)
    L.nr_rmsnorm.argtypes = [vp, vp, vp, vp, i64, i64, cint, f32, cint, vp]
    L.nr_qk_norm_rope.argtypes = [vp, vp, vp, vp, vp, vp, cint, vp, i64, i64, i64, i64, i64, i64,
                                  f32, f64, cint, cint, vp]
    L.nr_ln_modulate.argtypes = [vp, vp, vp, vp, i64, i64, i64, f32, cint, vp]
    L.nr_silu_and_mul.argtypes = [vp, vp, i64, i64, cint, vp]
    L.nr_gelu_and_mul.argtypes = [vp, vp, i64, i64, cint, vp]
    L.nr_rmsnorm_quant_fp8.argtypes = [vp, vp, vp, vp, vp, i64, i64, cint, f32, cint, f32, vp]
    L.nr_qk_norm_rope_ex.argtypes = [vp, vp, vp, vp, vp, vp, cint, vp, i64, i64, i64, i64, i64,
                                     i64, f32, cint, ctypes.POINTER(RopeConfig), cint, vp]
    L.nr_gated_residual_ln_modulate.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, f32, cint,
                                                vp]
    L.nr_test_wait_probe.argtypes = [i64, vp]
    L.nr_device_status.argtypes = [vp]
    L.nr_status_string.argtypes = [cint]
    L.nr_status_string.restype = ctypes.c_char_p
    L.nr_last_error_message.restype = ctypes.c_char_p
    return L


def declared_entry_points():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:nr_status|const char\*|int)\s+(nr_\w+)\s*\(", text, re.M)))


def test_header_declares_the_four_ops():
    names = declared_entry_points()
    for n in ("nr_rmsnorm", "nr_qk_norm_rope", "nr_ln_modulate", "nr_silu_and_mul",
              "nr_status_string", "nr_last_error_message", "nr_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_entry_points():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    assert lib.nr_status_string(OK) == b"NR_OK"
    assert lib.nr_status_string(ALIAS) == b"NR_ERR_ALIAS"
    assert lib.nr_status_string(TIMEOUT) == b"NR_ERR_TIMEOUT"
    assert lib.nr_status_string(99) == b"NR_ERR_UNKNOWN"
    assert lib.nr_version() >= 100


def rms(lib, out=A, x=A + 64 * MB, w=A + 128 * MB, res=None, rows=4, hidden=64, dtype=BF16,
        eps=1e-6, gemma=0):
    return lib.nr_rmsnorm(out, x, w, res, rows, hidden, dtype, eps, gemma, None)


def test_rmsnorm_validation(lib):
    assert rms(lib, rows=0, out=None, x=None, w=None) == OK  # zero rows: no launch
    assert rms(lib, dtype=7) == DTYPE
    assert rms(lib, rows=-1) == SHAPE
    assert rms(lib, hidden=0) == SHAPE
    assert rms(lib, x=None) == NULL
    assert rms(lib, w=None) == NULL
    assert rms(lib, hidden=12) == UNSUP  # bf16 needs hidden % 8 == 0
    assert rms(lib, hidden=12, dtype=F32, x=A + 2) == ALIGN  # f32 % 4 ok, x misaligned
    assert rms(lib, out=A + 8) == ALIGN
    assert rms(lib, eps=-1.0) == VALUE
    assert rms(lib, eps=float("nan")) == VALUE
    assert rms(lib, gemma=2) == VALUE
    assert rms(lib, out=A, x=A + 16) == ALIAS  # partial overlap of out and x
    assert rms(lib, res=A + 64 * MB) == ALIAS  # residual is x
    assert rms(lib, res=A) == ALIAS  # residual is out
    assert rms(lib, w=A + 32) == ALIAS  # w inside out


def test_rmsnorm_error_message_names_the_problem(lib):
    assert rms(lib, hidden=12) == UNSUP
    assert b"multiple of 8" in lib.nr_last_error_message()


def qk(lib, q_out=A, k_out=A + 64 * MB, q=A + 128 * MB, k=A + 192 * MB, wq=A + 256 * MB,
       wk=A + 257 * MB, w_dtype=F32, pos=A + 258 * MB, tokens=8, hq=4, hk=2, D=128, qs=None,
       ks=None, eps=1e-6, theta=1e4, gemma=0, dtype=BF16):
    qs = hq * D if qs is None else qs
    ks = hk * D if ks is None else ks
    return lib.nr_qk_norm_rope(q_out, k_out, q, k, wq, wk, w_dtype, pos, tokens, hq, hk, D, qs, ks,
                               eps, theta, gemma, dtype, None)


def test_qk_norm_rope_validation(lib):
    assert qk(lib, tokens=0, q_out=None, q=None, wq=None, pos=None) == OK
    assert qk(lib, dtype=5) == DTYPE
    assert qk(lib, w_dtype=5) == DTYPE
    assert qk(lib, hq=0) == SHAPE
    assert qk(lib, hk=-1) == SHAPE
    assert qk(lib, D=127) == SHAPE
    assert qk(lib, D=96) == UNSUP  # 96/16 = 6 lanes: not a power of two
    assert qk(lib, D=1024) == UNSUP
    assert qk(lib, D=8) == UNSUP  # bf16 needs >= 16
    assert qk(lib, theta=0.0) == VALUE
    assert qk(lib, theta=float("inf")) == VALUE
    assert qk(lib, eps=-1e-6) == VALUE
    assert qk(lib, qs=4 * 128 - 8) == SHAPE  # stride below heads * D
    assert qk(lib, q=None) == NULL
    assert qk(lib, pos=None) == NULL
    assert qk(lib, wk=None) == NULL
    assert qk(lib, hk=0, k=None, k_out=None, wk=None, ks=0) != NULL  # k optional when hk == 0
    assert qk(lib, qs=4 * 128 + 4) == ALIGN  # 8-byte token stride remainder
    assert qk(lib, q=A + 128 * MB + 8) == ALIGN
    assert qk(lib, pos=A + 258 * MB + 2) == ALIGN
    assert qk(lib, q_out=A + 192 * MB) == ALIAS  # q_out is k
    assert qk(lib, k_out=A) == ALIAS  # k_out is q_out
    assert qk(lib, q_out=A + 256 * MB) == ALIAS  # q_out over the weights


def ln(lib, out=A, x=A + 64 * MB, shift=A + 128 * MB, scale=A + 129 * MB, rows=4, hidden=64,
       rps=4, eps=1e-6, dtype=BF16):
    return lib.nr_ln_modulate(out, x, shift, scale, rows, hidden, rps, eps, dtype, None)


def test_ln_modulate_validation(lib):
    assert ln(lib, rows=0, out=None, x=None, shift=None, scale=None) == OK
    assert ln(lib, dtype=3) == DTYPE
    assert ln(lib, rps=0) == SHAPE
    assert ln(lib, hidden=-8) == SHAPE
    assert ln(lib, shift=None) == NULL
    assert ln(lib, hidden=20) == UNSUP
    assert ln(lib, scale=A + 129 * MB + 4) == ALIGN
    assert ln(lib, eps=float("inf")) == VALUE
    assert ln(lib, out=A + 64 * MB + 16) == ALIAS
    assert ln(lib, shift=A + 16) == ALIAS


@pytest.mark.parametrize("name", ["nr_silu_and_mul", "nr_gelu_and_mul"])
def test_act_and_mul_validation(lib, name):
    fn = getattr(lib, name)
    assert fn(None, None, 0, 64, BF16, None) == OK
    assert fn(A, A + MB, 4, 64, 9, None) == DTYPE
    assert fn(A, A + MB, -1, 64, BF16, None) == SHAPE
    assert fn(A, A + MB, 4, 0, BF16, None) == SHAPE
    assert fn(None, A + MB, 4, 64, BF16, None) == NULL
    assert fn(A, A + MB, 4, 60, BF16, None) == UNSUP
    assert fn(A + 4, A + MB, 4, 64, F32, None) == ALIGN
    assert fn(A, A + 256, 4, 64, BF16, None) == ALIAS  # out inside x
    assert name.encode() in lib.nr_last_error_message()


def gated(lib, out=A, res=A + 64 * MB, y=A + 128 * MB, gate=A + 192 * MB, shift=A + 193 * MB,
          scale=A + 194 * MB, rows=4, hidden=64, rps=4, eps=1e-6, dtype=BF16):
    return lib.nr_gated_residual_ln_modulate(out, res, y, gate, shift, scale, rows, hidden, rps,
                                             eps, dtype, None)


def test_gated_residual_ln_modulate_validation(lib):
    assert gated(lib, rows=0, out=None, res=None, y=None, gate=None, shift=None, scale=None) == OK
    assert gated(lib, dtype=4) == DTYPE
    assert gated(lib, rps=0) == SHAPE
    assert gated(lib, gate=None) == NULL
    assert gated(lib, hidden=20) == UNSUP
    assert gated(lib, hidden=8200) == UNSUP  # above 8192 for bf16
    assert gated(lib, hidden=4100, dtype=F32) == UNSUP  # above 4096 for f32
    assert gated(lib, y=A + 128 * MB + 8) == ALIGN
    assert gated(lib, eps=-0.5) == VALUE
    assert gated(lib, out=A + 64 * MB) == ALIAS  # out is the residual
    assert gated(lib, y=A + 64 * MB) == ALIAS  # y is the residual
    assert gated(lib, shift=A + 16) == ALIAS  # shift inside out


def qk_ex(lib, cfg=None, D=128, dtype=BF16, tokens=8, **over):
    if cfg is None:
        cfg = RopeConfig()
        cfg.theta = 1e4
    for k_, v in over.items():
        if k_ == "sections":
            for i, x in enumerate(v):
                cfg.mrope_section[i] = x
        else:
            setattr(cfg, k_, v)
    return lib.nr_qk_norm_rope_ex(A, A + 64 * MB, A + 128 * MB, A + 192 * MB, A + 256 * MB,
                                  A + 257 * MB, F32, A + 258 * MB, tokens, 4, 2, D, 4 * D, 2 * D,
                                  1e-6, 0, ctypes.byref(cfg), dtype, None)


def test_qk_norm_rope_ex_validation(lib):
    assert lib.nr_qk_norm_rope_ex(A, A, A, A, A, A, F32, A, 8, 4, 2, 128, 512, 256, 1e-6, 0,
                                  None, BF16, None) == NULL
    assert qk_ex(lib, tokens=0) == OK
    assert qk_ex(lib, rotary_dim=130) == SHAPE  # above head_dim
    assert qk_ex(lib, rotary_dim=63) == SHAPE  # odd
    assert qk_ex(lib, rotary_dim=40) == UNSUP  # rotate-half needs multiples of 16 (bf16)
    assert qk_ex(lib, rotary_dim=40, interleaved=1, sections=(0, 0, 0), theta=0.0) == VALUE
    assert qk_ex(lib, interleaved=2) == VALUE
    assert qk_ex(lib, llama3_factor=8.0) == VALUE  # factors missing
    assert qk_ex(lib, llama3_factor=8.0, llama3_low_freq_factor=4.0, llama3_high_freq_factor=1.0,
                 llama3_original_max_position=8192.0) == VALUE  # high < low
    assert qk_ex(lib, sections=(16, 24, 23)) == SHAPE  # sum != 64
    assert qk_ex(lib, sections=(-1, 33, 32)) == SHAPE


def quant(lib, codes=A, nb=A + 64 * MB, x=A + 128 * MB, w=A + 192 * MB, res=None, rows=4,
          hidden=64, dtype=BF16, eps=1e-6, gemma=0, scale=0.5):
    return lib.nr_rmsnorm_quant_fp8(codes, nb, x, w, res, rows, hidden, dtype, eps, gemma, scale,
                                    None)


def test_rmsnorm_quant_fp8_validation(lib):
    assert quant(lib, rows=0, codes=None, x=None, w=None) == OK
    assert quant(lib, dtype=2) == DTYPE
    assert quant(lib, scale=0.0) == VALUE
    assert quant(lib, scale=float("inf")) == VALUE
    assert quant(lib, scale=1e-40) == VALUE  # reciprocal overflows
    assert quant(lib, codes=None) == NULL
    assert quant(lib, hidden=12) == UNSUP
    assert quant(lib, hidden=32776) == UNSUP  # beyond 32768 for bf16
    assert quant(lib, codes=A + 8) == ALIGN
    assert quant(lib, codes=A + 128 * MB) == ALIAS  # codes over x
    assert quant(lib, nb=A) == ALIAS  # the two outputs
    assert quant(lib, res=A + 128 * MB) == ALIAS  # residual is x


def test_wait_probe_limit_is_validated_before_launch(lib):
    """Out-of-range limits are refused on the host (nothing is launched)."""
    assert lib.nr_test_wait_probe(0, None) == VALUE
    assert lib.nr_test_wait_probe(-5, None) == VALUE
    assert lib.nr_test_wait_probe((1 << 32) + 1, None) == VALUE
    assert b"limit_cycles" in lib.nr_last_error_message()
