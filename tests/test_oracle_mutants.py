"""The pins must catch plausible slips in the oracle.

Each case below plants one mistake in a copy of oracle.c (a dropped term, a
wrong sign, index or divisor, a misplaced eps, a missing rounding), compiles it
on the CPU, points the oracle module at the mutant and runs every pin in
test_oracle_pins.py.  At least one pin must fail for every mutant; the real
oracle is restored afterwards.

Rounding the residual sum to f32 before bf16 is deliberately absent: for two
bf16 operands it is an equivalent program (f32 keeps at least 2*8+2 bits, so
the second rounding cannot move), which is also why the GPU's f32 add is exact
against the oracle's single rounding.
"""
import ctypes
import inspect
import os

import numpy as np

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text in oracle.c, replacement)
MUTANTS = [
    ("bf16 ties away from zero", "nearbyint(scaled)", "floor(scaled + 0.5)"),
    ("bf16 truncation", "nearbyint(scaled)", "trunc(scaled)"),
    ("bf16 wrong significand width", "(e - 1) - 7", "(e - 1) - 8"),
    ("eps outside the sqrt", "1.0 / sqrt(ms + eps)", "1.0 / (sqrt(ms) + eps)"),
    ("mean over h-1", "sum_sq / (double)hidden", "sum_sq / (double)(hidden - 1)"),
    ("gemma dropped", "if (gemma) wj += 1.0;\n      const double yj",
     "if (gemma) wj += 0.0;\n      const double yj"),
    ("residual not rounded before squaring",
     "v = round_to(dtype, v + load(dtype, res_in, base + j));",
     "store(dtype, res_out, base + j, v + load(dtype, res_in, base + j)); v = v + load(dtype, res_in, base + j);"),
    ("output stored via f32 (double rounding)", "((uint16_t*)p)[i] = nro_bf16_round(v);",
     "((uint16_t*)p)[i] = nro_bf16_round((float)v);"),
    ("rope rotates the other way", "const double first = n[i] * c - n[i + half] * s;\n        const double second = n[i] * s + n[i + half] * c;",
     "const double first = n[i] * c + n[i + half] * s;\n        const double second = -n[i] * s + n[i + half] * c;"),
    ("rope sign slip in one half", "const double second = n[i] * s + n[i + half] * c;",
     "const double second = n[i] * s - n[i + half] * c;"),
    ("rope interleaved pairing", "n[i + half]", "n[(2 * i + 1) % D]"),
    ("rope frequency exponent -i/D", "-2.0 * (double)i / (double)D", "-(double)i / (double)D"),
    ("rope position off by one", "(double)pos[t] * freq", "(double)(pos[t] + 1) * freq"),
    ("rope weight reversed", "double wj = load(w_dtype, w, j);", "double wj = load(w_dtype, w, D - 1 - j);"),
    ("rope head norm over D-1", "sum_sq / (double)D + eps", "sum_sq / (double)(D - 1) + eps"),
    ("rope head stride", "const int64_t base = t * tok_stride + h * D;",
     "const int64_t base = t * tok_stride + h * half;"),
    ("ln unbiased variance", "sum_dev / (double)hidden", "sum_dev / (double)(hidden - 1)"),
    ("ln scale without the 1", "const double g = 1.0 + load(dtype, scale, sample + j);",
     "const double g = load(dtype, scale, sample + j);"),
    ("ln shift sign", "const double yj = xhat * g + sh;", "const double yj = xhat * g - sh;"),
    ("ln sample index", "(r / rows_per_sample) * hidden", "(r % rows_per_sample) * hidden"),
    ("ln eps outside the sqrt", "1.0 / sqrt(var + eps)", "1.0 / (sqrt(var) + eps)"),
    ("gated: gate ignored", "load(dtype, gate, sample + j) * load(dtype, y, r * hidden + j)",
     "load(dtype, y, r * hidden + j)"),
    ("gated: gate on the residual",
     "const double gy = load(dtype, gate, sample + j) * load(dtype, y, r * hidden + j);\n      const double v = sum_round_to_odd(load(dtype, residual, r * hidden + j), gy);",
     "const double gy = load(dtype, gate, sample + j) * load(dtype, residual, r * hidden + j);\n      const double v = sum_round_to_odd(load(dtype, y, r * hidden + j), gy);"),
    ("gated: sum rounded to nearest double, then to the dtype",
     "const double v = sum_round_to_odd(load(dtype, residual, r * hidden + j), gy);",
     "const double v = load(dtype, residual, r * hidden + j) + gy;"),
    ("gated: round to odd keeps the even neighbour", "return (bits & 1u) ? s : other;",
     "return (bits & 1u) ? other : s;"),
    ("gated: sample index", "const int64_t sample = (r / rows_per_sample) * hidden;\n    for (int64_t j = 0; j < hidden; j++) {\n      /* gate",
     "const int64_t sample = (r % rows_per_sample) * hidden;\n    for (int64_t j = 0; j < hidden; j++) {\n      /* gate"),
    ("rope-ex: head stride", "const int64_t row0 = t * tok_stride + h * D;",
     "const int64_t row0 = t * tok_stride + h * (D - 2);"),
    ("rope-ex: frequency over D, not rot", "pow(theta, -2.0 * (double)i / (double)rot)",
     "pow(theta, -2.0 * (double)i / (double)D)"),
    ("rope-ex: interleaved pairs (i, i+1)", "const int64_t a = interleaved ? 2 * i : i;",
     "const int64_t a = interleaved ? i : i;"),
    ("rope-ex: llama3 regions swapped", "if (wavelength > orig / low) return f / factor;",
     "if (wavelength > orig / low) return f;"),
    ("rope-ex: mrope interleaved off by one", "if (i % 3 == 1 && i / 3 < sections[1]) return 1;",
     "if (i % 3 == 1 && i / 3 <= sections[1]) return 1;"),
    ("rope-ex: mrope contiguous sections", "if (i < sections[0] + sections[1]) return 1;",
     "if (i < sections[1]) return 1;"),
    ("e4m3 exponent bias 8", "const int exp_field = (e - 1) + 7;", "const int exp_field = (e - 1) + 8;"),
    ("e4m3 no saturation", "if (r > 448.0) r = 448.0;", "if (r > 480.0) r = 448.0;"),
    ("e4m3 ties away", "double r = ldexp(nearbyint(ldexp(a, -quantum_exp)), quantum_exp);",
     "double r = ldexp(floor(ldexp(a, -quantum_exp) + 0.5), quantum_exp);"),
    ("fp8 code from the unrounded value", "const float t = (float)nro_bf16_value(nb) * inv_scale;",
     "const float t = (float)yj * inv_scale;"),
    ("fp8 scale applied the wrong way", "const float inv_scale = 1.0f / scale;",
     "const float inv_scale = scale;"),
    ("gelu cubic coefficient", "0.044715 * a * a * a", "0.044715 * a * a"),
    ("gelu missing half", "const double yj = 0.5 * a * one_plus_tanh * b;",
     "const double yj = a * one_plus_tanh * b;"),
    ("gelu 1 + tanh by direct sum", "z >= 0 ? 1.0 + tanh(z) :", "1 ? 1.0 + tanh(z) :"),
    ("gelu negative branch exponent", "2.0 * exp(2 * z) / (1.0 + exp(2 * z))",
     "2.0 * exp(z) / (1.0 + exp(2 * z))"),
    ("bf16 subnormal grid one step too fine", "if (quantum_exp < -133) quantum_exp = -133;",
     "if (quantum_exp < -134) quantum_exp = -134;"),
    ("rope-ex: llama3 blend weights swapped", "return (1.0 - s) * f / factor + s * f;",
     "return s * f / factor + (1.0 - s) * f;"),
    ("rope-ex: llama3 high-frequency bound uses low", "if (wavelength < orig / high) return f;",
     "if (wavelength < orig / low) return f;"),
    ("rope-ex: pass-through part not normed", "store(dtype, dst, row0 + j, n[j]);",
     "store(dtype, dst, row0 + j, load(dtype, src, row0 + j));"),
    ("rope-ex: partner at D/2 instead of rot/2", "const int64_t b = interleaved ? 2 * i + 1 : i + rot / 2;",
     "const int64_t b = interleaved ? 2 * i + 1 : i + D / 2;"),
    ("rope-ex: mrope positions read token-major", "(double)pos[axis * tokens + t]",
     "(double)pos[axis + 3 * t]"),
    ("rope-ex: mrope interleaved w axis test", "if (i % 3 == 2 && i / 3 < sections[2]) return 2;",
     "if (i % 3 == 2 && i / 3 < sections[1]) return 2;"),
    ("rope position through f32", "const double angle = (double)pos[t] * freq;",
     "const double angle = (double)(float)pos[t] * (double)(float)freq;"),
    ("e4m3 subnormal step 2^-10", "return (uint8_t)(sign | (uint8_t)ldexp(r, 9));",
     "return (uint8_t)(sign | (uint8_t)ldexp(r, 10));"),
    ("e4m3 sign dropped", "const uint8_t sign = signbit(f) ? (uint8_t)0x80 : (uint8_t)0;",
     "const uint8_t sign = 0;"),
    ("fp8: gemma ignored in the quantised norm", "if (gemma) wj += 1.0;\n      const double yj = v * inv * wj;\n      const uint16_t nb",
     "if (gemma) wj += 0.0;\n      const double yj = v * inv * wj;\n      const uint16_t nb"),
    ("rope: gemma ignored", "if (gemma) wj += 1.0;\n        n[j] = load(dtype, src, base + j) * inv * wj;",
     "if (gemma) wj += 0.0;\n        n[j] = load(dtype, src, base + j) * inv * wj;"),
    ("rope-ex: gemma ignored", "if (gemma) wj += 1.0;\n        n[j] = load(dtype, src, row0 + j) * inv * wj;",
     "if (gemma) wj += 0.0;\n        n[j] = load(dtype, src, row0 + j) * inv * wj;"),
    ("silu: up dropped", "const double yj = a / (1.0 + exp(-a)) * b;", "const double yj = a / (1.0 + exp(-a));"),
    ("gelu: up dropped", "const double yj = 0.5 * a * one_plus_tanh * b;",
     "const double yj = 0.5 * a * one_plus_tanh;"),
    ("ln: mean over hidden - 1", "const double mu = sum / (double)hidden;",
     "const double mu = sum / (double)(hidden - 1);"),
    ("gated: LayerNorm of the old residual", "nro_ln_modulate(dtype, rows, hidden, rows_per_sample, res_out,",
     "nro_ln_modulate(dtype, rows, hidden, rows_per_sample, residual,"),
    ("fp8: residual not rounded before squaring",
     "if (res_in != NULL) {\n        v = round_to(dtype, v + load(dtype, res_in, base + j));",
     "if (res_in != NULL) {\n        store(dtype, res_out, base + j, v + load(dtype, res_in, base + j)); v = v + load(dtype, res_in, base + j);"),
    ("fp8: eps outside the sqrt", "const double inv = 1.0 / sqrt(sum_sq / (double)hidden + eps);",
     "const double inv = 1.0 / (sqrt(sum_sq / (double)hidden) + eps);"),
    ("fp8: mean over h-1", "const double inv = 1.0 / sqrt(sum_sq / (double)hidden + eps);",
     "const double inv = 1.0 / sqrt(sum_sq / (double)(hidden - 1) + eps);"),
    ("silu exponent sign", "a / (1.0 + exp(-a)) * b", "a / (1.0 + exp(a)) * b"),
    ("silu gate and up swapped", "const double a = load(dtype, x, r * 2 * inter + j);\n      const double b = load(dtype, x, r * 2 * inter + inter + j);",
     "const double b = load(dtype, x, r * 2 * inter + j);\n      const double a = load(dtype, x, r * 2 * inter + inter + j);"),
]


def _pin_calls():
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if marks:
            argname, values = marks[0].args[0], marks[0].args[1]
            for v in values:
                calls.append((name, fn, {argname: v}))
        else:
            calls.append((name, fn, {}))
    return calls


def _caught(lib) -> list:
    saved = oracle._lib
    oracle._lib = lib
    failed = []
    try:
        # a mutant's garbage may overflow inside a pin's arithmetic: that pin fails anyway
        with np.errstate(all="ignore"):
            for name, fn, kw in _pin_calls():
                try:
                    fn(**kw)
                except (AssertionError, ValueError):
                    failed.append(name)
    finally:
        oracle._lib = saved
    return failed


def test_real_oracle_passes_all_pins():
    assert _caught(oracle._load()) == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation anchor not found: %r" % old
    mutated = src.replace(old, new, 1)  # the first occurrence only
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    lib_path = oracle.compile_source(str(path), str(tmp_path / "libmutant.so"))
    lib = oracle.configure(ctypes.CDLL(lib_path))
    failed = _caught(lib)
    assert failed, "no pin caught the mutant '%s'" % name
