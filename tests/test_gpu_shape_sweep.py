"""Seeded sweeps over many sizes, so that every launch configuration the
launchers can pick (vectors per thread, warps per row, the multi-pass
kernels for long rows, the Q/K kernels for each head size, variant and token
block) runs against the oracle.  Few rows each: the point is coverage of the
configuration space, not size."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import Guarded, dev, host_bits
from tests.parity import check_bf16, check_f32

pytestmark = pytest.mark.gpu
RNG = np.random.default_rng(2024)


def _sizes(n, lo, hi, mult):
    """n distinct multiples of `mult` in [lo, hi], log-spread, plus the ends."""
    vals = np.unique((np.exp(RNG.uniform(np.log(lo), np.log(hi), n)) // mult).astype(int) * mult)
    return sorted(set(int(v) for v in vals if lo <= v <= hi) | {lo, hi})


def _check(got, o_out, y=None, mag=None, k=None, dtype=torch.bfloat16, what=""):
    if dtype == torch.bfloat16:
        check_bf16(host_bits(got), o_out, y, mag, k_cancel=k, what=what)
    else:
        check_f32(host_bits(got), y, rel=1e-5, mag=mag, k_cancel=k, what=what)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_rmsnorm_hidden_sweep(nr, dtype):
    mult = 8 if dtype == torch.bfloat16 else 4
    for i, h in enumerate(_sizes(40, mult, 70000, mult)):
        x, res, w = synth.rmsnorm_inputs(3, h, 100 + i, dtype)
        rg = Guarded(res.shape, dtype, fill=res)
        out = nr.rmsnorm(dev(x), dev(w), residual=rg.t, gemma=bool(i % 2))
        torch.cuda.synchronize()
        rg.check()
        o_out, o_res, o_y = oracle.rmsnorm(host_bits(x), host_bits(w), residual=host_bits(res),
                                           gemma=bool(i % 2), want_y=True)
        assert np.array_equal(host_bits(rg.t), o_res), "residual, hidden %d" % h
        _check(out, o_out, o_y, dtype=dtype, what="rmsnorm hidden %d" % h)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_ln_modulate_hidden_sweep(nr, dtype):
    mult = 8 if dtype == torch.bfloat16 else 4
    for i, h in enumerate(_sizes(40, mult, 70000, mult)):
        x, sh, sc = synth.ln_inputs(3, h, 200 + i, dtype)
        out = nr.ln_modulate(dev(x), dev(sh), dev(sc))
        torch.cuda.synchronize()
        o_out, o_y, o_mag = oracle.ln_modulate(host_bits(x), host_bits(sh), host_bits(sc),
                                               want_y=True)
        _check(out, o_out, o_y, o_mag, k=64, dtype=dtype, what="ln hidden %d" % h)


def test_gated_and_quant_hidden_sweep(nr):
    """The gated op up to its limit (hidden 8192 bf16), the FP8 op up to its
    own (32768)."""
    for i, h in enumerate(_sizes(25, 8, 32768, 8)):
        if h > 8192:
            _quant_case(nr, h, i)
            continue
        res = synth.tensor(300 + i, 20, (3, h), torch.bfloat16)
        y = synth.tensor(300 + i, 21, (3, h), torch.bfloat16)
        gate, sh, sc = (synth.tensor(300 + i, j, (1, h), torch.bfloat16, std=0.3)
                        for j in (22, 23, 24))
        rd = dev(res)
        out = nr.gated_residual_ln_modulate(rd, dev(y), dev(gate), dev(sh), dev(sc))
        torch.cuda.synchronize()
        o_out, o_res, o_y, o_mag = oracle.gated_ln_modulate(
            host_bits(res), host_bits(y), host_bits(gate), host_bits(sh), host_bits(sc),
            want_y=True)
        assert np.array_equal(host_bits(rd), o_res), "gated residual, hidden %d" % h
        check_bf16(host_bits(out), o_out, o_y, o_mag, k_cancel=64, what="gated hidden %d" % h)
        _quant_case(nr, h, i)


def _quant_case(nr, h, i):
    x, _, w = synth.rmsnorm_inputs(3, h, 400 + i, torch.bfloat16, residual=False)
    codes, nb = nr.rmsnorm_quant_fp8(dev(x), dev(w), 0.03, out_bf16=True)
    torch.cuda.synchronize()
    o_codes, o_nb, _, _ = oracle.rmsnorm_quant_fp8(host_bits(x), host_bits(w), 0.03)
    check_bf16(host_bits(nb), o_nb, what="quant bf16 hidden %d" % h)
    same = host_bits(nb) == o_nb
    assert np.array_equal(codes.cpu().numpy()[same], o_codes[same]), "codes, hidden %d" % h


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_act_and_mul_sweep(nr, dtype):
    mult = 8 if dtype == torch.bfloat16 else 4
    for i, inter in enumerate(_sizes(25, mult, 100000, mult)):
        rows = 1 + i % 5
        g = synth.silu_inputs(rows, inter, 500 + i, dtype)
        for name, fn, ofn in (("silu", nr.silu_and_mul, oracle.silu_and_mul),
                              ("gelu", nr.gelu_and_mul, oracle.gelu_and_mul)):
            out = fn(dev(g))
            torch.cuda.synchronize()
            o_out, o_y = ofn(host_bits(g), want_y=True)
            _check(out, o_out, o_y, dtype=dtype, what="%s inter %d" % (name, inter))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_qk_shape_sweep(nr, dtype):
    """Head sizes from 2 to 32 lanes, MHA and GQA head counts, token counts
    from 1 to a few thousand, the plain rotation and each variant."""
    dims = [16, 32, 64, 128, 256, 512] if dtype == torch.bfloat16 else [8, 16, 32, 64, 128, 256]
    variants = [dict(), dict(rotary_dim="half"), dict(interleaved=True),
                dict(rotary_dim="half", interleaved=True), dict(mrope=True)]
    case = 0
    for D in dims:
        for var in variants:
            T = int(RNG.choice([1, 3, 17, 160, 1200, 3001]))
            hq = int(RNG.choice([1, 2, 5, 8, 16, 24]))
            hk = int(RNG.choice([0, 1, 2, hq]))
            q, k, wq, wk, pos = synth.qk_inputs(T, hq, hk, D, 600 + case, dtype, torch.float32)
            case += 1
            kw = {}
            if var.get("rotary_dim"):
                kw["rotary_dim"] = D // 2 if (D // 2) % (16 if dtype == torch.bfloat16 else 8) == 0 \
                    else D
            if var.get("interleaved"):
                kw["interleaved"] = True
            if var.get("mrope"):
                half = D // 2
                kw["mrope_sections"] = (half - 2 * (half // 3), half // 3, half // 3)
                pos = torch.stack([pos, pos // 3, pos // 7]).to(torch.int32).contiguous()
            qo, ko = nr.qk_norm_rope_ex(dev(q), dev(k), dev(wq), dev(wk), dev(pos), **kw)
            torch.cuda.synchronize()
            ref = oracle.qk_norm_rope_ex(host_bits(q), host_bits(k), host_bits(wq), host_bits(wk),
                                         pos.numpy(), want_y=True, **kw)
            what = "qk D %d T %d hq %d hk %d %s" % (D, T, hq, hk, kw)
            _check(qo, ref[0], ref[2], ref[4], k=32, dtype=dtype, what=what + " q")
            if hk:
                _check(ko, ref[1], ref[3], ref[5], k=32, dtype=dtype, what=what + " k")
