"""GPU parity: nr_gated_residual_ln_modulate against the oracle.

residual <- round(residual + gate * y) must be bit-exact (one rounding of the
exact value); out follows the LayerNorm + modulation rule of
test_gpu_ln_modulate.py (1 bf16 ulp, or the cancellation allowance K = 64).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import parity
from tests.gpu_util import Guarded, dev, host_bits
from tests.parity import check_bf16, check_f32

pytestmark = pytest.mark.gpu
K_LN = 64


def gated_inputs(rows, hidden, seed, samples=1, dtype=torch.bfloat16):
    res = synth.tensor(seed, 20, (rows, hidden), dtype)
    y = synth.tensor(seed, 21, (rows, hidden), dtype)
    gate = synth.tensor(seed, 22, (samples, hidden), dtype, std=0.5)
    shift = synth.tensor(seed, 23, (samples, hidden), dtype, std=0.1)
    scale = synth.tensor(seed, 24, (samples, hidden), dtype, std=0.1)
    return res, y, gate, shift, scale


def run_case(nr, res, y, gate, shift, scale, rps=None, chunk=None, eps=1e-6):
    rows, hidden = res.shape
    dtype = res.dtype
    rps = rows if rps is None else rps
    rg = Guarded(res.shape, dtype, fill=res)
    og = Guarded(res.shape, dtype)
    nr.gated_residual_ln_modulate(rg.t, dev(y), dev(gate), dev(shift), dev(scale), eps=eps,
                                  rows_per_sample=rps, out=og.t)
    torch.cuda.synchronize()
    rg.check()
    og.check()
    got_res, got_out = rg.t.cpu(), og.t.cpu()
    chunk = rows if chunk is None else chunk
    for r0 in range(0, rows, chunk):
        r1 = min(r0 + chunk, rows)
        s_idx = np.arange(r0, r1) // rps
        o_out, o_res, o_y, o_mag = oracle.gated_ln_modulate(
            host_bits(res[r0:r1]), host_bits(y[r0:r1]), host_bits(gate[s_idx]),
            host_bits(shift[s_idx]), host_bits(scale[s_idx]), eps=eps, rows_per_sample=1,
            want_y=True)
        assert np.array_equal(host_bits(got_res[r0:r1]), o_res), "residual not bit-exact"
        if dtype == torch.bfloat16:
            check_bf16(host_bits(got_out[r0:r1]), o_out, o_y, o_mag, k_cancel=K_LN,
                       what="gated ln rows %d.." % r0)
        else:
            check_f32(host_bits(got_out[r0:r1]), o_y, rel=1e-5, mag=o_mag, k_cancel=K_LN,
                      what="gated ln")


def test_dit_shape_26598x3072(nr):
    with parity.recording("gated residual + ln_modulate bf16 [26598, 3072]"):
        run_case(nr, *gated_inputs(26598, 3072, 5), chunk=4096)


def test_per_token_and_per_sample_modulation(nr):
    run_case(nr, *gated_inputs(12, 1024, 6, samples=12), rps=1)
    run_case(nr, *gated_inputs(12, 1024, 7, samples=3), rps=4)


@pytest.mark.parametrize("dtype,hidden", [(torch.bfloat16, h) for h in (8, 24, 1000, 3072, 5120,
                                                                         8192)]
                         + [(torch.float32, h) for h in (4, 12, 1000, 4096)])
def test_edge_hidden_sizes(nr, dtype, hidden):
    run_case(nr, *gated_inputs(5, hidden, hidden % 83, dtype=dtype))


def test_residual_rounds_the_exact_value_at_f32_midpoints(nr):
    """Cases where the f32 sum of g*y and r lands exactly on a bf16 midpoint
    while the exact value does not: g*y is itself a bf16 midpoint (an exact
    product of two bf16 values) and r is a tiny value of either sign, so f32
    rounds the sum onto the midpoint and ties-to-even would pick the wrong
    neighbour for one sign.  E.g. 1.75 * 37/64 = 1 + 3 * 2^-8."""
    hidden = 64
    gs, ys, rs = [], [], []
    rng = np.random.default_rng(9)
    while len(gs) < hidden:
        g = float(torch.tensor(rng.uniform(1, 2)).to(torch.bfloat16))
        y = float(torch.tensor(rng.uniform(0.5, 1)).to(torch.bfloat16))
        p = g * y  # exact in double
        b = torch.tensor([p], dtype=torch.float32).view(torch.int32).item()
        if (b & 0xFFFF) != 0x8000 or float(np.float32(p)) != p:
            continue  # want products that are exact bf16 midpoints
        for sign in (1.0, -1.0):
            gs.append(g)
            ys.append(y)
            rs.append(sign * 2.0 ** -25)
    gs, ys, rs = gs[:hidden], ys[:hidden], rs[:hidden]
    gate = torch.tensor([gs], dtype=torch.float32).to(torch.bfloat16)
    y = torch.tensor([ys], dtype=torch.float32).to(torch.bfloat16)
    res = torch.tensor([rs], dtype=torch.float32).to(torch.bfloat16)
    zero = torch.zeros(1, hidden, dtype=torch.bfloat16)
    # check the construction: f32 evaluation then RNE differs from the exact rounding
    f32_path = (gate.float() * y.float() + res.float()).to(torch.bfloat16)
    _, o_res, _, _ = oracle.gated_ln_modulate(host_bits(res), host_bits(y), host_bits(gate),
                                              host_bits(zero), host_bits(zero))
    assert (host_bits(f32_path) != o_res).sum() >= hidden // 4
    run_case(nr, res, y, gate, zero, zero)


def test_f32_residual_rounds_the_exact_value_near_f32_midpoints(nr):
    """f32 cases whose exact r + g*y sits 2^(e-70) j^2 away from an f32
    midpoint: r = m 2^e with m odd, g = 1 - j 2^-23, y = +-2^(e-24)(1 + j 2^-23),
    so g*y = +-(half an ulp of r)(1 - j^2 2^-46).  The sum rounded to double
    lands on the midpoint and ties to even, picking the wrong neighbour; the one
    rounding of the exact value keeps r.  Both signs of r and of y."""
    hidden = 256
    rng = np.random.default_rng(10)
    e = rng.integers(-20, 20, hidden)
    m = (2 ** 23 + 2 * rng.integers(0, 2 ** 22 - 1, hidden) + 1).astype(np.float64)  # odd
    r = np.ldexp(m, e - 23) * np.where(rng.random(hidden) < 0.5, -1.0, 1.0)
    j = rng.integers(1, 64, hidden).astype(np.float64)
    g = 1 - j * 2.0 ** -23
    y = np.ldexp(1 + j * 2.0 ** -23, e - 24) * np.where(rng.random(hidden) < 0.5, -1.0, 1.0)
    # m in (2^23, 2^24) keeps r +- half an ulp inside r's binade; all values are f32-exact
    r, g, y = (torch.from_numpy(a[None]).float() for a in (r, g, y))
    zero = torch.zeros(1, hidden, dtype=torch.float32)
    naive = (r.double() + g.double() * y.double()).float()
    _, o_res, _, _ = oracle.gated_ln_modulate(host_bits(r), host_bits(y), host_bits(g),
                                              host_bits(zero), host_bits(zero))
    assert (host_bits(naive) != o_res).sum() >= hidden // 4  # the construction bites
    assert np.array_equal(o_res, host_bits(r))  # exact value rounds back to r
    run_case(nr, r, y, g, zero, zero)


def test_zero_rows_is_a_no_op(nr):
    z = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    p = torch.zeros(1, 64, dtype=torch.bfloat16, device="cuda")
    assert nr.gated_residual_ln_modulate(z, z.clone(), p, p, p).shape == (0, 64)


def test_bf16_subnormal_operands_and_products(nr):
    """Gate and y down in the bf16 subnormal range and products that land
    there (r = 0 then keeps a tiny nonzero residual, which flushing subnormals
    to zero anywhere on the way would lose); bit-exact residual."""
    hidden = 256
    rng = np.random.default_rng(12)
    ex = rng.integers(-135, -60, (3, hidden)).astype(np.float64)
    sign = np.where(rng.random((3, hidden)) < 0.5, -1.0, 1.0)
    vals = sign * rng.uniform(1, 2, (3, hidden)) * np.exp2(ex)
    g = torch.from_numpy(vals[0][None]).to(torch.bfloat16)
    y = torch.from_numpy(vals[1][None]).to(torch.bfloat16)
    r = torch.from_numpy(vals[2][None]).to(torch.bfloat16)
    r[0, : hidden // 2] = 0.0                                 # residual 0: the product alone
    g[0, : hidden // 4] = torch.tensor(2.0 ** -70)            # products near 2^-130..2^-125
    y[0, : hidden // 4] = (torch.from_numpy(rng.uniform(1, 2, hidden // 4) * 2.0 ** -60)
                           .to(torch.bfloat16))
    zero = torch.zeros(1, hidden, dtype=torch.bfloat16)
    _, o_res, _, _ = oracle.gated_ln_modulate(host_bits(r), host_bits(y), host_bits(g),
                                              host_bits(zero), host_bits(zero))
    tiny = (o_res[0] & 0x7F80) == 0                           # bf16 subnormal or zero
    assert ((o_res[0] & 0x7FFF) != 0)[: hidden // 4].sum() >= hidden // 8  # nonzero tiny results
    assert tiny.sum() >= hidden // 8
    run_case(nr, r, y, g, zero, zero)
