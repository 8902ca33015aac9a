"""GPU parity: nr_ln_modulate (LayerNorm + adaLN modulation) against the oracle,
element by element, on seeded inputs.

Tolerance.  bf16 outputs: at most 1 bf16 ulp, except where xhat*(1+scale) and
shift cancel: there an element also passes when
|gpu - y| <= ulp_bf16(y) + K * 2^-24 * mag, K = 64, with
mag = (|x - mu| + mean|x|) * rstd * |1 + scale| + |shift| from the oracle.  K
counts the f32 roundings on the kernel's path: the row sum behind mu (up to
16 per thread + 5 butterfly + 6 cross-warp levels at hidden 3072, giving an
absolute error of ~27 * mean|x| in mu), the centred sum of squares and the
quotient and reciprocal square root behind rstd (~15 relative), and the final
products and fma.
The pages name the fusion (FastVideo PAN2 docs, "Performance switches",
dit_fused_kernels) without printing its formula.
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


def run_case(nr, rows, hidden, dtype=torch.bfloat16, samples=1, rps=None, eps=1e-6, seed=0,
             inplace=False, x=None, chunk=None):
    if x is None:
        x, shift, scale = synth.ln_inputs(rows, hidden, seed, dtype, samples=samples)
    else:
        _, shift, scale = synth.ln_inputs(rows, hidden, seed, dtype, samples=samples)
    rps = rows if rps is None else rps
    og = Guarded(x.shape, dtype, fill=x if inplace else None)
    xd = og.t if inplace else dev(x)
    nr.ln_modulate(xd, dev(shift), dev(scale), eps=eps, rows_per_sample=rps, out=og.t)
    torch.cuda.synchronize()
    og.check()
    got = og.t.cpu()
    chunk = rows if chunk is None else chunk
    for r0 in range(0, rows, chunk):
        r1 = min(r0 + chunk, rows)
        # sample index of a row depends on its global index: pass the matching shift rows
        s_idx = np.arange(r0, r1) // rps
        o_out, o_y, o_mag = oracle.ln_modulate(host_bits(x[r0:r1]), host_bits(shift[s_idx]),
                                               host_bits(scale[s_idx]), eps=eps,
                                               rows_per_sample=1, want_y=True)
        g = host_bits(got[r0:r1])
        if dtype == torch.bfloat16:
            check_bf16(g, o_out, o_y, o_mag, k_cancel=K_LN, what="ln_modulate rows %d.." % r0)
        else:
            check_f32(g, o_y, rel=1e-5, mag=o_mag, k_cancel=K_LN, what="ln_modulate")


def test_config_ln_modulate_26598x3072(nr):
    """The full workload the bench times: x [26598, 3072] bf16, one shift/scale
    sample for all rows; compared in row chunks."""
    c = synth.LN_MODULATE
    with parity.recording("ln_modulate bf16 [26598, 3072]"):
        run_case(nr, c["rows"], c["hidden"], eps=c["eps"], seed=c["seed"], chunk=4096)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("hidden", [8, 24, 1000, 3072, 5128, 32768, 32776, 65536])
def test_edge_hidden_sizes(nr, dtype, hidden):
    if dtype == torch.bfloat16 and hidden % 8:
        pytest.skip("bf16 needs hidden % 8 == 0")
    run_case(nr, 3, hidden, dtype=dtype, seed=hidden % 89)


def test_per_row_and_per_sample_modulation(nr):
    run_case(nr, 12, 1024, samples=12, rps=1, seed=3)  # one modulation row per token
    run_case(nr, 12, 1024, samples=3, rps=4, seed=4)   # 3 samples of 4 tokens


def test_in_place_out_is_x(nr):
    run_case(nr, 64, 3072, seed=6, inplace=True)


def test_constant_row_gives_shift_exactly(nr):
    """sigma^2 = 0: xhat = 0 and out = shift, bit for bit."""
    hidden = 3072
    _, shift, scale = synth.ln_inputs(4, hidden, 7, torch.bfloat16)
    x = torch.full((4, hidden), 0.7, dtype=torch.bfloat16)
    x[1] = -3.0
    x[2] = 0.0
    out = nr.ln_modulate(dev(x), dev(shift), dev(scale)).cpu()
    for r in range(4):
        assert torch.equal(out[r], shift[0])


def test_scale_minus_one_gives_shift(nr):
    x, shift, _ = synth.ln_inputs(8, 512, 8, torch.bfloat16)
    scale = torch.full((1, 512), -1.0, dtype=torch.bfloat16)
    out = nr.ln_modulate(dev(x), dev(shift), dev(scale)).cpu()
    assert torch.equal(out, shift.expand(8, 512))


def test_large_offset_rows(nr):
    """Rows with a large common offset (mean >> sigma) stay within the bound."""
    x, _, _ = synth.ln_inputs(16, 2048, 9, torch.float32)
    run_case(nr, 16, 2048, dtype=torch.bfloat16, x=(x * 0.5 + 40.0).to(torch.bfloat16), seed=9)


# Many rows (more than 64 per SM of a 152-SM GB300) at several row widths.
MANY_ROWS = 64 * 152


@pytest.mark.parametrize("hidden", [64, 1024, 2048, 3000, 3072, 4096])
def test_many_rows_hidden_sizes(nr, hidden):
    """One- and two-warp rows, a width that leaves lanes idle (3000 = 375
    vectors), and the smallest row."""
    run_case(nr, MANY_ROWS + 37, hidden, seed=hidden % 97, chunk=4096)


def test_many_rows_in_place_and_modulation_rows(nr):
    run_case(nr, MANY_ROWS + 5, 3072, seed=41, inplace=True, chunk=4096)
    run_case(nr, MANY_ROWS, 1024, samples=MANY_ROWS, rps=1, seed=42, chunk=4096)
    run_case(nr, MANY_ROWS + 3, 1024, samples=(MANY_ROWS + 3 + 99) // 100, rps=100, seed=43,
             chunk=4096)


def test_many_constant_rows_give_shift(nr):
    hidden = 3072
    _, shift, scale = synth.ln_inputs(1, hidden, 44, torch.bfloat16)
    x = torch.full((MANY_ROWS, hidden), 0.7, dtype=torch.bfloat16)
    out = nr.ln_modulate(dev(x), dev(shift), dev(scale)).cpu()
    assert torch.equal(out, shift.expand(MANY_ROWS, hidden))


def test_bf16_subnormal_inputs(nr):
    """Rows mixing bf16 subnormals with normal values, and rows of subnormals
    only (whose variance underflows to 0 in f32, leaving the shift)."""
    hidden = 1024
    rng = np.random.default_rng(45)
    x = rng.standard_normal((4, hidden))
    x[:, ::3] = np.sign(x[:, ::3]) * rng.uniform(1, 2, (4, (hidden + 2) // 3)) * 2.0 ** -130
    x[2:] = np.sign(x[2:]) * rng.uniform(1, 2, (2, hidden)) * 2.0 ** -128
    run_case(nr, 4, hidden, seed=46, x=torch.from_numpy(x).to(torch.bfloat16))
