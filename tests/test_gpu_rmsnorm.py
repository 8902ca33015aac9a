"""GPU parity: nr_rmsnorm (plain and with the fused residual add, gemma or not)
against the oracle, element by element, on seeded inputs.

bf16 outputs: at most 1 bf16 ulp; f32 outputs: relative error <= 1e-5;
residual write-back: bit-exact.  RMSNorm's last step is a product, so no
cancellation allowance applies.  Source: the vllm.cpp page src/vt/cuda/cuda_ops.cu,
its row-RMSNorm section and the residual-rounding helper before it.
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


def run_case(nr, rows, hidden, dtype, residual, gemma=False, eps=1e-6, seed=0, inplace=False,
             x=None, res=None, w=None):
    if x is None:
        x, res0, w = synth.rmsnorm_inputs(rows, hidden, seed, dtype, residual=residual)
        res = res0 if residual else None
    xo, wo = host_bits(x), host_bits(w)
    ro = None if res is None else host_bits(res)
    o_out, o_res, o_y = oracle.rmsnorm(xo, wo, residual=ro, eps=eps, gemma=gemma, want_y=True)

    xd, wd = dev(x), dev(w)
    rg = None if res is None else Guarded(res.shape, dtype, fill=res)
    if inplace:
        og = Guarded(x.shape, dtype, fill=x)
        xd = og.t
    else:
        og = Guarded(x.shape, dtype)
    nr.rmsnorm(xd, wd, residual=None if rg is None else rg.t, eps=eps, gemma=gemma, out=og.t)
    torch.cuda.synchronize()
    og.check()
    got = host_bits(og.t)
    if dtype == torch.bfloat16:
        rep = check_bf16(got, o_out, what="rmsnorm out")
    else:
        rep = check_f32(got, o_y, rel=1e-5, what="rmsnorm out")
    if rg is not None:
        rg.check()
        assert np.array_equal(host_bits(rg.t), o_res), "residual write-back is not bit-exact"
    return rep


def test_config_rmsnorm_f32_64x1024(nr):
    """fp32, 64 x 1024, no residual, gemma false, seed 0."""
    c = synth.RMSNORM_F32
    run_case(nr, c["rows"], c["hidden"], torch.float32, residual=False, eps=c["eps"], seed=c["seed"])


@pytest.mark.parametrize("gemma", [False, True])
def test_config_add_rmsnorm_bf16_8192x5120(nr, gemma):
    """bf16 add + RMSNorm, 8192 x 5120, residual in place, gemma false and true
    (the full workload the bench times, same entry point and launch)."""
    c = synth.ADD_RMSNORM
    with parity.recording("add_rmsnorm bf16 [8192, 5120], gemma %d" % gemma):
        run_case(nr, c["rows"], c["hidden"], torch.bfloat16, residual=True, gemma=gemma,
                 eps=c["eps"], seed=c["seed"])


@pytest.mark.parametrize("hidden", synth.DECODE["hidden"])
@pytest.mark.parametrize("rows", synth.DECODE["rows"])
def test_config_decode_add_rmsnorm(nr, rows, hidden):
    c = synth.DECODE
    run_case(nr, rows, hidden, torch.bfloat16, residual=True, eps=c["eps"], seed=c["seed"])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("hidden", [8, 16, 24, 296, 2040, 5128, 12288, 32768, 32776, 131072])
def test_edge_hidden_sizes(nr, dtype, residual, hidden):
    """Every vector-per-thread choice, ragged tails, the largest register-resident
    row (32768 bf16) and the multi-pass kernel beyond it."""
    run_case(nr, 3, hidden, dtype, residual=residual, gemma=True, seed=hidden % 97)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,hidden", [(1, 8192), (1, 8200), (2, 5128), (5, 1032), (19, 4096),
                                         (38, 2048), (75, 16392), (76, 4096), (77, 4096),
                                         (160, 8200), (160, 16384), (160, 32768), (256, 8192),
                                         (257, 8192), (1024, 5120), (1025, 5120)])
def test_few_and_many_rows(nr, dtype, rows, hidden):
    """Row counts below and above the SM count (one CTA per row either way),
    both sides of the few-row geometry (256 / 257 rows) and of the weight
    prefetch (1024 / 1025 rows), vectors-per-thread choices with idle slots,
    and the largest register-resident rows next to the multi-pass kernel
    (32768 f32)."""
    run_case(nr, rows, hidden, dtype, residual=True, gemma=True, seed=rows + hidden)


@pytest.mark.parametrize("rows", [1, 2, 7, 1000])
def test_edge_row_counts(nr, rows):
    run_case(nr, rows, 1024, torch.bfloat16, residual=True, seed=rows)


@pytest.mark.parametrize("residual", [False, True])
def test_in_place_out_is_x(nr, residual):
    run_case(nr, 16, 4096, torch.bfloat16, residual=residual, seed=5, inplace=True)


def test_zero_row_and_closed_forms(nr):
    """Zero row with eps > 0 gives 0; a row of 2s with eps = 0 gives w exactly."""
    hidden = 64
    x = torch.zeros(2, hidden, dtype=torch.bfloat16)
    x[1] = 2.0
    w = synth.tensor(3, 0, (hidden,), torch.bfloat16, mean=1.0, std=0.1)
    out = nr.rmsnorm(dev(x), dev(w), eps=0.0 + 1e-6)
    assert torch.all(out[0].cpu() == 0)
    out = nr.rmsnorm(dev(x[1:].contiguous()), dev(w), eps=0.0)
    assert torch.equal(out[0].cpu(), w)


def test_zero_rows_is_a_no_op(nr):
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    out = nr.rmsnorm(x, w)
    assert out.shape == (0, 64)


def test_zero_residual_equals_plain(nr):
    x, _, w = synth.rmsnorm_inputs(64, 2048, 8, torch.bfloat16, residual=False)
    zero = torch.zeros_like(x).cuda()
    a = nr.rmsnorm(dev(x), dev(w), residual=zero)
    b = nr.rmsnorm(dev(x), dev(w))
    assert torch.equal(a, b)
    assert torch.equal(zero.cpu(), x)


def test_residual_add_edge_values_bit_exact(nr):
    """The stored residual is round_bf16(x + residual) bit for bit over the
    whole bf16 range: exponent gaps from 0 to beyond 2^-24, subnormal
    operands and sums, exact cancellations (x = -residual, +-0 mixes), and
    ties between bf16 neighbours."""
    rng = np.random.default_rng(71)
    rows, hidden = 64, 1024
    n = rows * hidden
    mant = rng.uniform(1, 2, (2, n))
    ex = rng.integers(-140, 30, (2, n))  # down into the bf16 subnormal range
    sign = np.where(rng.random((2, n)) < 0.5, -1.0, 1.0)
    vals = sign * mant * np.exp2(ex.astype(np.float64))
    x = torch.from_numpy(vals[0]).to(torch.bfloat16)
    r = torch.from_numpy(vals[1]).to(torch.bfloat16)
    q = n // 8
    r[:q] = -x[:q]                       # exact cancellations
    x[q:2 * q] = 0.0                     # +0 + r
    r[2 * q:3 * q] = -0.0                # x + -0
    x[3 * q:3 * q + 64] = -0.0           # -0 + -0
    r[3 * q:3 * q + 64] = -0.0
    # ties: r is half an ulp of x (bf16 keeps 8 bits, so 2^-8 of x's binade)
    xt = x[4 * q:5 * q].float()
    r[4 * q:5 * q] = (torch.sign(xt) * torch.exp2(torch.floor(torch.log2(xt.abs().clamp_min(2.0 ** -120))) - 8)).to(torch.bfloat16)
    x = x.view(rows, hidden)
    r = r.view(rows, hidden)
    w = torch.ones(hidden, dtype=torch.bfloat16)
    run_case(nr, rows, hidden, torch.bfloat16, residual=True, x=x, res=r, w=w)
