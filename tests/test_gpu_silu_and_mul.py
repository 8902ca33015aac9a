"""GPU parity: nr_silu_and_mul against the oracle, element by element.

bf16 outputs: at most 1 bf16 ulp; f32 outputs: relative error <= 1e-5 (the op
is a product of silu(a) and b, so there is no cancellation).  Source: vllm.cpp
src/vt/cuda/cuda_ops.cu, SiLU gated-activation section (gate first, up second)."""
import pytest
import torch

import oracle
import synth
from tests.gpu_util import Guarded, dev, host_bits
from tests.parity import check_bf16, check_f32

pytestmark = pytest.mark.gpu


def run_case(nr, rows, inter, dtype=torch.bfloat16, seed=0, x=None):
    if x is None:
        x = synth.silu_inputs(rows, inter, seed, dtype)
    og = Guarded((rows, inter), dtype)
    nr.silu_and_mul(dev(x), out=og.t)
    torch.cuda.synchronize()
    og.check()
    o_out, o_y = oracle.silu_and_mul(host_bits(x), want_y=True)
    got = host_bits(og.t)
    if dtype == torch.bfloat16:
        check_bf16(got, o_out, what="silu_and_mul")
    else:
        check_f32(got, o_y, rel=1e-5, what="silu_and_mul")


@pytest.mark.parametrize("hidden", synth.DECODE["hidden"])
@pytest.mark.parametrize("rows", synth.DECODE["rows"])
def test_config_decode_silu_and_mul(nr, rows, hidden):
    """x [rows, 2I] with I = 3 * hidden, the decode sweep's cells."""
    run_case(nr, rows, 3 * hidden, seed=synth.DECODE["seed"])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,inter", [(1, 8), (3, 24), (5, 1032), (2, 65536 + 8), (512, 4096)])
def test_edge_shapes(nr, dtype, rows, inter):
    run_case(nr, rows, inter, dtype=dtype, seed=rows + inter)


def test_more_rows_than_one_grid_column(nr):
    """70000 rows exceed the 65535 grid rows of one launch: the kernel loops."""
    run_case(nr, 70000, 16, seed=1)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_extreme_gates(nr, dtype):
    """Gates where e^-a overflows or vanishes in f32.  The gates -89, -90 and
    -91 (e^-a beyond the f32 range, a * e^a still a normal f32) are paired with
    ups of +-1e30, so that the product sits far above the comparison's absolute
    floor and its relative error is what is checked."""
    gates = [-120.0, -100.0, -88.0, -87.0, -50.0, -20.0, -1.0, 0.0, 1.0, 20.0, 50.0, 88.0, 100.0,
             120.0, -0.0, 1e-30, -89.0, -90.0, -91.0]
    n = len(gates)
    x = torch.empty(1, 2 * n, dtype=torch.float32)
    x[0, :n] = torch.tensor(gates)
    x[0, n:] = torch.linspace(-2, 2, n)
    if dtype == torch.float32:
        x[0, 2 * n - 3:] = torch.tensor([1e30, -1e30, 1e30])
    n8 = (n + 7) // 8 * 8
    xp = torch.zeros(1, 2 * n8, dtype=torch.float32)
    xp[0, :n] = x[0, :n]
    xp[0, n8:n8 + n] = x[0, n:]
    run_case(nr, 1, n8, dtype=dtype, x=xp.to(dtype))
