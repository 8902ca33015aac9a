"""GPU parity: nr_gelu_and_mul against the oracle, element by element.

bf16 outputs: at most 1 bf16 ulp; f32 outputs: relative error <= 1e-5 (a
product of gelu_tanh(a) and b, no cancellation; the f32 kernel carries 2z in
two floats so that e^{2z} keeps its relative accuracy for negative gates).
Source: vllm.cpp src/vt/cuda/cuda_ops.cu, GELU gated-activation section (gate first, up
second, the tanh form of GELU)."""
import numpy as np
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
    nr.gelu_and_mul(dev(x), out=og.t)
    torch.cuda.synchronize()
    og.check()
    o_out, o_y = oracle.gelu_and_mul(host_bits(x), want_y=True)
    got = host_bits(og.t)
    if dtype == torch.bfloat16:
        check_bf16(got, o_out, what="gelu_and_mul")
    else:
        check_f32(got, o_y, rel=1e-5, what="gelu_and_mul")


@pytest.mark.parametrize("hidden", synth.DECODE["hidden"])
@pytest.mark.parametrize("rows", [1, 32, 256])
def test_decode_cells(nr, rows, hidden):
    """x [rows, 2I] with I = 3 * hidden."""
    run_case(nr, rows, 3 * hidden, seed=synth.DECODE["seed"])


def test_prefill_8192x15360(nr):
    """The bench's prefill shape; checked on every element (the oracle takes a
    few seconds)."""
    run_case(nr, 8192, 3 * 5120, seed=6)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,inter", [(1, 8), (3, 24), (5, 1032), (2, 65536 + 8), (512, 4096)])
def test_edge_shapes(nr, dtype, rows, inter):
    run_case(nr, rows, inter, dtype=dtype, seed=rows + inter)


def test_more_rows_than_one_grid_column(nr):
    """70000 rows exceed the 65535 grid rows of one launch: the kernel loops."""
    run_case(nr, 70000, 16, seed=1)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_gates_across_the_range(nr, dtype):
    """Gates from -25 to 25 in steps of 1/64 (every value exact in bf16 and
    f32): where e^{2z} falls towards the f32 subnormals, where the sigmoid
    saturates, both sides of the clamp at |a| = 20, signed zeros, tiny and
    huge gates."""
    gates = np.concatenate([np.arange(-25 * 64, 25 * 64 + 1) / 64.0,
                            [-0.0, 1e-30, -1e-30, 3e30, -3e30, 1e-3, -1e-3]])
    n = (len(gates) + 7) // 8 * 8
    x = torch.zeros(1, 2 * n, dtype=torch.float32)
    x[0, :len(gates)] = torch.from_numpy(gates)
    x[0, n:n + len(gates)] = torch.from_numpy(np.linspace(-2, 2, len(gates)))
    run_case(nr, 1, n, dtype=dtype, x=x.to(dtype))


def test_zero_rows_is_a_no_op(nr):
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    assert nr.gelu_and_mul(x).shape == (0, 32)
