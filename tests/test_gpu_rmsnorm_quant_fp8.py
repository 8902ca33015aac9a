"""GPU parity: nr_rmsnorm_quant_fp8 (RMSNorm + static e4m3 quantisation).

The bf16 intermediate follows the RMSNorm rule (1 bf16 ulp; residual bit-exact).
The e4m3 code is decided in f32 from that bf16 value on both sides, so it must
be bit-exact wherever the GPU's bf16 value equals the oracle's, and elsewhere
equal to the oracle's conversion of the GPU's own bf16 value.  Source: vllm.cpp
src/vt/cuda/cuda_ops.cu, its fused RMSNorm + static FP8 section."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import Guarded, dev, host_bits
from tests.parity import bf16_to_f64, check_bf16

pytestmark = pytest.mark.gpu


def run_case(nr, rows, hidden, dtype=torch.bfloat16, residual=True, scale=0.02, gemma=False,
             seed=0):
    x, res, w = synth.rmsnorm_inputs(rows, hidden, seed, dtype, residual=residual)
    codes_ref, nb_ref, res_ref, _ = oracle.rmsnorm_quant_fp8(
        host_bits(x), host_bits(w), scale, residual=None if res is None else host_bits(res),
        gemma=gemma)
    rg = None if res is None else Guarded(res.shape, dtype, fill=res)
    codes = torch.zeros((rows, hidden), dtype=torch.uint8, device="cuda")
    nbg = Guarded((rows, hidden), torch.bfloat16)
    nr.rmsnorm_quant_fp8(dev(x), dev(w), scale, residual=None if rg is None else rg.t,
                         gemma=gemma, codes=codes, out_bf16=nbg.t)
    torch.cuda.synchronize()
    nbg.check()
    if rg is not None:
        rg.check()
        assert np.array_equal(host_bits(rg.t), res_ref), "residual not bit-exact"
    nb = host_bits(nbg.t)
    check_bf16(nb, nb_ref, what="fp8 bf16 intermediate")
    got = codes.cpu().numpy()
    same = nb == nb_ref
    assert np.array_equal(got[same], codes_ref[same])
    t = (bf16_to_f64(nb[~same]).astype(np.float32)
         * (np.float32(1.0) / np.float32(scale)))
    assert np.array_equal(got[~same], oracle.e4m3_array(t))
    return got


@pytest.mark.parametrize("gemma", [False, True])
def test_dense_workload_8192x5120(nr, gemma):
    run_case(nr, 8192, 5120, gemma=gemma, seed=1)


def test_saturation_and_subnormal_codes(nr):
    """A small scale pushes many codes to +-448 (satfinite); a large one makes
    subnormal codes."""
    got = run_case(nr, 16, 1024, scale=1e-3, seed=2)
    assert ((got & 0x7F) == 0x7E).mean() > 0.3
    got = run_case(nr, 16, 1024, scale=200.0, seed=3)
    assert ((got & 0x78) == 0).mean() > 0.3


@pytest.mark.parametrize("dtype,hidden", [(torch.bfloat16, h) for h in (8, 24, 4096, 8200, 32768)]
                         + [(torch.float32, h) for h in (4, 12, 4096, 8200, 16384)])
def test_edge_sizes(nr, dtype, hidden):
    """Down to one vector per row and up to the largest supported hidden
    (32768 bf16 / 16384 f32: 4096 vectors of 16 bytes held in registers)."""
    run_case(nr, 3, hidden, dtype=dtype, residual=hidden % 3 == 0, seed=hidden % 31)


@pytest.mark.parametrize("dtype,hidden", [(torch.bfloat16, 32768), (torch.bfloat16, 5128),
                                          (torch.float32, 16384)])
@pytest.mark.parametrize("rows", [1, 19, 160])
def test_few_and_many_rows(nr, rows, dtype, hidden):
    """One row, fewer rows than SMs and more, at the largest supported hidden."""
    run_case(nr, rows, hidden, dtype=dtype, residual=True, seed=rows)


def test_hidden_above_the_register_limit_is_refused(nr):
    x = torch.zeros(2, 16388, dtype=torch.float32, device="cuda")
    w = torch.ones(16388, dtype=torch.float32, device="cuda")
    with pytest.raises(nr.NrError, match="UNSUPPORTED"):
        nr.rmsnorm_quant_fp8(x, w, 1.0)


def test_codes_only_without_bf16_copy(nr):
    x, res, w = synth.rmsnorm_inputs(4, 2048, 4, torch.bfloat16)
    a = nr.rmsnorm_quant_fp8(dev(x), dev(w), 0.05)
    b, _ = nr.rmsnorm_quant_fp8(dev(x), dev(w), 0.05, out_bf16=True)
    assert torch.equal(a, b)
