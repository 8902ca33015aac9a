"""GPU parity: nr_qk_norm_rope_ex (RoPE variants) against the oracle.

Same tolerance as test_gpu_qk_norm_rope.py (1 bf16 ulp, or the cancellation
allowance with K = 32).  Sources: vllm.cpp src/vt/cuda/cuda_ops.cu, the NeoX RoPE
section (Llama-3 rescale), the cache-driven RoPE section (GPT-J pairs, M-RoPE
axis selection), the fused attention-preamble section (partial rotary)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import parity
from tests.gpu_util import Guarded, dev, host_bits
from tests.parity import check_bf16, check_f32

pytestmark = pytest.mark.gpu
K_ROPE = 32
LLAMA3 = (8.0, 1.0, 4.0, 8192.0)


def run_variant(nr, tokens, hq, hk, D, dtype=torch.bfloat16, seed=0, pos=None, **kw):
    q, k, wq, wk, p = synth.qk_inputs(tokens, hq, hk, D, seed, dtype, torch.float32)
    if pos is not None:
        p = pos
    qg, kg = Guarded(q.shape, dtype), Guarded(k.shape, dtype)
    nr.qk_norm_rope_ex(dev(q), dev(k), dev(wq), dev(wk), dev(p), q_out=qg.t, k_out=kg.t, **kw)
    torch.cuda.synchronize()
    qg.check()
    kg.check()
    ref = oracle.qk_norm_rope_ex(host_bits(q), host_bits(k), host_bits(wq), host_bits(wk),
                                 p.numpy(), want_y=True, **kw)
    for got, o, y, m, name in ((qg.t, ref[0], ref[2], ref[4], "q"),
                               (kg.t, ref[1], ref[3], ref[5], "k")):
        g = host_bits(got)
        if dtype == torch.bfloat16:
            check_bf16(g, o, y, m, k_cancel=K_ROPE, what="rope-ex " + name)
        else:
            check_f32(g, y, rel=1e-5, mag=m, k_cancel=K_ROPE, what="rope-ex " + name)
    return qg.t, kg.t


def test_defaults_match_the_plain_entry_point(nr):
    q, k, wq, wk, p = synth.qk_inputs(40, 8, 2, 128, 3, torch.bfloat16, torch.float32)
    a = nr.qk_norm_rope(dev(q), dev(k), dev(wq), dev(wk), dev(p))
    b = nr.qk_norm_rope_ex(dev(q), dev(k), dev(wq), dev(wk), dev(p))
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("D,rot", [(128, 64), (128, 32), (128, 16), (256, 64), (64, 32)])
def test_partial_rotary(nr, D, rot):
    run_variant(nr, 37, 4, 2, D, seed=rot, rotary_dim=rot)


@pytest.mark.parametrize("D,rot", [(128, 128), (128, 64), (128, 24), (64, 8), (256, 256)])
def test_interleaved_pairs(nr, D, rot):
    run_variant(nr, 29, 3, 3, D, seed=D + rot, rotary_dim=rot, interleaved=True)


def test_llama3_rescale_long_positions(nr):
    pos = torch.arange(0, 131072, 131072 // 64, dtype=torch.int32)
    run_variant(nr, 64, 4, 2, 128, seed=5, pos=pos, theta=500000.0, llama3=LLAMA3)


@pytest.mark.parametrize("interleaved", [False, True])
def test_mrope_sections(nr, interleaved):
    T = 33
    rng = np.random.default_rng(7)
    pos = torch.from_numpy(rng.integers(0, 8192, (3, T)).astype(np.int32))
    run_variant(nr, T, 6, 2, 128, seed=8, pos=pos, mrope_sections=(16, 24, 24),
                mrope_interleaved=interleaved, theta=1e6)


def _mrope_positions(T, seed):
    rng = np.random.default_rng(seed)
    return torch.from_numpy(rng.integers(0, 8192, (3, T)).astype(np.int32))


@pytest.mark.parametrize("D,dtype,hq,hk,T", [
    (256, torch.bfloat16, 3, 1, 45),    # 128 pairs: one per thread of the bulk kernel
    (512, torch.bfloat16, 2, 1, 19),    # 256 pairs: more than its threads, the ring kernel
    (64, torch.float32, 3, 1, 21),
    (256, torch.float32, 2, 2, 17),     # f32, 128 pairs
    (128, torch.bfloat16, 7, 3, 3001),  # GQA, passes that straddle Q/K or end past the heads
], ids=["bf16_256", "bf16_512_ring", "f32_64", "f32_256", "gqa_many_tokens"])
def test_mrope_whole_head_sizes_and_paths(nr, D, dtype, hq, hk, T):
    """M-RoPE over the whole head at each kernel's edge, sections in the
    16:24:24 proportion of the benchmark."""
    half = D // 2
    sections = (half // 4, 3 * half // 8, half - half // 4 - 3 * half // 8)
    run_variant(nr, T, hq, hk, D, dtype=dtype, seed=D + T, pos=_mrope_positions(T, D),
                mrope_sections=sections, theta=1e6)


@pytest.mark.parametrize("interleaved", [False, True])
def test_mrope_partial_rotary_runs_the_ring_kernel(nr, interleaved):
    """M-RoPE on the first 64 of 128 dims (sections sum to 32 pairs), with
    rotate-half or GPT-J pairs: layouts the full-head kernel does not take."""
    T = 41
    run_variant(nr, T, 4, 2, 128, seed=23, pos=_mrope_positions(T, 23), rotary_dim=64,
                interleaved=interleaved, mrope_sections=(8, 12, 12), theta=1e6)


@pytest.mark.parametrize("kw", [dict(rotary_dim=64), dict(interleaved=True),
                                dict(rotary_dim=32, interleaved=True)])
def test_f32_variants(nr, kw):
    run_variant(nr, 21, 3, 1, 64, dtype=torch.float32, seed=11, **kw)


def test_all_at_once(nr):
    """Partial rotary, interleaved pairs, Llama-3 and interleaved M-RoPE together."""
    T = 17
    rng = np.random.default_rng(12)
    pos = torch.from_numpy(rng.integers(-1000, 100000, (3, T)).astype(np.int32))
    run_variant(nr, T, 5, 3, 256, seed=13, pos=pos, rotary_dim=128, interleaved=True,
                llama3=LLAMA3, mrope_sections=(24, 20, 20), mrope_interleaved=True)


@pytest.mark.parametrize("kw", [dict(rotary_dim=64), dict(rotary_dim=64, interleaved=True),
                                dict(interleaved=True),
                                dict(mrope_sections=(16, 24, 24), theta=1e6)],
                         ids=["partial", "gptj_partial", "gptj", "mrope"])
def test_variants_at_the_benchmark_shape(nr, kw):
    """Q, K [26598, 24, 128] bf16 as in the benchmark: every block cycles its
    stages through ~35 tokens.  Compared with the oracle on every element, in
    token chunks."""
    c = synth.QK_NORM_ROPE
    T = c["tokens"]
    q, k, wq, wk, pos = synth.qk_inputs(T, c["hq"], c["hk"], c["head_dim"], 17, torch.bfloat16,
                                        torch.float32)
    if kw.get("mrope_sections"):
        pos = torch.stack([pos // 1024, (pos // 32) % 32, pos % 32]).to(torch.int32).contiguous()
    qd, kd = dev(q), dev(k)
    qo, ko = nr.qk_norm_rope_ex(qd, kd, dev(wq), dev(wk), dev(pos), **kw)
    torch.cuda.synchronize()
    gq, gk = host_bits(qo), host_bits(ko)
    qb, kb = host_bits(q), host_bits(k)
    name = ",".join("%s=%s" % kv for kv in sorted(kw.items()))
    with parity.recording("rope variant %s bf16 [26598, 24+24, 128]" % name):
        for t0 in range(0, T, 4096):
            t1 = min(t0 + 4096, T)
            p = pos[..., t0:t1].contiguous().numpy()
            ref = oracle.qk_norm_rope_ex(qb[t0:t1], kb[t0:t1], host_bits(wq), host_bits(wk), p,
                                         want_y=True, **kw)
            check_bf16(gq[t0:t1], ref[0], ref[2], ref[4], k_cancel=K_ROPE,
                       what="rope-ex q %d" % t0)
            check_bf16(gk[t0:t1], ref[1], ref[3], ref[5], k_cancel=K_ROPE,
                       what="rope-ex k %d" % t0)


def test_gptj_partial_many_tokens_gqa_and_odd_head_counts(nr):
    """GQA (more Q heads than K heads) with head counts that leave the last
    pass of a token partly empty, many tokens per block."""
    run_variant(nr, 5003, 7, 3, 128, seed=19, rotary_dim=96, interleaved=True)
    run_variant(nr, 4001, 5, 1, 64, seed=20, rotary_dim=32)
