"""GPU parity: nr_qk_norm_rope (per-head Q/K RMSNorm + NeoX RoPE) against the
oracle, element by element, on seeded inputs.

Tolerance.  bf16 outputs: at most 1 bf16 ulp, except where the rotation's two
products cancel: there an element also passes when
|gpu - y| <= ulp_bf16(y) + K * 2^-24 * (|n_i| + |n_{i+D/2}|), K = 32.  K counts
the kernel's f32 roundings: ~19 in the head's sum of squares (16 per lane +
3 butterfly levels), rsqrtf (2 ulp), two products forming n (so ~14 relative
on n), ~4 absolute on cos/sin (argument conversion + sincospif) plus the
oracle's own double rounding of pos*freq at |pos| up to 2^31 (~4), and the
final product and fma: < 32 in all.  f32 outputs: relative 1e-5 plus the same
allowance.  Sources: the vllm.cpp page src/vt/cuda/cuda_ops.cu,
its fused attention-preamble and NeoX RoPE sections.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import parity
from tests.gpu_util import Guarded, dev, host_bits
from tests.parity import bf16_ulp_distance, check_bf16, check_f32

pytestmark = pytest.mark.gpu
K_ROPE = 32


def _compare(got_q, got_k, q, k, wq, wk, pos, eps, theta, gemma, dtype, t_lo=0, t_hi=None):
    """Compare GPU outputs (host copies, [T, H, D] views) on tokens [t_lo, t_hi)."""
    t_hi = q.shape[0] if t_hi is None else t_hi
    sl = slice(t_lo, t_hi)
    qo, ko, qy, ky, qm, km = oracle.qk_norm_rope(host_bits(q[sl]), host_bits(k[sl]),
                                                 host_bits(wq), host_bits(wk), pos[sl].numpy(),
                                                 eps=eps, theta=theta, gemma=gemma, want_y=True)
    reps = []
    for got, o, y, m, name in ((got_q, qo, qy, qm, "q"), (got_k, ko, ky, km, "k")):
        g = host_bits(got[sl].contiguous())
        if dtype == torch.bfloat16:
            reps.append(check_bf16(g, o, y, m, k_cancel=K_ROPE, what="rope " + name))
        else:
            reps.append(check_f32(g, y, rel=1e-5, mag=m, k_cancel=K_ROPE, what="rope " + name))
    return reps


def run_case(nr, tokens, hq, hk, D, dtype=torch.bfloat16, w_dtype=torch.float32, eps=1e-6,
             theta=10000.0, gemma=False, seed=0, pos=None, chunk=None):
    q, k, wq, wk, p = synth.qk_inputs(tokens, hq, hk, D, seed, dtype, w_dtype)
    if pos is not None:
        p = pos
    qg, kg = Guarded(q.shape, dtype), Guarded(k.shape, dtype)
    nr.qk_norm_rope(dev(q), dev(k), dev(wq), dev(wk), dev(p), eps=eps, theta=theta, gemma=gemma,
                    q_out=qg.t, k_out=kg.t)
    torch.cuda.synchronize()
    qg.check()
    kg.check()
    gq, gk = qg.t.cpu(), kg.t.cpu()
    chunk = tokens if chunk is None else chunk
    reps = []
    for t0 in range(0, tokens, chunk):
        reps += _compare(gq, gk, q, k, wq, wk, p, eps, theta, gemma, dtype, t0,
                         min(t0 + chunk, tokens))
    return reps


@pytest.mark.parametrize("w_dtype", [torch.float32, torch.bfloat16])
def test_config_qk_norm_rope_26598x24x128(nr, w_dtype):
    """The full workload the bench times: Q, K [26598, 24, 128] bf16,
    positions 0..26597, theta 1e4; compared in token chunks."""
    c = synth.QK_NORM_ROPE
    with parity.recording("qk_norm_rope bf16 [26598, 24+24, 128], %s weights"
                          % str(w_dtype).split(".")[-1]):
        reps = run_case(nr, c["tokens"], c["hq"], c["hk"], c["head_dim"], w_dtype=w_dtype,
                        eps=c["eps"], theta=c["theta"], seed=c["seed"], chunk=2048)
    total = sum(r["n"] for r in reps)
    assert total == 2 * c["tokens"] * c["hq"] * c["head_dim"]


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, d) for d in (16, 32, 64, 128, 256, 512)]
                         + [(torch.float32, d) for d in (8, 16, 32, 64, 128, 256)])
def test_every_head_dim(nr, dtype, D):
    run_case(nr, 37, 3, 2, D, dtype=dtype, gemma=True, seed=D)


@pytest.mark.parametrize("tokens,hq,hk", [(1, 1, 1), (1, 24, 24), (5, 7, 1), (300, 32, 8),
                                          (17, 1, 0), (64, 2, 2)])
def test_token_and_head_counts(nr, tokens, hq, hk):
    run_case(nr, tokens, hq, hk, 128, seed=tokens + hq)


@pytest.mark.parametrize("dtype,tokens,hq,hk,D", [(torch.bfloat16, 9, 48, 16, 512),
                                                  (torch.float32, 7, 64, 64, 256)])
def test_token_blocks_too_large_for_the_bulk_stages(nr, dtype, tokens, hq, hk, D):
    """64 KB / 128 KB of Q and K rows per token: more than the bulk-copy
    stages hold, so the per-warp ring kernel runs instead."""
    run_case(nr, tokens, hq, hk, D, dtype=dtype, seed=hq + D)


def test_many_tokens_per_block_with_gqa(nr):
    """Enough tokens that every block cycles through its stages many times,
    with fewer K heads than Q heads (a K block smaller than the Q block)."""
    run_case(nr, 20000, 16, 2, 128, seed=41, chunk=5000)


def test_large_and_negative_positions(nr):
    """Positions across the whole int32 range, in random order: the angle is
    reduced exactly, so large positions keep full accuracy."""
    rng = np.random.default_rng(3)
    p = rng.integers(-2 ** 31, 2 ** 31, 200, dtype=np.int64).astype(np.int32)
    p[:4] = [0, 2 ** 31 - 1, -2 ** 31, 1]
    run_case(nr, 200, 4, 2, 128, pos=torch.from_numpy(p), seed=11)


@pytest.mark.parametrize("theta", [10.0, 500000.0, 1e6])
def test_theta(nr, theta):
    run_case(nr, 50, 2, 2, 64, theta=theta, seed=13)


def test_position_zero_is_plain_head_rmsnorm(nr):
    """At position 0 the rotation is the identity: the output equals the RMSNorm
    kernel's result on the same head rows (bf16 weights), within 1 ulp."""
    q, k, wq, wk, _ = synth.qk_inputs(8, 4, 4, 128, 21, torch.bfloat16, torch.bfloat16)
    zero = torch.zeros(8, dtype=torch.int32)
    qo, ko = nr.qk_norm_rope(dev(q), dev(k), dev(wq), dev(wk), dev(zero))
    rq = nr.rmsnorm(dev(q.reshape(-1, 128)), dev(wq))
    d = bf16_ulp_distance(host_bits(qo.reshape(-1, 128)), host_bits(rq))
    assert d.max() <= 1


def test_fused_qkv_layout_and_in_place(nr):
    """Q and K as token-strided views into one fused [T, (hq + 2 hk) * D] row
    (V untouched), rotated in place."""
    T, hq, hk, D = 33, 8, 2, 128
    width = (hq + 2 * hk) * D
    fused = synth.tensor(17, 5, (T, width), torch.bfloat16)
    _, _, wq, wk, pos = synth.qk_inputs(T, hq, hk, D, 17, torch.bfloat16, torch.float32)
    q = fused[:, :hq * D].reshape(T, hq, D)  # strided views (token stride = width)
    k = fused[:, hq * D:(hq + hk) * D].reshape(T, hk, D)
    fd = fused.cuda()
    qd = fd[:, :hq * D].view(T, hq, D)
    kd = fd[:, hq * D:(hq + hk) * D].view(T, hk, D)
    assert qd.stride(0) == width
    nr.qk_norm_rope(qd, kd, dev(wq), dev(wk), dev(pos), q_out=qd, k_out=kd)
    torch.cuda.synchronize()
    res = fd.cpu()
    assert torch.equal(res[:, (hq + hk) * D:], fused[:, (hq + hk) * D:])  # V untouched
    _compare(res[:, :hq * D].reshape(T, hq, D), res[:, hq * D:(hq + hk) * D].reshape(T, hk, D),
             q, k, wq, wk, pos, 1e-6, 10000.0, False, torch.bfloat16)


def test_out_of_place_strided_outputs(nr):
    T, hq, hk, D = 20, 4, 4, 64
    width = (hq + hk) * D + 64  # padded rows
    buf_in = synth.tensor(19, 6, (T, width), torch.bfloat16)
    _, _, wq, wk, pos = synth.qk_inputs(T, hq, hk, D, 19, torch.bfloat16, torch.bfloat16)
    bi = buf_in.cuda()
    bo = torch.zeros_like(bi)
    qi, ki = bi[:, :hq * D].view(T, hq, D), bi[:, hq * D:(hq + hk) * D].view(T, hk, D)
    qo, ko = bo[:, :hq * D].view(T, hq, D), bo[:, hq * D:(hq + hk) * D].view(T, hk, D)
    nr.qk_norm_rope(qi, ki, dev(wq), dev(wk), dev(pos), q_out=qo, k_out=ko)
    torch.cuda.synchronize()
    assert torch.equal(bi.cpu(), buf_in)
    assert torch.all(bo[:, (hq + hk) * D:].cpu() == 0)  # padding untouched
    _compare(qo.cpu(), ko.cpu(), buf_in[:, :hq * D].reshape(T, hq, D),
             buf_in[:, hq * D:(hq + hk) * D].reshape(T, hk, D), wq, wk, pos, 1e-6, 10000.0,
             False, torch.bfloat16)


def test_zero_tokens_is_a_no_op(nr):
    q = torch.empty(0, 2, 128, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(128, device="cuda")
    p = torch.empty(0, dtype=torch.int32, device="cuda")
    qo, ko = nr.qk_norm_rope(q, q.clone(), w, w, p)
    assert qo.shape == (0, 2, 128)


def test_no_k_heads_without_wk(nr):
    """With no K heads the K weight may be None (a NULL pointer through the
    C ABI): Q is the same as with a K weight given."""
    q, k, wq, wk, p = synth.qk_inputs(17, 3, 0, 128, 5, torch.bfloat16, torch.float32)
    qo, ko = nr.qk_norm_rope(dev(q), dev(k), dev(wq), None, dev(p))
    qo2, _ = nr.qk_norm_rope(dev(q), dev(k), dev(wq), dev(wk), dev(p))
    torch.cuda.synchronize()
    assert ko.shape == (17, 0, 128)
    assert torch.equal(qo.cpu(), qo2.cpu())
