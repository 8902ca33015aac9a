"""Chains of dependent calls on one stream, with no synchronisation between
them.

Every kernel is launched with programmatic stream serialisation and may be
scheduled while its predecessor is still running; it must not read anything
before the predecessor has finished.  Here each call reads what the call
before it wrote (out of place, in place, and across different kernels), at
sizes where the predecessor runs for tens of microseconds, and every stage is
checked against the oracle applied to the GPU's own previous result -- a
stage that read stale or partly written data would fail."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import host_bits
from tests.parity import check_bf16

pytestmark = pytest.mark.gpu
K_LN = 64


def _ln_check(got, x_bits, shift, scale, what):
    o_out, o_y, o_mag = oracle.ln_modulate(x_bits, host_bits(shift), host_bits(scale),
                                           want_y=True)
    check_bf16(host_bits(got), o_out, o_y, o_mag, k_cancel=K_LN, what=what)


def test_layernorm_chain_out_of_place_then_in_place(nr):
    rows, hidden = 8192, 3072
    x = synth.tensor(61, 0, (rows, hidden), torch.bfloat16).cuda()
    sh = synth.tensor(61, 1, (1, hidden), torch.bfloat16, std=0.1).cuda()
    sc = synth.tensor(61, 2, (1, hidden), torch.bfloat16, std=0.1).cuda()
    y1 = nr.ln_modulate(x, sh, sc)
    y2 = nr.ln_modulate(y1, sc, sh)  # reads y1 while it may still be being written
    y3 = y2.clone()                   # (a torch copy in between)
    nr.ln_modulate(y3, sh, sc, out=y3)  # in place
    torch.cuda.synchronize()
    _ln_check(y1, host_bits(x), sh, sc, "ln stage 1")
    _ln_check(y2, host_bits(y1), sc, sh, "ln stage 2")
    _ln_check(y3, host_bits(y2), sh, sc, "ln stage 3 (in place)")


def test_residual_chain_is_bit_exact(nr):
    """residual <- x1 + residual, then residual <- x2 + residual, then a third
    add: the final residual is the exact rounded sums, bit for bit."""
    rows, hidden = 8192, 5120
    x1, res, w = synth.rmsnorm_inputs(rows, hidden, 62, torch.bfloat16)
    x2 = synth.tensor(62, 9, (rows, hidden), torch.bfloat16)
    x3 = synth.tensor(62, 10, (rows, hidden), torch.bfloat16)
    r = res.cuda()
    o1 = nr.rmsnorm(x1.cuda(), w.cuda(), residual=r)
    o2 = nr.rmsnorm(x2.cuda(), w.cuda(), residual=r)
    o3 = nr.rmsnorm(x3.cuda(), w.cuda(), residual=r, gemma=True)
    torch.cuda.synchronize()
    e1, r1, _ = oracle.rmsnorm(host_bits(x1), host_bits(w), residual=host_bits(res))
    e2, r2, _ = oracle.rmsnorm(host_bits(x2), host_bits(w), residual=r1)
    e3, r3, _ = oracle.rmsnorm(host_bits(x3), host_bits(w), residual=r2, gemma=True)
    assert np.array_equal(host_bits(r), r3)
    for got, exp, name in ((o1, e1, "1"), (o2, e2, "2"), (o3, e3, "3")):
        check_bf16(host_bits(got), exp, what="chained add+rmsnorm " + name)


def test_qk_rope_chain_in_place(nr):
    """Q/K rotated in place twice at different positions; the second call
    reads the first call's output."""
    T, hq, hk, D = 4096, 24, 8, 128
    q, k, wq, wk, pos = synth.qk_inputs(T, hq, hk, D, 63, torch.bfloat16, torch.float32)
    pos2 = torch.flip(pos, [0]).contiguous()
    qd, kd = q.cuda(), k.cuda()
    nr.qk_norm_rope(qd, kd, wq.cuda(), wk.cuda(), pos.cuda(), q_out=qd, k_out=kd)
    q1, k1 = qd.clone(), kd.clone()  # snapshot of stage 1, ordered on the stream
    nr.qk_norm_rope(qd, kd, wq.cuda(), wk.cuda(), pos2.cuda(), q_out=qd, k_out=kd)
    torch.cuda.synchronize()
    for inp_q, inp_k, p, got_q, got_k, name in (
            (host_bits(q), host_bits(k), pos, q1, k1, "stage 1"),
            (host_bits(q1), host_bits(k1), pos2, qd, kd, "stage 2")):
        qo, ko, qy, ky, qm, km = oracle.qk_norm_rope(inp_q, inp_k, host_bits(wq), host_bits(wk),
                                                     p.numpy(), want_y=True)
        check_bf16(host_bits(got_q), qo, qy, qm, k_cancel=32, what="rope q " + name)
        check_bf16(host_bits(got_k), ko, ky, km, k_cancel=32, what="rope k " + name)


def test_across_kernels(nr):
    """RMSNorm -> silu_and_mul -> LayerNorm + modulation -> gelu_and_mul, each
    reading the previous call's output."""
    rows, width = 4096, 6144
    x = synth.tensor(64, 0, (rows, width), torch.bfloat16).cuda()
    w = synth.tensor(64, 1, (width,), torch.bfloat16, std=0.1, mean=1.0).cuda()
    sh = synth.tensor(64, 2, (1, width // 2), torch.bfloat16, std=0.1).cuda()
    sc = synth.tensor(64, 3, (1, width // 2), torch.bfloat16, std=0.1).cuda()
    a = nr.rmsnorm(x, w)                 # [rows, 6144]
    b = nr.silu_and_mul(a)               # [rows, 3072]
    c = nr.ln_modulate(b, sh, sc)        # [rows, 3072]
    d = nr.gelu_and_mul(c)               # [rows, 1536]
    torch.cuda.synchronize()
    ea, _, _ = oracle.rmsnorm(host_bits(x), host_bits(w))
    check_bf16(host_bits(a), ea, what="stage rmsnorm")
    check_bf16(host_bits(b), oracle.silu_and_mul(host_bits(a))[0], what="stage silu")
    _ln_check(c, host_bits(b), sh, sc, "stage ln")
    check_bf16(host_bits(d), oracle.gelu_and_mul(host_bits(c))[0], what="stage gelu")


def test_host_threads_on_their_own_streams(nr):
    """Four host threads, each on its own stream, launch Q/K calls with
    different head layouts (first use of each launch configuration races in
    the library's host-side caches) and LayerNorm calls; every result matches
    the oracle."""
    import threading

    layouts = [(300, 8, 2, 128), (300, 16, 4, 64), (200, 32, 8, 128), (200, 4, 4, 256)]
    inputs = [synth.qk_inputs(T, hq, hk, D, 70 + i, torch.bfloat16, torch.float32)
              for i, (T, hq, hk, D) in enumerate(layouts)]
    results = [None] * len(layouts)
    errors = []

    def work(i):
        try:
            q, k, wq, wk, pos = inputs[i]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                qd, kd = q.cuda(non_blocking=False), k.cuda(non_blocking=False)
                for _ in range(3):
                    out = nr.qk_norm_rope(qd, kd, wq.cuda(), wk.cuda(), pos.cuda())
                x = synth.tensor(80 + i, 0, (64, 1024), torch.bfloat16).cuda()
                p = torch.zeros(1, 1024, dtype=torch.bfloat16, device="cuda")
                ln = nr.ln_modulate(x, p, p)
            s.synchronize()
            results[i] = (out[0].cpu(), out[1].cpu(), x.cpu(), ln.cpu())
        except Exception as exc:  # reported below, in the main thread
            errors.append(exc)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(layouts))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for (q, k, wq, wk, pos), (gq, gk, x, ln) in zip(inputs, results):
        qo, ko, qy, ky, qm, km = oracle.qk_norm_rope(host_bits(q), host_bits(k), host_bits(wq),
                                                     host_bits(wk), pos.numpy(), want_y=True)
        check_bf16(host_bits(gq), qo, qy, qm, k_cancel=32, what="threaded rope q")
        check_bf16(host_bits(gk), ko, ky, km, k_cancel=32, what="threaded rope k")
        zero = np.zeros((1, 1024), np.uint16)
        o_out, o_y, o_mag = oracle.ln_modulate(host_bits(x), zero, zero, want_y=True)
        check_bf16(host_bits(ln), o_out, o_y, o_mag, k_cancel=K_LN, what="threaded ln")
