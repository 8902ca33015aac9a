"""Every entry point captured into one CUDA graph and replayed.

The kernels are launched with programmatic stream serialisation; under stream
capture those launches become graph nodes with programmatic dependencies.
Here a graph holds one call of each op, in a dependent order (the in-place
residual and the in-place Q/K feed the next replay), is replayed twice, and
every output is checked against the oracle (applied twice where state carries
over, to the GPU's own first-replay values where they are rounded results) --
a replay that read a predecessor's output early, or a launch attribute lost in
capture, would fail."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import host_bits
from tests.parity import check_bf16

pytestmark = pytest.mark.gpu


def test_all_ops_in_one_graph_replayed_twice(nr):
    bf = torch.bfloat16
    x, res, w = synth.rmsnorm_inputs(512, 4096, 71, bf)
    q, k, wq, wk, pos = synth.qk_inputs(300, 8, 4, 128, 72, bf, torch.float32, pos_start=50)
    lx, sh, sc = synth.ln_inputs(384, 3072, 73, bf)
    gres = synth.tensor(74, 1, (384, 3072), bf)
    gate = synth.tensor(74, 2, (1, 3072), bf, std=0.5)
    sx = synth.silu_inputs(64, 3 * 2048, 75, bf)

    d = {n: t.cuda() for n, t in dict(x=x, res=res, w=w, q=q, k=k, wq=wq, wk=wk, pos=pos, lx=lx,
                                      sh=sh, sc=sc, gres=gres, gate=gate, sx=sx).items()}
    out = torch.empty_like(d["x"])
    codes = torch.empty(d["x"].shape, dtype=torch.uint8, device="cuda")
    nb = torch.empty_like(d["x"])
    lout = torch.empty_like(d["lx"])
    gout = torch.empty_like(d["gres"])
    sout = torch.empty((64, 3 * 2048), dtype=bf, device="cuda")
    gelu_out = torch.empty_like(sout)

    def step():
        nr.rmsnorm(d["x"], d["w"], residual=d["res"], out=out)           # residual in place
        nr.rmsnorm_quant_fp8(out, d["w"], 0.05, codes=codes, out_bf16=nb)  # reads out
        nr.qk_norm_rope(d["q"], d["k"], d["wq"], d["wk"], d["pos"], q_out=d["q"], k_out=d["k"])
        nr.ln_modulate(d["lx"], d["sh"], d["sc"], out=lout)
        nr.gated_residual_ln_modulate(d["gres"], lout, d["gate"], d["sh"], d["sc"], out=gout)
        nr.silu_and_mul(d["sx"], out=sout)
        nr.gelu_and_mul(d["sx"], out=gelu_out)

    # warm-up outside the capture (first-call set-up in the library), on copies
    # of the tensors that the graph updates in place
    saved = {n: d[n].clone() for n in ("res", "q", "k", "gres")}
    step()
    torch.cuda.synchronize()
    for n, t in saved.items():
        d[n].copy_(t)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            step()
    # capture launches nothing: the in-place tensors still hold their inputs
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(d["res"]), host_bits(res))
    graph.replay()
    torch.cuda.synchronize()
    # Q/K after one replay: the second replay normalises and rotates these
    # rounded values again, so it is checked against the oracle applied to them
    q1, k1 = host_bits(d["q"]), host_bits(d["k"])
    graph.replay()
    torch.cuda.synchronize()
    nr.device_status()

    # oracle, twice where state carries over
    o_out, r1, _ = oracle.rmsnorm(host_bits(x), host_bits(w), residual=host_bits(res))
    o_out, r2, _ = oracle.rmsnorm(host_bits(x), host_bits(w), residual=r1)
    assert np.array_equal(host_bits(d["res"]), r2), "residual after two replays"
    check_bf16(host_bits(out), o_out, what="graph rmsnorm")
    c_ref, nb_ref, _, _ = oracle.rmsnorm_quant_fp8(host_bits(out), host_bits(w), 0.05)
    check_bf16(host_bits(nb), nb_ref, what="graph fp8 bf16 copy")
    same = host_bits(nb) == nb_ref
    assert np.array_equal(codes.cpu().numpy()[same], c_ref[same])

    for got_q, got_k, qb, kb, what in ((q1, k1, host_bits(q), host_bits(k), "replay 1"),
                                       (host_bits(d["q"]), host_bits(d["k"]), q1, k1,
                                        "replay 2")):
        r = oracle.qk_norm_rope(qb, kb, host_bits(wq), host_bits(wk), pos.numpy(), want_y=True)
        check_bf16(got_q, r[0], r[2], r[4], k_cancel=32, what="graph q, " + what)
        check_bf16(got_k, r[1], r[3], r[5], k_cancel=32, what="graph k, " + what)

    l_out, l_y, l_mag = oracle.ln_modulate(host_bits(lx), host_bits(sh), host_bits(sc),
                                           want_y=True)
    check_bf16(host_bits(lout), l_out, l_y, l_mag, k_cancel=64, what="graph ln")
    # the gated residual was updated by both replays, with the GPU's own LN output
    g1 = oracle.gated_ln_modulate(host_bits(gres), host_bits(lout), host_bits(gate),
                                  host_bits(sh), host_bits(sc), want_y=True)
    g2 = oracle.gated_ln_modulate(g1[1], host_bits(lout), host_bits(gate), host_bits(sh),
                                  host_bits(sc), want_y=True)
    assert np.array_equal(host_bits(d["gres"]), g2[1]), "gated residual after two replays"
    check_bf16(host_bits(gout), g2[0], g2[2], g2[3], k_cancel=64, what="graph gated ln")

    check_bf16(host_bits(sout), oracle.silu_and_mul(host_bits(sx))[0], what="graph silu")
    check_bf16(host_bits(gelu_out), oracle.gelu_and_mul(host_bits(sx))[0], what="graph gelu")
