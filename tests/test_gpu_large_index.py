"""GPU parity past 2^31 elements: every op on a tensor whose element offsets
leave the int32 range, checked against the oracle on sampled rows.

The bulk of each tensor is filled on the device from a seeded torch generator;
the sampled rows (the first, those around element 2^31 and the last) are
overwritten with the counter-based synthetic inputs generated on the host, and
only those rows' outputs are compared, so the oracle sees host-generated
inputs only.  Each case holds 13-20 GB on the device and frees it afterwards.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import host_bits
from tests.parity import check_bf16

pytestmark = pytest.mark.gpu

BIG = 2 ** 31
K_ROPE, K_LN = 32, 64


def sample_rows(rows, row_elems):
    """Rows to check: the first, the rows around element 2^31, the last."""
    edge = BIG // row_elems
    picks = {0, 1, edge - 1, edge, edge + 1, rows - 2, rows - 1}
    return sorted(r for r in picks if 0 <= r < rows)


def fill(t, seed):
    g = torch.Generator(device=t.device).manual_seed(seed)
    t.normal_(generator=g)
    return t


def place(big, rows_idx, small):
    """Write host rows `small` [len(rows_idx), ...] into `big` at rows_idx."""
    big[torch.tensor(rows_idx, device=big.device)] = small.to(big.device)


def test_add_rmsnorm_past_2_31_elements(nr):
    hidden = 4096
    rows = BIG // hidden + 1000
    picks = sample_rows(rows, hidden)
    dev = torch.device("cuda")
    x = fill(torch.empty(rows, hidden, dtype=torch.bfloat16, device=dev), 1)
    res = fill(torch.empty(rows, hidden, dtype=torch.bfloat16, device=dev), 2)
    xs, rs, w = synth.rmsnorm_inputs(len(picks), hidden, 61, torch.bfloat16)
    place(x, picks, xs)
    place(res, picks, rs)
    out = nr.rmsnorm(x, w.to(dev), residual=res)
    torch.cuda.synchronize()
    o_out, o_res, _ = oracle.rmsnorm(host_bits(xs), host_bits(w), residual=host_bits(rs))
    idx = torch.tensor(picks, device=dev)
    assert np.array_equal(host_bits(res[idx]), o_res), "residual not bit-exact"
    check_bf16(host_bits(out[idx]), o_out, what="add + RMSNorm past 2^31")
    del x, res, out
    torch.cuda.empty_cache()


def test_ln_modulate_and_gated_past_2_31_elements(nr):
    hidden = 3072
    rows = BIG // hidden + 700
    picks = sample_rows(rows, hidden)
    dev = torch.device("cuda")
    x = fill(torch.empty(rows, hidden, dtype=torch.bfloat16, device=dev), 3)
    xs, sh, sc = synth.ln_inputs(len(picks), hidden, 62, torch.bfloat16)
    place(x, picks, xs)
    out = nr.ln_modulate(x, sh.to(dev), sc.to(dev))
    torch.cuda.synchronize()
    idx = torch.tensor(picks, device=dev)
    o_out, o_y, o_mag = oracle.ln_modulate(host_bits(xs), host_bits(sh), host_bits(sc),
                                           want_y=True)
    check_bf16(host_bits(out[idx]), o_out, o_y, o_mag, k_cancel=K_LN, what="LN past 2^31")
    # the gated kernel on the same rows: x as the residual, a fresh y
    y = fill(torch.empty_like(x), 4)
    ys = synth.tensor(63, 21, (len(picks), hidden), torch.bfloat16)
    gate = synth.tensor(63, 22, (1, hidden), torch.bfloat16, std=0.5)
    place(y, picks, ys)
    out = nr.gated_residual_ln_modulate(x, y, gate.to(dev), sh.to(dev), sc.to(dev))
    torch.cuda.synchronize()
    g_out, g_res, g_y, g_mag = oracle.gated_ln_modulate(host_bits(xs), host_bits(ys),
                                                         host_bits(gate), host_bits(sh),
                                                         host_bits(sc), want_y=True)
    assert np.array_equal(host_bits(x[idx]), g_res), "gated residual not bit-exact"
    check_bf16(host_bits(out[idx]), g_out, g_y, g_mag, k_cancel=K_LN, what="gated past 2^31")
    del x, y, out
    torch.cuda.empty_cache()


def test_qk_norm_rope_past_2_31_elements(nr):
    hq = hk = 24
    D = 128
    tokens = BIG // (hq * D) + 500
    picks = sample_rows(tokens, hq * D)
    dev = torch.device("cuda")
    q = fill(torch.empty(tokens, hq, D, dtype=torch.bfloat16, device=dev), 5)
    k = fill(torch.empty(tokens, hk, D, dtype=torch.bfloat16, device=dev), 6)
    qs, ks, wq, wk, _ = synth.qk_inputs(len(picks), hq, hk, D, 64, torch.bfloat16,
                                         torch.float32)
    place(q, picks, qs)
    place(k, picks, ks)
    pos = torch.arange(tokens, dtype=torch.int32, device=dev)
    qo, ko = nr.qk_norm_rope(q, k, wq.to(dev), wk.to(dev), pos)
    torch.cuda.synchronize()
    idx = torch.tensor(picks, device=dev)
    ref = oracle.qk_norm_rope(host_bits(qs), host_bits(ks), host_bits(wq), host_bits(wk),
                              np.array(picks, dtype=np.int32), want_y=True)
    check_bf16(host_bits(qo[idx]), ref[0], ref[2], ref[4], k_cancel=K_ROPE, what="Q past 2^31")
    check_bf16(host_bits(ko[idx]), ref[1], ref[3], ref[5], k_cancel=K_ROPE, what="K past 2^31")
    del q, k, qo, ko
    torch.cuda.empty_cache()


@pytest.mark.parametrize("act", ["silu", "gelu"])
def test_gated_activation_past_2_31_elements(nr, act):
    inter = 12288
    rows = BIG // (2 * inter) + 300
    picks = sample_rows(rows, 2 * inter)
    dev = torch.device("cuda")
    x = fill(torch.empty(rows, 2 * inter, dtype=torch.bfloat16, device=dev), 7)
    xs = synth.silu_inputs(len(picks), inter, 65, torch.bfloat16)
    place(x, picks, xs)
    fn = nr.silu_and_mul if act == "silu" else nr.gelu_and_mul
    out = fn(x)
    torch.cuda.synchronize()
    idx = torch.tensor(picks, device=dev)
    ofn = oracle.silu_and_mul if act == "silu" else oracle.gelu_and_mul
    o_out, _ = ofn(host_bits(xs))
    check_bf16(host_bits(out[idx]), o_out, what="%s past 2^31" % act)
    del x, out
    torch.cuda.empty_cache()
