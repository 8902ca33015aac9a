"""Pins for the CPU oracle: closed forms, invariants, library special cases and
exact brute force, each chosen so that a plausible slip in the oracle (a dropped
term, a wrong sign, index or operand order, a misplaced eps, a missing rounding)
fails at least one of them.  The oracle is never compared with itself here.

Sources (page, section): vllm.cpp src/vt/cuda/cuda_ops.cu -- the bf16
load/store helpers, the residual-rounding helper, the row-RMSNorm, NeoX RoPE,
fused attention-preamble and gated-activation sections; FastVideo PAN2 docs,
"Performance switches" (dit_fused_kernels: LayerNorm + modulation).
"""
import math
import os
from fractions import Fraction

import mpmath
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.parity import bf16_to_f64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(vals):
    """bf16 bits of values that are exactly representable (asserted)."""
    t = torch.tensor(vals, dtype=torch.float64)
    b = t.to(torch.bfloat16)
    assert torch.equal(b.double(), t), "value not exactly representable in bf16"
    return b.view(torch.int16).numpy().view(np.uint16)


def f32(vals):
    return np.asarray(vals, dtype=np.float32)


# --------------------------------------------------------------------------
# bf16 rounding
# --------------------------------------------------------------------------
def test_bf16_rounding_golden_cases():
    n = 0
    with open(os.path.join(GOLDEN, "bf16_rounding.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            hexval, bits, _ = line.split(None, 2)
            d = float.fromhex(hexval)
            assert oracle.bf16_round(d) == int(bits, 16), line
            n += 1
    assert n >= 12


def test_bf16_rounding_matches_torch_on_f32_values():
    """For values that are f32, rounding the double straight to bf16 must agree
    with torch's f32 -> bf16 conversion (a library round-to-nearest-even)."""
    rng = np.random.default_rng(7)
    hi = np.arange(0, 1 << 16, dtype=np.uint32)
    hi = hi[(hi & 0x7F80) != 0x7F80]  # finite values only
    lows = [0x0000, 0x7FFF, 0x8000, 0x8001, 0xFFFF]
    words = np.concatenate([(hi << 16) | np.uint32(lo) for lo in lows]
                           + [(hi << 16) | rng.integers(0, 1 << 16, hi.size).astype(np.uint32)])
    f = words.view(np.float32)
    ours = oracle.bf16_round_array(f.astype(np.float64))
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    mism = np.nonzero(ours != ref)[0]
    assert mism.size == 0, "first mismatch: f32 bits 0x%08x" % words[mism[0]]


def _nearest_bf16_exact(d: float) -> int:
    """Brute force: the bf16 pattern nearest to d in exact rational arithmetic,
    ties to the even pattern, among the patterns around torch's f32 guess."""
    guess = int(torch.tensor([d], dtype=torch.float32).to(torch.bfloat16)
                .view(torch.int16).item()) & 0xFFFF
    x = Fraction(d)
    best = None
    for b in range(max(guess - 3, 0), guess + 4):
        if ((b >> 7) & 0xFF) == 0xFF or (b & 0x8000) != (guess & 0x8000):
            continue
        v = Fraction(bf16_to_f64(np.array([b], np.uint16))[0])
        key = (abs(v - x), b & 1)
        if best is None or key < best[0]:
            best = (key, b)
    return best[1]


def _nearest_f32_exact(x: Fraction) -> Fraction:
    """Brute force: the f32 value nearest to the rational x, ties to the even
    pattern, among the five values around a guess (normal range only)."""
    guess = np.float32(float(x))
    cands = [guess]
    for _ in range(2):
        cands = ([np.nextafter(cands[0], np.float32(-np.inf), dtype=np.float32)] + cands
                 + [np.nextafter(cands[-1], np.float32(np.inf), dtype=np.float32)])
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - x),
                                     int(np.array([c], np.float32).view(np.uint32)[0]) & 1))
    return Fraction(float(best))


def test_bf16_rounding_exact_brute_force_on_doubles():
    rng = np.random.default_rng(11)
    d = rng.standard_normal(4000) * np.exp2(rng.integers(-120, 120, 4000))
    # add doubles sitting just off bf16 midpoints, where rounding via f32 would differ
    mids = bf16_to_f64(rng.integers(0x0100, 0x7E00, 500).astype(np.uint16)) * (1 + 2.0 ** -8)
    d = np.concatenate([d, mids * (1 + 2.0 ** -40), mids * (1 - 2.0 ** -40)])
    ours = oracle.bf16_round_array(d)
    for i in range(d.size):
        assert ours[i] == _nearest_bf16_exact(float(d[i])), d[i]


def test_e4m3_golden_cases():
    n = 0
    with open(os.path.join(GOLDEN, "e4m3_rounding.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            hexval, code, _ = line.split(None, 2)
            v = np.array([float.fromhex(hexval)], np.float32)
            assert oracle.e4m3_array(v)[0] == int(code, 16), line
            n += 1
    assert n >= 12


def test_e4m3_matches_torch_within_range():
    """Inside +-448 the oracle's e4m3 rounding agrees with torch's f32 ->
    float8_e4m3fn conversion (a library round-to-nearest-even)."""
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(17)
    v = np.concatenate([rng.uniform(-448, 448, 20000), rng.standard_normal(20000) * 2.0 ** -7,
                        np.arange(-448, 448.01, 1 / 64.0)]).astype(np.float32)
    ours = oracle.e4m3_array(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


# --------------------------------------------------------------------------
# residual add
# --------------------------------------------------------------------------
def _random_bf16_pairs(n, seed):
    """bf16 pairs spread over every exponent gap between the operands."""
    rng = np.random.default_rng(seed)
    a = rng.standard_normal(n) * np.exp2(rng.integers(-30, 30, n))
    b = rng.standard_normal(n) * np.exp2(rng.integers(-30, 30, n))
    ab = torch.from_numpy(a).to(torch.bfloat16)
    bb = torch.from_numpy(b).to(torch.bfloat16)
    return ab, bb


def test_residual_add_is_one_exact_rounding():
    """res <- round_bf16(x + res), the exact sum rounded once.  Checked against
    exact rational rounding, and against torch's f32 add followed by its bf16
    conversion (the GPU's evaluation: f32 keeps 24 >= 2*8+2 bits, so rounding
    through f32 first cannot change the result)."""
    xa, ra = _random_bf16_pairs(8 * 512, 3)
    x = synth.to_oracle(xa).reshape(512, 8)
    r = synth.to_oracle(ra).reshape(512, 8)
    w = bf16([1.0] * 8)
    _, res_out, _ = oracle.rmsnorm(x, w, residual=r, eps=1e-6)
    via_f32 = (xa.float() + ra.float()).to(torch.bfloat16)
    assert np.array_equal(res_out.reshape(-1), synth.to_oracle(via_f32))
    xs, rs = bf16_to_f64(x.reshape(-1)), bf16_to_f64(r.reshape(-1))
    for i in range(0, xs.size, 7):
        assert res_out.reshape(-1)[i] == _nearest_bf16_exact(float(Fraction(xs[i]) + Fraction(rs[i])))


def test_residual_add_f32_is_ieee_add():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((64, 8)) * np.exp2(rng.integers(-40, 40, (64, 8)))).astype(np.float32)
    r = (rng.standard_normal((64, 8)) * np.exp2(rng.integers(-40, 40, (64, 8)))).astype(np.float32)
    _, res_out, _ = oracle.rmsnorm(x, f32([1.0] * 8), residual=r)
    assert np.array_equal(res_out, x + r)  # numpy's f32 add is the IEEE add


def test_residual_is_rounded_before_it_is_squared():
    """x = 1, res = 2^-9 rounds to exactly 1 in bf16, so a row of such sums has
    mean square exactly 1 and, with eps = 0, out = w exactly.  Squaring the
    unrounded sum 1 + 2^-9 would give a different y."""
    x = bf16([[1.0] * 8])
    r = bf16([[2.0 ** -9] + [0.0] * 7])
    wv = [0.5, 0.75, 1.0, 1.25, 1.5, 1.75, 2.0, 2.25]
    out, res_out, y = oracle.rmsnorm(x, bf16(wv), residual=r, eps=0.0, want_y=True)
    assert np.array_equal(res_out, bf16([[1.0] * 8]))
    assert np.array_equal(y[0], np.array(wv))


# --------------------------------------------------------------------------
# RMSNorm
# --------------------------------------------------------------------------
W8 = [0.5, -0.75, 1.0, 1.25, -1.5, 1.75, 2.0, 0.125]


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_rmsnorm_constant_row_gives_w(dt):
    """A row of 2s has mean square 4; with eps = 0, out = 2/2 * w = w (catches a
    1/(h-1) mean, a wrong weight index)."""
    mk = bf16 if dt == "bf16" else f32
    _, _, y = oracle.rmsnorm(mk([[2.0] * 8] * 4), mk(W8), eps=0.0, want_y=True)
    assert np.array_equal(y, np.tile(np.array(W8), (4, 1)))


def test_rmsnorm_output_rounds_once_from_the_exact_value():
    """x = e_0 of length 8 and w = 1 give y_0 = 1/sqrt(1/8 + eps).  eps is set so
    that y_0 sits 2^-30 (relative) above the bf16 midpoint 1 + 2^-8: the single
    rounding goes up to 1 + 2^-7 (0x3f81); rounding through f32 first would land
    on the midpoint and tie down to 1.0.  Just below the midpoint it goes down."""
    x = bf16([[1.0] + [0.0] * 7])
    w = bf16([1.0] * 8)
    for target, bits in (((1 + 2.0 ** -8) * (1 + 2.0 ** -30), 0x3F81),
                         ((1 + 2.0 ** -8) * (1 - 2.0 ** -30), 0x3F80)):
        eps = 1.0 / target ** 2 - 1.0 / 8
        out, _, y = oracle.rmsnorm(x, w, eps=eps, want_y=True)
        assert abs(y[0, 0] / target - 1) < 1e-14
        assert out[0, 0] == bits


def test_rmsnorm_alternating_row():
    """[a, -a, a, -a, ...] has mean square a^2: out_j = sign_j * w_j."""
    a = 3.0
    x = bf16([[a if j % 2 == 0 else -a for j in range(8)]])
    _, _, y = oracle.rmsnorm(x, bf16(W8), eps=0.0, want_y=True)
    assert np.allclose(y[0], [w if j % 2 == 0 else -w for j, w in enumerate(W8)], rtol=0,
                       atol=1e-15)


def test_rmsnorm_eps_inside_the_sqrt():
    """Constant row c = 1 with eps = 3: inv = 1/sqrt(1 + 3) = 1/2 exactly.
    eps outside the sqrt (1/(1+3)) or added to the rms would give 1/4."""
    _, _, y = oracle.rmsnorm(bf16([[1.0] * 8]), bf16(W8), eps=3.0, want_y=True)
    assert np.array_equal(y[0], np.array(W8) / 2)


def test_rmsnorm_gemma_adds_one_to_w():
    """gemma with w equals plain with w + 1 (values chosen so w + 1 is exact)."""
    xs, _, _ = synth.rmsnorm_inputs(6, 64, 9, torch.bfloat16, residual=False)
    x = synth.to_oracle(xs)
    w = np.arange(64) / 64.0 - 0.5
    o1, _, y1 = oracle.rmsnorm(x, bf16(list(w)), gemma=True, want_y=True)
    o2, _, y2 = oracle.rmsnorm(x, bf16(list(w + 1.0)), gemma=False, want_y=True)
    assert np.array_equal(o1, o2) and np.array_equal(y1, y2)
    o3, _, _ = oracle.rmsnorm(x, bf16(list(w)), gemma=False)
    assert not np.array_equal(o1, o3)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_rmsnorm_zero_residual_reduces_to_plain(dtype):
    x, _, w = synth.rmsnorm_inputs(16, 96, 12, dtype, residual=False)
    zero = torch.zeros_like(x)
    o1, r1, y1 = oracle.rmsnorm(synth.to_oracle(x), synth.to_oracle(w),
                                residual=synth.to_oracle(zero), want_y=True)
    o2, _, y2 = oracle.rmsnorm(synth.to_oracle(x), synth.to_oracle(w), want_y=True)
    assert np.array_equal(o1, o2) and np.array_equal(y1, y2)
    assert np.array_equal(r1, synth.to_oracle(x))


def test_rmsnorm_scale_invariance():
    """With eps = 0, RMSNorm(4x) = RMSNorm(x) exactly (power-of-two scaling)."""
    x, _, w = synth.rmsnorm_inputs(8, 40, 13, torch.float32, residual=False)
    _, _, y1 = oracle.rmsnorm(synth.to_oracle(x), synth.to_oracle(w), eps=0.0, want_y=True)
    _, _, y2 = oracle.rmsnorm(synth.to_oracle(x * 4), synth.to_oracle(w), eps=0.0, want_y=True)
    assert np.allclose(y1, y2, rtol=1e-15, atol=0)


def test_rmsnorm_brute_force_4x8():
    """4x8 random rows against a 50-digit evaluation of sum/sqrt, element by element."""
    mpmath.mp.dps = 50
    xt, rt, wt = synth.rmsnorm_inputs(4, 8, 21, torch.bfloat16)
    x, r, w = synth.to_oracle(xt), synth.to_oracle(rt), synth.to_oracle(wt)
    out, res_out, y = oracle.rmsnorm(x, w, residual=r, eps=1e-6, gemma=True, want_y=True)
    xv, rv, wv = bf16_to_f64(x), bf16_to_f64(r), bf16_to_f64(w)
    for i in range(4):
        v = [_nearest_bf16_exact(float(Fraction(xv[i, j]) + Fraction(rv[i, j]))) for j in range(8)]
        assert list(res_out[i]) == v
        vals = [mpmath.mpf(float(bf16_to_f64(np.array([b], np.uint16))[0])) for b in v]
        ms = sum(t * t for t in vals) / 8
        inv = 1 / mpmath.sqrt(ms + mpmath.mpf(1e-6))
        for j in range(8):
            exact = vals[j] * inv * (mpmath.mpf(float(wv[j])) + 1)
            assert abs(y[i, j] - float(exact)) <= 4e-16 * abs(float(exact))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_rmsnorm_quant_fp8_composition(dtype):
    """The fused op equals RMSNorm (pinned above) rounded to bf16, then the
    e4m3 code of the f32 product with 1/scale (numpy f32 arithmetic and
    torch's e4m3 conversion, for codes inside the range)."""
    x, res, w = synth.rmsnorm_inputs(8, 256, 14, dtype)
    scale = 0.0123
    codes, nb, r_out, y = oracle.rmsnorm_quant_fp8(synth.to_oracle(x), synth.to_oracle(w), scale,
                                                   residual=synth.to_oracle(res), gemma=True,
                                                   want_y=True)
    o, r2, y2 = oracle.rmsnorm(synth.to_oracle(x), synth.to_oracle(w),
                               residual=synth.to_oracle(res), gemma=True, want_y=True)
    assert np.array_equal(r_out, r2) and np.array_equal(y, y2)
    assert np.array_equal(nb, oracle.bf16_round_array(y2))
    t = bf16_to_f64(nb).astype(np.float32) * (np.float32(1.0) / np.float32(scale))
    assert np.array_equal(codes, oracle.e4m3_array(t))
    if hasattr(torch, "float8_e4m3fn"):
        inside = np.abs(t) <= 448
        ref = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(codes[inside], ref[inside])
        assert inside.mean() > 0.5 and (~inside).any()  # both regimes exercised
        assert np.all(codes[~inside] & 0x7F == 0x7E)


# --------------------------------------------------------------------------
# Q/K RMSNorm + NeoX RoPE
# --------------------------------------------------------------------------
def _qk_small(tokens=3, hq=2, hk=1, D=16, seed=31):
    q, k, wq, wk, pos = synth.qk_inputs(tokens, hq, hk, D, seed, torch.bfloat16, torch.float32)
    return (synth.to_oracle(q), synth.to_oracle(k), synth.to_oracle(wq), synth.to_oracle(wk),
            pos.numpy())


def test_rope_position_zero_is_the_plain_head_norm():
    """At position 0 every angle is 0: the output is the per-head RMSNorm
    (checked against the separately pinned RMSNorm of the same head rows)."""
    q, k, wq, wk, _ = _qk_small(tokens=4, hq=3, hk=2, D=32)
    wqb = synth.to_oracle(torch.from_numpy(wq).to(torch.bfloat16))
    wkb = synth.to_oracle(torch.from_numpy(wk).to(torch.bfloat16))
    qo, ko, qy, ky, _, _ = oracle.qk_norm_rope(q, k, wqb, wkb, np.zeros(4, np.int32), want_y=True)
    ro, _, ry = oracle.rmsnorm(q.reshape(-1, 32), wqb, want_y=True)
    assert np.array_equal(qo.reshape(-1, 32), ro) and np.array_equal(qy.reshape(-1, 32), ry)
    ro, _, ry = oracle.rmsnorm(k.reshape(-1, 32), wkb, want_y=True)
    assert np.array_equal(ko.reshape(-1, 32), ro) and np.array_equal(ky.reshape(-1, 32), ry)


def test_rope_preserves_each_pair_norm():
    q, k, wq, wk, _ = _qk_small(tokens=5, hq=2, hk=2, D=64)
    pos = np.array([0, 1, 77, 4096, 26597], np.int32)
    _, _, qy, ky, _, _ = oracle.qk_norm_rope(q, k, wq, wk, pos, want_y=True)
    _, _, q0, k0, _, _ = oracle.qk_norm_rope(q, k, wq, wk, np.zeros(5, np.int32), want_y=True)
    for yr, y0 in ((qy, q0), (ky, k0)):
        a = yr[..., :32] ** 2 + yr[..., 32:] ** 2
        b = y0[..., :32] ** 2 + y0[..., 32:] ** 2
        assert np.allclose(a, b, rtol=1e-12, atol=0)


def _onehot_case(idx, p, D=128, theta=10000.0, wq=None):
    """One q head whose only nonzero element is at idx (value 1), eps = 0, so the
    normed vector is sqrt(D) * w_idx at idx."""
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, idx] = 1.0
    q = synth.to_oracle(torch.from_numpy(q).to(torch.bfloat16))
    k = q.copy()
    if wq is None:
        wq = (1.0 + np.arange(D) / 256.0).astype(np.float32)  # w_i != w_{i+D/2}
    _, _, qy, _, _, _ = oracle.qk_norm_rope(q, k, wq, wq, np.array([p], np.int32), eps=0.0,
                                            theta=theta, want_y=True)
    return qy[0, 0], wq


def test_rope_rotation_direction_and_pairing():
    """One-hot at i = 0 (frequency 1) and position 1: the pair (0, 64) becomes
    n*(cos 1, sin 1) -- rotate-half pairing, positive sine on the second half,
    weight of the first element (norm before rotation); all else stays 0."""
    y, w = _onehot_case(0, 1)
    n = math.sqrt(128) * float(w[0])
    assert abs(y[0] - n * math.cos(1.0)) < 1e-13 and abs(y[64] - n * math.sin(1.0)) < 1e-13
    rest = np.delete(y, [0, 64])
    assert np.all(rest == 0)


def test_rope_second_half_rotates_the_other_way():
    """One-hot at 64 + 5: y_5 = -n sin(a), y_69 = n cos(a) with a = p * theta^(-10/128)."""
    p = 3
    y, w = _onehot_case(69, p)
    n = math.sqrt(128) * float(w[69])
    a = p * 10000.0 ** (-10 / 128)
    assert abs(y[5] + n * math.sin(a)) < 1e-13 and abs(y[69] - n * math.cos(a)) < 1e-13


def test_rope_frequency_exponent():
    """i = 32 of D = 128: freq = 10000^(-64/128) = 1/100, so position 100 turns
    the pair (32, 96) by exactly 1 radian; theta = 500, i = 16: freq = 500^(-1/4)."""
    y, w = _onehot_case(32, 100)
    n = math.sqrt(128) * float(w[32])
    assert abs(y[32] - n * math.cos(1.0)) < 1e-12 and abs(y[96] - n * math.sin(1.0)) < 1e-12
    y, w = _onehot_case(16, 7, theta=500.0)
    n = math.sqrt(128) * float(w[16])
    a = 7 * 500.0 ** -0.25
    assert abs(y[16] - n * math.cos(a)) < 1e-12 and abs(y[80] - n * math.sin(a)) < 1e-12


def test_rope_q_and_k_use_their_own_weights_and_heads():
    """Two q heads and one k head with one-hot inputs at distinct indices and
    distinct weights: each output is the closed form with its own tensor's weight."""
    D = 16
    q = np.zeros((2, 2, D), np.float32)
    k = np.zeros((2, 1, D), np.float32)
    q[:, 0, 1] = 1.0
    q[:, 1, 2] = 1.0
    k[:, 0, 3] = 1.0
    qb = synth.to_oracle(torch.from_numpy(q).to(torch.bfloat16))
    kb = synth.to_oracle(torch.from_numpy(k).to(torch.bfloat16))
    wq = (1.0 + np.arange(D) / 32.0).astype(np.float32)
    wk = (2.0 - np.arange(D) / 32.0).astype(np.float32)
    pos = np.array([5, 9], np.int32)
    _, _, qy, ky, _, _ = oracle.qk_norm_rope(qb, kb, wq, wk, pos, eps=0.0, theta=10.0, want_y=True)
    s = math.sqrt(D)
    for t, p in enumerate(pos):
        for (y, i, wv) in ((qy[t, 0], 1, wq), (qy[t, 1], 2, wq), (ky[t, 0], 3, wk)):
            a = p * 10.0 ** (-2 * i / D)
            assert abs(y[i] - s * float(wv[i]) * math.cos(a)) < 1e-12
            assert abs(y[i + D // 2] - s * float(wv[i]) * math.sin(a)) < 1e-12


def test_rope_relative_position_invariance():
    """<R(p+s) q, R(p'+s) k> = <R(p) q, R(p') k> for every head pair."""
    q, k, wq, wk, _ = _qk_small(tokens=2, hq=2, hk=2, D=32, seed=41)

    def dots(p0, p1):
        _, _, qy, ky, _, _ = oracle.qk_norm_rope(q[:1], k[1:], wq, wk, np.array([p0], np.int32),
                                                 want_y=True)
        _, _, _, ky1, _, _ = oracle.qk_norm_rope(q[:1], k[1:], wq, wk, np.array([p1], np.int32),
                                                 want_y=True)
        return np.einsum("hd,gd->hg", qy[0], ky1[0])

    base = dots(10, 3)
    for s in (1, 250, 9000):
        assert np.allclose(dots(10 + s, 3 + s), base, rtol=0, atol=1e-9)


def test_rope_strided_input_matches_dense():
    """q/k given as views into a wider row (token stride > heads*D)."""
    q, k, wq, wk, pos = _qk_small(tokens=3, hq=2, hk=2, D=16)
    wide = np.zeros((3, 7, 16), np.uint16)
    wide[:, 1:3] = q
    wide[:, 4:6] = k
    a = oracle.qk_norm_rope(q, k, wq, wk, pos)
    b = oracle.qk_norm_rope(wide[:, 1:3], wide[:, 4:6], wq, wk, pos)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_rope_brute_force_4_tokens():
    """4 tokens x 1 head x 8 dims (pairs (i, i+4)) against a 50-digit evaluation."""
    mpmath.mp.dps = 50
    q, k, wq, wk, _ = _qk_small(tokens=4, hq=1, hk=1, D=8, seed=51)
    pos = np.array([0, 3, 1000, 26597], np.int32)
    _, _, qy, _, _, _ = oracle.qk_norm_rope(q, k, wq, wk, pos, eps=1e-6, theta=10000.0,
                                            want_y=True)
    qv = bf16_to_f64(q)
    for t in range(4):
        v = [mpmath.mpf(float(a)) for a in qv[t, 0]]
        inv = 1 / mpmath.sqrt(sum(a * a for a in v) / 8 + mpmath.mpf(1e-6))
        n = [v[j] * inv * mpmath.mpf(float(wq[j])) for j in range(8)]
        for i in range(4):
            # the frequency is the double pow result (the method's own rounding)
            f = mpmath.mpf(10000.0 ** (-2.0 * i / 8))
            a = int(pos[t]) * f
            e0 = n[i] * mpmath.cos(a) - n[i + 4] * mpmath.sin(a)
            e1 = n[i] * mpmath.sin(a) + n[i + 4] * mpmath.cos(a)
            assert abs(qy[t, 0, i] - float(e0)) < 1e-11
            assert abs(qy[t, 0, i + 4] - float(e1)) < 1e-11


# --------------------------------------------------------------------------
# RoPE variants
# --------------------------------------------------------------------------
def test_rope_ex_defaults_equal_the_plain_rope():
    q, k, wq, wk, _ = _qk_small(tokens=4, hq=2, hk=2, D=64, seed=91)
    pos = np.array([0, 5, 300, 26000], np.int32)
    a = oracle.qk_norm_rope(q, k, wq, wk, pos, want_y=True)
    b = oracle.qk_norm_rope_ex(q, k, wq, wk, pos, want_y=True)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("variant", [{}, {"rotary_dim": 32}, {"interleaved": True}])
def test_rope_gemma_adds_one_to_both_weights(variant):
    """gemma uses w + 1 for the head norm (fused attention-preamble section): with
    weights whose w + 1 is exact, gemma on w equals gemma off on w + 1, for Q
    and for K, in the plain kernel and the variants."""
    q, k, _, _, _ = _qk_small(tokens=3, hq=2, hk=2, D=64, seed=94)
    wq = ((np.arange(64) % 7) - 3).astype(np.float32) / 8
    wk = ((np.arange(64) % 5) - 2).astype(np.float32) / 4
    pos = np.array([0, 9, 4000], np.int32)
    fn = oracle.qk_norm_rope_ex if variant else oracle.qk_norm_rope
    a = fn(q, k, wq, wk, pos, gemma=True, want_y=True, **variant)
    b = fn(q, k, wq + 1, wk + 1, pos, gemma=False, want_y=True, **variant)
    for x, y in zip(a[:4], b[:4]):
        assert np.array_equal(x, y)
    c = fn(q, k, wq, wk, pos, gemma=False, want_y=True, **variant)
    assert not np.array_equal(a[2], c[2]) and not np.array_equal(a[3], c[3])


def _onehot_ex(idx, p, D=128, **kw):
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, idx] = 1.0
    q = synth.to_oracle(torch.from_numpy(q).to(torch.bfloat16))
    w = (1.0 + np.arange(D) / 256.0).astype(np.float32)
    pos = kw.pop("pos", np.array([p], np.int32))
    _, _, qy, _, _, _ = oracle.qk_norm_rope_ex(q, q.copy(), w, w, pos, eps=0.0, want_y=True, **kw)
    return qy[0, 0], math.sqrt(D) * float(w[idx])


def test_rope_partial_rotary_pairs_and_unrotated_tail():
    """rot = 64 of D = 128: pair (i, i + 32) with freq theta^(-2i/64); elements
    64..127 keep their normed value whatever the position."""
    y, n = _onehot_ex(0, 1, rotary_dim=64)
    assert abs(y[0] - n * math.cos(1.0)) < 1e-12 and abs(y[32] - n * math.sin(1.0)) < 1e-12
    assert y[64] == 0.0
    y, n = _onehot_ex(16, 100, rotary_dim=64)  # 10000^(-32/64) = 1/100
    assert abs(y[16] - n * math.cos(1.0)) < 1e-12 and abs(y[48] - n * math.sin(1.0)) < 1e-12
    y, n = _onehot_ex(100, 12345, rotary_dim=64)
    assert abs(y[100] - n) < 1e-12 and np.count_nonzero(y) == 1
    q, k, wq, wk, _ = _qk_small(tokens=3, hq=2, hk=1, D=64, seed=92)
    wb = synth.to_oracle(torch.from_numpy(wq).to(torch.bfloat16))
    out = oracle.qk_norm_rope_ex(q, k, wb, wb, np.array([7, 70, 700], np.int32), rotary_dim=32,
                                 want_y=True)
    ro, _, ry = oracle.rmsnorm(q.reshape(-1, 64), wb, want_y=True)
    assert np.array_equal(out[2].reshape(-1, 64)[:, 32:], ry[:, 32:])
    # the stored tail too: the rounded normed value, not the input
    assert np.array_equal(out[0].reshape(-1, 64)[:, 32:], ro[:, 32:])


def test_rope_interleaved_pairs():
    """GPT-J pairing: (2i, 2i + 1), freq theta^(-2i/rot)."""
    y, n = _onehot_ex(0, 1, interleaved=True)
    assert abs(y[0] - n * math.cos(1.0)) < 1e-12 and abs(y[1] - n * math.sin(1.0)) < 1e-12
    y, n = _onehot_ex(65, 100, interleaved=True)  # pair 32 (odd member): freq 1/100
    assert abs(y[64] + n * math.sin(1.0)) < 1e-12 and abs(y[65] - n * math.cos(1.0)) < 1e-12


def test_rope_llama3_rescale_regions():
    """orig 8192, low 1, high 4, factor 8: wavelengths below 2048 keep f, above
    8192 divide f by 8, in between interpolate with s = (8192/L - 1)/3."""
    D, theta = 128, 500000.0
    f = [theta ** (-2 * i / D) for i in range(D // 2)]
    L = [2 * math.pi / x for x in f]
    i_hi = max(i for i in range(64) if L[i] < 2048)
    i_lo = min(i for i in range(64) if L[i] > 8192)
    i_mid = next(i for i in range(64) if 2048 <= L[i] <= 8192)
    for i, expect in ((i_hi, f[i_hi]), (i_lo, f[i_lo] / 8),
                      (i_mid, (1 - (8192 / L[i_mid] - 1) / 3) * f[i_mid] / 8
                       + (8192 / L[i_mid] - 1) / 3 * f[i_mid])):
        p = 3
        y, n = _onehot_ex(i, p, theta=theta, llama3=(8.0, 1.0, 4.0, 8192.0))
        assert abs(y[i] - n * math.cos(p * expect)) < 1e-12
        assert abs(y[i + 64] - n * math.sin(p * expect)) < 1e-12
    y1, _ = _onehot_ex(5, 77, theta=theta, llama3=(1.0, 1.0, 4.0, 8192.0))  # factor 1: no change
    y0, _ = _onehot_ex(5, 77, theta=theta)
    assert np.allclose(y1, y0, rtol=0, atol=1e-15)


@pytest.mark.parametrize("interleaved", [False, True])
def test_mrope_axis_selection(interleaved):
    """Three equal position rows reproduce plain RoPE; changing only the h row
    changes exactly the pairs of axis h."""
    D, T = 32, 3  # 16 pairs
    sec = (8, 3, 5)
    q, k, wq, wk, _ = _qk_small(tokens=T, hq=1, hk=1, D=D, seed=93)
    base = np.array([11, 222, 3333], np.int32)
    same = np.stack([base, base, base])
    a = oracle.qk_norm_rope(q, k, wq, wk, base, want_y=True)
    b = oracle.qk_norm_rope_ex(q, k, wq, wk, same, mrope_sections=sec,
                               mrope_interleaved=interleaved, want_y=True)
    assert np.array_equal(a[2], b[2])
    moved = same.copy()
    moved[1] += 1000
    c = oracle.qk_norm_rope_ex(q, k, wq, wk, moved, mrope_sections=sec,
                               mrope_interleaved=interleaved, want_y=True)
    if interleaved:
        h_pairs = [i for i in range(16) if i % 3 == 1 and i // 3 < sec[1]]
    else:
        h_pairs = list(range(sec[0], sec[0] + sec[1]))
    changed = [i for i in range(16) if not np.allclose(c[2][..., i], b[2][..., i], atol=1e-14)]
    assert changed == h_pairs
    # Moving one axis row at a time: each axis owns as many frequency pairs as
    # its section says, and the three sets split the pairs between them.
    owned = []
    for axis in range(3):
        moved = same.copy()
        moved[axis] += 1000
        c = oracle.qk_norm_rope_ex(q, k, wq, wk, moved, mrope_sections=sec,
                                   mrope_interleaved=interleaved, want_y=True)
        owned.append({i for i in range(16)
                      if not np.allclose(c[2][..., i], b[2][..., i], atol=1e-14)})
    assert [len(s) for s in owned] == list(sec)
    assert set().union(*owned) == set(range(16))


# --------------------------------------------------------------------------
# LayerNorm + adaLN modulation
# --------------------------------------------------------------------------
def test_ln_row_1_to_8_closed_form():
    """x = 1..8: mean 4.5, biased variance 5.25; with eps = 1, sqrt(6.25) = 2.5,
    so xhat_j = (j - 4.5) / 2.5 (an unbiased variance or eps outside the sqrt
    would differ)."""
    x = bf16([[float(j) for j in range(1, 9)]])
    zero = bf16([0.0] * 8)
    _, y, _ = oracle.ln_modulate(x, zero, zero, eps=1.0, want_y=True)
    assert np.allclose(y[0], (np.arange(1, 9) - 4.5) / 2.5, rtol=0, atol=1e-15)
    _, y, _ = oracle.ln_modulate(x, zero, zero, eps=0.0, want_y=True)
    assert np.allclose(y[0], (np.arange(1, 9) - 4.5) / math.sqrt(5.25), rtol=0, atol=1e-15)


def test_ln_rows_have_mean_zero_and_variance_var_over_var_plus_eps():
    xt, _, _ = synth.ln_inputs(32, 3072, 61, torch.bfloat16)
    x = synth.to_oracle(xt)
    zero = bf16([0.0] * 3072)
    eps = 1e-2
    _, y, _ = oracle.ln_modulate(x, zero, zero, eps=eps, want_y=True)
    xv = bf16_to_f64(x)
    var = xv.var(axis=1)
    assert np.all(np.abs(y.mean(axis=1)) < 1e-12)
    assert np.allclose(y.var(axis=1), var / (var + eps), rtol=1e-12, atol=0)


def test_ln_scale_minus_one_gives_shift_and_constant_row_gives_shift():
    xt, st, _ = synth.ln_inputs(4, 64, 62, torch.bfloat16, samples=2)
    x, shift = synth.to_oracle(xt), synth.to_oracle(st)
    minus1 = bf16([[-1.0] * 64] * 2)
    out, y, _ = oracle.ln_modulate(x, shift, minus1, rows_per_sample=2, want_y=True)
    assert np.array_equal(out, shift[[0, 0, 1, 1]])  # row r uses sample r // 2
    const = bf16([[0.75] * 64] * 4)
    scale = synth.to_oracle(synth.tensor(62, 99, (2, 64), torch.bfloat16, std=0.1))
    out, y, _ = oracle.ln_modulate(const, shift, scale, rows_per_sample=2, want_y=True)
    assert np.array_equal(out, shift[[0, 0, 1, 1]])


def test_ln_zero_modulation_is_plain_ln_and_shift_invariant():
    """scale = shift = 0 gives plain LN: odd in x and invariant to adding a
    constant (to 1e-12), with the mean/variance pins above fixing its values."""
    xt, _, _ = synth.ln_inputs(8, 256, 63, torch.float32)
    x = synth.to_oracle(xt)
    zero = f32([0.0] * 256)
    _, y, _ = oracle.ln_modulate(x, zero, zero, want_y=True)
    _, yn, _ = oracle.ln_modulate(-x, zero, zero, want_y=True)
    _, ys, _ = oracle.ln_modulate(x + np.float32(8.0), zero, zero, want_y=True)
    assert np.array_equal(yn, -y)
    assert np.allclose(ys, y, rtol=0, atol=1e-5)  # x + 8 is rounded to f32 once


def test_ln_modulation_uses_one_plus_scale():
    """y = xhat * (1 + scale) + shift: with scale = 1, shift = 0.5 the result is
    2 * xhat + 0.5 (scale used alone would give xhat + 0.5)."""
    x = bf16([[float(j) for j in range(1, 9)]])
    _, y, _ = oracle.ln_modulate(x, bf16([0.5] * 8), bf16([1.0] * 8), eps=1.0, want_y=True)
    assert np.allclose(y[0], 2 * (np.arange(1, 9) - 4.5) / 2.5 + 0.5, rtol=0, atol=1e-15)


# --------------------------------------------------------------------------
# gated residual + LayerNorm + modulation
# --------------------------------------------------------------------------
def _gated_inputs(rows, hidden, seed, samples=1, dtype=torch.bfloat16):
    res = synth.tensor(seed, 20, (rows, hidden), dtype)
    y = synth.tensor(seed, 21, (rows, hidden), dtype)
    gate = synth.tensor(seed, 22, (samples, hidden), dtype, std=0.5)
    shift = synth.tensor(seed, 23, (samples, hidden), dtype, std=0.1)
    scale = synth.tensor(seed, 24, (samples, hidden), dtype, std=0.1)
    return [synth.to_oracle(t) for t in (res, y, gate, shift, scale)]


def test_gated_zero_gate_is_plain_ln_modulate():
    res, y, gate, shift, scale = _gated_inputs(6, 64, 81)
    zero = np.zeros_like(gate)
    out, res_out, yv, _ = oracle.gated_ln_modulate(res, y, zero, shift, scale, want_y=True)
    assert np.array_equal(res_out, res)
    o2, y2, _ = oracle.ln_modulate(res, shift, scale, want_y=True)
    assert np.array_equal(out, o2) and np.array_equal(yv, y2)


def test_gated_unit_gate_is_the_residual_add():
    """gate = 1: the residual update is the plain residual add (pinned above)."""
    res, y, gate, shift, scale = _gated_inputs(6, 64, 82)
    one = bf16([[1.0] * 64])
    out, res_out, _, _ = oracle.gated_ln_modulate(res, y, one, shift, scale)
    _, r2, _ = oracle.rmsnorm(y, bf16([1.0] * 64), residual=res)
    assert np.array_equal(res_out, r2)
    # and the LayerNorm + modulation is taken of the updated residual
    o2, _, _ = oracle.ln_modulate(r2, shift, scale, want_y=True)
    assert np.array_equal(out, o2)


def test_gated_residual_is_one_exact_rounding():
    """round(r + g*y) against exact rational arithmetic, over wide exponent gaps."""
    rng = np.random.default_rng(83)
    n = 16 * 64

    def spread(seed_shift):
        a = rng.standard_normal(n) * np.exp2(rng.integers(-20, 20, n))
        return torch.from_numpy(a).to(torch.bfloat16)

    r, g, yy = spread(0), spread(1), spread(2)
    ro, go, yo = (synth.to_oracle(t) for t in (r, g, yy))
    zero = np.zeros((1, 64), np.uint16)
    for i in range(16):
        sl = slice(i * 64, (i + 1) * 64)
        _, res_out, _, _ = oracle.gated_ln_modulate(ro[sl].reshape(1, 64), yo[sl].reshape(1, 64),
                                                    go[sl].reshape(1, 64), zero, zero)
        rv, gv, yv = (bf16_to_f64(a[sl]) for a in (ro, go, yo))
        for j in range(0, 64, 3):
            exact = Fraction(rv[j]) + Fraction(gv[j]) * Fraction(yv[j])
            assert res_out[0, j] == _nearest_bf16_exact(float(exact)) or \
                bf16_to_f64(np.array([res_out[0, j]], np.uint16))[0] == float(exact)


def test_gated_residual_rounds_exactly_at_f32_midpoints():
    """g*y an exact bf16 midpoint (1.75 * 37/64 = 1 + 3*2^-8) plus a tiny r:
    the exact sum is just off the midpoint, so the single rounding goes the
    way r points (an f32 sum would land on the midpoint and tie to even)."""
    g, yv = bf16([[1.75, 1.75]]), bf16([[37 / 64, 37 / 64]])
    r = bf16([[2.0 ** -25, -(2.0 ** -25)]])
    zero = bf16([[0.0, 0.0]])
    _, res_out, _, _ = oracle.gated_ln_modulate(r, yv, g, zero, zero)
    mid = 1 + 3 * 2.0 ** -8
    for j in range(2):
        exact = Fraction(mid) + Fraction(bf16_to_f64(r)[0, j])
        assert res_out[0, j] == _nearest_bf16_exact(float(exact))
    assert list(res_out[0]) == [0x3F82, 0x3F81]


def test_gated_f32_residual_rounds_once_below_a_midpoint():
    """f32: r = 1 + 2^-23, g = 1 - 2^-23, y = 2^-24 (1 + 2^-23).  The exact
    r + g*y is 1 + 2^-23 + 2^-24 - 2^-70, just below the midpoint between
    1 + 2^-23 and 1 + 2^-22, so the one rounding gives 1 + 2^-23 (0x3f800001).
    Rounding the sum to double first lands on the midpoint, which then ties to
    even (0x3f800002): the double rounding this pin rules out."""
    r = f32([[1 + 2.0 ** -23, -(1 + 2.0 ** -23)]])
    g = f32([[1 - 2.0 ** -23, 1 - 2.0 ** -23]])
    yv = f32([[2.0 ** -24 * (1 + 2.0 ** -23), -(2.0 ** -24 * (1 + 2.0 ** -23))]])
    zero = f32([[0.0, 0.0]])
    _, res_out, _, _ = oracle.gated_ln_modulate(r, yv, g, zero, zero)
    assert list(res_out.view(np.uint32)[0]) == [0x3F800001, 0xBF800001]


def test_gated_f32_residual_is_one_exact_rounding():
    """f32 round(r + g*y) against exact rational arithmetic, with g*y placed
    near the f32 rounding midpoints of r (where a second rounding would show)
    and over wide exponent gaps."""
    rng = np.random.default_rng(84)
    rows, hidden = 8, 64
    r = (rng.standard_normal((rows, hidden)) * np.exp2(rng.integers(-8, 8, (rows, hidden))))
    r = r.astype(np.float32)
    g = (1 + rng.integers(-2 ** 20, 2 ** 20, (rows, hidden)) * 2.0 ** -23).astype(np.float32)
    # y near half an f32 ulp of r (divided by g), nudged by a few ulps of y
    half_ulp = np.spacing(np.abs(r)).astype(np.float64) / 2
    y = (half_ulp / g.astype(np.float64)).astype(np.float32)
    y = (y * (1 + rng.integers(-3, 4, (rows, hidden)) * 2.0 ** -23)).astype(np.float32)
    y[rows // 2:] = (rng.standard_normal((rows - rows // 2, hidden))
                     * np.exp2(rng.integers(-30, 10, (rows - rows // 2, hidden)))).astype(np.float32)
    y *= np.where(rng.random((rows, hidden)) < 0.5, -1, 1).astype(np.float32)
    zero = np.zeros((1, hidden), np.float32)
    for i in range(rows):
        _, res_out, _, _ = oracle.gated_ln_modulate(r[i:i + 1], y[i:i + 1], g[i:i + 1], zero, zero)
        for j in range(hidden):
            exact = Fraction(float(r[i, j])) + Fraction(float(g[i, j])) * Fraction(float(y[i, j]))
            assert Fraction(float(res_out[0, j])) == _nearest_f32_exact(exact), (i, j)


def test_gated_per_sample_gate_rows():
    """Row r uses gate row r // rows_per_sample: with y = 1 and residual = 0
    the updated residual is the gate row itself."""
    res = np.zeros((4, 8), np.uint16)
    y = bf16([[1.0] * 8] * 4)
    gate = bf16([[0.5] * 8, [-2.0] * 8])
    zero = np.zeros((2, 8), np.uint16)
    _, res_out, _, _ = oracle.gated_ln_modulate(res, y, gate, zero, zero, rows_per_sample=2)
    assert np.array_equal(res_out, gate[[0, 0, 1, 1]])


# --------------------------------------------------------------------------
# silu_and_mul
# --------------------------------------------------------------------------
def test_silu_closed_forms_and_operand_order():
    """Row layout [gate | up].  silu(0) = 0; up = 0 gives 0; up = 1 gives
    silu(gate); silu(ln 3) = (3/4) ln 3 (with e^{+a} it would be ln3/4)."""
    ln3 = math.log(3.0)
    a = [0.0, ln3, -2.0, 40.0]
    x = np.array([a + [1.0, 1.0, 1.0, 1.0], a + [0.0, 0.0, 0.0, 0.0]], np.float32)
    out, y = oracle.silu_and_mul(x, want_y=True)
    assert y[0, 0] == 0.0
    # the stored gate is ln 3 rounded to f32 (off by < 6e-8; silu' < 1 there)
    assert abs(y[0, 1] - 0.75 * ln3) < 1e-7
    assert abs(y[0, 2] - (-2.0 / (1 + math.e ** 2))) < 1e-15
    assert abs(y[0, 3] - 40.0 * (1 - math.exp(-40.0))) < 1e-12
    assert np.all(y[1] == 0.0)


def test_silu_odd_part_identity():
    """silu(a) - silu(-a) = a for every a (catches a sign slip in the exponent)."""
    g = synth.tensor(71, 0, (1, 64), torch.float32).numpy()
    ones = np.ones_like(g)
    _, yp = oracle.silu_and_mul(np.concatenate([g, ones], axis=1), want_y=True)
    _, ym = oracle.silu_and_mul(np.concatenate([-g, ones], axis=1), want_y=True)
    assert np.allclose(yp - ym, g.astype(np.float64), rtol=1e-15, atol=1e-15)


def test_silu_up_multiplies():
    """out is linear in up: doubling the up half doubles y exactly."""
    x = synth.tensor(72, 0, (3, 32), torch.float32).numpy()
    x2 = x.copy()
    x2[:, 16:] *= 2
    _, y1 = oracle.silu_and_mul(x, want_y=True)
    _, y2 = oracle.silu_and_mul(x2, want_y=True)
    assert np.array_equal(y2, 2 * y1)


# --------------------------------------------------------------------------
# gelu_and_mul (tanh GELU)
# --------------------------------------------------------------------------
def test_gelu_matches_torch_tanh_gelu_and_operand_order():
    """up = 1: y is torch's tanh-approximated GELU (float64, a library routine);
    up = 0: y = 0; doubling up doubles y."""
    g = synth.tensor(73, 0, (2, 64), torch.float32)
    x = torch.cat([g, torch.ones_like(g)], dim=1)
    _, y = oracle.gelu_and_mul(synth.to_oracle(x), want_y=True)
    ref = torch.nn.functional.gelu(g.double(), approximate="tanh").numpy()
    assert np.allclose(y, ref, rtol=1e-14, atol=1e-300)
    x0 = torch.cat([g, torch.zeros_like(g)], dim=1)
    _, y0 = oracle.gelu_and_mul(synth.to_oracle(x0), want_y=True)
    assert np.all(y0 == 0)
    x2 = torch.cat([g, 2 * torch.ones_like(g)], dim=1)
    _, y2 = oracle.gelu_and_mul(synth.to_oracle(x2), want_y=True)
    assert np.array_equal(y2, 2 * y)


def test_gelu_against_150_digit_evaluation():
    """Gates from -12 to 12, where for strongly negative gates 1 + tanh(z) is
    below double's resolution near -1 (down to 1e-71 at a = -12): y within
    1e-13 (relative) of the tanh formula evaluated with 150 significant
    digits, enough to resolve 1 + tanh(z) there."""
    mpmath.mp.dps = 150
    g = np.concatenate([np.linspace(-12, 12, 97), [-0.5, 1e-30, -1e-30, 0.0]])[None, :]
    g = g.astype(np.float32)
    x = np.concatenate([g, np.full_like(g, 1.5)], axis=1)
    _, y = oracle.gelu_and_mul(x, want_y=True)
    k = mpmath.sqrt(2 / mpmath.pi)
    for a, got in zip(g[0], y[0]):
        am = mpmath.mpf(float(a))
        ref = mpmath.mpf("0.5") * am * (1 + mpmath.tanh(k * (am + mpmath.mpf("0.044715") * am**3)))
        ref = float(ref * mpmath.mpf("1.5"))
        assert abs(got - ref) <= 1e-13 * abs(ref), (a, got, ref)


def test_gelu_odd_part_identity():
    """gelu(a) - gelu(-a) = a (tanh is odd)."""
    g = synth.tensor(74, 0, (1, 64), torch.float32).numpy()
    ones = np.ones_like(g)
    _, yp = oracle.gelu_and_mul(np.concatenate([g, ones], axis=1), want_y=True)
    _, ym = oracle.gelu_and_mul(np.concatenate([-g, ones], axis=1), want_y=True)
    assert np.allclose(yp - ym, g.astype(np.float64), rtol=1e-14, atol=1e-15)
