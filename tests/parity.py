"""Comparison rules between the CUDA path and the oracle.

bf16 outputs: at most 1 bf16 ulp, measured as the distance between the two bit
patterns on the monotone integer map of bf16 (+0 and -0 map to the same point).

Where an op's last step adds terms that can cancel (the RoPE rotation, the
LayerNorm modulation), an f32 evaluation carries an absolute error of a few
f32 roundings of the terms' magnitudes, which near a cancellation is larger
than one bf16 ulp of the small result.  For those outputs an element also
passes when |gpu - y| <= ulp_bf16(y) + K * 2^-24 * mag, where y is the oracle's
exact pre-rounding value and mag the sum of magnitudes of the combined terms
(both from the oracle).  K is derived from the number of f32 roundings on the
kernel's path and is stated where each test uses it.

f32 outputs: |gpu - y| <= 1e-5 * |y| (plus the same cancellation allowance where
it applies), with an absolute floor of 1e-30 for exact zeros.

Residual write-back: bit-exact.
"""
from __future__ import annotations

import contextlib

import numpy as np

U32 = 2.0 ** -24  # unit roundoff of f32

# Reports of the checks made inside recording(name) blocks, as (name, report);
# tests/conftest.py prints one line per name at the end of the run, so the
# use of the cancellation allowance on the full-size cases is on record.
REPORTS: list = []
_recording: list = []


@contextlib.contextmanager
def recording(name: str):
    """Record the report of every check made inside the block under `name`."""
    _recording.append(name)
    try:
        yield
    finally:
        _recording.pop()


def _record(report: dict) -> dict:
    if _recording:
        REPORTS.append((_recording[-1], report))
    return report


def summarize_reports():
    """One dict per recorded name: elements checked, elements beyond 1 bf16 ulp
    (or beyond the f32 relative bound), how many of those the cancellation
    allowance admitted, and the largest error over mag in units of 2^-24."""
    out = {}
    for name, r in REPORTS:
        s = out.setdefault(name, {"n": 0, "over_1ulp": 0, "cancel_allowance_used": 0,
                                  "max_err_over_mag_u": 0.0, "max_ulp": 0})
        s["n"] += r.get("n", 0)
        s["over_1ulp"] += r.get("over_1ulp", r.get("over_rel", 0))
        s["cancel_allowance_used"] += r.get("cancel_allowance_used", 0)
        s["max_err_over_mag_u"] = max(s["max_err_over_mag_u"], r.get("max_err_over_mag_u", 0.0))
        s["max_ulp"] = max(s["max_ulp"], r.get("max_ulp", 0))
    return out


def bf16_ordinal(bits: np.ndarray) -> np.ndarray:
    """Monotone integer map of bf16 bit patterns; +0 and -0 both map to 0."""
    b = bits.astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def bf16_ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    return np.abs(bf16_ordinal(a_bits) - bf16_ordinal(b_bits))


def bf16_ulp_at(y: np.ndarray) -> np.ndarray:
    """Spacing of the bf16 grid at |y| (2^-133 below the normal range)."""
    a = np.abs(y)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, e, -133.0)
    return np.exp2(np.maximum(e - 7.0, -133.0))


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_bf16(gpu_bits, oracle_bits, y=None, mag=None, k_cancel=None, what=""):
    """Assert the bf16 rule; returns a small report dict."""
    gpu_bits = np.asarray(gpu_bits).reshape(-1)
    oracle_bits = np.asarray(oracle_bits).reshape(-1)
    assert gpu_bits.shape == oracle_bits.shape, what
    d = bf16_ulp_distance(gpu_bits, oracle_bits)
    bad = d > 1
    report = {"n": int(d.size), "max_ulp": int(d.max()) if d.size else 0,
              "over_1ulp": int(bad.sum())}
    if bad.any():
        if k_cancel is None or y is None or mag is None:
            i = int(np.argmax(d))
            raise AssertionError("%s: %d of %d elements beyond 1 bf16 ulp (max %d at flat index %d:"
                                 " gpu 0x%04x oracle 0x%04x)" % (what, int(bad.sum()), d.size,
                                                                d.max(), i, gpu_bits[i],
                                                                oracle_bits[i]))
        y = np.asarray(y).reshape(-1)[bad]
        mag = np.asarray(mag).reshape(-1)[bad]
        g = bf16_to_f64(gpu_bits[bad])
        allow = bf16_ulp_at(y) + k_cancel * U32 * mag
        err = np.abs(g - y)
        fail = err > allow
        report["cancel_allowance_used"] = int(bad.sum())
        report["max_err_over_mag_u"] = float(np.max(err / np.maximum(mag, 1e-300)) / U32)
        if fail.any():
            i = int(np.argmax(err - allow))
            raise AssertionError("%s: %d elements beyond 1 ulp and beyond the cancellation"
                                 " allowance (worst: gpu %r, exact %r, mag %r, allowed %r)"
                                 % (what, int(fail.sum()), g[i], y[i], mag[i], allow[i]))
        # The allowance is for rare cancellations, not a blanket widening.
        assert bad.mean() < 1e-3, "%s: %.2e of elements needed the allowance" % (what, bad.mean())
    return _record(report)


def check_f32(gpu, y, rel=1e-5, mag=None, k_cancel=None, what=""):
    gpu = np.asarray(gpu, dtype=np.float64).reshape(-1)
    y = np.asarray(y, dtype=np.float64).reshape(-1)
    plain = np.maximum(rel * np.abs(y), 1e-30)
    allow = plain
    err = np.abs(gpu - y)
    report = {"n": int(gpu.size),
              "max_rel": float(np.max(err / np.maximum(np.abs(y), 1e-30))) if gpu.size else 0.0}
    if mag is not None and k_cancel is not None:
        mag = np.asarray(mag).reshape(-1)
        allow = plain + k_cancel * U32 * mag
        over = err > plain
        report["over_rel"] = int(over.sum())
        report["cancel_allowance_used"] = int((over & (err <= allow)).sum())
        if over.any():
            report["max_err_over_mag_u"] = float(np.max(err[over] / np.maximum(mag[over], 1e-300))
                                                 / U32)
    fail = err > allow
    if fail.any():
        i = int(np.argmax(err / allow))
        raise AssertionError("%s: %d of %d f32 elements beyond tolerance (worst: gpu %r exact %r)"
                             % (what, int(fail.sum()), gpu.size, gpu[i], y[i]))
    return _record(report)
