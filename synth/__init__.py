"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module holds none of the method's arithmetic: it only draws numbers.  Both
the CUDA path and the CPU oracle receive the exact same bits from it.

Generator: splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; the 64-bit finaliser as published by Vigna),
used counter-based: element k of tensor ``tensor_id`` under ``seed`` is the
finaliser applied to ``key + (k + 1) * golden_gamma`` with
``key = mix(seed * golden_gamma + tensor_id)``.  Normal deviates come from the
Box-Muller transform in double precision on consecutive pairs of uniforms.
Values are then converted to the storage dtype by torch (round to nearest even).

Workload recipes (shapes, distributions and seeds of the five benchmark
configurations) are the module-level dicts and ``*_inputs`` helpers below.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 20


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, tensor_id: int) -> np.uint64:
    with np.errstate(over="ignore"):
        z = np.array([np.uint64(seed) * _GAMMA + np.uint64(tensor_id)], dtype=np.uint64)
        return _mix(z)[0]


def uniform_bits(seed: int, tensor_id: int, start: int, count: int) -> np.ndarray:
    """64-bit words number start .. start+count-1 of the stream (seed, tensor_id)."""
    key = _key(seed, tensor_id)
    with np.errstate(over="ignore"):
        ctr = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        return _mix(key + ctr * _GAMMA)


def _normal_pairs(seed: int, tensor_id: int, p0: int, pc: int) -> np.ndarray:
    """Box-Muller deviates from uniform pairs p0 .. p0+pc-1 (2*pc values)."""
    words = uniform_bits(seed, tensor_id, 2 * p0, 2 * pc)
    # 53-bit uniforms; u1 in (0, 1] keeps the logarithm finite.
    u1 = ((words[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (words[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * math.pi * u2
    z = np.empty(2 * pc, np.float64)
    z[0::2] = r * np.cos(t)
    z[1::2] = r * np.sin(t)
    return z


def normal(seed: int, tensor_id: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """n normal deviates N(mean, std^2) as float64.

    Chunks are drawn on a thread pool (numpy releases the GIL); the values do not
    depend on the chunking or the thread count."""
    out = np.empty(n, np.float64)
    pairs = (n + 1) // 2
    starts = list(range(0, pairs, _CHUNK))

    def work(p0):
        pc = min(_CHUNK, pairs - p0)
        z = _normal_pairs(seed, tensor_id, p0, pc)
        take = min(2 * pc, n - 2 * p0)
        out[2 * p0:2 * p0 + take] = z[:take]

    if len(starts) <= 1:
        for p0 in starts:
            work(p0)
    else:
        workers = min(len(starts), os.cpu_count() or 1, 16)
        with ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(work, starts))
    return mean + std * out


def tensor(seed: int, tensor_id: int, shape, dtype, mean: float = 0.0, std: float = 1.0):
    """A CPU torch tensor of the given shape and dtype (torch.float32 / torch.bfloat16)."""
    import torch

    n = 1
    for s in shape:
        n *= int(s)
    vals = normal(seed, tensor_id, n, mean, std).astype(np.float32)
    t = torch.from_numpy(vals).reshape(tuple(int(s) for s in shape))
    return t.to(dtype)


def to_oracle(t) -> np.ndarray:
    """The storage bits of a CPU torch tensor as the oracle takes them."""
    import torch

    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError("oracle storage is bf16 or f32, got %s" % t.dtype)


def from_oracle(a: np.ndarray):
    """A CPU torch tensor holding the oracle's stored bits."""
    import torch

    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a))


# --------------------------------------------------------------------------
# Workload recipes: shapes, distributions and seeds of the five benchmark
# configurations.  Tensor ids are fixed per tensor so that a shard or a
# sub-case draws the same stream.
# --------------------------------------------------------------------------
RMSNORM_F32 = dict(name="rmsnorm_f32_64x1024", rows=64, hidden=1024, seed=0, eps=1e-6)
ADD_RMSNORM = dict(name="add_rmsnorm_bf16_8192x5120", rows=8192, hidden=5120, seed=1, eps=1e-6)
QK_NORM_ROPE = dict(name="qk_norm_rope_bf16_26598x24x128", tokens=26598, hq=24, hk=24,
                    head_dim=128, seed=2, eps=1e-6, theta=10000.0)
LN_MODULATE = dict(name="ln_modulate_bf16_26598x3072", rows=26598, hidden=3072, seed=3, eps=1e-6)
DECODE = dict(name="decode_sweep_bf16", rows=(1, 8, 32, 128, 256), hidden=(4096, 5120, 8192),
              seed=4, eps=1e-6)

# tensor ids
T_X, T_RES, T_W, T_Q, T_K, T_WQ, T_WK, T_SHIFT, T_SCALE, T_GATEUP = range(10)


def rmsnorm_inputs(rows, hidden, seed, dtype, residual=True, id_offset=0):
    """x, residual ~ N(0,1) [rows, hidden]; w ~ N(1, 0.1) [hidden]."""
    x = tensor(seed, T_X + id_offset, (rows, hidden), dtype)
    res = tensor(seed, T_RES + id_offset, (rows, hidden), dtype) if residual else None
    w = tensor(seed, T_W + id_offset, (hidden,), dtype, mean=1.0, std=0.1)
    return x, res, w


def qk_inputs(tokens, hq, hk, head_dim, seed, dtype, w_dtype, pos_start=0):
    """Q [tokens, hq, D], K [tokens, hk, D] ~ N(0,1); wq, wk ~ N(1, 0.1) [D],
    drawn in double, stored bf16 then widened to w_dtype (identical values for
    either weight dtype); positions pos_start .. pos_start+tokens-1 (int32)."""
    import torch

    q = tensor(seed, T_Q, (tokens, hq, head_dim), dtype)
    k = tensor(seed, T_K, (tokens, hk, head_dim), dtype)
    wq = tensor(seed, T_WQ, (head_dim,), torch.bfloat16, mean=1.0, std=0.1).to(w_dtype)
    wk = tensor(seed, T_WK, (head_dim,), torch.bfloat16, mean=1.0, std=0.1).to(w_dtype)
    pos = torch.arange(pos_start, pos_start + tokens, dtype=torch.int32)
    return q, k, wq, wk, pos


def ln_inputs(rows, hidden, seed, dtype, samples=1):
    """x ~ N(0,1) [rows, hidden]; shift, scale ~ N(0, 0.1) [samples, hidden]."""
    x = tensor(seed, T_X, (rows, hidden), dtype)
    shift = tensor(seed, T_SHIFT, (samples, hidden), dtype, std=0.1)
    scale = tensor(seed, T_SCALE, (samples, hidden), dtype, std=0.1)
    return x, shift, scale


def silu_inputs(rows, inter, seed, dtype):
    """x ~ N(0,1) [rows, 2*inter] (gate | up)."""
    return tensor(seed, T_GATEUP, (rows, 2 * inter), dtype)
