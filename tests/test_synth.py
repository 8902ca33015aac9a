"""The seeded input generator that both the CUDA path and the oracle read
(CPU).  Its finaliser is the published splitmix64 one, its values do not
depend on how the draw is chunked over threads, streams are distinct per seed
and tensor, and the normal deviates have the stated moments."""
import numpy as np
import torch

import synth

# splitmix64 from state 0: the first three outputs of the published generator
SPLITMIX64_SEED0 = (0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F)


def test_finaliser_is_splitmix64():
    gamma = 0x9E3779B97F4A7C15
    states = np.array([(k * gamma) % (1 << 64) for k in (1, 2, 3)], dtype=np.uint64)
    with np.errstate(over="ignore"):
        got = synth._mix(states)
    assert [int(v) for v in got] == list(SPLITMIX64_SEED0)


def test_values_do_not_depend_on_chunking():
    chunk = synth._CHUNK
    short = synth.normal(3, 7, 2 * chunk + 7)      # crosses two chunk boundaries of pairs
    long = synth.normal(3, 7, 6 * chunk + 1)       # more chunks, more threads, odd length
    assert np.array_equal(short, long[:short.size])
    # and one word at a time from the counter agrees with the bulk draw
    words = synth.uniform_bits(3, 7, 0, 64)
    for k in (0, 1, 31, 63):
        assert words[k] == synth.uniform_bits(3, 7, k, 1)[0]


def test_streams_are_distinct_and_reproducible():
    a = synth.normal(1, 0, 4096)
    assert np.array_equal(a, synth.normal(1, 0, 4096))
    assert not np.array_equal(a, synth.normal(1, 1, 4096))
    assert not np.array_equal(a, synth.normal(2, 0, 4096))
    assert np.abs(np.corrcoef(a, synth.normal(1, 1, 4096))[0, 1]) < 0.1


def test_normal_moments_and_storage():
    z = synth.normal(11, 3, 1 << 20)
    assert abs(z.mean()) < 0.005 and abs(z.std() - 1.0) < 0.005
    w = synth.normal(11, 4, 1 << 20, mean=1.0, std=0.1)
    assert abs(w.mean() - 1.0) < 0.001 and abs(w.std() - 0.1) < 0.001
    t = synth.tensor(11, 3, (4, 1 << 18), torch.bfloat16)
    assert t.shape == (4, 1 << 18) and t.dtype == torch.bfloat16
    # storage is the deviates rounded to the dtype, and to_oracle/from_oracle round-trip
    assert torch.equal(synth.from_oracle(synth.to_oracle(t)), t)
    bits = synth.uniform_bits(5, 5, 0, 1 << 16)
    ones = np.unpackbits(bits.view(np.uint8)).mean()
    assert abs(ones - 0.5) < 0.002
