"""Device-side failure report: bounded waits, the status word, the probe.

The bulk-copy path of the Q/K kernel waits on shared-memory barriers for its
copies; every such wait is bounded and, when it runs out, sets a bit of the
library's device status word, which nr_device_status reads and clears.  A
wait that nothing completes is made here with the library's probe (bounded
to a fraction of a millisecond): no fault, no hang, and the context stays
usable afterwards."""
import pytest
import torch

import synth
from tests.gpu_util import dev
from tests.test_gpu_qk_norm_rope import run_case

pytestmark = pytest.mark.gpu


def test_status_is_clear_after_normal_work(nr):
    nr.device_status()  # clears anything left by earlier tests
    run_case(nr, 257, 24, 8, 128, seed=31)
    nr.device_status()  # raises if any bounded wait ran out


def test_probe_timeout_is_reported_once_and_context_survives(nr):
    nr.device_status()
    nr.wait_probe(200000)
    with pytest.raises(nr.NrError, match="TIMEOUT"):
        nr.device_status()
    nr.device_status()  # read-and-clear: the second check is clean
    # the context is still usable: a full Q/K call still matches the oracle
    run_case(nr, 64, 8, 2, 128, seed=32)
    nr.device_status()


def test_probe_on_a_side_stream(nr):
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        nr.wait_probe(50000)
        with pytest.raises(nr.NrError, match="TIMEOUT"):
            nr.device_status()
    nr.device_status()


def test_a_bit_set_while_another_stream_reads_is_not_lost(nr):
    """A probe on stream A sets its bit about 0.1 s after launch, while the host
    keeps reading the status through stream B (which does not wait for A).
    Each read clears only the bits it saw, so the probe's bit is reported by
    exactly one read: one of B's reads, or the final read on A."""
    nr.device_status()
    a, b = torch.cuda.Stream(), torch.cuda.Stream()
    done = torch.cuda.Event()
    with torch.cuda.stream(a):
        nr.wait_probe(200_000_000)  # ~0.1 s of SM clock
        done.record(a)
    seen = 0
    reads = 0
    while True:
        finished = done.query()
        with torch.cuda.stream(b):
            try:
                nr.device_status()
            except nr.NrError as err:
                assert "TIMEOUT" in str(err)
                seen += 1
        reads += 1
        if finished:
            break
    with torch.cuda.stream(a):
        try:
            nr.device_status()
        except nr.NrError:
            seen += 1
    assert reads >= 2
    assert seen == 1, "the probe's bit was reported %d times" % seen
    nr.device_status()


def test_bits_read_are_cleared_and_later_bits_kept(nr):
    """Back-to-back probes on two streams, read in turn: each read reports the
    bit left since the previous read, and a clean read follows the last."""
    a, b = torch.cuda.Stream(), torch.cuda.Stream()
    nr.device_status()
    for s in (a, b, a):
        with torch.cuda.stream(s):
            nr.wait_probe(20000)
            with pytest.raises(nr.NrError, match="TIMEOUT"):
                nr.device_status()
    with torch.cuda.stream(b):
        nr.device_status()
