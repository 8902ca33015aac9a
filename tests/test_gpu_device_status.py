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
