"""Helpers for the GPU parity tests: device copies and guarded outputs."""
from __future__ import annotations

import numpy as np
import torch

import synth

GUARD = 256  # elements of canary on each side of a guarded output
CANARY_BITS = {torch.bfloat16: 0x7FBF, torch.float32: 0x7FBFBFBF}  # quiet-NaN patterns


def dev(t):
    return None if t is None else t.cuda()


def host_bits(t) -> np.ndarray:
    """Storage bits of a tensor (any device) in the oracle's convention."""
    return synth.to_oracle(t.detach().cpu())


class Guarded:
    """An output tensor with canary bands before and after it in one allocation."""

    def __init__(self, shape, dtype, fill=None):
        n = int(np.prod(shape)) if len(shape) else 1
        itype = torch.int16 if dtype == torch.bfloat16 else torch.int32
        raw = torch.full((n + 2 * GUARD,), CANARY_BITS[dtype], dtype=itype)
        self.buf = raw.view(dtype).cuda()
        self.t = self.buf[GUARD:GUARD + n].view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def check(self):
        itype = torch.int16 if self.buf.dtype == torch.bfloat16 else torch.int32
        b = self.buf.view(itype).cpu()
        canary = CANARY_BITS[self.buf.dtype]
        assert torch.all(b[:GUARD] == canary), "write before the output buffer"
        assert torch.all(b[-GUARD:] == canary), "write after the output buffer"
