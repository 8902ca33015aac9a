"""The C ABI used from plain C: tests/c_consumer/nr_consumer.c includes only
include/nr.h and the CUDA runtime header, links libnormrope.so and the CUDA
runtime, and calls the ops on device buffers it allocates itself (no Python
or torch in that process).

CPU: the program compiles with gcc as C11 (-Wall -Wextra -Werror) and links
against the library, so the header is valid C and every symbol it uses
resolves.  GPU: the program runs on seeded inputs written as raw files, and
what it writes back is checked against the oracle (bf16: at most 1 ulp plus
the derived cancellation allowance; residual write-back bit-exact)."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.parity import check_bf16

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_consumer", "nr_consumer.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")

# rows, hidden | tokens, hq, hk, head_dim | ln_rows, ln_hidden | act_rows, inter
SIZES = dict(rows=37, hidden=4096, tokens=21, hq=6, hk=2, D=128, ln_rows=19, ln_hidden=3072,
             act_rows=5, inter=2048)


def _compile(lib_path, exe):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    if not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime_api.h")):
        pytest.skip("no CUDA runtime headers")
    libdir = os.path.dirname(lib_path)
    cmd = [cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-O2",
           "-I" + os.path.join(ROOT, "include"), "-I" + os.path.join(CUDA, "include"), SRC,
           "-L" + libdir, "-l:" + os.path.basename(lib_path),
           "-L" + os.path.join(CUDA, "lib64"), "-lcudart",
           "-Wl,-rpath," + libdir, "-Wl,-rpath," + os.path.join(CUDA, "lib64"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, "C consumer failed to build:\n%s%s" % (r.stdout, r.stderr)


def test_c_consumer_builds_against_header_and_library(lib_path, tmp_path):
    _compile(lib_path, str(tmp_path / "nr_consumer"))
    assert os.path.exists(tmp_path / "nr_consumer")


@pytest.mark.gpu
def test_c_consumer_matches_the_oracle(lib_path, tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = str(tmp_path / "nr_consumer")
    _compile(lib_path, exe)
    s = SIZES
    bf = torch.bfloat16
    x, res, w = synth.rmsnorm_inputs(s["rows"], s["hidden"], 81, bf)
    q, k, wq, wk, pos = synth.qk_inputs(s["tokens"], s["hq"], s["hk"], s["D"], 82, bf,
                                        torch.float32, pos_start=700)
    lx, sh, sc = synth.ln_inputs(s["ln_rows"], s["ln_hidden"], 83, bf)
    ax = synth.silu_inputs(s["act_rows"], s["inter"], 84, bf)
    arrays = dict(x=x, res=res, w=w, q=q, k=k, wq=wq, wk=wk, pos=pos, lx=lx, shift=sh,
                  scale=sc, ax=ax)
    for name, t in arrays.items():
        host = t.numpy().astype(np.int32) if t.dtype == torch.int32 else synth.to_oracle(t)
        host.tofile(str(tmp_path / (name + ".bin")))
    args = [str(tmp_path)] + [str(s[n]) for n in ("rows", "hidden", "tokens", "hq", "hk", "D",
                                                  "ln_rows", "ln_hidden", "act_rows", "inter")]
    r = subprocess.run([exe] + args, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, "nr_consumer: %s%s" % (r.stdout, r.stderr)

    def got(name, shape):
        return np.fromfile(str(tmp_path / (name + ".bin")), dtype=np.uint16).reshape(shape)

    o_out, o_res, _ = oracle.rmsnorm(synth.to_oracle(x), synth.to_oracle(w),
                                     residual=synth.to_oracle(res), gemma=True)
    check_bf16(got("rms_out", o_out.shape), o_out, what="C consumer rmsnorm")
    assert np.array_equal(got("rms_res", o_res.shape), o_res), "residual not bit-exact"

    rq = oracle.qk_norm_rope(synth.to_oracle(q), synth.to_oracle(k), synth.to_oracle(wq),
                             synth.to_oracle(wk), pos.numpy(), want_y=True)
    check_bf16(got("q_out", rq[0].shape), rq[0], rq[2], rq[4], k_cancel=32, what="C consumer q")
    check_bf16(got("k_out", rq[1].shape), rq[1], rq[3], rq[5], k_cancel=32, what="C consumer k")

    l_out, l_y, l_mag = oracle.ln_modulate(synth.to_oracle(lx), synth.to_oracle(sh),
                                           synth.to_oracle(sc), want_y=True)
    check_bf16(got("ln_out", l_out.shape), l_out, l_y, l_mag, k_cancel=64, what="C consumer ln")

    s_out, _ = oracle.silu_and_mul(synth.to_oracle(ax))
    check_bf16(got("silu_out", s_out.shape), s_out, what="C consumer silu")
