"""The Python binding on the CPU: it declares every C entry point with the
argument count include/nr.h gives it, refuses tensors that are not on a CUDA
device before calling the library, and fails loudly at import when the
library has not been built (there is no fallback)."""
import importlib.util
import os
import re
import shutil

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nr.h")
PKG = os.path.join(ROOT, "normalisation_rope_transformers_gb300")


def header_param_counts():
    """Number of parameters of every nr_* function declared in the header."""
    text = open(HEADER).read()
    counts = {}
    for m in re.finditer(r"^\s*(?:nr_status|const char\*|int)\s+(nr_\w+)\s*\(([^)]*)\)\s*;", text,
                         re.M):
        params = m.group(2).strip()
        counts[m.group(1)] = 0 if params in ("", "void") else len(params.split(","))
    return counts


@pytest.fixture(scope="module")
def binding(lib_path):
    import normalisation_rope_transformers_gb300 as nrt
    return nrt


def test_argtypes_match_the_header(binding):
    counts = header_param_counts()
    assert set(binding.ENTRY_POINTS) == set(counts), "binding and header list different entry points"
    for name, n in counts.items():
        fn = getattr(binding.lib, name)
        assert len(fn.argtypes) == n, "%s: %d argtypes, header declares %d" % (
            name, len(fn.argtypes), n)
        assert fn.restype is not None


def test_cpu_tensors_are_refused_before_the_library_is_called(binding):
    x = torch.zeros(2, 64, dtype=torch.bfloat16)
    w = torch.ones(64, dtype=torch.bfloat16)
    calls = [
        lambda: binding.rmsnorm(x, w),
        lambda: binding.rmsnorm_quant_fp8(x, w, 1.0),
        lambda: binding.ln_modulate(x, w[None], w[None]),
        lambda: binding.silu_and_mul(x),
        lambda: binding.gelu_and_mul(x),
        lambda: binding.gated_residual_ln_modulate(x, x, w[None], w[None], w[None]),
        lambda: binding.qk_norm_rope(x.view(2, 1, 64), x.view(2, 1, 64), w.float(), w.float(),
                                     torch.zeros(2, dtype=torch.int32)),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="CUDA"):
            call()


def test_import_without_the_library_fails_loudly(tmp_path):
    pkg = tmp_path / "nr_unbuilt"
    pkg.mkdir()
    shutil.copy(os.path.join(PKG, "__init__.py"), pkg / "__init__.py")
    spec = importlib.util.spec_from_file_location("nr_unbuilt", str(pkg / "__init__.py"))
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError, match="build"):
        spec.loader.exec_module(mod)
