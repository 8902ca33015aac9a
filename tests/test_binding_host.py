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


def _bf(*shape):
    return torch.zeros(*shape, dtype=torch.bfloat16)


MISMATCHED = {
    # rmsnorm: weight length, residual / out shape and dtype
    "rmsnorm short w": lambda b: b.rmsnorm(_bf(4, 64), _bf(32)),
    "rmsnorm f32 w next to bf16 x": lambda b: b.rmsnorm(_bf(4, 64), torch.ones(64)),
    "rmsnorm short residual": lambda b: b.rmsnorm(_bf(4, 64), _bf(64), residual=_bf(3, 64)),
    "rmsnorm f32 residual": lambda b: b.rmsnorm(_bf(4, 64), _bf(64), residual=torch.zeros(4, 64)),
    "rmsnorm strided residual": lambda b: b.rmsnorm(_bf(4, 64), _bf(64), residual=_bf(4, 128)[:, :64]),
    "rmsnorm short out": lambda b: b.rmsnorm(_bf(4, 64), _bf(64), out=_bf(4, 32)),
    "fp8 short codes": lambda b: b.rmsnorm_quant_fp8(_bf(4, 64), _bf(64), 1.0,
                                                     codes=torch.zeros(4, 32, dtype=torch.uint8)),
    "fp8 codes not bytes": lambda b: b.rmsnorm_quant_fp8(_bf(4, 64), _bf(64), 1.0, codes=_bf(4, 64)),
    "fp8 out_bf16 f32": lambda b: b.rmsnorm_quant_fp8(_bf(4, 64), _bf(64), 1.0,
                                                      out_bf16=torch.zeros(4, 64)),
    "fp8 short w": lambda b: b.rmsnorm_quant_fp8(_bf(4, 64), _bf(8), 1.0),
    # qk_norm_rope: token counts, head_dim, positions, weights, outputs
    "qk k with fewer tokens": lambda b: b.qk_norm_rope(_bf(4, 2, 64), _bf(3, 1, 64), torch.ones(64),
                                                       torch.ones(64), torch.zeros(4, dtype=torch.int32)),
    "qk k head_dim": lambda b: b.qk_norm_rope(_bf(4, 2, 64), _bf(4, 1, 32), torch.ones(64),
                                              torch.ones(64), torch.zeros(4, dtype=torch.int32)),
    "qk short positions": lambda b: b.qk_norm_rope(_bf(4, 2, 64), _bf(4, 1, 64), torch.ones(64),
                                                   torch.ones(64), torch.zeros(3, dtype=torch.int32)),
    "qk int64 positions": lambda b: b.qk_norm_rope(_bf(4, 2, 64), _bf(4, 1, 64), torch.ones(64),
                                                   torch.ones(64), torch.zeros(4, dtype=torch.int64)),
    "qk strided positions": lambda b: b.qk_norm_rope(_bf(4, 2, 64), _bf(4, 1, 64), torch.ones(64),
                                                     torch.ones(64),
                                                     torch.zeros(8, dtype=torch.int32)[::2]),
    "qk short wq": lambda b: b.qk_norm_rope(_bf(4, 2, 64), _bf(4, 1, 64), torch.ones(32),
                                            torch.ones(64), torch.zeros(4, dtype=torch.int32)),
    "qk wk None with K heads": lambda b: b.qk_norm_rope(_bf(4, 2, 64), _bf(4, 1, 64), torch.ones(64),
                                                         None, torch.zeros(4, dtype=torch.int32)),
    "qk wq wk dtypes": lambda b: b.qk_norm_rope(_bf(4, 2, 64), _bf(4, 1, 64), torch.ones(64),
                                                _bf(64), torch.zeros(4, dtype=torch.int32)),
    "qk q k dtypes": lambda b: b.qk_norm_rope(_bf(4, 2, 64), torch.zeros(4, 1, 64), torch.ones(64),
                                              torch.ones(64), torch.zeros(4, dtype=torch.int32)),
    "qk short q_out": lambda b: b.qk_norm_rope(_bf(4, 2, 64), _bf(4, 1, 64), torch.ones(64),
                                               torch.ones(64), torch.zeros(4, dtype=torch.int32),
                                               q_out=_bf(3, 2, 64)),
    "qk k_out dtype": lambda b: b.qk_norm_rope(_bf(4, 2, 64), _bf(4, 1, 64), torch.ones(64),
                                               torch.ones(64), torch.zeros(4, dtype=torch.int32),
                                               k_out=torch.zeros(4, 1, 64)),
    "qk-ex mrope positions [tokens]": lambda b: b.qk_norm_rope_ex(
        _bf(4, 2, 64), _bf(4, 1, 64), torch.ones(64), torch.ones(64),
        torch.zeros(4, dtype=torch.int32), mrope_sections=(16, 8, 8)),
    "qk-ex short positions": lambda b: b.qk_norm_rope_ex(
        _bf(4, 2, 64), _bf(4, 1, 64), torch.ones(64), torch.ones(64),
        torch.zeros(2, dtype=torch.int32)),
    # ln_modulate / gated: sample rows, dtypes, widths
    "ln shift too few samples": lambda b: b.ln_modulate(_bf(6, 64), _bf(2, 64), _bf(3, 64),
                                                        rows_per_sample=2),
    "ln scale width": lambda b: b.ln_modulate(_bf(6, 64), _bf(1, 64), _bf(1, 32)),
    "ln f32 shift": lambda b: b.ln_modulate(_bf(6, 64), torch.zeros(1, 64), _bf(1, 64)),
    "ln out shape": lambda b: b.ln_modulate(_bf(6, 64), _bf(1, 64), _bf(1, 64), out=_bf(5, 64)),
    "ln rows_per_sample 0": lambda b: b.ln_modulate(_bf(6, 64), _bf(1, 64), _bf(1, 64),
                                                    rows_per_sample=0),
    "gated short y": lambda b: b.gated_residual_ln_modulate(_bf(6, 64), _bf(5, 64), _bf(1, 64),
                                                            _bf(1, 64), _bf(1, 64)),
    "gated per-token gate too short": lambda b: b.gated_residual_ln_modulate(
        _bf(6, 64), _bf(6, 64), _bf(5, 64), _bf(6, 64), _bf(6, 64), rows_per_sample=1),
    "gated f32 y": lambda b: b.gated_residual_ln_modulate(_bf(6, 64), torch.zeros(6, 64), _bf(1, 64),
                                                          _bf(1, 64), _bf(1, 64)),
    "gated out dtype": lambda b: b.gated_residual_ln_modulate(_bf(6, 64), _bf(6, 64), _bf(1, 64),
                                                              _bf(1, 64), _bf(1, 64),
                                                              out=torch.zeros(6, 64)),
    # activations: output shape and dtype
    "silu out width": lambda b: b.silu_and_mul(_bf(4, 128), out=_bf(4, 128)),
    "gelu out dtype": lambda b: b.gelu_and_mul(_bf(4, 128), out=torch.zeros(4, 64)),
}


@pytest.mark.parametrize("case", sorted(MISMATCHED))
def test_mismatched_operands_are_refused_before_any_launch(binding, case):
    """Every operand's dtype, shape and layout is checked against the main
    tensor before the library is called: the C ABI takes bare pointers, so a
    short or mistyped operand would otherwise be read or written past its end.
    On this CPU-only machine the tensors are host tensors, so a check that
    came after the device check would surface as the "CUDA" error instead."""
    with pytest.raises((ValueError, TypeError)) as err:
        MISMATCHED[case](binding)
    assert "CUDA" not in str(err.value), str(err.value)


def test_well_formed_operands_reach_the_device_check(binding):
    """The same calls with matching operands pass every shape check and stop
    only at the device check (the tensors here are on the host)."""
    p4 = torch.zeros(4, dtype=torch.int32)
    calls = [
        lambda: binding.rmsnorm(_bf(4, 64), _bf(64), residual=_bf(4, 64), out=_bf(4, 64)),
        lambda: binding.rmsnorm_quant_fp8(_bf(4, 64), _bf(64), 1.0, out_bf16=True),
        lambda: binding.qk_norm_rope(_bf(4, 2, 64), _bf(4, 1, 64), torch.ones(64), torch.ones(64), p4),
        lambda: binding.qk_norm_rope_ex(_bf(4, 2, 64), _bf(4, 1, 64), torch.ones(64), torch.ones(64),
                                        torch.zeros(3, 4, dtype=torch.int32),
                                        mrope_sections=(16, 8, 8)),
        lambda: binding.ln_modulate(_bf(6, 64), _bf(3, 64), _bf(3, 64), rows_per_sample=2),
        lambda: binding.ln_modulate(_bf(6, 64), _bf(64), _bf(1, 64)),
        lambda: binding.gated_residual_ln_modulate(_bf(6, 64), _bf(6, 64), _bf(6, 64), _bf(6, 64),
                                                   _bf(6, 64), rows_per_sample=1),
        lambda: binding.silu_and_mul(_bf(4, 128), out=_bf(4, 64)),
        # no K heads: wk may be None
        lambda: binding.qk_norm_rope(_bf(4, 2, 64), _bf(4, 0, 64), torch.ones(64), None, p4),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="CUDA"):
            call()
