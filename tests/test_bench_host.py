"""Host-side pieces of bench.py that every reported number depends on: the
algorithmic bytes of each call (the numerator of every GB/s and of the
roofline's `achieved`) and the config object both arms print.  CPU only.

The expected byte counts are worked out here from the workload shapes alone
(elements read plus elements written, times the element size), independently
of how bench.py totals them."""
import bench
import synth

MB = 1e6


def test_algorithmic_bytes_of_each_call():
    got = {name: (nbytes, rows, unit) for name, nbytes, rows, unit in bench.step_shapes(synth)}
    # RMSNorm f32 [64, 1024]: read x and w, write out
    assert got["rmsnorm_f32_64x1024"] == (4 * (64 * 1024 + 1024 + 64 * 1024), 64, "rows")
    # add + RMSNorm bf16 [8192, 5120]: read x, residual, w; write residual, out
    add = 2 * (8192 * 5120 * 2 + 5120 + 8192 * 5120 * 2)
    assert got["add_rmsnorm_bf16_8192x5120_gemma0"] == (add, 8192, "rows")
    assert got["add_rmsnorm_bf16_8192x5120_gemma1"] == (add, 8192, "rows")
    assert abs(add / MB - 335.55) < 0.01
    # Q/K [26598, 24 + 24, 128] bf16: read Q, K; write Q', K'; f32 weights; int32 positions
    qk_rows = 26598 * 48
    qk = 2 * 128 * qk_rows * 2 + 2 * 4 * 128 + 4 * 26598
    assert got["qk_norm_rope_bf16_26598x24x128"] == (qk, qk_rows, "head rows")
    assert abs(qk / MB - 653.78) < 0.01
    # LN + modulation bf16 [26598, 3072]: read x, shift, scale; write out
    ln = 2 * (26598 * 3072 * 2 + 2 * 3072)
    assert got["ln_modulate_bf16_26598x3072"] == (ln, 26598, "rows")
    assert abs(ln / MB - 326.85) < 0.01
    # decode add + RMSNorm [256, 8192] and silu_and_mul [256, 2 x 24576]
    assert got["add_rmsnorm_bf16_256x8192"] == (2 * (4 * 256 * 8192 + 8192), 256, "rows")
    assert got["silu_and_mul_bf16_256x49152"] == (2 * (256 * 49152 + 256 * 24576), 256, "rows")
    assert len(got) == 7


def test_config_is_the_same_object_for_both_arms():
    shapes = bench.step_shapes(synth)
    cfg = bench.step_config(shapes, 1)
    assert cfg["bytes_per_step"] == sum(s[1] for s in shapes) == 1706808216
    assert cfg["workload"].startswith("dit_norm_step: rmsnorm_f32_64x1024 + ")
    assert cfg["rows_per_step"]["qk_norm_rope_bf16_26598x24x128"] == 26598 * 48
    assert cfg["parallelism"].startswith("dp1")
    assert bench.step_config(shapes, 4)["parallelism"].startswith("dp4")


def test_algorithmic_bytes_of_the_next_rows():
    """The next rows' byte counts at a few rows (device buffers built on the
    CPU; nothing is launched)."""
    import torch

    r = 4
    cases = dict(bench.next_row_cases(None, synth, torch, torch.device("cpu"), rows_override=r))
    want = {
        # read residual, y, gate, shift, scale; write residual, out
        "gated_residual_ln_modulate_bf16_26598x3072": 2 * (4 * r * 3072 + 3 * 3072),
        # read x, residual, w; write residual (bf16) and the codes (1 byte)
        "rmsnorm_quant_fp8_bf16_8192x5120": 2 * (3 * r * 5120 + 5120) + r * 5120,
        # read gate and up (2 x 15360), write out (15360)
        "gelu_and_mul_bf16_8192x30720": 2 * (r * 30720 + r * 15360),
    }
    qk = 2 * 2 * r * 48 * 128 + 2 * 4 * 128
    want["qk_norm_rope_mrope_bf16_26598x24x128"] = qk + 3 * 4 * r  # three position rows
    want["qk_norm_rope_gptj_rot64_bf16_26598x24x128"] = qk + 4 * r
    want["qk_norm_rope_llama3_bf16_26598x24x128"] = qk + 4 * r
    assert set(cases) == set(want)
    for name, make in cases.items():
        _, nbytes, rows = make()
        assert (nbytes, rows) == (want[name], r), name


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one
    JSON line with the GPU arm's metric, unit and config, and a cpu_baseline
    and an e2e object with no host-device bytes."""
    import json
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] >= 3
    assert d["config"] == bench.step_config(bench.step_shapes(synth), 1)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] > 0
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    """Under torchrun only rank 0 runs the reference arm; the others exit 0
    without work or output."""
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"], capture_output=True,
                       text=True, timeout=300, cwd=root, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_config_flag_selects_each_workloads_calls():
    """--config N keeps the calls of workload N only, in both arms' config."""
    all_names = [s[0] for s in bench.step_shapes(synth)]
    covered = []
    for n, names in bench.CONFIG_CALLS.items():
        shapes = bench.step_shapes(synth, names)
        assert [s[0] for s in shapes] == list(names), n
        covered += names
        cfg = bench.step_config(shapes, 1)
        assert cfg["bytes_per_step"] == sum(s[1] for s in shapes)
    assert sorted(covered) == sorted(all_names)  # every call belongs to exactly one workload
    small = bench.step_config(bench.step_shapes(synth, bench.CONFIG_CALLS[1]), 1)
    assert "fits in the 129 MB L2" in small["l2"]
    big = bench.step_config(bench.step_shapes(synth, bench.CONFIG_CALLS[3]), 1)
    assert ">> 129 MB L2" in big["l2"]


def test_seed_flag_replaces_every_workload_seed():
    import argparse
    import copy

    saved = {k: copy.deepcopy(getattr(synth, k)) for k in
             ("RMSNORM_F32", "ADD_RMSNORM", "QK_NORM_ROPE", "LN_MODULATE", "DECODE")}
    try:
        sel = bench.apply_workload_args(argparse.Namespace(seed=77, config=4), synth)
        assert sel == bench.CONFIG_CALLS[4]
        assert all(getattr(synth, k)["seed"] == 77 for k in saved)
        assert bench.apply_workload_args(argparse.Namespace(seed=None, config=None), synth) is None
    finally:
        for k, v in saved.items():
            getattr(synth, k).clear()
            getattr(synth, k).update(v)


def test_reference_arm_with_config_and_seed():
    import json
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--config", "1", "--seed", "5"],
                       capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["config"] == bench.step_config(bench.step_shapes(synth, bench.CONFIG_CALLS[1]), 1)
    assert "rmsnorm_f32" in d["cpu_baseline"]["sample"] and "qk_norm" not in d["cpu_baseline"]["sample"]
