"""The benchmark's reference arm on CPU: one JSON line with the contract's
keys, the oracle timed on the host cores, and the other ranks silent under
torchrun.  (The GPU arm's line is checked on the GPU machine by running
bench.py; here only what needs no GPU.)"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=e,
                       capture_output=True, text=True, timeout=600)
    return r


def gpu_arm_config(workload, gpus=1):
    """The config dict bench.py's GPU arm builds for `--workload <workload>`
    (it needs no device: the planner's choices go to a separate key)."""
    sys.path.insert(0, ROOT)
    import bench
    args = bench.argparse.Namespace(workload=workload, batch=None, seq_len=None, num_splits=None,
                                    n_sink=4, window=64, gpus=gpus, graph=0, phi=6.5,
                                    plant_frac=0.001, split_sweep=False)
    return bench.workload_config(args)


def test_default_workload_is_the_largest_single_gpu_config():
    c = gpu_arm_config("million")
    assert (c["B"], c["Hq"], c["Hkv"], c["d"], c["L"]) == (1, 32, 8, 128, 1 << 20)
    with open(os.path.join(ROOT, "bench.py")) as f:
        assert 'ap.add_argument("--workload", default="million"' in f.read()


def test_inputs_exceed_l2_or_are_flushed():
    # every workload's timed calls read HBM: caches under twice the L2 rotate
    # through copies, the tiny config empties L2 before each call
    sys.path.insert(0, ROOT)
    import bench
    for name, (B, Hq, Hkv, L, d) in bench.FULL_SHAPES.items():
        c = gpu_arm_config(name)
        if name == "tiny":
            assert "512 MiB write before each call" in c["l2"]
            continue
        if name.endswith("_fp4"):
            per_token = 2 * (d // 2 + d // 32)
        elif name.endswith("_fp8"):
            per_token = 2 * (d + 4)
        else:
            per_token = 4 * d
        if name == "ladder" or "paged" in name:
            continue  # the ladder rotates its own copies; the paged pools are > 1 GB
        nbytes = B * Hkv * L * per_token * bench.encoded_copies(name, B, L, Hkv, d)
        assert nbytes >= 2 * bench.L2_BYTES or name.startswith("ffd"), (name, nbytes)
    assert bench.encoded_copies("mha32k_fp4", 1, 32768, 32, 128) == 3
    assert "3 copies of the encoded cache" in gpu_arm_config("mha32k_fp4")["l2"]


@pytest.mark.timeout(600)
@pytest.mark.parametrize("workload", ["tiny", "mha32k_fp8", "ffd_topdelta5", "ffd_sparse_topdelta5_union"])
def test_reference_arm_json_line(workload):
    r = run_bench(["--impl", "reference", "--workload", workload, "--steps", "3", "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["steps"] == 3 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["config"]["workload"] == workload
    # the GPU arm prints the same config dict for the same command line
    assert d["config"] == gpu_arm_config(workload)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


@pytest.mark.timeout(600)
def test_reference_arm_other_ranks_print_nothing():
    r = run_bench(["--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3"],
                  env={"RANK": "1", "WORLD_SIZE": "1", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_algorithmic_flops():
    # 4d per (query head, attended token); the top-delta scan adds 2d per (query head, scanned token)
    from types import SimpleNamespace
    sys.path.insert(0, ROOT)
    import bench
    p = SimpleNamespace(Hq=32, Hkv=8, d=128)
    dense = SimpleNamespace(p=p, kv_tokens=1 << 20, topdelta=None)
    assert bench.Workload.algorithmic_flops(dense) == (1 << 20) * 32 * 4 * 128
    sel = {"selected_per_query": 0.25, "union_tokens": 3 * 1000}
    td = SimpleNamespace(p=p, kv_tokens=4000, topdelta=5.0, sel_stats=sel, group_union=False)
    assert bench.Workload.algorithmic_flops(td) == 4000 * 32 * 2 * 128 + 0.25 * 4000 * 32 * 4 * 128
    tu = SimpleNamespace(p=p, kv_tokens=4000, topdelta=5.0, sel_stats=sel, group_union=True)
    assert bench.Workload.algorithmic_flops(tu) == 4000 * 32 * 2 * 128 + 3000 * 4 * 4 * 128
