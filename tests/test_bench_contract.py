"""bench.py's reference arm (the CPU oracle timed as it stands) keeps the JSON-line
contract on a machine without a GPU: one line with the metric, the workload, the
oracle's cpu_baseline and an end-to-end figure that moves no host-device bytes;
under torchrun only rank 0 prints."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(extra_env=None, *args):
    env = dict(os.environ)
    env.update(extra_env or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *args],
                       capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    return [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]


def test_reference_arm_json_line():
    lines = run_bench(None, "--steps", "2", "--warmup", "3")
    assert len(lines) == 1
    d = lines[0]
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config"):
        assert k in d, k
    assert d["impl"] == "reference"
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["workload"] == "resnet50_w8_allreduce"
    # the same workload as the GPU arm's step: all five buckets, every algorithmic byte
    assert d["config"]["buckets"] == 5 and d["config"]["bytes_per_step"] == 1_635_650_048
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert cb["sample"].startswith("the whole workload: all 5 buckets")
    th = cb["threaded"]
    assert th["threads"] >= 1 and th["value"] > 0
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_print_nothing():
    lines = run_bench({"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"}, "--steps", "1", "--warmup", "3",
                      "--no-threaded")
    assert lines == []


def test_rotation_copies():
    """Steps smaller than twice the L2 rotate over enough input copies to exceed it."""
    sys.path.insert(0, ROOT)
    import bench

    l2 = 135_528_448                                    # GB300's L2 as the device reports it
    assert bench.rotation_copies(1_635_650_048, l2) == 1          # ResNet-50 W=8: far above
    assert bench.rotation_copies(2 * l2, l2) == 1
    r = bench.rotation_copies(6_390_080, l2)                       # the MLP W=4 step
    assert r == 44 and r * 6_390_080 > 2 * l2
    assert bench.rotation_copies(1000, l2) == 64                   # capped
    assert bench.rotation_copies(6_390_080, l2, micro_steps=4) == 1
