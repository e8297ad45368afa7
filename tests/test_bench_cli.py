"""bench.py's command line on the CPU: it parses, lists every workload and keeps the
per-launch traffic table consistent with the sources it was measured on."""
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

WORKLOADS = ["single_decode", "batched_decode", "causal_prefill", "mixed_batch", "prefix_shared_decode",
             "layered_decode", "batched_decode_fp8", "prefix_shared_decode_cascade", "qkv_append"]


def test_help_lists_every_workload():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--help"], capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr
    for w in WORKLOADS:
        assert w in r.stdout


def test_traffic_entries_name_existing_sources():
    for name, entry in bench.TRAFFIC.items():
        assert entry["bytes_per_launch"] > 0
        for src in entry["sources"]:
            assert os.path.exists(os.path.join(ROOT, "paged_gqa_attention_gb300", "csrc", src)), (name, src)
        # a stale entry reports null rather than a number taken on other sources
        fresh = bench.source_hash(*entry["sources"]) == entry["sha"]
        assert (bench.traffic_for(name) is not None) == fresh


def test_traffic_only_for_the_captured_workload():
    # a capture's bytes describe a launch of the captured size: a line of another workload
    # (another size of launch of the same kernel) reports null
    for name, entry in bench.TRAFFIC.items():
        assert entry["workload"] in WORKLOADS, name
        fresh = bench.source_hash(*entry["sources"]) == entry["sha"]
        got = bench.traffic_for(name, entry["workload"])
        assert got == (entry["bytes_per_launch"] if fresh else None)
        others = [w for w in WORKLOADS if w != entry["workload"]]
        assert all(bench.traffic_for(name, w) is None for w in others)


def _reference_run(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--workload", "single_decode", "--steps", "3", "--warmup", "1",
                           "--cpu-seconds", "0.3"], capture_output=True, text=True, env=env, timeout=600)


def test_reference_arm_rank0_prints_other_ranks_exit():
    import json
    r0 = _reference_run(0, 2)
    assert r0.returncode == 0, r0.stderr[-2000:]
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    r1 = _reference_run(1, 2)
    assert r1.returncode == 0, r1.stderr[-2000:]
    assert r1.stdout.strip() == ""
