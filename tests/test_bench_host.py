"""Host logic of bench.py: workload sizes, algorithmic bytes, and the multi-rank
(weak scaling) timing reduction, the latter over two gloo ranks on the CPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_algorithmic_bytes_of_each_workload():
    # x read once + y written once + gamma/beta read once, fp32
    assert bench.algorithmic_bytes(bench.CONFIGS["rms_small"]) == 1_048_576
    assert bench.algorithmic_bytes(bench.CONFIGS["ln"]) == 570_425_344
    assert bench.algorithmic_bytes(bench.CONFIGS["gn"]) == 67_174_400
    assert bench.algorithmic_bytes(bench.CONFIGS["rms"]) == 15_032_385_536
    assert bench.algorithmic_bytes(bench.CONFIGS["ln_stress"]) == 570_425_344
    assert bench.elements(bench.CONFIGS["rms"]) == 112 * 64 * 512 * 512


def test_weak_scaling_value():
    # 2 ranks, each moving 1e9 bytes per step, slowest rank 0.5 ms per step -> 4000 GB/s
    assert bench.weak_scaling_value(10**9, 2, 0.5e-3) == pytest.approx(4000.0)
    assert bench.weak_scaling_value(10**9, 1, 1e-3) == pytest.approx(1000.0)


def test_peak_prefers_measured_file():
    peak, note = bench.hbm_peak()
    if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        assert "measured" in note and peak > 1000
    else:
        assert peak == bench.FALLBACK_HBM_GBS


def test_reference_arm_non_zero_ranks_exit_without_work():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "3", "--warmup", "3"], env={**os.environ, "RANK": "1", "WORLD_SIZE": "2",
                                                                 "LOCAL_RANK": "1"},
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_line_shape():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "gn",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=300,
                       env={k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")})
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


WORKER = r"""
import os, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
rank = int(os.environ["RANK"]); world = int(os.environ["WORLD_SIZE"])
bench.dist_init(world, "gloo")
# each rank reports its own step time; the slowest one decides the job's throughput
mx = bench.dist_max(0.001 * (rank + 1), world)
bench.dist_barrier(world)
val = bench.weak_scaling_value(10**9, world, mx)
print(f"RESULT {{rank}} {{mx}} {{val}}", flush=True)
dist.destroy_process_group()
"""


def test_two_gloo_ranks_reduce_max_time(tmp_path):
    script = tmp_path / "worker.py"
    script.write_text(WORKER.format(root=ROOT))
    env = {**os.environ, "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": "29517", "WORLD_SIZE": "2"}
    procs = [subprocess.Popen([sys.executable, str(script)], env={**env, "RANK": str(r), "LOCAL_RANK": str(r)},
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True) for r in range(2)]
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (out, err) in zip(procs, outs):
        assert p.returncode == 0, err
    results = sorted(l.split()[1:] for out, _ in outs for l in out.splitlines() if l.startswith("RESULT"))
    assert len(results) == 2
    for rank, mx, val in results:
        assert float(mx) == pytest.approx(0.002)
        assert float(val) == pytest.approx(2 * 1e9 / 0.002 / 1e9)


def test_buffer_sets_keep_every_step_out_of_l2():
    l2 = 126 * 2**20
    # one LayerNorm step moves 512 MiB of x and y: larger than twice the L2 by itself
    assert bench.buffer_sets(bench.CONFIGS["ln"], l2) == 1
    assert bench.buffer_sets(bench.CONFIGS["rms"], l2) == 1
    # GroupNorm (64 MiB) and the small RMSNorm (1 MiB) rotate through >= 3 L2s of sets
    for name in ("gn", "rms_small"):
        cfg = bench.CONFIGS[name]
        n = bench.buffer_sets(cfg, l2)
        assert n > 1 and n * 8 * bench.elements(cfg) >= 3 * l2
        assert (n - 1) * 8 * bench.elements(cfg) < 3 * l2
    assert "rotate through" in bench.l2_note(bench.CONFIGS["gn"], l2)


def test_kernel_source_hash_ignores_comments():
    import bench
    a = "int f(int x) { return x + 1; } // add one\n/* block\n comment */ int g;"
    b = "// header\nint   f(int x)\n{\n    return x + 1; /* inline */\n}\nint g;"
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only("int f(int x) { return x + 2; }") != bench.code_only(a)
    for op in bench.KERNEL_SOURCES:
        assert len(bench.kernel_source_hash(op)) == 16


def test_main_kernel_of_group_norm_workloads():
    assert bench.main_kernel_name(bench.CONFIGS["gn"]) == "gn_vec4_kernel"
    assert bench.main_kernel_name(bench.CONFIGS["gn_m48"]) == "gns_team_kernel"
    assert bench.main_kernel_name(dict(op="gn", C=4096, G=4)) == "gns_team_kernel"  # 256 vectors a group
    assert bench.main_kernel_name(dict(op="gn", C=4096, G=4, bf16=True)) == "gns_reg_kernel"
    assert bench.main_kernel_name(dict(op="gn", C=960, G=32)) == "gns_team_kernel"  # pairs of elements
