"""Host-side logic of bench.py: clock parsing, peaks, traffic lookup, and the
multi-rank helpers run as two gloo ranks on the CPU."""
import json
import os
import socket
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reduce_max_and_barrier_two_gloo_ranks(tmp_path):
    script = tmp_path / "ranks.py"
    script.write_text(textwrap.dedent("""
        import os, sys
        sys.path.insert(0, %r)
        import torch.distributed as dist
        import bench
        dist.init_process_group("gloo")
        world, rank, local = bench.dist_setup()
        bench.barrier(world)
        m = bench.reduce_max(1.5 + rank, world)
        print("RANK%%d %%d %%.3f" %% (rank, world, m))
        dist.destroy_process_group()
    """ % ROOT))
    env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()), WORLD_SIZE="2")
    procs = []
    for r in range(2):
        e = dict(env, RANK=str(r), LOCAL_RANK=str(r))
        procs.append(subprocess.Popen([sys.executable, str(script)], env=e, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    lines = sorted(l for o, _ in outs for l in o.split("\n") if l.startswith("RANK"))
    assert lines == ["RANK0 2 2.500", "RANK1 2 2.500"]


def test_single_rank_helpers_are_identity():
    assert bench.reduce_max(3.25, 1) == 3.25
    bench.barrier(1)


def test_peaks_fallback_and_measured(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.load_peaks()
    assert p["source"] == "fallback" and p["bf16_tflops"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"gb300": {"hbm_gbs": 7000.0, "bf16_tflops": 2010.0, "bf16_tflops_sustained": 1800.0}}))
    p = bench.load_peaks()
    assert p["source"] == "measured" and p["bf16_tflops"] == 2010.0 and p["bf16_tflops_sustained"] == 1800.0


def test_traffic_only_for_matching_kernel(tmp_path, monkeypatch):
    f = tmp_path / "t.json"
    f.write_text(json.dumps({"w": {"kernel_sha": bench.kernel_hash(), "dram_bytes_per_launch": 123}}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.load_traffic("w") == 123
    f.write_text(json.dumps({"w": {"kernel_sha": "0" * 16, "dram_bytes_per_launch": 123}}))
    assert bench.load_traffic("w") is None
    assert bench.load_traffic("other") is None


def test_workload_config_and_flops():
    from fa_inputs import make_dense, make_varlen
    small = make_dense(1, 2, 2, 16, 16, 64, seed=0, causal=True)
    cfg = bench.workload_config(small, "x")
    assert cfg["flop_per_step"] == 4 * 2 * 16 * 16 * 64 / 2
    v = make_varlen([3, 5], 2, 2, 64, seed=0, causal=False)
    cfg = bench.workload_config(v, "v")
    assert cfg["seqlens"] == [3, 5] and cfg["total_tokens"] == 8
    assert cfg["flop_per_step"] == 4 * 2 * (9 + 25) * 64


def test_rotated_inputs_exceed_l2():
    # The timed steps cycle through enough input copies that together they
    # hold more than twice the L2 (shape-only stand-ins of the dense workloads;
    # step_bytes reads only the array sizes and the head dim).
    from types import SimpleNamespace
    from fa_inputs import WORKLOADS
    for name, w in WORKLOADS.items():
        if w["kind"] != "dense":
            continue
        arr = lambda h, n: SimpleNamespace(size=w["B"] * h * n * w["d"])
        prob = SimpleNamespace(q=arr(w["Hq"], w["Nq"]), k=arr(w["Hkv"], w["Nk"]), v=arr(w["Hkv"], w["Nk"]), d=w["d"])
        for bwd in (False, True):
            for fp8 in (False, True):
                rot = bench.rotation(prob, bwd, fp8)
                assert bench.ROTATE_MIN <= rot <= bench.ROTATE_MAX, name
                assert rot == bench.ROTATE_MAX or rot * bench.step_bytes(prob, bwd, fp8) > 2 * bench.L2_BYTES, name


def test_oracle_sample_reports_threads():
    from fa_inputs import make_dense
    prob = make_dense(1, 2, 2, 64, 64, 64, seed=1, causal=True)
    v, threads, desc, dt = bench.oracle_sample(prob, 0.0)
    assert v > 0 and threads >= 1 and "head" in desc
