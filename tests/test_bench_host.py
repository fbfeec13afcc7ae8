"""Host-side pieces of bench.py: the multi-rank reduction (gloo, world size 2,
on CPU), the reference arm (the oracle) under torchrun, and the roofline
byte counts."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    bench.dist_init(world, "gloo")
    bench.barrier(world)
    m = bench.reduce_max(10.0 + rank, world)
    q.put((rank, m))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 11.0, 1: 11.0}


def test_reference_arm_under_torchrun_rank0_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3", "--ref-budget-s", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["config"]["workload"] == bench.HEADLINE
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_roofline_byte_counts():
    from mamba_ssd_selective_gb300 import inputs
    w = inputs.WORKLOADS[bench.HEADLINE]
    b = bench.ssd_compulsory_bytes(w)
    # x and y: 4096 tokens x 24 heads x 64 x 2 bytes each
    assert b["x"] == 4096 * 24 * 64 * 2 == b["y"]
    assert b["total"] == b["x"] + b["y"] + b["dt"] + b["B"] + b["C"] + b["final_state"]
    # 28.2 MB per step: zero initial state, so only the final state is moved
    assert abs(b["total"] / 1e6 - 28.25) < 0.01
    assert bench.stage_algorithmic_bytes(w, "chunk_scan") == b["x"] + b["dt"] + b["B"] + b["C"] + b["y"]


def test_traffic_records_are_well_formed():
    """profiles/traffic.json: one record per dominant kernel the bench reports,
    naming a kernel that exists in its source file, with a positive per-launch
    byte count and the capture it came from; a record whose source has changed
    since is reported as null by the bench, never as a stale number."""
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        recs = json.load(f)
    assert set(recs) >= {"chunk_scan", "decode_step", "diag_scan"}
    for key, rec in recs.items():
        src = os.path.join(ROOT, "mamba_ssd_selective_gb300", "csrc", rec["source"])
        assert os.path.exists(src), key
        with open(src) as f:
            assert rec["kernel"] in f.read(), key
        assert int(rec["bytes_per_launch"]) > 0 and rec["capture"], key
        got = bench._traffic_for(key)
        assert got is None or got == rec["bytes_per_launch"], key
    assert bench._traffic_for("no_such_kernel") is None
