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
    # x and y: 8 x 2048 tokens x 80 heads x 64 x 2 bytes each
    assert b["x"] == 8 * 2048 * 80 * 64 * 2 == b["y"]
    assert b["total"] == b["x"] + b["y"] + b["dt"] + b["B"] + b["C"] + b["final_state"]
    # 367.5 MB per step: zero initial state, so only the final state is moved
    assert abs(b["total"] / 1e6 - 367.53) < 0.01
    assert bench.stage_algorithmic_bytes(w, "chunk_scan") == b["x"] + b["dt"] + b["B"] + b["C"] + b["y"]
    # the single-pass kernel moves the whole step's compulsory bytes
    assert bench.stage_algorithmic_bytes(w, "chunk_fused") == b["total"]
    w130 = inputs.WORKLOADS["ssd_m2_130m_L4096"]
    assert abs(bench.ssd_compulsory_bytes(w130)["total"] / 1e6 - 28.25) < 0.01


def test_traffic_records_are_well_formed():
    """profiles/traffic.json: per-step records ("step:<workload>:<path>:<chunk>")
    and per-kernel records ("kernel:<name>") with DRAM read and write bytes,
    the kernels and the source files they come from (every kernel name found in
    them), a hash of those sources and the capture's command; a record whose
    sources have changed since is reported as null by the bench, never as a
    stale number."""
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        recs = json.load(f)
    assert any(k.startswith("step:" + bench.HEADLINE) for k in recs)
    for key, rec in recs.items():
        assert key.startswith(("step:", "kernel:")), key
        srcs = [os.path.join(ROOT, "mamba_ssd_selective_gb300", "csrc", s) for s in rec["sources"]]
        text = ""
        for src in srcs:
            assert os.path.exists(src), key
            with open(src) as f:
                text += f.read()
        for k in rec["kernels"]:
            assert k in text, (key, k)
        assert int(rec["read"]) > 0 and int(rec["write"]) >= 0 and rec["capture"] and rec["command"], key
        got = bench._traffic_record(key)
        assert got is None or got == rec, key
    assert bench._traffic_record("kernel:no_such_kernel") is None
