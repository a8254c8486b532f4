"""The multi-process path of bench.py on the CPU: two gloo ranks (replicas
only, no data-path collective) agree on the slowest rank's time, and the
reference arm under torchrun prints exactly one JSON line from rank 0."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, _ = bench.dist_setup(world)
    bench.barrier(w)
    out[r] = bench.max_over_ranks(10.0 + r, w)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    port = free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(2, port, out), nprocs=2, start_method="spawn")
        assert dict(out) == {0: 11.0, 1: 11.0}


def test_reference_arm_under_torchrun_prints_one_line():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1", "--oracle-pairs", "40000"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_traffic_is_reported_only_for_the_captured_sources(tmp_path, monkeypatch):
    """roofline.traffic comes from the committed ncu capture only while the
    kernel sources it lists still hash to the recorded value."""
    import hashlib
    import shutil
    sys.path.insert(0, ROOT)
    import bench
    name = "traffic_bwd_main_llama8b_chunk_64k.json"
    with open(os.path.join(ROOT, "profiles", name)) as f:
        d = json.load(f)
    (tmp_path / "profiles").mkdir()
    h = hashlib.sha256()
    for src in d["sources"]:
        dst = tmp_path / src
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(ROOT, src), dst)
        h.update(dst.read_bytes())
    d["sources_sha256"] = h.hexdigest()
    (tmp_path / "profiles" / name).write_text(json.dumps(d))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic() == int(d["dram_read_bytes"]) + int(d["dram_write_bytes"])
    changed = tmp_path / d["sources"][0]
    changed.write_bytes(changed.read_bytes() + b"\n")
    assert bench.measured_traffic() is None
