"""The benchmark's host-side logic on the CPU: its multi-rank timing (gloo,
world size 2) and the roofline's recorded traffic.

The decode read shards by rows with no exchange step, so N GPUs run N
independent batches; the only cross-rank operations are the timing barrier
and the max-over-ranks reduction, tested here without a GPU.
"""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 0.5 * rank])
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got))


def test_max_over_ranks_gloo_world2():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [2.0, 10.0, 0.5]


def test_whole_job_value_is_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_gbs(1e9, 1, 1.0)
    two = bench.whole_job_gbs(1e9, 2, 1.0)
    assert one == pytest.approx(1000.0) and two == pytest.approx(2000.0)
    assert bench.whole_job_gbs(1e9, 2, 2.0) == pytest.approx(1000.0)


def test_reference_arm_under_torchrun_prints_one_line():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "2", "--warmup", "1", "--workload", "tiny_f32", "--cpu-seconds", "0.5"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["unit"] == "GB/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_recorded_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    """roofline.traffic comes from the committed ncu capture only while the
    decode kernel's source is the one it was taken on: every consumer form
    has an entry for the current source, and a changed source gives null."""
    sys.path.insert(0, ROOT)
    import bench
    got = {c: bench.recorded_traffic(c, 1e9) for c in (1, 2, 3, 4)}
    assert all(v is not None for v in got.values()), got
    # the captured kernels read their unique bytes about once
    assert all(0.9e9 < v < 1.1e9 for v in got.values()), got
    changed = tmp_path / "decode.cu"
    changed.write_bytes(open(bench.DECODE_SRC, "rb").read() + b"\n// changed\n")
    monkeypatch.setattr(bench, "DECODE_SRC", str(changed))
    assert all(bench.recorded_traffic(c, 1e9) is None for c in (1, 2, 3, 4))
