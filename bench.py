"""Benchmark of one serving step: KV append + batched paged decode read.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl nsv|reference]
                    [--workload headline_bf16]

Prints ONE JSON line (rank 0).  A step is the whole hot path over one batch,
through the fused entry point nsv_decode_step: the KV append (one kernel,
which also zeroes the read's merge counters) then the decode read (one
kernel, launched programmatically dependent on the append), on the headline
workload by default (256 rows, 32 heads, head_dim 128, block 16, width 8192,
lengths uniform in [512, 8192], bf16, seeded synthetic data).

value     = algorithmic bytes of a step (unique K+V read + q + out + the
            append's read and write) x ranks / max-over-ranks seconds per
            step, inputs resident in HBM; the step's inputs (18.8 GB) are far
            larger than L2, so no flush is needed between steps.
e2e       = the same metric through the C ABI with the step's inputs in
            pinned host memory: every step copies q, k_new, v_new,
            write_slots, block_tables and context_lens host->device (packed
            in one staging buffer, one copy) and the output device->host
            inside the timed region (the KV pool is the resident cache and
            stays on the device).
roofline  = the decode read alone, timed in a separate loop of
            nsv_paged_decode_ws calls (the counter-zeroing kernel + the read,
            each between its own CUDA events): read bytes (K+V + q + out) /
            its time, against the measured HBM copy bandwidth in
            MEASURED_PEAKS.json (a read+write copy, which a read-only
            stream such as this one can exceed).  Workloads smaller than 4x L2
            flush L2 (a 256 MB write) before every step and every read,
            outside the timed spans.
cpu_baseline = the oracle (plain C, fp64) timed on this host's cores on a
            time-bounded sample of rows of the same workload.

--impl reference times that oracle as the reference arm (host cores only).
Under torchrun each rank runs its own batch (weak scaling, no collective on
the data path; the barrier and the max-over-ranks reduction are timing only).
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode-attention KV GB/s (% of GB300 HBM peak) and µs/step"
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_kernel_traffic.json")
DECODE_SRC = os.path.join(ROOT, "paged_kv_decode_nsv_gb300", "csrc", "decode.cu")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["nsv", "reference"], default="nsv")
    ap.add_argument("--workload", default="headline_bf16")
    ap.add_argument("--e2e-steps", type=int, default=0,
                    help="steps of the host-buffer measurement (default: min(steps, 100))")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="time budget of the oracle sample")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(values, device="cpu"):
    """Element-wise max of `values` over all ranks (identity on one rank)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_gbs(bytes_per_step_per_rank, world, ms_per_step):
    """Weak scaling: every rank moves its own batch; the slowest rank sets the time."""
    return bytes_per_step_per_rank * world / (ms_per_step * 1e-3) / 1e9


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(consumer, read_bytes):
    """DRAM bytes per decode-kernel launch, from the committed ncu capture of
    the same consumer variant taken on the kernel source as it is now (else
    None): the capture's traffic/algorithmic ratio times this launch's
    algorithmic read bytes."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        with open(DECODE_SRC, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
        if d.get("decode_cu_sha256") != sha:
            return None
        cap = d["captures"][{1: "cuda", 2: "tensor", 3: "tensor_vector_rows",
                             4: "tensor_tmem"}[consumer]]
        return cap["traffic_over_algorithmic"] * read_bytes
    except (OSError, ValueError, KeyError):
        return None


# ---------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_uuid=None):
        self.proc = None
        self.uuid = device_uuid

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [r[0] for r in rows]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, _, parts in rows:
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(r[1] for r in rows),
                "sm_mhz_min": min(sm), "samples": len(rows), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# the oracle on host cores (cpu_baseline and the reference arm)


_SAMPLE_CACHE = {}


def oracle_throughput(wl, budget_s, threads=0, seed=12345):
    """Run the oracle on consecutive rows of `wl` until `budget_s` passes.

    Inputs: the sampled rows' own blocks as a compact pool drawn on the host
    (same shapes, lengths and distribution as the workload).  Returns
    (GB/s of the sample's algorithmic read bytes, rows done, seconds, threads).
    """
    import torch

    import oracle
    from paged_kv_decode_nsv_gb300 import workloads as W

    threads = threads or os.cpu_count() or oracle.max_threads()
    done, t_total, bytes_total, r0 = 0, 0.0, 0, 0
    per_call = max(1, threads)
    while t_total < budget_s and r0 < wl.rows:
        rows = tuple(range(r0, min(wl.rows, r0 + per_call)))
        key = (wl.name, rows, seed)
        if key not in _SAMPLE_CACHE:
            blocks, tables, _ = W.compact_rows(wl, rows)
            # at least one real block: a sample of empty rows still has a pool
            shape = (max(len(blocks), 1) + 1, wl.kv_heads, wl.block_size, wl.head_dim)
            gen = torch.Generator().manual_seed(seed * 100003 + r0)

            def draw(s):
                x = torch.randn(s, generator=gen, dtype=torch.float32)
                if wl.dtype == "bf16":
                    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
                return x.numpy()
            _SAMPLE_CACHE[key] = (draw(shape), draw(shape),
                                  draw((len(rows), wl.heads, wl.head_dim)), tables)
        kp, vp, q, tables = _SAMPLE_CACHE[key]
        ctx = wl.context_lens[list(rows)]
        t0 = time.perf_counter()
        oracle.paged_decode(q, kp, vp, tables, ctx, wl.scale, threads=threads)
        t_total += time.perf_counter() - t0
        kv = int(ctx.astype(np.int64).sum()) * wl.kv_heads * wl.head_dim * 2 * wl.elem_bytes
        bytes_total += kv + 2 * len(rows) * wl.heads * wl.head_dim * wl.elem_bytes
        done += len(rows)
        r0 += len(rows)
    return bytes_total / t_total / 1e9, done, t_total, threads


def run_reference(args, wl):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_throughput(wl, per_step)
    vals, rows_done, secs = [], 0, 0.0
    threads = 0
    for _ in range(args.steps):
        gbs, n, t, threads = oracle_throughput(wl, per_step)
        vals.append(gbs)
        rows_done += n
        secs += t
    value = float(np.median(vals))
    sample = ("%d rows of %s (first rows, each step about %.1f s of oracle time; "
              "compact host pool of the rows' own blocks)" % (rows_done // max(1, args.steps),
                                                               wl.name, per_step))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        # each timed step is a bounded sample of the workload (see the sample)
        "ms_per_step": 1e3 * secs / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": workload_config(wl),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(wl):
    return {"workload": wl.name, "rows": wl.rows, "heads": wl.heads, "kv_heads": wl.kv_heads,
            "head_dim": wl.head_dim, "block_size": wl.block_size, "width": wl.width,
            "total_tokens": wl.total_tokens, "kv_dtype": wl.dtype, "accumulate": "f32",
            "step": "kv_append + decode_read",
            "l2": "inputs larger than L2 (no flush)" if wl.step_bytes() > 4 * 129e6
                  else "L2 flushed between steps"}


# ---------------------------------------------------------------------------
# the GPU arm


def run_nsv(args, wl):
    # the library first: without it this arm stops here (ImportError), before
    # any device work, and has no other path to take
    from paged_kv_decode_nsv_gb300 import nsv
    from paged_kv_decode_nsv_gb300 import workloads as W
    import torch
    import torch.distributed as dist

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    # The oracle sample runs first, on the host, before the GPU work starts.
    cpu = cpu1 = None
    if rank == 0 and ws == 1 and args.cpu_seconds > 0:
        cpu = oracle_throughput(wl, args.cpu_seconds)
        # and on one core, a shorter sample
        cpu1 = oracle_throughput(wl, max(1.0, args.cpu_seconds / 4), threads=1)

    stream = torch.cuda.current_stream()
    q, kp, vp, kn, vn = W.device_values(wl, "cuda")
    bt = torch.from_numpy(wl.block_tables).cuda()
    ctx = torch.from_numpy(wl.context_lens).cuda()
    slots = torch.from_numpy(wl.write_slots).cuda()
    out = torch.empty_like(q)
    shape = nsv.shape_of(q, kp, bt)
    plan = nsv.plan_split(shape)
    wsp = nsv.workspace_for(plan)
    # nsv_decode_step launches two kernels per step: kv_write_kernel (which
    # also zeroes the read's merge counters) and decode_kernel, the read
    # launched programmatically dependent on the append.  No memset.
    launches_per_step = 2
    small_l2 = wl.step_bytes() <= 4 * 129e6
    # L2 flush for small workloads: write a buffer larger than L2, then read
    # another one, so that L2 holds clean lines and no write-back of the
    # flush lands inside the next timed span.
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda") if small_l2 else None
    flush_rd = torch.ones(32 << 20, dtype=torch.int64, device="cuda") if small_l2 else None

    def flush_l2():
        if flush is not None:
            flush.zero_()
            flush_rd.sum()

    def step(ev_s=None, ev_e=None):
        """One serving step through the fused entry point (the timed unit)."""
        flush_l2()
        if ev_s is not None:
            ev_s.record(stream)
        nsv.decode_step(q, kn, vn, slots, kp, vp, bt, ctx, wl.scale, out, workspace=wsp,
                        plan=plan)
        if ev_e is not None:
            ev_e.record(stream)

    def read(ev_s=None, ev_e=None):
        """The decode read alone (its counter-zeroing kernel and the read), for the
        roofline of the dominant kernel."""
        flush_l2()
        if ev_s is not None:
            ev_s.record(stream)
        nsv.paged_decode_ws(q, kp, vp, bt, ctx, wl.scale, out, workspace=wsp, plan=plan)
        if ev_e is not None:
            ev_e.record(stream)

    nsv.device_status(clear=True)
    for _ in range(max(3, args.warmup)):
        step()
        read()
    torch.cuda.synchronize()
    st, _ = nsv.device_status(clear=True)
    if st:
        raise RuntimeError("device status %#x after warm-up" % st)

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(local).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid)
    sampler.start()

    K = args.steps
    # The timed region: K fused steps.  Without a flush the events bracket
    # the whole loop; with one, each step has its own pair and the flushes
    # sit between the timed spans.
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(2)) for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for k in range(K):
        if flush is None:
            step()
        else:
            step(*ev[k])
    end.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    if flush is None:
        total_ms = start.elapsed_time(end)
    else:
        total_ms = sum(a.elapsed_time(b) for a, b in ev)

    # The read alone, each launch between its own pair of events on the
    # launching stream (the roofline's kernel time).
    rev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(2)) for _ in range(K)]
    for k in range(K):
        read(*rev[k])
    torch.cuda.synchronize()
    read_ms = [a.elapsed_time(b) for a, b in rev]

    # end to end through the C ABI from pinned host buffers.  The step's
    # inputs are packed into one pinned staging buffer and copied to one
    # device buffer with a single copy (as a serving loop stages a step's
    # metadata); the kernels read views into it.
    E = args.e2e_steps or min(K, 100)
    parts = [q, kn, vn, bt, ctx, slots]
    offs, size = [], 0
    for t in parts:
        offs.append(size)
        size += -(-t.numel() * t.element_size() // 256) * 256
    h_buf = torch.empty(size, dtype=torch.uint8).pin_memory()
    d_buf = torch.empty(size, dtype=torch.uint8, device="cuda")

    def view(buf, t, off):
        return buf[off:off + t.numel() * t.element_size()].view(t.dtype).view(t.shape)

    for t, off in zip(parts, offs):
        view(h_buf, t, off).copy_(t.cpu())
    d_q, d_kn, d_vn, d_bt, d_ctx, d_slots = (view(d_buf, t, off) for t, off in zip(parts, offs))
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in parts)
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step(ev_s=None, ev_e=None):
        if flush is not None:
            flush.zero_()
            flush_rd.sum()
        if ev_s is not None:
            ev_s.record(stream)
        d_buf.copy_(h_buf, non_blocking=True)
        nsv.decode_step(d_q, d_kn, d_vn, d_slots, kp, vp, d_bt, d_ctx, wl.scale, out,
                        workspace=wsp, plan=plan)
        h_out.copy_(out, non_blocking=True)
        if ev_e is not None:
            ev_e.record(stream)

    for _ in range(3):
        e2e_step()
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    eev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(2)) for _ in range(E)]
    for k in range(E):
        e2e_step(*eev[k])
    torch.cuda.synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in eev) / E
    clocks = sampler.stop()
    st, _ = nsv.device_status(clear=True)
    if st:
        raise RuntimeError("device status %#x after the timed steps" % st)

    ms_step = total_ms / K
    ms_read = float(np.mean(read_ms))
    ms_step, e2e_ms, ms_read = max_over_ranks([ms_step, e2e_ms, ms_read], device="cuda")
    if ws > 1:
        dist.destroy_process_group()
    if rank != 0:
        return 0

    step_bytes = wl.step_bytes()
    value = whole_job_gbs(step_bytes, ws, ms_step)
    peak, peak_kind = measured_peak()
    achieved = wl.read_bytes() / (ms_read * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "us_per_step": ms_step * 1e3,
        "pct_of_hbm_peak": 100.0 * value / ws / peak,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic (seeded N(0,1) values, seeded lengths and block permutation)",
        "config": dict(workload_config(wl), plan=plan.as_dict()),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "peak_source": (peak_kind + " (MEASURED_PEAKS.json hbm_gbs: a read+write "
                                     "copy's bandwidth; a read-only stream can exceed it)")
                     if peak_kind == "measured" else "fallback",
                     "kernel": "decode read (decode_kernel, %s consumer)"
                               % {1: "CUDA-core", 2: "tensor-core",
                                  3: "tensor-core, vectors as rows",
                                  4: "tcgen05, tensor-memory accumulators"}[plan.consumer],
                     "bytes_per_launch": wl.read_bytes(), "us_per_launch": ms_read * 1e3,
                     "traffic": recorded_traffic(plan.consumer, wl.read_bytes())},
        "e2e": {"value": whole_job_gbs(step_bytes, ws, e2e_ms), "unit": "GB/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": K * launches_per_step,
        "gpu_launches_note": "timed region = K nsv_decode_step calls: kv_write_kernel + "
                             "decode_kernel each; the roofline's read-only loop is timed "
                             "separately (the counter-zeroing kernel + decode_kernel per launch)",
        "clocks": clocks,
    }
    if cpu is not None:
        gbs, nrows, secs, threads = cpu
        line["cpu_baseline"] = {
            "value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": "%d of %d rows of %s, %.1f s of oracle time (fp64, full-width rectangle "
                      "per row)" % (nrows, wl.rows, wl.name, secs)}
        if cpu1 is not None:
            g1, n1, s1, _ = cpu1
            line["cpu_baseline"]["single_core"] = {
                "value": g1, "unit": "GB/s", "cores": 1,
                "sample": "%d rows of %s, %.1f s of oracle time" % (n1, wl.name, s1)}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    from paged_kv_decode_nsv_gb300 import workloads as W
    wl = W.WORKLOADS[args.workload]()
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_nsv(args, wl)


if __name__ == "__main__":
    sys.exit(main())
