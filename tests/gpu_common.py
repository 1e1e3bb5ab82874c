"""Helpers shared by the GPU parity tests: run a step through the C ABI and
compute the same step with the oracle on the same seeded inputs.

Tolerances (the bar the path is held to):
  fp32 KV   max |gpu - oracle| <= 1e-5 over every output element
  bf16 KV   per (row, head): max |gpu - oracle| / max(max |oracle|, 1e-6) <= 2e-2
            (the oracle sees the same bf16 values, widened exactly)
  append    bit-exact
"""

import numpy as np

import oracle
from paged_kv_decode_nsv_gb300 import workloads as W

F32_ABS_TOL = 1e-5
BF16_REL_TOL = 2e-2


def torch_mod():
    import torch
    return torch


def device_inputs(wl, value_seed=None):
    torch = torch_mod()
    q, kp, vp, kn, vn = W.device_values(wl, "cuda", value_seed)
    return dict(q=q, k_pool=kp, v_pool=vp, k_new=kn, v_new=vn,
                block_tables=torch.from_numpy(wl.block_tables).cuda(),
                context_lens=torch.from_numpy(wl.context_lens).cuda(),
                write_slots=torch.from_numpy(wl.write_slots).cuda())


def host_copy(inp):
    """Numpy copies of the device inputs (take them before any step runs)."""
    return {k: W.to_numpy(inp[k]) for k in ("q", "k_pool", "v_pool", "k_new", "v_new")}


def default_plan(inp):
    from paged_kv_decode_nsv_gb300 import nsv
    return nsv.plan_split(nsv.shape_of(inp["q"], inp["k_pool"], inp["block_tables"]))


def gpu_step(wl, inp, plan=None, library_workspace=False, out=None):
    """kv_write + decode through nsv_decode_step; returns the output tensor."""
    from paged_kv_decode_nsv_gb300 import nsv
    torch = torch_mod()
    if out is None:
        out = torch.empty_like(inp["q"])
    ws = None
    if not library_workspace:
        if plan is None:
            plan = default_plan(inp)
        ws = nsv.workspace_for(plan)
    nsv.decode_step(inp["q"], inp["k_new"], inp["v_new"], inp["write_slots"], inp["k_pool"],
                    inp["v_pool"], inp["block_tables"], inp["context_lens"], wl.scale, out,
                    workspace=ws, plan=None if library_workspace else plan)
    torch.cuda.synchronize()
    return out


def gpu_read(wl, inp, plan=None, out=None):
    """Decode read only (no append), caller workspace."""
    from paged_kv_decode_nsv_gb300 import nsv
    torch = torch_mod()
    if out is None:
        out = torch.empty_like(inp["q"])
    if plan is None:
        plan = default_plan(inp)
    ws = nsv.workspace_for(plan)
    nsv.paged_decode_ws(inp["q"], inp["k_pool"], inp["v_pool"], inp["block_tables"],
                        inp["context_lens"], wl.scale, out, workspace=ws, plan=plan)
    torch.cuda.synchronize()
    return out


def oracle_step(wl, host, rows=None, threads=0):
    """The oracle's append then read on host copies; fp64 [rows, H, D]."""
    kp = host["k_pool"].copy()
    vp = host["v_pool"].copy()
    oracle.kv_write(_flat(host["k_new"]), _flat(host["v_new"]),
                    np.asarray(wl.write_slots).reshape(-1), kp, vp)
    return oracle.paged_decode(host["q"], kp, vp, wl.block_tables, wl.context_lens, wl.scale,
                               rows=rows, threads=threads)


def _flat(new):
    """[R, NQ, Hkv, D] new tokens -> [R*NQ, Hkv, D] (the append is per token)."""
    return new.reshape(-1, new.shape[-2], new.shape[-1])


def oracle_read(wl, host, rows=None, threads=0):
    """The oracle's read alone on host copies."""
    return oracle.paged_decode(host["q"], host["k_pool"], host["v_pool"], wl.block_tables,
                               wl.context_lens, wl.scale, rows=rows, threads=threads)


def oracle_step_sampled(wl, inp, rows, threads=0):
    """The oracle on a compact host copy of just `rows`' blocks (pre-step).

    Call it before the GPU step modifies the pool.  Relabelling physical
    blocks is an invariance of the read, so the compact pool gives the same
    result as the full one.
    """
    torch = torch_mod()
    rows = list(rows)
    blocks, tables, slots = W.compact_rows(wl, rows)
    idx = torch.from_numpy(blocks).cuda()
    # the sink block (and a spare real block when every sampled row is empty)
    sink = torch.zeros((1 if len(blocks) else 2,) + tuple(inp["k_pool"].shape[1:]),
                       dtype=inp["k_pool"].dtype, device="cuda")
    kp = W.to_numpy(torch.cat([inp["k_pool"].index_select(0, idx), sink]))
    vp = W.to_numpy(torch.cat([inp["v_pool"].index_select(0, idx), sink]))
    ridx = torch.tensor(rows, dtype=torch.long, device="cuda")
    q = W.to_numpy(inp["q"].index_select(0, ridx))
    kn = W.to_numpy(inp["k_new"].index_select(0, ridx))
    vn = W.to_numpy(inp["v_new"].index_select(0, ridx))
    ctx = wl.context_lens[rows]
    oracle.kv_write(_flat(kn), _flat(vn), slots.reshape(-1), kp, vp)
    return oracle.paged_decode(q, kp, vp, tables, ctx, wl.scale, threads=threads)


def gpu_out_f64(out):
    torch = torch_mod()
    return out.detach().to(torch.float64).cpu().numpy()


def max_rel_per_head(got, ref):
    num = np.max(np.abs(got - ref), axis=-1)
    den = np.maximum(np.max(np.abs(ref), axis=-1), 1e-6)
    return float(np.max(num / den)) if num.size else 0.0


def assert_parity(dtype, got, ref):
    """got, ref: float64 arrays of one shape; returns the error measured."""
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), "non-finite GPU output"
    if dtype == "f32":
        err = float(np.max(np.abs(got - ref))) if got.size else 0.0
        assert err <= F32_ABS_TOL, "fp32 max-abs error %.3g > %.0e" % (err, F32_ABS_TOL)
        return err
    err = max_rel_per_head(got, ref)
    assert err <= BF16_REL_TOL, "bf16 max-rel error %.3g > %.0e" % (err, BF16_REL_TOL)
    return err


def status(clear=True):
    from paged_kv_decode_nsv_gb300 import nsv
    return nsv.device_status(clear)
