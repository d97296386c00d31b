"""Shared test helpers: oracle calls on the exact values handed to the GPU, the
error metric, and small input builders."""
import numpy as np
import torch

import oracle

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def f64(t):
    """Exact values of a tensor (BF16 upcast, not regenerated) as float64 NumPy."""
    if t is None:
        return None
    return t.detach().to("cpu", torch.float64).numpy()


def rel_err(x, ref, rows=None):
    """max |x - ref| / max |ref| over the defined rows (axis 1 of [B,T,...])."""
    x = f64(x) if isinstance(x, torch.Tensor) else np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    if rows is not None:
        x = x[:, rows]
        ref = ref[:, rows]
    den = np.abs(ref).max()
    return float(np.abs(x - ref).max() / (den if den > 0 else 1.0))


def active_rows(T, cu):
    if cu is None:
        return np.arange(T)
    cu = [int(c) for c in cu]
    return np.arange(cu[0], cu[-1])


def oracle_fwd(inp, scale=None, heads=None):
    """Oracle forward on a dict of torch inputs (optionally on a subset of heads)."""
    q, k, v, g, b = (f64(inp[n]) for n in ("q", "k", "v", "gate", "beta"))
    s0 = f64(inp.get("initial_state"))
    cu = inp.get("cu_seqlens")
    cu = None if cu is None else cu.cpu().numpy()
    if heads is not None:
        q, k, v, g, b = q[:, :, heads], k[:, :, heads], v[:, :, heads], g[:, :, heads], b[:, :, heads]
        s0 = None if s0 is None else s0[:, heads]
    return oracle.gdn_fwd(q, k, v, g, b, s0, cu_seqlens=cu, scale=scale)


def oracle_bwd(inp, scale=None):
    q, k, v, g, b = (f64(inp[n]) for n in ("q", "k", "v", "gate", "beta"))
    cu = inp.get("cu_seqlens")
    cu = None if cu is None else cu.cpu().numpy()
    return oracle.gdn_bwd(q, k, v, g, b, f64(inp.get("initial_state")), f64(inp["d_out"]),
                          f64(inp.get("d_final_state")), cu_seqlens=cu, scale=scale)


def small_inputs(B, T, H, D, dtype, seed, s0=True, lengths=None, grads=False, device="cuda"):
    """Config-0 distributions at arbitrary sizes (seeded)."""
    from chunked_linear_recurrence_gb300.workloads import Workload, make_inputs
    w = Workload("small", B, T, H, D, D, dtype, seed=seed, s0_std=0.1 if s0 else None,
                 lengths=lengths, with_grads=grads)
    return make_inputs(w, device)
