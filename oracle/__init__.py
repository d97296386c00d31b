"""FP64 CPU oracle for the gated delta rule -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library
(``chunked_linear_recurrence_gb300``) never imports it, and the two share no
code: the oracle is the plain token-by-token definition from the Attention Gym
"Linear Attention" page, section "Gated Delta Rule", written in C
(``gdn_oracle.c``) and run in FP64 on the host.

Functions take and return NumPy float64 arrays in the library's layouts::

    q, k [B,T,HK,K]   v, out [B,T,H,V]   g, beta [B,T,H]   state [N,H,V,K]

HK divides H (grouped heads, the chunk_gdn parameter table of the same page):
value head h reads query/key head h // (H // HK), i.e. each block of H // HK
consecutive value heads shares one query/key head.  The oracle takes that
definition literally: q and k are repeated per block before the per-head
recurrence, and the gradient of a shared query/key head is the sum over its block.

Pins (see ``tests/test_oracle_pins.py``): closed forms for beta = 0, for the
delta rule's exact write, for orthonormal keys and for T = 1; an exact
rational brute force of the transition products; split == sequential;
affine-map and scan identities; finite differences and an adjoint test for the
backward.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (-O2, OpenMP).  Returns the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int32)
            I = ctypes.c_int
            lib.oracle_gdn_fwd.argtypes = [I, I, I, I, I, I, ip, dp, dp, dp, dp, dp, dp,
                                           ctypes.c_double, dp, dp]
            lib.oracle_gdn_bwd.argtypes = [I, I, I, I, I, I, ip, dp, dp, dp, dp, dp, dp,
                                           ctypes.c_double, dp, dp, dp, dp, dp, dp, dp, dp]
            lib.oracle_gdn_summary.argtypes = [I, I, I, I, I, dp, dp, dp, dp, ip, I, dp, dp]
            lib.oracle_state_scan.argtypes = [I, I, I, I, dp, dp, dp, dp, dp]
            for f in (lib.oracle_gdn_fwd, lib.oracle_gdn_bwd, lib.oracle_gdn_summary,
                      lib.oracle_state_scan):
                f.restype = I
            lib.oracle_num_threads.restype = I
            _lib = lib
    return _lib


def _d(a):
    """Contiguous float64 copy (or None) and its ctypes pointer."""
    if a is None:
        return None, None
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _i(a):
    if a is None:
        return None, None
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def num_threads() -> int:
    """OpenMP threads the oracle runs with (OMP_NUM_THREADS, else all cores)."""
    return int(_load().oracle_num_threads())


def _shape(q, v, cu_seqlens):
    B, T, H, K = q.shape
    V = v.shape[-1]
    N = B if cu_seqlens is None else len(cu_seqlens) - 1
    return B, T, H, K, V, N


def _per_value_head(x, H):
    """[B,T,HK,K] query/key heads -> [B,T,H,K]: value head h reads head h // (H // HK)."""
    x = np.asarray(x, np.float64)
    HK = x.shape[2]
    if H % HK:
        raise ValueError(f"query/key heads {HK} do not divide value heads {H}")
    return np.repeat(x, H // HK, axis=2) if HK != H else x


def _per_shared_head(dx, HK):
    """Gradients per value head [B,T,H,K] -> per shared query/key head [B,T,HK,K] (sum
    over each block of H // HK consecutive value heads)."""
    B, T, H, K = dx.shape
    return dx.reshape(B, T, HK, H // HK, K).sum(axis=3) if HK != H else dx


def gdn_fwd(q, k, v, g, beta, initial_state=None, cu_seqlens=None, scale=None):
    """Token-by-token forward.  Returns (out [B,T,H,V], final_state [N,H,V,K]).

    Rows of ``out`` outside every sequence are NaN.
    """
    lib = _load()
    Hv = np.asarray(v).shape[2]
    q, qp = _d(_per_value_head(q, Hv)); k, kp = _d(_per_value_head(k, Hv))
    v, vp = _d(v); g, gp = _d(g); beta, bp = _d(beta)
    B, T, H, K, V, N = _shape(q, v, cu_seqlens)
    s0, s0p = _d(initial_state)
    cu, cup = _i(cu_seqlens)
    if scale is None:
        scale = 1.0 / np.sqrt(K)
    out = np.full((B, T, H, V), np.nan)
    fin = np.zeros((N, H, V, K))
    rc = lib.oracle_gdn_fwd(B, T, H, K, V, N, cup, qp, kp, vp, gp, bp, s0p, float(scale),
                            out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                            fin.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    if rc != 0:
        raise ValueError("oracle_gdn_fwd: malformed arguments")
    return out, fin


def gdn_bwd(q, k, v, g, beta, initial_state, d_out, d_final_state=None,
            cu_seqlens=None, scale=None):
    """Reverse-mode gradients of (out, final_state) w.r.t. every input.

    Returns dict with dq, dk, dv, dg, dbeta, d_initial_state (FP64); dq and dk have the
    shape of q and k (grouped heads: summed over each head's block of value heads).
    """
    lib = _load()
    HK = np.asarray(q).shape[2]
    Hv = np.asarray(v).shape[2]
    q, qp = _d(_per_value_head(q, Hv)); k, kp = _d(_per_value_head(k, Hv))
    v, vp = _d(v); g, gp = _d(g); beta, bp = _d(beta)
    B, T, H, K, V, N = _shape(q, v, cu_seqlens)
    s0, s0p = _d(initial_state)
    do, dop = _d(d_out)
    dsf, dsfp = _d(d_final_state)
    cu, cup = _i(cu_seqlens)
    if scale is None:
        scale = 1.0 / np.sqrt(K)
    res = {n: np.zeros(s) for n, s in (("dq", q.shape), ("dk", k.shape), ("dv", v.shape),
                                       ("dg", g.shape), ("dbeta", beta.shape),
                                       ("d_initial_state", (N, H, V, K)))}
    ptr = {n: a.ctypes.data_as(ctypes.POINTER(ctypes.c_double)) for n, a in res.items()}
    rc = lib.oracle_gdn_bwd(B, T, H, K, V, N, cup, qp, kp, vp, gp, bp, s0p, float(scale),
                            dop, dsfp, ptr["dq"], ptr["dk"], ptr["dv"], ptr["dg"],
                            ptr["dbeta"], ptr["d_initial_state"])
    if rc != 0:
        raise ValueError("oracle_gdn_bwd: malformed arguments")
    res["dq"] = _per_shared_head(res["dq"], HK)
    res["dk"] = _per_shared_head(res["dk"], HK)
    return res


def segment_summary(k, v, g, beta, bounds):
    """Affine map of each token range by probing.  bounds: int [R,2] flattened rows.

    Returns (P [R,H,K,K], E [R,H,V,K]) with S_out = S_in @ P + E.
    """
    lib = _load()
    k, kp = _d(_per_value_head(k, np.asarray(v).shape[2]))
    v, vp = _d(v); g, gp = _d(g); beta, bp = _d(beta)
    B, T, H, K = k.shape
    V = v.shape[-1]
    bd, bdp = _i(np.asarray(bounds).reshape(-1, 2))
    R = bd.shape[0]
    P = np.zeros((R, H, K, K))
    E = np.zeros((R, H, V, K))
    rc = lib.oracle_gdn_summary(B, T, H, K, V, kp, vp, gp, bp, bdp, R,
                                P.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                E.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    if rc != 0:
        raise ValueError("oracle_gdn_summary: malformed bounds")
    return P, E


def state_scan(P, E, initial_state=None):
    """Exclusive scan: entry_0 = S0, entry_{j+1} = entry_j @ P_j + E_j.

    Returns (entry_states [R,H,V,K], final_state [H,V,K]).
    """
    lib = _load()
    P, Pp = _d(P); E, Ep = _d(E)
    R, H, K, _ = P.shape
    V = E.shape[2]
    s0, s0p = _d(initial_state)
    entry = np.zeros((R, H, V, K))
    fin = np.zeros((H, V, K))
    lib.oracle_state_scan(R, H, K, V, Pp, Ep, s0p,
                          entry.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                          fin.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return entry, fin


def segment_reverse_summary(q, k, g, beta, d_out, seg_offsets):
    """Reverse (cotangent) map of each segment by probing, the backward counterpart of
    ``segment_summary`` (Attention Gym "Linear Attention", section "Context Parallelism":
    the backward carries the state cotangent from the end of the sequence to its start,
    and every token step's adjoint is affine in it).

    Segments are consecutive token ranges of one batch row, given as offsets [R+1] with the
    cu_seqlens convention (q, k, d_out [1,T,...]).  The cotangent at a segment's start is
    dS_entry = dS_exit @ P^T + C, with P the segment's forward transition; C is the
    cotangent that the segment's own output gradients produce at its start when nothing
    flows in at its end.  It is probed here by the backward of each segment run as its own
    sequence with a zero exit cotangent (zero values and entry state: the cotangent chain
    reads neither).  Returns C [R,H,V,K].
    """
    q = np.asarray(q, np.float64)
    d_out = np.asarray(d_out, np.float64)
    B, T, H, V = d_out.shape
    K = np.asarray(k).shape[-1]
    R = len(seg_offsets) - 1
    v0 = np.zeros((B, T, H, V))
    s0 = np.zeros((R, H, V, K))
    res = gdn_bwd(q, k, v0, g, beta, s0, d_out, np.zeros((R, H, V, K)), cu_seqlens=seg_offsets)
    return res["d_initial_state"]


def state_scan_reverse(P, C, d_final_state=None):
    """Exclusive scan of the cotangent maps from the last segment to the first:
    exit_{R-1} = dS_final, exit_{j-1} = exit_j @ P_j^T + C_j; the cotangent at the start of
    segment 0 is exit_0 @ P_0^T + C_0.  Returns (exit cotangents [R,H,V,K], d_initial [H,V,K]).
    """
    P = np.asarray(P, np.float64)
    C = np.asarray(C, np.float64)
    R, H, K, _ = P.shape
    V = C.shape[2]
    cur = np.zeros((H, V, K)) if d_final_state is None else np.array(d_final_state, np.float64)
    exits = np.zeros((R, H, V, K))
    for j in range(R - 1, -1, -1):
        exits[j] = cur
        cur = np.einsum("hvk,hjk->hvj", cur, P[j]) + C[j]
    return exits, cur


def paged_chunk_fwd(q, k, v, g, beta, state_cache, state_indices, has_initial_state=None,
                    cu_seqlens=None, scale=None):
    """The forward advancing a paged state cache (Attention Gym "Linear Attention",
    paged_chunk_gdn): sequence n starts from slot state_indices[n] (from zero when
    has_initial_state[n] is False) and leaves its final state there; an index outside
    [1, num_slots) is padding -- zero output rows, the cache untouched.

    Returns (out [B,T,H,V], the advanced cache)."""
    cache = np.array(state_cache, np.float64)
    idx = np.asarray(state_indices).astype(np.int64)
    N = len(idx)
    num_slots = cache.shape[0]
    live = (idx > 0) & (idx < num_slots)
    load_ = live if has_initial_state is None else live & np.asarray(has_initial_state, bool)
    S0 = np.zeros((N,) + cache.shape[1:])
    for n in range(N):
        if load_[n]:
            S0[n] = cache[idx[n]]
    out, fin = gdn_fwd(q, k, v, g, beta, S0, cu_seqlens=cu_seqlens, scale=scale)
    for n in range(N):
        if live[n]:
            cache[idx[n]] = fin[n]
        elif cu_seqlens is None:
            out[n] = 0.0
        else:
            out[:, int(cu_seqlens[n]):int(cu_seqlens[n + 1])] = 0.0
    return out, cache
