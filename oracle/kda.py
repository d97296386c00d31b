"""FP64 CPU oracle for Kimi Delta Attention (KDA) -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
use this module; the product library never imports it.

The per-token rule (Attention Gym "Linear Attention", section "Kimi Delta Attention",
chunk_kda / recurrent_kda parameter tables): the same delta rule as the gated delta rule,
except that the gate is a per-channel natural-log decay shaped like q, [B,T,H,K], and the
previous state is multiplied channelwise (along K) by exp(gate).  With the V-major state
S [V,K] of each (sequence, head):

    decayed  = S * exp(g_t)[None, :]          (column k scaled by exp(g_t[k]))
    residual = beta_t * (v_t - decayed @ k_t)
    S        = decayed + outer(residual, k_t)
    out_t    = scale * S @ q_t                (the query reads the updated state)

scale defaults to 1/sqrt(K).  Sequences are dense batch rows or packed cu_seqlens ranges;
rows outside every sequence are NaN in ``out``.  Plain Python over tokens, NumPy for the
per-token vector work; small cases only.
"""
from __future__ import annotations

import numpy as np


def _spans(B, T, cu_seqlens):
    if cu_seqlens is None:
        return [(b, 0, T) for b in range(B)]                  # (batch row, start, stop)
    cu = [int(c) for c in cu_seqlens]
    return [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]


def kda_fwd(q, k, v, g, beta, initial_state=None, cu_seqlens=None, scale=None):
    """Token-by-token forward.  q, k, g [B,T,H,K]; v [B,T,H,V]; beta [B,T,H];
    initial_state [N,H,V,K] or None.  Returns (out [B,T,H,V], final_state [N,H,V,K])."""
    q, k, v, g, beta = (np.asarray(x, np.float64) for x in (q, k, v, g, beta))
    B, T, H, K = q.shape
    V = v.shape[-1]
    scale = 1.0 / np.sqrt(K) if scale is None else float(scale)
    spans = _spans(B, T, cu_seqlens)
    out = np.full((B, T, H, V), np.nan)
    fin = np.zeros((len(spans), H, V, K))
    for n, (b, t0, t1) in enumerate(spans):
        for h in range(H):
            S = np.zeros((V, K)) if initial_state is None else np.array(initial_state[n, h], np.float64)
            for t in range(t0, t1):
                dec = S * np.exp(g[b, t, h])[None, :]
                r = beta[b, t, h] * (v[b, t, h] - dec @ k[b, t, h])
                S = dec + np.outer(r, k[b, t, h])
                out[b, t, h] = scale * (S @ q[b, t, h])
            fin[n, h] = S
    return out, fin


def kda_bwd(q, k, v, g, beta, initial_state, d_out, d_final_state=None, cu_seqlens=None,
            scale=None):
    """Reverse-mode gradients of <d_out, out> + <d_final_state, final_state> with respect
    to every input (the forward differentiated token by token, states recomputed).
    Returns dict dq, dk, dv, dg (per channel, [B,T,H,K]), dbeta, d_initial_state."""
    q, k, v, g, beta, d_out = (np.asarray(x, np.float64) for x in (q, k, v, g, beta, d_out))
    B, T, H, K = q.shape
    V = v.shape[-1]
    scale = 1.0 / np.sqrt(K) if scale is None else float(scale)
    spans = _spans(B, T, cu_seqlens)
    N = len(spans)
    res = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v),
               dg=np.zeros_like(g), dbeta=np.zeros_like(beta),
               d_initial_state=np.zeros((N, H, V, K)))
    for n, (b, t0, t1) in enumerate(spans):
        for h in range(H):
            S = np.zeros((V, K)) if initial_state is None else np.array(initial_state[n, h], np.float64)
            saved = []                                    # (S_prev, decayed, residual, S)
            for t in range(t0, t1):
                dec = S * np.exp(g[b, t, h])[None, :]
                r = beta[b, t, h] * (v[b, t, h] - dec @ k[b, t, h])
                S_new = dec + np.outer(r, k[b, t, h])
                saved.append((S, dec, r, S_new))
                S = S_new
            dS = np.zeros((V, K)) if d_final_state is None else np.array(d_final_state[n, h], np.float64)
            for t in range(t1 - 1, t0 - 1, -1):
                S_prev, dec, r, S_t = saved[t - t0]
                qt, kt, vt, bt = q[b, t, h], k[b, t, h], v[b, t, h], beta[b, t, h]
                do = d_out[b, t, h]
                # out = scale S_t q
                dS = dS + scale * np.outer(do, qt)
                res["dq"][b, t, h] = scale * (S_t.T @ do)
                # S_t = dec + r k^T
                dr = dS @ kt
                dk = dS.T @ r
                # r = beta (v - dec k)
                res["dv"][b, t, h] = bt * dr
                res["dbeta"][b, t, h] = dr @ (vt - dec @ kt)
                ddec = dS - bt * np.outer(dr, kt)
                dk = dk - bt * (dec.T @ dr)
                res["dk"][b, t, h] = dk
                # dec = S_prev * exp(g): column-wise
                res["dg"][b, t, h] = (ddec * dec).sum(axis=0)
                dS = ddec * np.exp(g[b, t, h])[None, :]
            res["d_initial_state"][n, h] = dS
    return res
