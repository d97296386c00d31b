"""FP64 NumPy statement of the chunk-parallel form of the gated delta rule.

Test-only design aid (never imported by the library): it writes out, per
64-token chunk, the algebra the CUDA kernels implement, so the tests can check
that algebra against the token-by-token oracle before any kernel is trusted.
The pages name the pieces (WY factors, a hierarchical triangular solve, raw
QK/KK contracted before masked non-positive decay differences, corrected
values V_new) but print no formulas; the derivation here is this library's
reading of them.

For a chunk with entry state S [V,K], per-token gates g, gamma_i = sum_{m<=i} g_m:

    A_ij   = beta_i e^{gamma_i - gamma_j} (k_i . k_j)          (j < i)
    T      = (I + A)^{-1}                                       (unit lower)
    U      = T diag(beta) V,    W = T diag(beta e^gamma) K
    Delta  = U - W S^T                                          (V_new)
    O      = scale (diag(e^gamma) Q S^T + (M o Gamma o Q K^T) Delta)
    S_next = e^{gamma_C} S + Delta^T diag(e^{gamma_C - gamma}) K

and the chunk's affine map S_next = S P_c + E_c:

    P_c = e^{gamma_C} I - W^T diag(e^{gamma_C - gamma}) K,
    E_c = U^T diag(e^{gamma_C - gamma}) K.
"""
import numpy as np

CHUNK = 64


def chunk_terms(k, v, g, beta):
    """Per-chunk factors for one (sequence, head): k [L,K], v [L,V], g, beta [L]."""
    L = k.shape[0]
    gam = np.cumsum(g)
    Gam = np.exp(np.minimum(gam[:, None] - gam[None, :], 0.0))
    A = np.tril(beta[:, None] * Gam * (k @ k.T), -1)
    T = np.linalg.inv(np.eye(L) + A)
    U = T @ (beta[:, None] * v)
    W = T @ ((beta * np.exp(gam))[:, None] * k)
    dec = np.exp(gam[-1] - gam)
    return gam, Gam, U, W, dec


def fwd_seq(q, k, v, g, beta, S, scale, C=CHUNK):
    """Chunked forward of one sequence/head.  Returns (out [L,V], S_final)."""
    L = q.shape[0]
    out = np.zeros((L, v.shape[1]))
    for c0 in range(0, L, C):
        sl = slice(c0, min(c0 + C, L))
        qc, kc = q[sl], k[sl]
        gam, Gam, U, W, dec = chunk_terms(kc, v[sl], g[sl], beta[sl])
        Delta = U - W @ S.T
        Aqk = np.tril(Gam * (qc @ kc.T))
        out[sl] = scale * (np.exp(gam)[:, None] * (qc @ S.T) + Aqk @ Delta)
        S = np.exp(gam[-1]) * S + Delta.T @ (dec[:, None] * kc)
    return out, S


def summary_seq(k, v, g, beta, C=CHUNK):
    """Chunk-composed affine map (P [K,K], E [V,K]) of one token range."""
    Kd = k.shape[1]
    P = np.eye(Kd)
    E = np.zeros((v.shape[1], Kd))
    for c0 in range(0, k.shape[0], C):
        sl = slice(c0, min(c0 + C, k.shape[0]))
        gam, _, U, W, dec = chunk_terms(k[sl], v[sl], g[sl], beta[sl])
        Pc = np.exp(gam[-1]) * np.eye(Kd) - W.T @ (dec[:, None] * k[sl])
        Ec = U.T @ (dec[:, None] * k[sl])
        P, E = P @ Pc, E @ Pc + Ec
    return P, E


def bwd_chunk(q, k, v, g, beta, S, dO, dSn, scale):
    """Chunk-form backward of one chunk (L <= 64 rows) given its entry state S
    and the cotangent dSn of its exit state.  Returns (dq, dk, dv, dg, dbeta,
    dS_entry).  This is the algebra the CUDA backward follows, step by step."""
    L, Kd = k.shape
    gam = np.cumsum(g)
    eg = np.exp(gam)
    dec = np.exp(gam[-1] - gam)
    Gam = np.exp(np.minimum(gam[:, None] - gam[None, :], 0.0))
    low = np.tril(np.ones((L, L)), -1)
    lowd = np.tril(np.ones((L, L)))
    Ak = low * Gam * (k @ k.T)                 # A = diag(beta) Ak
    T = np.linalg.inv(np.eye(L) + beta[:, None] * Ak)
    Aqk = lowd * Gam * (q @ k.T)
    W = T @ ((beta * eg)[:, None] * k)
    U = T @ (beta[:, None] * v)
    Delta = U - W @ S.T
    dgam = np.zeros(L)
    # reverse chain pieces
    dDelta = scale * Aqk.T @ dO + dec[:, None] * (k @ dSn.T)
    dS_entry = eg[-1] * dSn + scale * dO.T @ (eg[:, None] * q) - dDelta.T @ W
    # output: O = scale (diag(eg) Q S^T + Aqk Delta)
    dAqk = scale * dO @ Delta.T
    rho = dAqk * Aqk
    dgam += rho.sum(1) - rho.sum(0)
    G = dAqk * Gam * lowd
    dQfirst = scale * eg[:, None] * (dO @ S)
    dq = dQfirst + G @ k
    dk = G.T @ q
    dgam += (q * dQfirst).sum(1)
    # exit state: S_next = eg_C S + Delta^T diag(dec) K
    Z = Delta @ dSn
    dk += dec[:, None] * Z
    ddec = (k * Z).sum(1)
    dgam -= dec * ddec
    dgam[-1] += (dec * ddec).sum() + eg[-1] * (dSn * S).sum()
    # Delta = U - W S^T
    dW = -dDelta @ S
    TtdU = T.T @ dDelta
    dv = beta[:, None] * TtdU
    dbeta = (v * TtdU).sum(1)
    dT = dDelta @ (beta[:, None] * v).T
    TtdW = T.T @ dW
    dk += (beta * eg)[:, None] * TtdW
    kt = (k * TtdW).sum(1)
    dbeta += eg * kt
    dgam += beta * eg * kt
    dT += dW @ ((beta * eg)[:, None] * k).T
    dA = -(T.T @ dT @ T.T) * low
    dbeta += (dA * Ak).sum(1)
    rhoA = dA * beta[:, None] * Ak
    dgam += rhoA.sum(1) - rhoA.sum(0)
    dKK = dA * beta[:, None] * Gam * low
    dk += dKK @ k + dKK.T @ k
    dg = np.cumsum(dgam[::-1])[::-1]
    return dq, dk, dv, dg, dbeta, dS_entry


def bwd_seq(q, k, v, g, beta, S0, dO, dSf, scale, C=CHUNK):
    """Chunk-form backward of one sequence: replay entry states, then walk the
    chunks in reverse carrying the state cotangent."""
    L = q.shape[0]
    starts = list(range(0, L, C))
    ents = []
    S = S0
    for c0 in starts:
        ents.append(S)
        sl = slice(c0, min(c0 + C, L))
        _, S = fwd_seq(q[sl], k[sl], v[sl], g[sl], beta[sl], S, scale, C)
    grads = [np.zeros_like(x) for x in (q, k, v, g, beta)]
    dS = dSf
    for c0, Sc in zip(reversed(starts), reversed(ents)):
        sl = slice(c0, min(c0 + C, L))
        dq, dk, dv, dg, db, dS = bwd_chunk(q[sl], k[sl], v[sl], g[sl], beta[sl], Sc,
                                          dO[sl], dS, scale)
        for gr, x in zip(grads, (dq, dk, dv, dg, db)):
            gr[sl] = x
    return (*grads, dS)
