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
