"""FP64 NumPy statement of the chunk-parallel form of Kimi Delta Attention (KDA).

Test-only design aid (never imported by the library), the KDA counterpart of
chunk_form.py: it writes out per 64-token chunk the algebra a chunked KDA kernel would
implement, so that the algebra is checked against the token-by-token oracle
(oracle/kda.py) before any kernel exists.  The pages give the per-token rule only; the
derivation is this library's reading of it.

Within a chunk with entry state S [V,K] and per-channel cumulative gates
gamma_i = sum_{m<=i} g_m (vectors over K), write the state in decay-normalised
coordinates S~_i = S_i diag(e^{-gamma_i}).  The token rule then becomes an ungated delta
rule that reads with K o e^{gamma} and writes with K o e^{-gamma}, which gives (all
exponents below are gamma_i - gamma_j <= 0 for j <= i, since gates are non-positive):

    Akk_ij = sum_c k_i[c] k_j[c] e^{gamma_i[c] - gamma_j[c]}      (j < i)
    Aqk_ij = sum_c q_i[c] k_j[c] e^{gamma_i[c] - gamma_j[c]}      (j <= i)
    T      = (I + diag(beta) Akk)^{-1}
    U      = T diag(beta) V,       W = T diag(beta) (K o e^{gamma})
    Delta  = U - W S^T
    O      = scale ((Q o e^{gamma}) S^T + Aqk Delta)
    S_next = S diag(e^{gamma_C}) + Delta^T (K o e^{gamma_C - gamma})

and the chunk's affine map S_next = S P_c + E_c:

    P_c = diag(e^{gamma_C}) - W^T (K o e^{gamma_C - gamma}),   E_c = U^T (K o e^{gamma_C - gamma}).
"""
import numpy as np

CHUNK = 64


def chunk_terms(q, k, v, g, beta):
    """Per-chunk factors for one (sequence, head): q, k, g [L,K], v [L,V], beta [L]."""
    L = k.shape[0]
    gam = np.cumsum(g, axis=0)                                       # [L, K]
    diff = np.minimum(gam[:, None, :] - gam[None, :, :], 0.0)        # [L, L, K], <= 0
    E = np.exp(diff)
    Akk = np.tril(np.einsum("ic,jc,ijc->ij", k, k, E), -1)
    Aqk = np.tril(np.einsum("ic,jc,ijc->ij", q, k, E))
    T = np.linalg.inv(np.eye(L) + beta[:, None] * Akk)
    U = T @ (beta[:, None] * v)
    W = T @ (beta[:, None] * (k * np.exp(gam)))
    kdec = k * np.exp(gam[-1][None, :] - gam)                        # K o e^{gamma_C - gamma}
    return gam, Aqk, U, W, kdec


def fwd_seq(q, k, v, g, beta, S, scale, C=CHUNK):
    """Chunked forward of one sequence/head.  Returns (out [L,V], S_final)."""
    L = q.shape[0]
    out = np.zeros((L, v.shape[1]))
    for c0 in range(0, L, C):
        sl = slice(c0, min(c0 + C, L))
        gam, Aqk, U, W, kdec = chunk_terms(q[sl], k[sl], v[sl], g[sl], beta[sl])
        Delta = U - W @ S.T
        out[sl] = scale * ((q[sl] * np.exp(gam)) @ S.T + Aqk @ Delta)
        S = S * np.exp(gam[-1])[None, :] + Delta.T @ kdec
    return out, S


def summary_seq(q, k, v, g, beta, C=CHUNK):
    """Chunk-composed affine map (P [K,K], E [V,K]) of one token range."""
    Kd = k.shape[1]
    P = np.eye(Kd)
    E = np.zeros((v.shape[1], Kd))
    for c0 in range(0, k.shape[0], C):
        sl = slice(c0, min(c0 + C, k.shape[0]))
        gam, _, U, W, kdec = chunk_terms(q[sl], k[sl], v[sl], g[sl], beta[sl])
        Pc = np.diag(np.exp(gam[-1])) - W.T @ kdec
        Ec = U.T @ kdec
        P, E = P @ Pc, E @ Pc + Ec
    return P, E


def bwd_chunk(q, k, v, g, beta, S, dO, dSn, scale):
    """Chunk-form backward of one chunk (L <= 64 rows) from its entry state S and the
    cotangent dSn of its exit state.  Returns (dq, dk, dv, dg [L,K], dbeta, dS_entry).

    The chunk algebra above, with read keys Kh = K o e^{gamma}, Qh = Q o e^{gamma}, write
    keys Kv = K o e^{-gamma} (Akk = tril(Kh Kv^T, -1), Aqk = tril(Qh Kv^T)) and end keys
    Kt = K o e^{gamma_C - gamma}, differentiated term by term; the gate gradient is the
    per-channel reverse cumulative sum of dgamma.  FP64 design aid: e^{-gamma} is formed
    directly, so keep gates moderate."""
    L, Kd = k.shape
    gam = np.cumsum(g, axis=0)
    Eh = np.exp(gam)
    Ev = np.exp(-gam)
    EC = np.exp(gam[-1])
    Kh, Qh, Kv = k * Eh, q * Eh, k * Ev
    Kt = Kv * EC[None, :]
    Akk = np.tril(Kh @ Kv.T, -1)
    A = beta[:, None] * Akk
    T = np.linalg.inv(np.eye(L) + A)
    U = T @ (beta[:, None] * v)
    W = T @ (beta[:, None] * Kh)
    Delta = U - W @ S.T
    Aqk = np.tril(Qh @ Kv.T)
    # S_next = S diag(EC) + Delta^T Kt
    dS = dSn * EC[None, :]
    dDelta = Kt @ dSn.T
    dKt = Delta @ dSn
    dEC = (dSn * S).sum(axis=0)
    # O = scale (Qh S^T + Aqk Delta)
    dQh = scale * dO @ S
    dS += scale * dO.T @ Qh
    dAqk = np.tril(scale * dO @ Delta.T)
    dDelta += scale * Aqk.T @ dO
    dQh += dAqk @ Kv
    dKv = dAqk.T @ Qh
    # Delta = U - W S^T
    dU = dDelta
    dW = -dDelta @ S
    dS += -dDelta.T @ W
    # U = T diag(beta) V ;  W = T diag(beta) Kh
    dT = dU @ (beta[:, None] * v).T + dW @ (beta[:, None] * Kh).T
    TU, TW = T.T @ dU, T.T @ dW
    dv = beta[:, None] * TU
    dbeta = (v * TU).sum(axis=1) + (Kh * TW).sum(axis=1)
    dKh = beta[:, None] * TW
    # T = (I + A)^{-1};  A = diag(beta) tril(Kh Kv^T, -1)
    dA = np.tril(-T.T @ dT @ T.T, -1)
    dbeta += (dA * Akk).sum(axis=1)
    dM = beta[:, None] * dA
    dKh += dM @ Kv
    dKv += dM.T @ Kh
    # back to Q, K and gamma
    dq = dQh * Eh
    dk = dKh * Eh + dKv * Ev + dKt * np.exp(gam[-1][None, :] - gam)
    dgam = dQh * q * Eh + dKh * k * Eh - dKv * Kv - dKt * Kt
    dgamC = (dKt * Kt).sum(axis=0) + dEC * EC
    dgam[-1] += dgamC
    dg = np.cumsum(dgam[::-1], axis=0)[::-1]
    return dq, dk, dv, dg, dbeta, dS


def bwd_seq(q, k, v, g, beta, S0, dO, dSf, scale, C=CHUNK):
    """Chunk-form backward of one sequence/head: the forward's chunk-entry states, then the
    chunks in reverse with the cotangent carried from each chunk's start to the one before."""
    L = q.shape[0]
    starts = list(range(0, L, C))
    entries, S = [], S0
    for c0 in starts:
        sl = slice(c0, min(c0 + C, L))
        entries.append(S)
        _, S = fwd_seq(q[sl], k[sl], v[sl], g[sl], beta[sl], S, scale, C)
    grads = [np.zeros_like(x) for x in (q, k, v, g, beta)]
    dS = dSf
    for ci in range(len(starts) - 1, -1, -1):
        sl = slice(starts[ci], min(starts[ci] + C, L))
        r = bwd_chunk(q[sl], k[sl], v[sl], g[sl], beta[sl], entries[ci], dO[sl], dS, scale)
        for gr, part in zip(grads, r[:5]):
            gr[sl] = part
        dS = r[5]
    return (*grads, dS)


def decay_products_stable(x, k, g, sub=16, dtype=np.float32):
    """Aq_ij = sum_c x_i[c] k_j[c] e^{gamma_i[c] - gamma_j[c]} for j <= i (x = q or k), in a
    form whose exponentials stay bounded: the chunk is cut into `sub`-token blocks with the
    reference point r_I at the start of block I.  For j in an earlier block J,
    e^{gamma_i - gamma_j} = e^{gamma_i - gamma_rI} e^{gamma_rI - gamma_j}, both exponents <= 0,
    so block (I, J) is one product of two bounded factors; within a block the per-entry
    exponentials e^{gamma_i - gamma_j} <= 1 are formed directly.  Computed in `dtype`."""
    x, k, g = (np.asarray(a, dtype) for a in (x, k, g))
    L, Kd = k.shape
    gam = np.cumsum(g, axis=0, dtype=dtype)
    out = np.zeros((L, L), dtype)
    for I0 in range(0, L, sub):
        I = slice(I0, min(I0 + sub, L))
        ref = gam[I0]
        xa = x[I] * np.exp(np.minimum(gam[I] - ref, 0))             # rows of block I, <= 1
        if I0 > 0:
            J = slice(0, I0)
            kb = k[J] * np.exp(np.minimum(ref - gam[J], 0))          # earlier columns, <= 1
            out[I, J] = xa @ kb.T
        d = np.minimum(gam[I][:, None, :] - gam[I][None, :, :], 0)  # within the block
        out[I, I] = np.tril(np.einsum("ic,jc,ijc->ij", x[I], k[I], np.exp(d)))
    return out
