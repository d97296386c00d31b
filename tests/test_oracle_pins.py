"""Pins for the FP64 oracle, checked against facts that do not come from the
oracle itself: closed forms, an exact rational brute force, finite
differences, affine/scan identities and the pages' worked offset example.

Each pin targets a class of mistake: a wrong decay order or base (beta = 0),
a wrong residual sign or pre-/post-update read (the delta write and the
interpolation property), a transposed state (K != V everywhere), a wrong
index in a closed-form sum (orthonormal keys), any algebra slip (exact
rationals), and any backward slip (finite differences + adjoint).
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(1234)
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_inputs(B, T, H, K, V, rng, s0=True, normalise=True):
    q = rng.normal(size=(B, T, H, K))
    k = rng.normal(size=(B, T, H, K))
    if normalise:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.normal(size=(B, T, H, V))
    g = -np.log1p(np.exp(rng.normal(size=(B, T, H))))
    beta = 1.0 / (1.0 + np.exp(-rng.normal(size=(B, T, H))))
    S0 = rng.normal(size=(B, H, V, K)) * 0.3 if s0 else None
    return q, k, v, g, beta, S0


# ---------------------------------------------------------------- closed forms
def test_beta_zero_is_pure_decay():
    """beta = 0: S_T = exp(sum g) S0 and out_t = scale exp(gamma_t) S0 q_t."""
    B, T, H, K, V = 2, 9, 2, 3, 5
    q, k, v, g, beta, S0 = rand_inputs(B, T, H, K, V, RNG)
    beta[:] = 0.0
    out, fin = oracle.gdn_fwd(q, k, v, g, beta, S0, scale=0.7)
    gam = np.cumsum(g, axis=1)                                   # [B,T,H]
    exp_out = 0.7 * np.exp(gam)[..., None] * np.einsum("bhvk,bthk->bthv", S0, q)
    np.testing.assert_allclose(out, exp_out, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(fin, np.exp(gam[:, -1])[..., None, None] * S0,
                               rtol=1e-13, atol=1e-15)


def test_delta_rule_write_and_interpolation():
    """Unit-norm key: after one token, S k = (1-beta) exp(g) S0 k + beta v, and
    directions orthogonal to k only decay: S u = exp(g) S0 u."""
    K, V = 4, 6
    for trial in range(5):
        q, k, v, g, beta, S0 = rand_inputs(1, 1, 1, K, V, RNG)
        kk = k[0, 0, 0]
        # read S k through the output by querying with q = k, scale 1
        out_k, fin = oracle.gdn_fwd(k, k, v, g, beta, S0, scale=1.0)
        a, b = math.exp(g[0, 0, 0]), beta[0, 0, 0]
        want = (1 - b) * a * (S0[0, 0] @ kk) + b * v[0, 0, 0]
        np.testing.assert_allclose(out_k[0, 0, 0], want, rtol=1e-12, atol=1e-13)
        u = RNG.normal(size=K)
        u -= (u @ kk) * kk
        np.testing.assert_allclose(fin[0, 0] @ u, a * (S0[0, 0] @ u), rtol=1e-11, atol=1e-13)
    # beta = 1, no decay: the state stores v exactly under key k
    q, k, v, g, beta, S0 = rand_inputs(1, 6, 1, K, V, RNG)
    beta[:] = 1.0
    g[:] = 0.0
    out, _ = oracle.gdn_fwd(k, k, v, g, beta, S0, scale=1.0)
    np.testing.assert_allclose(out[0, :, 0], v[0, :, 0], rtol=1e-12, atol=1e-12)


def test_orthonormal_keys_reduce_to_gated_linear_attention():
    """k_t = e_t (T <= K), S0 = 0: the delta correction vanishes and
    S_T = sum_t beta_t e^{gamma_T - gamma_t} v_t e_t^T,
    out_t = scale sum_{j<=t} beta_j e^{gamma_t - gamma_j} (q_t)_j v_j."""
    T, K, V = 7, 9, 4
    q, _, v, g, beta, _ = rand_inputs(1, T, 1, K, V, RNG)
    k = np.zeros((1, T, 1, K))
    for t in range(T):
        k[0, t, 0, t] = 1.0
    out, fin = oracle.gdn_fwd(q, k, v, g, beta, None, scale=0.5)
    gam = np.cumsum(g[0, :, 0])
    S_want = np.zeros((V, K))
    for t in range(T):
        S_want[:, t] = beta[0, t, 0] * math.exp(gam[-1] - gam[t]) * v[0, t, 0]
    np.testing.assert_allclose(fin[0, 0], S_want, rtol=1e-12, atol=1e-14)
    for t in range(T):
        o = sum(beta[0, j, 0] * math.exp(gam[t] - gam[j]) * q[0, t, 0, j] * v[0, j, 0]
                for j in range(t + 1))
        np.testing.assert_allclose(out[0, t, 0], 0.5 * o, rtol=1e-12, atol=1e-14)


def test_exact_rational_transition_products():
    """Brute force in exact rationals: with F_t = a_t (I - beta_t k_t k_t^T),
    S_t = S0 F_1..F_t + sum_{j<=t} beta_j v_j k_j^T F_{j+1}..F_t and
    out_t = scale S_t q_t.  The oracle gets g_t = log(a_t)."""
    rng = np.random.default_rng(7)
    T, K, V = 5, 3, 2

    def rat(lo, hi, den=8):
        return Fraction(int(rng.integers(lo * den, hi * den + 1)), den)

    a = [rat(0, 1) or Fraction(1, 2) for _ in range(T)]
    bt = [rat(0, 1) for _ in range(T)]
    kv = [[rat(-1, 1) for _ in range(K)] for _ in range(T)]
    qv = [[rat(-1, 1) for _ in range(K)] for _ in range(T)]
    vv = [[rat(-2, 2) for _ in range(V)] for _ in range(T)]
    S0 = [[rat(-1, 1) for _ in range(K)] for _ in range(V)]
    scale = Fraction(1, 2)

    def matmul(X, Y):
        return [[sum(X[i][m] * Y[m][j] for m in range(len(Y))) for j in range(len(Y[0]))]
                for i in range(len(X))]

    def F(t):
        return [[a[t] * ((1 if i == j else 0) - bt[t] * kv[t][i] * kv[t][j]) for j in range(K)]
                for i in range(K)]

    outs = []
    for t in range(T):
        S = S0
        for s in range(t + 1):
            S = matmul(S, F(s))
        for j in range(t + 1):
            term = [[bt[j] * vv[j][i] * kv[j][c] for c in range(K)] for i in range(V)]
            for s in range(j + 1, t + 1):
                term = matmul(term, F(s))
            S = [[S[i][c] + term[i][c] for c in range(K)] for i in range(V)]
        outs.append([scale * sum(S[i][c] * qv[t][c] for c in range(K)) for i in range(V)])
    S_T = S

    f = lambda X: np.array([[float(x) for x in row] for row in X])
    q = f(qv)[None, :, None, :]
    k = f(kv)[None, :, None, :]
    v = f(vv)[None, :, None, :]
    g = np.log(np.array([float(x) for x in a]))[None, :, None]
    b = np.array([float(x) for x in bt])[None, :, None]
    out, fin = oracle.gdn_fwd(q, k, v, g, b, f(S0)[None, None], scale=0.5)
    np.testing.assert_allclose(out[0, :, 0], f(outs), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(fin[0, 0], f(S_T), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------- state passing
def test_split_equals_sequential_bitwise():
    """[SF] Eq. 4-5: running [0,T1) then [T1,T) from the carried state is the
    same token sequence, so it is bit-identical to one pass."""
    B, T, H, K, V = 1, 50, 2, 4, 3
    q, k, v, g, beta, S0 = rand_inputs(B, T, H, K, V, RNG)
    out, fin = oracle.gdn_fwd(q, k, v, g, beta, S0)
    T1 = 21
    o1, f1 = oracle.gdn_fwd(q[:, :T1], k[:, :T1], v[:, :T1], g[:, :T1], beta[:, :T1], S0)
    o2, f2 = oracle.gdn_fwd(q[:, T1:], k[:, T1:], v[:, T1:], g[:, T1:], beta[:, T1:], f1)
    assert np.array_equal(np.concatenate([o1, o2], axis=1), out)
    assert np.array_equal(f2, fin)


def test_packed_equals_per_sequence_bitwise():
    """Packed stream with cu_seqlens == each sequence run alone (bitwise);
    an empty sequence passes its initial state through."""
    cu = [0, 40, 40, 232, 384]
    H, K, V = 2, 5, 3
    T = cu[-1] + 10                               # tail past cu[-1] is inactive
    q, k, v, g, beta, _ = rand_inputs(1, T, H, K, V, RNG)
    S0 = RNG.normal(size=(len(cu) - 1, H, V, K))
    out, fin = oracle.gdn_fwd(q, k, v, g, beta, S0, cu_seqlens=cu)
    for n in range(len(cu) - 1):
        s, e = cu[n], cu[n + 1]
        o1, f1 = oracle.gdn_fwd(q[:, s:e], k[:, s:e], v[:, s:e], g[:, s:e], beta[:, s:e],
                                S0[n:n + 1])
        assert np.array_equal(out[:, s:e], o1)
        assert np.array_equal(fin[n:n + 1], f1)
    assert np.isnan(out[:, cu[-1]:]).all()        # inactive rows untouched
    assert np.array_equal(fin[1], S0[1])          # empty sequence


def test_summary_is_the_affine_map_of_the_range():
    """[AG-CP]: S_out = S_in P + E for ANY entry state; linearity of
    S_in -> S_out - E; an empty range is the identity map."""
    B, T, H, K, V = 1, 70, 2, 5, 3
    q, k, v, g, beta, _ = rand_inputs(B, T, H, K, V, RNG)
    bounds = np.array([[0, 70], [13, 45], [30, 30]], dtype=np.int32)
    P, E = oracle.segment_summary(k, v, g, beta, bounds)
    for r, (s, e) in enumerate(bounds):
        for _ in range(3):
            Sin = RNG.normal(size=(1, H, V, K))
            _, fin = oracle.gdn_fwd(q[:, s:e], k[:, s:e], v[:, s:e], g[:, s:e],
                                    beta[:, s:e], Sin)
            np.testing.assert_allclose(fin[0], np.einsum("hvk,hkj->hvj", Sin[0], P[r]) + E[r],
                                       rtol=1e-11, atol=1e-12)
    assert np.array_equal(P[2], np.broadcast_to(np.eye(K), (H, K, K)))
    assert not E[2].any()


def test_scan_equals_carried_state_loop():
    """Entry states from the exclusive scan of the segment maps equal the
    states a carried-state segment loop reaches ([SF] Eq. 5)."""
    B, T, H, K, V = 1, 96, 2, 4, 6
    q, k, v, g, beta, S0 = rand_inputs(B, T, H, K, V, RNG)
    g *= 0.05                                      # keep the maps away from 0
    seg = [(0, 30), (30, 64), (64, 96)]
    P, E = oracle.segment_summary(k, v, g, beta, np.array(seg))
    entry, final = oracle.state_scan(P, E, S0[0])
    S = S0
    for j, (s, e) in enumerate(seg):
        np.testing.assert_allclose(entry[j], S[0], rtol=1e-11, atol=1e-13)
        _, S = oracle.gdn_fwd(q[:, s:e], k[:, s:e], v[:, s:e], g[:, s:e], beta[:, s:e], S)
    np.testing.assert_allclose(final, S[0], rtol=1e-11, atol=1e-13)


def _fragments_to_spans(cu_global, fragments):
    """Cut each rank's fragments at sequence boundaries; return per rank the
    list of (global_start, global_end, sequence) pieces, in listed order."""
    spans = []
    for frs in fragments:
        pieces = []
        for (fs, fe) in frs:
            for n in range(len(cu_global) - 1):
                s, e = max(fs, cu_global[n]), min(fe, cu_global[n + 1])
                if s < e:
                    pieces.append((s, e, n))
        spans.append(pieces)
    return spans


def test_page_offset_example_and_state_passing_over_ranks():
    """Golden: the page's zig-zag example.  Local cu_seqlens derived from the
    fragment table equal the printed ones; composing the pieces' summaries in
    slot order and running each piece from its composed entry state reproduces
    the single-stream outputs and final states."""
    with open(os.path.join(GOLDEN, "cp_offsets_example.json")) as f:
        gold = json.load(f)
    cu_g = gold["cu_seqlens_global"]
    spans = _fragments_to_spans(cu_g, gold["fragments_global"])
    for r, pieces in enumerate(spans):
        local = [0]
        for (s, e, _) in pieces:
            local.append(local[-1] + (e - s))
        assert local == gold["local_cu_seqlens"][r]

    H, K, V = 2, 4, 3
    T = cu_g[-1]
    q, k, v, g, beta, _ = rand_inputs(1, T, H, K, V, RNG)
    g *= 0.1
    S0 = RNG.normal(size=(3, H, V, K))
    out_ref, fin_ref = oracle.gdn_fwd(q, k, v, g, beta, S0, cu_seqlens=cu_g)

    # every piece's summary, then per sequence an exclusive scan in token order
    pieces = sorted({p for sp in spans for p in sp})
    P, E = oracle.segment_summary(k, v, g, beta, np.array([(s, e) for s, e, _ in pieces]))
    entry = {}
    fin = np.zeros_like(fin_ref)
    for n in range(3):
        idx = [i for i, p in enumerate(pieces) if p[2] == n]
        ent, f_n = oracle.state_scan(P[idx], E[idx], S0[n])
        for j, i in enumerate(idx):
            entry[pieces[i]] = ent[j]
        fin[n] = f_n
    np.testing.assert_allclose(fin, fin_ref, rtol=1e-10, atol=1e-12)
    # each rank runs its span packed, with per-piece entry states
    for pieces_r, cu_local in zip(spans, gold["local_cu_seqlens"]):
        rows = np.concatenate([np.arange(s, e) for s, e, _ in pieces_r])
        S_in = np.stack([entry[p] for p in pieces_r])
        o, _ = oracle.gdn_fwd(q[:, rows], k[:, rows], v[:, rows], g[:, rows], beta[:, rows],
                              S_in, cu_seqlens=cu_local)
        np.testing.assert_allclose(o[0], out_ref[0, rows], rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- backward
def _loss(inputs, dO, dSf, cu=None):
    q, k, v, g, beta, S0 = inputs
    out, fin = oracle.gdn_fwd(q, k, v, g, beta, S0, cu_seqlens=cu)
    m = ~np.isnan(out)
    return float((np.where(m, out, 0.0) * dO).sum() + (fin * dSf).sum())


@pytest.mark.parametrize("K,V,cu", [(8, 8, None), (5, 7, None), (4, 3, [0, 11, 11, 32])])
def test_backward_matches_central_differences(K, V, cu):
    """Every gradient (q, k, v, gate, beta, initial state) against FP64 central
    differences of <dO, out> + <dS_T, S_T>, h = 1e-6, relative error <= 1e-6."""
    T, H = 32, 1
    B = 2 if cu is None else 1
    rng = np.random.default_rng(K * 100 + V)
    q, k, v, g, beta, S0 = rand_inputs(B, T, H, K, V, rng, normalise=False)
    q *= 0.4; k *= 0.4
    N = B if cu is None else len(cu) - 1
    S0 = rng.normal(size=(N, H, V, K)) * 0.3
    dO = rng.normal(size=(B, T, H, V))
    dSf = rng.normal(size=(N, H, V, K))
    grads = oracle.gdn_bwd(q, k, v, g, beta, S0, dO, dSf, cu_seqlens=cu)
    inputs = [q, k, v, g, beta, S0]
    names = ["dq", "dk", "dv", "dg", "dbeta", "d_initial_state"]
    h = 1e-6
    for i, name in enumerate(names):
        x = inputs[i]
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = [a.copy() for a in inputs]
            xp[i][idx] += h
            lp = _loss(xp, dO, dSf, cu)
            xp[i][idx] -= 2 * h
            lm = _loss(xp, dO, dSf, cu)
            fd[idx] = (lp - lm) / (2 * h)
        an = grads[name]
        if cu is not None and name in ("dq", "dk", "dv", "dg", "dbeta"):
            an = an.copy()
            an[:, cu[-1]:] = 0.0                  # inactive rows: no gradient defined
        err = np.abs(an - fd).max() / max(np.abs(fd).max(), 1e-300)
        assert err <= 1e-6, (name, err)


def test_backward_adjoint_at_head_dim_64():
    """Directional derivative along a random direction of ALL inputs equals
    <grad, direction> (d = 64, two chunks' worth of tokens)."""
    B, T, H, K, V = 1, 40, 1, 64, 64
    rng = np.random.default_rng(99)
    q, k, v, g, beta, S0 = rand_inputs(B, T, H, K, V, rng)
    dO = rng.normal(size=(B, T, H, V))
    dSf = rng.normal(size=(B, H, V, K))
    grads = oracle.gdn_bwd(q, k, v, g, beta, S0, dO, dSf)
    inputs = [q, k, v, g, beta, S0]
    dirs = [rng.normal(size=x.shape) for x in inputs]
    h = 1e-6
    lp = _loss([x + h * d for x, d in zip(inputs, dirs)], dO, dSf)
    lm = _loss([x - h * d for x, d in zip(inputs, dirs)], dO, dSf)
    fd = (lp - lm) / (2 * h)
    an = sum((grads[n] * d).sum() for n, d in
             zip(["dq", "dk", "dv", "dg", "dbeta", "d_initial_state"], dirs))
    assert abs(fd - an) <= 1e-6 * max(abs(an), 1.0), (fd, an)


# ---------------------------------------------------------------- grouped heads
def test_grouped_heads_are_consecutive_blocks():
    """H = 4 value heads over HK = 2 query/key heads: heads 0, 1 read query/key head 0 and
    heads 2, 3 head 1 (consecutive blocks, not h % HK).  Changing query/key head 1 moves
    value heads 2 and 3 only; each value head equals a one-head run on its own q/k."""
    B, T, H, HK, K, V = 1, 20, 4, 2, 4, 3
    rng = np.random.default_rng(7)
    q, k, v, g, beta, S0 = rand_inputs(B, T, H, K, V, rng)
    q, k = q[:, :, :HK].copy(), k[:, :, :HK].copy()
    out, fin = oracle.gdn_fwd(q, k, v, g, beta, S0)
    q2, k2 = q.copy(), k.copy()
    q2[:, :, 1] = rng.normal(size=(B, T, K))
    k2[:, :, 1] = k2[:, :, 1][:, ::-1]
    out2, fin2 = oracle.gdn_fwd(q2, k2, v, g, beta, S0)
    assert np.array_equal(out[:, :, :2], out2[:, :, :2]) and np.array_equal(fin[:, :2], fin2[:, :2])
    assert not np.allclose(out[:, :, 2:], out2[:, :, 2:])
    for h in range(H):
        hk = h // (H // HK)
        o1, f1 = oracle.gdn_fwd(q[:, :, hk:hk + 1], k[:, :, hk:hk + 1], v[:, :, h:h + 1],
                                g[:, :, h:h + 1], beta[:, :, h:h + 1], S0[:, h:h + 1])
        assert np.array_equal(o1[:, :, 0], out[:, :, h]) and np.array_equal(f1[:, 0], fin[:, h])


def test_grouped_heads_gradients_match_central_differences():
    """dq and dk of shared query/key heads (H = 4 over HK = 2, and H = 3 over HK = 1)
    against FP64 central differences: the gradient of a shared head sums its block."""
    for H, HK in ((4, 2), (3, 1)):
        B, T, K, V = 1, 12, 4, 3
        rng = np.random.default_rng(10 * H + HK)
        q, k, v, g, beta, S0 = rand_inputs(B, T, H, K, V, rng, normalise=False)
        q, k = 0.4 * q[:, :, :HK], 0.4 * k[:, :, :HK]
        dO = rng.normal(size=(B, T, H, V))
        dSf = rng.normal(size=(B, H, V, K))
        grads = oracle.gdn_bwd(q, k, v, g, beta, S0, dO, dSf)
        inputs = [q, k, v, g, beta, S0]
        h = 1e-6
        for i, name in ((0, "dq"), (1, "dk")):
            x = inputs[i]
            assert grads[name].shape == x.shape
            fd = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp = [a.copy() for a in inputs]
                xp[i][idx] += h
                lp = _loss(xp, dO, dSf)
                xp[i][idx] -= 2 * h
                lm = _loss(xp, dO, dSf)
                fd[idx] = (lp - lm) / (2 * h)
            err = np.abs(grads[name] - fd).max() / np.abs(fd).max()
            assert err <= 1e-6, (H, HK, name, err)


def test_grouped_heads_summary_is_the_affine_map():
    """Segment summaries with shared keys: S_out = S_in @ P + S_ext for the forward run of
    the same range from a random S_in (H = 4 over HK = 2)."""
    B, T, H, HK, K, V = 1, 40, 4, 2, 5, 3
    rng = np.random.default_rng(11)
    q, k, v, g, beta, S0 = rand_inputs(B, T, H, K, V, rng)
    k = k[:, :, :HK].copy()
    q = q[:, :, :HK].copy()
    bounds = np.array([[7, 31]])
    P, E = oracle.segment_summary(k, v, g, beta, bounds)
    sl = slice(7, 31)
    _, fin = oracle.gdn_fwd(q[:, sl], k[:, sl], v[:, sl], g[:, sl], beta[:, sl], S0)
    assert np.allclose(fin[0], np.einsum("hvk,hkj->hvj", S0[0], P[0]) + E[0], atol=1e-12)


# ---------------------------------------------------------------- reverse (cotangent) maps
def test_reverse_map_is_affine_with_the_transposed_forward_transition():
    """For a segment, the backward's cotangent at its start equals dS_exit @ P^T + C for
    any exit cotangent, entry state and values: P from the forward summary (identity
    probing), C from the reverse summary (zero probing), the left side from the plain
    backward -- three oracle routines that share nothing but the token rule."""
    B, T, H, K, V = 1, 45, 2, 5, 3
    rng = np.random.default_rng(21)
    q, k, v, g, beta, S0 = rand_inputs(B, T, H, K, V, rng)
    g *= 0.3
    dO = rng.normal(size=(B, T, H, V))
    offs = [0, 19, 19, 45]
    P, _ = oracle.segment_summary(k, v, g, beta, np.array([[0, 19], [19, 19], [19, 45]]))
    C = oracle.segment_reverse_summary(q, k, g, beta, dO, offs)
    dSf = rng.normal(size=(3, H, V, K))
    S0r = rng.normal(size=(3, H, V, K))
    got = oracle.gdn_bwd(q, k, v, g, beta, S0r, dO, dSf, cu_seqlens=offs)["d_initial_state"]
    want = np.einsum("rhvk,rhjk->rhvj", dSf, P) + C
    assert np.allclose(got, want, rtol=1e-11, atol=1e-12)
    assert np.array_equal(C[1], np.zeros_like(C[1]))          # an empty segment adds nothing


def test_reverse_scan_equals_the_single_pass_backward():
    """Segment maps composed from the end reproduce the single-pass cotangents: the exit
    cotangent of each segment is the d_initial_state of the backward of everything after
    it, and the scan's last value is the whole sequence's d_initial_state."""
    B, T, H, K, V = 1, 60, 1, 4, 4
    rng = np.random.default_rng(22)
    q, k, v, g, beta, S0 = rand_inputs(B, T, H, K, V, rng)
    g *= 0.2
    dO = rng.normal(size=(B, T, H, V))
    dSf = rng.normal(size=(1, H, V, K))
    offs = [0, 17, 40, 60]
    bounds = np.array([[offs[i], offs[i + 1]] for i in range(3)])
    P, _ = oracle.segment_summary(k, v, g, beta, bounds)
    C = oracle.segment_reverse_summary(q, k, g, beta, dO, offs)
    exits, d0 = oracle.state_scan_reverse(P, C, dSf[0])
    full = oracle.gdn_bwd(q, k, v, g, beta, S0, dO, dSf)
    assert np.allclose(d0, full["d_initial_state"][0], rtol=1e-10, atol=1e-12)
    for j in range(3):
        sl = slice(offs[j + 1], T)
        tail = oracle.gdn_bwd(q[:, sl], k[:, sl], v[:, sl], g[:, sl], beta[:, sl],
                              S0, dO[:, sl], dSf)["d_initial_state"][0]
        if offs[j + 1] == T:
            tail = dSf[0]
        assert np.allclose(exits[j], tail, rtol=1e-10, atol=1e-12), j


# ---------------------------------------------------------------- paged state cache
def test_paged_cache_advances_like_one_pass():
    """Prefill through the cache in two calls (the first from fresh slots full of NaN,
    has_initial_state False) equals one forward over the whole sequences; padding rows are
    zero and every slot not selected keeps its bits."""
    B, T, H, K, V = 1, 40, 2, 4, 3
    rng = np.random.default_rng(31)
    q, k, v, g, beta, _ = rand_inputs(B, T, H, K, V, rng)
    lengths = [(9, 6), (0, 11), (7, 7)]                       # (first call, second call) per sequence
    whole_cu = np.cumsum([0] + [a + b for a, b in lengths])
    slots = np.array([3, -1, 1], np.int32)                    # sequence 1 is padding
    cache = rng.normal(size=(5, H, V, K))
    cache[3] = np.nan                                         # garbage: must never be read
    cache[1] = np.nan

    def part(which):
        rows = np.concatenate([np.arange(whole_cu[n] + (0 if which == 0 else lengths[n][0]),
                                         whole_cu[n] + lengths[n][0] + (0 if which == 0 else lengths[n][1]))
                               for n in range(3)]).astype(int)
        cu = np.cumsum([0] + [lengths[n][which] for n in range(3)])
        sl = lambda a: a[:, rows]
        return sl(q), sl(k), sl(v), sl(g), sl(beta), cu, rows

    q1, k1, v1, g1, b1, cu1, r1 = part(0)
    out1, c1 = oracle.paged_chunk_fwd(q1, k1, v1, g1, b1, cache, slots,
                                      has_initial_state=[False, True, False], cu_seqlens=cu1)
    q2, k2, v2, g2, b2, cu2, r2 = part(1)
    out2, c2 = oracle.paged_chunk_fwd(q2, k2, v2, g2, b2, c1, slots, cu_seqlens=cu2)
    ref_out, ref_fin = oracle.gdn_fwd(q, k, v, g, beta, None, cu_seqlens=whole_cu)
    for n, s in ((0, 3), (2, 1)):
        assert np.allclose(c2[s], ref_fin[n], rtol=1e-12, atol=1e-12)
    full = np.full_like(ref_out, np.nan)
    full[:, r1] = out1
    full[:, r2] = out2
    for n in (0, 2):
        rows = slice(whole_cu[n], whole_cu[n + 1])
        assert np.allclose(full[:, rows], ref_out[:, rows], rtol=1e-12, atol=1e-12)
    assert not full[:, whole_cu[1]:whole_cu[2]].any()         # padding: zero output
    for s in (0, 2, 4):
        assert np.array_equal(c2[s], cache[s])                # unselected slots keep their bits
