"""Pins for the KDA oracle (oracle/kda.py), against facts that do not come from it: with
one gate value for every channel KDA is the gated delta rule, so it must match the C GDN
oracle forward and backward; a beta = 0 closed form with K != V (catches decaying rows
instead of columns); an orthonormal-key closed form (per-channel decay indices); central
differences of every gradient; packed == per-sequence."""
import numpy as np
import pytest

import oracle
from oracle import kda


def _inputs(B, T, H, K, V, rng, per_channel=True):
    q = rng.normal(size=(B, T, H, K))
    k = rng.normal(size=(B, T, H, K))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.normal(size=(B, T, H, V))
    g = -np.log1p(np.exp(rng.normal(size=(B, T, H, K if per_channel else 1))))
    beta = 1.0 / (1.0 + np.exp(-rng.normal(size=(B, T, H))))
    return q, k, v, g, beta


def test_equal_channels_reduce_to_the_gated_delta_rule():
    B, T, H, K, V = 2, 37, 2, 5, 4
    rng = np.random.default_rng(41)
    q, k, v, g1, beta = _inputs(B, T, H, K, V, rng, per_channel=False)
    S0 = rng.normal(size=(B, H, V, K)) * 0.3
    dO = rng.normal(size=(B, T, H, V))
    dSf = rng.normal(size=(B, H, V, K))
    gK = np.repeat(g1, K, axis=-1)
    out, fin = kda.kda_fwd(q, k, v, gK, beta, S0)
    ref_out, ref_fin = oracle.gdn_fwd(q, k, v, g1[..., 0], beta, S0)
    assert np.allclose(out, ref_out, rtol=1e-12, atol=1e-12)
    assert np.allclose(fin, ref_fin, rtol=1e-12, atol=1e-12)
    gr = kda.kda_bwd(q, k, v, gK, beta, S0, dO, dSf)
    ref = oracle.gdn_bwd(q, k, v, g1[..., 0], beta, S0, dO, dSf)
    for n in ("dq", "dk", "dv", "dbeta", "d_initial_state"):
        assert np.allclose(gr[n], ref[n], rtol=1e-10, atol=1e-12), n
    assert np.allclose(gr["dg"].sum(-1), ref["dg"], rtol=1e-10, atol=1e-12)


def test_beta_zero_is_channelwise_decay():
    """beta = 0: S_t = S0 scaled column k by exp(sum_{s<=t} g_s[k]), out_t = scale S_t q_t
    (K = 5 != V = 3, so decaying rows instead of columns cannot pass)."""
    B, T, H, K, V = 1, 9, 1, 5, 3
    rng = np.random.default_rng(42)
    q, k, v, g, _ = _inputs(B, T, H, K, V, rng)
    S0 = rng.normal(size=(1, H, V, K))
    out, fin = kda.kda_fwd(q, k, v, g, np.zeros((B, T, H)), S0)
    cum = np.cumsum(g[0, :, 0], axis=0)                   # [T, K]
    for t in range(T):
        St = S0[0, 0] * np.exp(cum[t])[None, :]
        assert np.allclose(out[0, t, 0], (St @ q[0, t, 0]) / np.sqrt(K), rtol=1e-12)
    assert np.allclose(fin[0, 0], S0[0, 0] * np.exp(cum[-1])[None, :], rtol=1e-12)


def test_orthonormal_keys_closed_form():
    """k_t = e_t (T <= K), S0 = 0: column t is written once, with beta_t v_t, then decays by
    exp(g_s[t]) for s > t; out_t = scale sum_{j<=t} beta_j v_j q_t[j] exp(sum_{j<s<=t} g_s[j])."""
    B, T, H, K, V = 1, 6, 1, 8, 3
    rng = np.random.default_rng(43)
    q, _, v, g, beta = _inputs(B, T, H, K, V, rng)
    k = np.zeros((B, T, H, K))
    for t in range(T):
        k[0, t, 0, t] = 1.0
    out, fin = kda.kda_fwd(q, k, v, g, beta, None)
    G = g[0, :, 0]                                        # [T, K]
    for t in range(T):
        want = np.zeros(V)
        for j in range(t + 1):
            want += beta[0, j, 0] * v[0, j, 0] * q[0, t, 0, j] * np.exp(G[j + 1:t + 1, j].sum())
        assert np.allclose(out[0, t, 0], want / np.sqrt(K), rtol=1e-12), t
    for j in range(T):
        assert np.allclose(fin[0, 0][:, j], beta[0, j, 0] * v[0, j, 0] * np.exp(G[j + 1:, j].sum()),
                           rtol=1e-12)


def _loss(inputs, dO, dSf, cu=None):
    q, k, v, g, beta, S0 = inputs
    out, fin = kda.kda_fwd(q, k, v, g, beta, S0, cu_seqlens=cu)
    m = ~np.isnan(out)
    return float((np.where(m, out, 0.0) * dO).sum() + (fin * dSf).sum())


@pytest.mark.parametrize("cu", [None, [0, 5, 5, 13]])
def test_backward_matches_central_differences(cu):
    B = 2 if cu is None else 1
    T, H, K, V = 13, 1, 4, 3
    rng = np.random.default_rng(44)
    q, k, v, g, beta = _inputs(B, T, H, K, V, rng)
    q *= 0.7
    k *= 0.7
    N = B if cu is None else len(cu) - 1
    S0 = rng.normal(size=(N, H, V, K)) * 0.3
    dO = rng.normal(size=(B, T, H, V))
    dSf = rng.normal(size=(N, H, V, K))
    gr = kda.kda_bwd(q, k, v, g, beta, S0, dO, dSf, cu_seqlens=cu)
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
        an = gr[name]
        if cu is not None and name != "d_initial_state":
            an = an.copy()
            an[:, cu[-1]:] = 0.0
        err = np.abs(an - fd).max() / max(np.abs(fd).max(), 1e-300)
        assert err <= 1e-6, (name, err)


def test_packed_equals_per_sequence():
    rng = np.random.default_rng(45)
    lengths = [7, 0, 12]
    T = sum(lengths) + 3
    q, k, v, g, beta = _inputs(1, T, 2, 4, 4, rng)
    cu = np.cumsum([0] + lengths)
    S0 = rng.normal(size=(3, 2, 4, 4))
    out, fin = kda.kda_fwd(q, k, v, g, beta, S0, cu_seqlens=cu)
    for n in range(3):
        sl = slice(cu[n], cu[n + 1])
        o1, f1 = kda.kda_fwd(q[:, sl], k[:, sl], v[:, sl], g[:, sl], beta[:, sl], S0[n:n + 1])
        assert np.array_equal(out[:, sl], o1) and np.array_equal(fin[n], f1[0]), n
    assert np.isnan(out[:, cu[-1]:]).all()
