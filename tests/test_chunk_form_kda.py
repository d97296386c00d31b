"""The KDA chunk-form algebra (chunk_form_kda.py) equals the token-by-token KDA oracle:
forward over several chunks with a ragged tail, and the chunk-composed affine map equals
the probing construction (run from S0 = I without values, and from S0 = 0)."""
import numpy as np

import chunk_form_kda as cf
from oracle import kda


def _inputs(T, K, V, rng):
    q = rng.normal(size=(T, K))
    k = rng.normal(size=(T, K))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.normal(size=(T, V))
    g = -np.log1p(np.exp(rng.normal(size=(T, K)))) * 0.3
    beta = 1.0 / (1.0 + np.exp(-rng.normal(size=T)))
    return q, k, v, g, beta


def test_chunk_form_forward_equals_oracle():
    rng = np.random.default_rng(51)
    T, K, V = 150, 8, 6                      # three chunks, the last one partial
    q, k, v, g, beta = _inputs(T, K, V, rng)
    S0 = rng.normal(size=(V, K)) * 0.3
    out, S = cf.fwd_seq(q, k, v, g, beta, S0.copy(), 1.0 / np.sqrt(K))
    ref_out, ref_fin = kda.kda_fwd(q[None, :, None], k[None, :, None], v[None, :, None],
                                   g[None, :, None], beta[None, :, None], S0[None, None])
    assert np.allclose(out, ref_out[0, :, 0], rtol=1e-10, atol=1e-12)
    assert np.allclose(S, ref_fin[0, 0], rtol=1e-10, atol=1e-12)


def test_chunk_form_summary_equals_probing():
    rng = np.random.default_rng(52)
    T, K, V = 130, 6, 5
    q, k, v, g, beta = _inputs(T, K, V, rng)
    P, E = cf.summary_seq(q, k, v, g, beta)
    _, fP = kda.kda_fwd(q[None, :, None], k[None, :, None], np.zeros((1, T, 1, K)),
                        g[None, :, None], beta[None, :, None], np.eye(K)[None, None])
    _, fE = kda.kda_fwd(q[None, :, None], k[None, :, None], v[None, :, None],
                        g[None, :, None], beta[None, :, None], None)
    assert np.allclose(P, fP[0, 0], rtol=1e-10, atol=1e-12)
    assert np.allclose(E, fE[0, 0], rtol=1e-10, atol=1e-12)


def test_chunk_form_backward_equals_oracle():
    rng = np.random.default_rng(53)
    T, K, V = 150, 6, 5
    q, k, v, g, beta = _inputs(T, K, V, rng)
    g *= 0.5                                     # e^{-gamma} is formed directly here
    S0 = rng.normal(size=(V, K)) * 0.3
    dO = rng.normal(size=(T, V))
    dSf = rng.normal(size=(V, K))
    scale = 1.0 / np.sqrt(K)
    dq, dk, dv, dg, dbeta, dS0 = cf.bwd_seq(q, k, v, g, beta, S0, dO, dSf, scale)
    ref = kda.kda_bwd(q[None, :, None], k[None, :, None], v[None, :, None], g[None, :, None],
                      beta[None, :, None], S0[None, None], dO[None, :, None], dSf[None, None])
    for name, got, want in (("dq", dq, ref["dq"][0, :, 0]), ("dk", dk, ref["dk"][0, :, 0]),
                            ("dv", dv, ref["dv"][0, :, 0]), ("dg", dg, ref["dg"][0, :, 0]),
                            ("dbeta", dbeta, ref["dbeta"][0, :, 0]),
                            ("dS0", dS0, ref["d_initial_state"][0, 0])):
        err = np.abs(got - want).max() / np.abs(want).max()
        assert err <= 1e-9, (name, err)


def test_stable_decay_products_match_and_survive_extreme_gates():
    """The sub-blocked form of Aqk / Akk equals the direct one, and with gates at the pages'
    bound (about -5.9 per token: gamma falls to about -380 over 64 tokens) it stays finite in
    FP32 where the read/write-key factorisation Kh Kv^T overflows."""
    rng = np.random.default_rng(54)
    L, K, V = 64, 8, 4
    q, k, v, g, beta = _inputs(L, K, V, rng)
    _, Aqk, _, _, _ = cf.chunk_terms(q, k, v, g, beta)
    got = cf.decay_products_stable(q, k, g, dtype=np.float64)
    assert np.allclose(got, Aqk, rtol=1e-12, atol=1e-14)
    gx = -5.9 * np.ones((L, K))                           # every 16-token sum is -94.4
    gx[:, ::2] = -5.4                                     # (-86.4 on half the channels)
    s32 = cf.decay_products_stable(q, k, gx, dtype=np.float32)
    assert np.isfinite(s32).all()
    gam = np.cumsum(gx, axis=0)
    with np.errstate(over="ignore", invalid="ignore"):
        naive = (q.astype(np.float32) * np.exp(gam).astype(np.float32)) @ \
                (k.astype(np.float32) * np.exp(-gam).astype(np.float32)).T
    assert not np.isfinite(naive).all()
    ref = np.tril(np.einsum("ic,jc,ijc->ij", q, k,
                            np.exp(np.minimum(gam[:, None, :] - gam[None, :, :], 0))))
    # error relative to the largest entry (the parity tests' metric): FP32 rounding of the
    # cumulative gates moves a few tiny cancelling entries by ~1e-4 of themselves only
    assert np.abs(s32 - ref).max() <= 1e-6 * np.abs(ref).max()
