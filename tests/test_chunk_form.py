"""The chunk-parallel algebra (the kernels' reading of the WY/UT form) equals
the token-by-token oracle in FP64, for whole and partial chunks."""
import numpy as np
import pytest

import oracle
from chunk_form import fwd_seq, summary_seq
from test_oracle_pins import rand_inputs


@pytest.mark.parametrize("T,K,V", [(64, 16, 16), (200, 8, 12), (130, 32, 32), (1, 4, 4)])
def test_chunk_form_forward_equals_oracle(T, K, V):
    rng = np.random.default_rng(T + K)
    q, k, v, g, beta, S0 = rand_inputs(1, T, 1, K, V, rng)
    out, fin = oracle.gdn_fwd(q, k, v, g, beta, S0, scale=0.3)
    o2, f2 = fwd_seq(q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0], beta[0, :, 0],
                     S0[0, 0], 0.3)
    np.testing.assert_allclose(o2, out[0, :, 0], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(f2, fin[0, 0], rtol=1e-10, atol=1e-12)


def test_chunk_form_summary_equals_probing():
    rng = np.random.default_rng(5)
    q, k, v, g, beta, _ = rand_inputs(1, 150, 1, 8, 6, rng)
    g *= 0.05
    P, E = oracle.segment_summary(k, v, g, beta, np.array([[0, 150]]))
    P2, E2 = summary_seq(k[0, :, 0], v[0, :, 0], g[0, :, 0], beta[0, :, 0])
    np.testing.assert_allclose(P2, P[0, 0], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(E2, E[0, 0], rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("T,K,V", [(64, 8, 8), (150, 6, 10), (1, 4, 4)])
def test_chunk_form_backward_equals_oracle(T, K, V):
    from chunk_form import bwd_seq
    rng = np.random.default_rng(T * 3 + K)
    q, k, v, g, beta, S0 = rand_inputs(1, T, 1, K, V, rng)
    dO = rng.normal(size=(1, T, 1, V))
    dSf = rng.normal(size=(1, 1, V, K))
    ref = oracle.gdn_bwd(q, k, v, g, beta, S0, dO, dSf, scale=0.3)
    got = bwd_seq(q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0], beta[0, :, 0], S0[0, 0],
                  dO[0, :, 0], dSf[0, 0], 0.3)
    for name, x in zip(["dq", "dk", "dv", "dg", "dbeta"], got[:5]):
        np.testing.assert_allclose(x, ref[name][0, :, 0], rtol=1e-9, atol=1e-11, err_msg=name)
    np.testing.assert_allclose(got[5], ref["d_initial_state"][0, 0], rtol=1e-9, atol=1e-11)
