"""Backward parity: every gradient of L = <d_out, out> + <dS_T, S_T> against
the oracle's reverse-mode gradients (themselves pinned by finite differences)."""
import numpy as np
import pytest
import torch

from helpers import TOL, active_rows, oracle_bwd, rel_err, small_inputs

pytestmark = pytest.mark.gpu

NAMES = ["dq", "dk", "dv", "dgate", "dbeta", "d_initial_state"]
ORACLE = {"dq": "dq", "dk": "dk", "dv": "dv", "dgate": "dg", "dbeta": "dbeta",
          "d_initial_state": "d_initial_state"}


def run_bwd(inp):
    import chunked_linear_recurrence_gb300 as sf
    return sf.sf_gdn_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                               inp.get("initial_state"), inp["d_out"], inp.get("d_final_state"),
                               cu_seqlens=inp.get("cu_seqlens"))


def check_bwd(inp, tol):
    got = run_bwd(inp)
    torch.cuda.synchronize()
    ref = oracle_bwd(inp)
    rows = active_rows(inp["q"].shape[1], inp.get("cu_seqlens"))
    errs = {}
    for n in NAMES:
        if n == "d_initial_state":
            errs[n] = rel_err(got[n], ref[ORACLE[n]])
        else:
            errs[n] = rel_err(got[n], ref[ORACLE[n]], rows)
    bad = {n: e for n, e in errs.items() if not e <= tol}
    assert not bad, errs
    return errs


@pytest.mark.parametrize("B,T,H", [(1, 64, 1), (2, 200, 2), (1, 1, 1), (1, 130, 3)])
def test_bwd_f32_d64(B, T, H):
    inp = small_inputs(B, T, H, 64, torch.float32, seed=B + T + H, grads=True)
    check_bwd(inp, 1e-4)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B,T,H", [(1, 64, 1), (2, 200, 2), (1, 333, 2)])
def test_bwd_bf16(D, B, T, H):
    inp = small_inputs(B, T, H, D, torch.bfloat16, seed=D + B + T, grads=True)
    check_bwd(inp, 2e-2)


@pytest.mark.parametrize("dtype,D", [(torch.float32, 64), (torch.bfloat16, 128)])
def test_bwd_packed_varlen(dtype, D):
    lengths = [0, 70, 1, 128, 0, 45]
    T = sum(lengths) + 20
    inp = small_inputs(1, T, 2, D, dtype, seed=4, lengths=lengths, grads=True)
    check_bwd(inp, TOL[dtype])


def test_bwd_without_initial_state_or_final_cotangent():
    inp = small_inputs(1, 150, 2, 64, torch.float32, seed=8, s0=False, grads=True)
    inp["d_final_state"] = None
    check_bwd(inp, 1e-4)


def test_bwd_unsupported_f32_d128():
    import chunked_linear_recurrence_gb300 as sf
    inp = small_inputs(1, 64, 1, 128, torch.float32, seed=1, grads=True)
    with pytest.raises(sf.SfError) as ei:
        run_bwd(inp)
    assert ei.value.status == 2


def test_bwd_bf16_one_long_chain():
    """Dense K = V = 128 with one (sequence, head) chain of 32 chunks: in the launch that runs
    the reverse chain beside the token gradients, every gradient CTA but the first waits for
    that one chain's exit cotangents, in the order the chain writes them."""
    inp = small_inputs(1, 2048, 1, 128, torch.bfloat16, seed=2048, grads=True)
    check_bwd(inp, 2e-2)


def test_bwd_bf16_sixty_four_chains():
    """Dense K = V = 128 with 64 chains (B = 32, H = 2, a partial last chunk): the most
    chains the shared launch takes; each chain CTA joins the token gradients after its
    chain."""
    inp = small_inputs(32, 130, 2, 128, torch.bfloat16, seed=64, grads=True)
    check_bwd(inp, 2e-2)
