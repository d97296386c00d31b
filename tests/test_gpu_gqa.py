"""Grouped query/key heads (HK divides H; value head h reads query/key head h // (H // HK)):
forward, segment summaries and backward through the C ABI against the FP64 oracle, which
takes the same definition literally (q and k repeated per block, gradients of a shared
head summed over its block)."""
import pytest
import torch

from helpers import TOL, active_rows, oracle_bwd, oracle_fwd, rel_err, small_inputs

import oracle
from helpers import f64

pytestmark = pytest.mark.gpu
BF16 = torch.bfloat16


def grouped(inp, HK):
    """The first HK query/key heads of a small_inputs dict (values stay L2-normalised)."""
    out = dict(inp)
    out["q"] = inp["q"][:, :, :HK].contiguous()
    out["k"] = inp["k"][:, :, :HK].contiguous()
    return out


def _sf():
    import chunked_linear_recurrence_gb300 as sf
    return sf


@pytest.mark.parametrize("dtype,D,HK", [(BF16, 128, 2), (BF16, 128, 1), (BF16, 64, 2),
                                        (torch.float32, 64, 2)])
def test_forward_dense(dtype, D, HK):
    inp = grouped(small_inputs(2, 200, 4, D, dtype, seed=300 + D + HK), HK)
    out, fin = _sf().sf_gdn_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                                      inp["initial_state"], output_final_state=True)
    torch.cuda.synchronize()
    assert out.shape == inp["v"].shape
    ref_out, ref_fin = oracle_fwd(inp)
    assert rel_err(out, ref_out) <= TOL[dtype]
    assert rel_err(fin, ref_fin) <= TOL[dtype]


def test_forward_packed_one_shared_head():
    """Packed sequences (one empty, ragged tails) with all four value heads on one q/k head."""
    lengths = [130, 0, 64, 201]
    T = sum(lengths) + 9
    inp = grouped(small_inputs(1, T, 4, 128, BF16, seed=310, lengths=lengths), 1)
    out = torch.full(inp["v"].shape, float("nan"), dtype=BF16, device="cuda")
    _, fin = _sf().sf_gdn_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                                    inp["initial_state"], cu_seqlens=inp["cu_seqlens"],
                                    output_final_state=True, out=out)
    torch.cuda.synchronize()
    ref_out, ref_fin = oracle_fwd(inp)
    rows = active_rows(T, inp["cu_seqlens"])
    assert rel_err(out, ref_out, rows) <= TOL[BF16]
    assert rel_err(fin, ref_fin) <= TOL[BF16]
    assert torch.isnan(out[:, sum(lengths):].float()).all()      # inactive rows untouched


def test_summary_shared_keys():
    inp = grouped(small_inputs(2, 300, 4, 128, BF16, seed=320, s0=False), 2)
    inp["gate"] *= 0.02
    bounds = torch.tensor([[0, 300], [13, 140], [300, 300], [300, 600]], dtype=torch.int32)
    P, E = _sf().sf_gdn_segment_summary(inp["k"], inp["v"], inp["gate"], inp["beta"],
                                        bounds.cuda())
    torch.cuda.synchronize()
    Pr, Er = oracle.segment_summary(f64(inp["k"]), f64(inp["v"]), f64(inp["gate"]),
                                    f64(inp["beta"]), bounds.numpy())
    for r in (0, 1, 3):
        assert rel_err(P[r], Pr[r]) <= TOL[BF16], r
        assert rel_err(E[r], Er[r]) <= TOL[BF16], r
    assert torch.equal(P[2], torch.eye(128, device="cuda").expand(4, 128, 128))


NAMES = {"dq": "dq", "dk": "dk", "dv": "dv", "dgate": "dg", "dbeta": "dbeta",
         "d_initial_state": "d_initial_state"}


@pytest.mark.parametrize("dtype,D,HK", [(BF16, 128, 2), (BF16, 64, 1), (torch.float32, 64, 2)])
def test_backward_dense(dtype, D, HK):
    inp = grouped(small_inputs(2, 150, 4, D, dtype, seed=330 + D + HK, grads=True), HK)
    got = _sf().sf_gdn_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                                 inp["initial_state"], inp["d_out"], inp["d_final_state"])
    torch.cuda.synchronize()
    assert got["dq"].shape == inp["q"].shape and got["dk"].shape == inp["k"].shape
    ref = oracle_bwd(inp)
    errs = {n: rel_err(got[n], ref[r]) for n, r in NAMES.items()}
    assert all(e <= TOL[dtype] for e in errs.values()), errs


def test_backward_packed_inactive_rows_untouched():
    """Packed BF16 K = 128, four value heads on two q/k heads: every gradient against the
    oracle on the active rows; dq and dk rows past the last offset keep their contents."""
    lengths = [70, 0, 129]
    T = sum(lengths) + 23
    inp = grouped(small_inputs(1, T, 4, 128, BF16, seed=340, lengths=lengths, grads=True), 2)
    sf = _sf()
    grads = {n: torch.full_like(inp[src], float("nan")) for n, src in
             (("dq", "q"), ("dk", "k"), ("dv", "v"), ("dgate", "gate"), ("dbeta", "beta"))}
    grads["d_initial_state"] = torch.empty_like(inp["initial_state"])
    got = sf.sf_gdn_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                              inp["initial_state"], inp["d_out"], inp["d_final_state"],
                              cu_seqlens=inp["cu_seqlens"], grads=grads)
    torch.cuda.synchronize()
    ref = oracle_bwd(inp)
    rows = active_rows(T, inp["cu_seqlens"])
    for n, r in NAMES.items():
        e = rel_err(got[n], ref[r]) if n == "d_initial_state" else rel_err(got[n], ref[r], rows)
        assert e <= TOL[BF16], (n, e)
    end = sum(lengths)
    assert torch.isnan(got["dq"][:, end:].float()).all() and torch.isnan(got["dk"][:, end:].float()).all()


def test_backward_noalloc_grouped():
    """The allocation-free entry point with grouped heads agrees with the workspace one (dgate
    and dbeta sum through shared-memory atomics, so their last bits vary from run to run)."""
    sf = _sf()
    from chunked_linear_recurrence_gb300 import _native
    inp = grouped(small_inputs(1, 256, 4, 128, BF16, seed=350, grads=True), 1)
    args = (inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"], inp["initial_state"],
            inp["d_out"], inp["d_final_state"])
    a = sf.sf_gdn_chunk_bwd(*args)
    b = _native.sf_gdn_chunk_bwd_noalloc(*args)
    torch.cuda.synchronize()
    for n in NAMES:
        assert rel_err(a[n], f64(b[n])) <= 1e-5, n
