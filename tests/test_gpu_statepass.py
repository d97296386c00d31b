"""Segment summaries, the exclusive scan and segment-parallel forward from the
scanned entry states (boundary-state passing), against the oracle and against
the single sequential pass."""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL, f64, oracle_fwd, rel_err, small_inputs

pytestmark = pytest.mark.gpu


def _sf():
    import chunked_linear_recurrence_gb300 as sf
    return sf


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("D", [64, 128])
def test_summary_matches_oracle(dtype, D):
    inp = small_inputs(2, 300, 2, D, dtype, seed=21 + D, s0=False)
    inp["gate"] *= 0.02                      # keep P away from zero so it is tested
    bounds = torch.tensor([[0, 300], [13, 140], [300, 300], [300, 600], [450, 451], [64, 64]],
                          dtype=torch.int32)
    P, E = _sf().sf_gdn_segment_summary(inp["k"], inp["v"], inp["gate"], inp["beta"],
                                        bounds.cuda())
    torch.cuda.synchronize()
    Pr, Er = oracle.segment_summary(f64(inp["k"]), f64(inp["v"]), f64(inp["gate"]),
                                    f64(inp["beta"]), bounds.numpy())
    tol = TOL[dtype]
    for r in range(bounds.shape[0]):
        assert rel_err(P[r], Pr[r]) <= tol, r
        assert rel_err(E[r], Er[r]) <= tol or np.abs(Er[r]).max() == 0, r
    # empty ranges: identity map exactly
    eye = torch.eye(D, device="cuda").expand(2, D, D)
    assert torch.equal(P[2], eye) and torch.equal(P[5], eye)
    assert not E[2].any() and not E[5].any()


@pytest.mark.parametrize("dtype,D", [(torch.float32, 64), (torch.bfloat16, 128)])
def test_summary_invalid_bounds_give_nan(dtype, D):
    inp = small_inputs(2, 100, 1, D, dtype, seed=2, s0=False)
    bounds = torch.tensor([[0, 50], [90, 110], [-1, 5], [10, 5], [0, 201]], dtype=torch.int32)
    P, E = _sf().sf_gdn_segment_summary(inp["k"], inp["v"], inp["gate"], inp["beta"],
                                        bounds.cuda())
    torch.cuda.synchronize()
    assert torch.isfinite(P[0]).all() and torch.isfinite(E[0]).all()
    for r in (1, 2, 3, 4):      # crosses a batch row / negative / reversed / past the end
        assert torch.isnan(P[r]).all() and torch.isnan(E[r]).all(), r


def test_summary_more_ranges_than_chain_ctas():
    """BF16, K = V = 128: 23 ranges x 2 heads = 46 (range, head) chains, more than the 32
    chain CTAs that own record streams (each with its P twin), so some walk two chains;
    range lengths from 0 to 7 chunks, starts not on chunk boundaries, a partial last chunk."""
    B, T, H, D = 2, 520, 2, 128
    inp = small_inputs(B, T, H, D, torch.bfloat16, seed=77, s0=False)
    inp["gate"] *= 0.05
    g = torch.Generator().manual_seed(5)
    rows = []
    for r in range(23):
        b = r % B
        n = int(torch.randint(0, 450, (1,), generator=g))
        st = int(torch.randint(0, T - n + 1, (1,), generator=g))
        rows.append((b * T + st, b * T + st + n))
    rows[4] = (600, 600)             # empty
    rows[9] = (T, 2 * T)             # a whole batch row
    bounds = torch.tensor(rows, dtype=torch.int32)
    P, E = _sf().sf_gdn_segment_summary(inp["k"], inp["v"], inp["gate"], inp["beta"],
                                        bounds.cuda())
    torch.cuda.synchronize()
    Pr, Er = oracle.segment_summary(f64(inp["k"]), f64(inp["v"]), f64(inp["gate"]),
                                    f64(inp["beta"]), bounds.numpy())
    tol = TOL[torch.bfloat16]
    for r in range(len(rows)):
        assert rel_err(P[r], Pr[r]) <= tol, r
        assert rel_err(E[r], Er[r]) <= tol or np.abs(Er[r]).max() == 0, r
    assert torch.equal(P[4], torch.eye(D, device="cuda").expand(H, D, D)) and not E[4].any()


@pytest.mark.parametrize("D", [64, 128])
def test_scan_matches_oracle(D):
    g = torch.Generator().manual_seed(D)
    R, H = 5, 3
    P = (torch.randn(R, H, D, D, generator=g) / D ** 0.5).float()
    E = torch.randn(R, H, D, D, generator=g).float()
    S0 = torch.randn(H, D, D, generator=g).float()
    ent, fin = _sf().sf_state_scan(P.cuda(), E.cuda(), S0.cuda())
    torch.cuda.synchronize()
    ent_r, fin_r = oracle.state_scan(f64(P), f64(E), f64(S0))
    assert rel_err(ent, ent_r) <= 1e-5 and rel_err(fin, fin_r) <= 1e-5
    ent0, fin0 = _sf().sf_state_scan(P.cuda(), E.cuda(), None)
    ent0_r, fin0_r = oracle.state_scan(f64(P), f64(E), None)
    assert rel_err(ent0, ent0_r) <= 1e-5 and rel_err(fin0, fin0_r) <= 1e-5


def state_passing(inp, segments):
    """summary -> scan -> packed forward of all segments from their entry states."""
    sf = _sf()
    B, T, H, D = inp["q"].shape
    L = T // segments
    bounds = torch.tensor([(i * L, (i + 1) * L) for i in range(segments)], dtype=torch.int32,
                          device="cuda")
    P, E = sf.sf_gdn_segment_summary(inp["k"], inp["v"], inp["gate"], inp["beta"], bounds)
    s0 = inp.get("initial_state")
    ent, fin = sf.sf_state_scan(P, E, None if s0 is None else s0[0])
    cu = torch.arange(0, T + 1, L, dtype=torch.int32, device="cuda")
    out, seg_fin = sf.sf_gdn_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                                       ent, cu_seqlens=cu, output_final_state=True)
    return out, fin, seg_fin, ent


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_state_passing_equals_single_pass(dtype):
    """Segments run in parallel from scanned entry states == one sequential
    pass == the carried-state segment loop (low-decay inputs so the entry
    states matter)."""
    T, segments, D = 1024, 4, 128
    inp = small_inputs(1, T, 2, D, dtype, seed=31)
    inp["gate"] *= 1e-3
    inp["beta"] *= 0.1
    out, fin, seg_fin, ent = state_passing(inp, segments)
    ref_out, ref_fin = oracle_fwd(inp)
    tol = TOL[dtype]
    assert rel_err(out, ref_out) <= tol
    assert rel_err(fin, ref_fin[0]) <= tol
    assert rel_err(seg_fin[-1], ref_fin[0]) <= tol
    # carried-state loop through the forward entry point
    sf = _sf()
    L = T // segments
    S = inp["initial_state"]
    for j in range(segments):
        assert rel_err(ent[j], f64(S)[0]) <= tol, j
        part = {x: inp[x][:, j * L:(j + 1) * L].contiguous() for x in ("q", "k", "v", "gate", "beta")}
        _, S = sf.sf_gdn_chunk_fwd(part["q"], part["k"], part["v"], part["gate"], part["beta"], S,
                                   output_final_state=True)
    assert rel_err(S[0], ref_fin[0]) <= tol
