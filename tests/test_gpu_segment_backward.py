"""Segment-parallel backward: the cotangent maps of consecutive segments (dS_entry =
dS_exit @ P^T + C), their reverse scan, and the full pipeline -- forward summaries and
scan for the entry states, reverse summaries and reverse scan for the exit cotangents,
then one packed backward over all segments -- against the FP64 oracle's single pass."""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL, f64, oracle_bwd, rel_err, small_inputs

pytestmark = pytest.mark.gpu
BF16 = torch.bfloat16


def _sf():
    import chunked_linear_recurrence_gb300 as sf
    return sf


@pytest.mark.parametrize("dtype,D", [(BF16, 128), (BF16, 64), (torch.float32, 64)])
def test_reverse_summary_matches_oracle(dtype, D):
    """Segments of 70, 0, 130 and 133 tokens (an empty one, partial last chunks)."""
    offs = [0, 70, 70, 200, 333]
    inp = small_inputs(1, 340, 2, D, dtype, seed=500 + D, grads=True)
    inp["gate"] *= 0.05
    cu = torch.tensor(offs, dtype=torch.int32, device="cuda")
    C = _sf().sf_gdn_segment_reverse_summary(inp["q"], inp["k"], inp["gate"], inp["beta"],
                                             inp["d_out"], cu)
    torch.cuda.synchronize()
    Cr = oracle.segment_reverse_summary(f64(inp["q"]), f64(inp["k"]), f64(inp["gate"]),
                                        f64(inp["beta"]), f64(inp["d_out"]), offs)
    for r in (0, 2, 3):
        assert rel_err(C[r], Cr[r]) <= TOL[dtype], r
    assert not C[1].any()                               # an empty segment adds nothing


@pytest.mark.parametrize("D", [64, 128])
def test_reverse_scan_matches_oracle(D):
    g = torch.Generator().manual_seed(D + 1)
    R, H = 5, 3
    P = (torch.randn(R, H, D, D, generator=g) / D ** 0.5).float()
    C = torch.randn(R, H, D, D, generator=g).float()
    dSf = torch.randn(H, D, D, generator=g).float()
    ex, d0 = _sf().sf_state_scan_reverse(P.cuda(), C.cuda(), dSf.cuda())
    torch.cuda.synchronize()
    ex_r, d0_r = oracle.state_scan_reverse(f64(P), f64(C), f64(dSf))
    assert rel_err(ex, ex_r) <= 1e-5 and rel_err(d0, d0_r) <= 1e-5
    ex0, d00 = _sf().sf_state_scan_reverse(P.cuda(), C.cuda(), None)
    ex0_r, d00_r = oracle.state_scan_reverse(f64(P), f64(C), None)
    assert rel_err(ex0, ex0_r) <= 1e-5 and rel_err(d00, d00_r) <= 1e-5


@pytest.mark.parametrize("dtype,D", [(BF16, 128), (torch.float32, 64)])
def test_segment_parallel_backward_equals_single_pass(dtype, D):
    """Four segments of one 1024-token sequence (low decay, so entry states and cotangents
    cross segment boundaries): every gradient of the segment-parallel pipeline against the
    oracle's single pass, and each segment's entry cotangent against the reverse scan."""
    T, R, H = 1024, 4, 2
    L = T // R
    inp = small_inputs(1, T, H, D, dtype, seed=520 + D, grads=True)
    inp["gate"] *= 1e-3
    inp["beta"] *= 0.1
    sf = _sf()
    offs = torch.arange(0, T + 1, L, dtype=torch.int32, device="cuda")
    bounds = torch.stack([offs[:-1], offs[1:]], 1).contiguous()
    P, E = sf.sf_gdn_segment_summary(inp["k"], inp["v"], inp["gate"], inp["beta"], bounds)
    entry, _ = sf.sf_state_scan(P, E, inp["initial_state"][0])
    C = sf.sf_gdn_segment_reverse_summary(inp["q"], inp["k"], inp["gate"], inp["beta"],
                                          inp["d_out"], offs)
    exits, d0 = sf.sf_state_scan_reverse(P, C, inp["d_final_state"][0])
    got = sf.sf_gdn_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"], entry,
                              inp["d_out"], exits, cu_seqlens=offs)
    torch.cuda.synchronize()
    ref = oracle_bwd(inp)
    tol = TOL[dtype]
    for n, r in (("dq", "dq"), ("dk", "dk"), ("dv", "dv"), ("dgate", "dg"), ("dbeta", "dbeta")):
        assert rel_err(got[n], ref[r]) <= tol, n
    assert rel_err(d0, ref["d_initial_state"][0]) <= tol
    assert rel_err(got["d_initial_state"][0], ref["d_initial_state"][0]) <= tol
    for j in range(1, R):      # a segment's entry cotangent is the previous one's exit
        assert rel_err(got["d_initial_state"][j], f64(exits[j - 1])) <= tol, j
