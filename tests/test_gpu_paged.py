"""Paged-cache prefill (paged_chunk_gdn) through the C ABI against the FP64 oracle: entry
states gathered from cache slots, final states written back in place, padding sequences
(index <= 0 or >= num_slots) with zero output and untouched slots, has_initial_state False
ignoring the slot's (garbage) contents, and two prefill calls equal to one."""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL, active_rows, f64, rel_err, small_inputs

pytestmark = pytest.mark.gpu
BF16 = torch.bfloat16


def _sf():
    import chunked_linear_recurrence_gb300 as sf
    return sf


def _cache(H, D, slots, seed):
    g = torch.Generator().manual_seed(seed)
    c = (torch.randn(slots, H, D, D, generator=g) * 0.1).cuda()
    return c


@pytest.mark.parametrize("dtype,D", [(BF16, 128), (BF16, 64), (torch.float32, 64)])
def test_paged_packed_matches_oracle(dtype, D):
    lengths = [130, 0, 64, 201, 45]
    T = sum(lengths) + 11
    inp = small_inputs(1, T, 2, D, dtype, seed=600 + D, lengths=lengths)
    cache = _cache(2, D, 8, 601 + D)
    cache[6] = float("nan")                       # read by nobody (has_initial_state False)
    before = cache.clone()
    idx = torch.tensor([2, 6, -1, 5, 9], dtype=torch.int32, device="cuda")   # -1, 9: padding
    has = torch.tensor([True, False, True, True, True], device="cuda")
    out = torch.full(inp["v"].shape, float("nan"), dtype=dtype, device="cuda")
    _sf().sf_gdn_paged_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"], cache,
                                 idx, cu_seqlens=inp["cu_seqlens"], has_initial_state=has,
                                 out=out)
    torch.cuda.synchronize()
    cu = inp["cu_seqlens"].cpu().numpy()
    ref_out, ref_cache = oracle.paged_chunk_fwd(
        f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["gate"]), f64(inp["beta"]),
        f64(before), idx.cpu().numpy(), has_initial_state=has.cpu().numpy(), cu_seqlens=cu)
    rows = active_rows(T, cu)
    assert rel_err(out, ref_out, rows) <= TOL[dtype]
    for s in (2, 6, 5):
        assert rel_err(cache[s], ref_cache[s]) <= TOL[dtype], s
    for s in (0, 1, 3, 4, 7):                     # not selected: bits unchanged
        assert torch.equal(cache[s], before[s]), s
    assert not out[:, cu[2]:cu[3]].float().any() and not out[:, cu[4]:cu[5]].float().any()
    assert torch.isnan(out[:, cu[-1]:].float()).all()        # rows past the offsets untouched


def test_paged_dense_two_calls_equal_one():
    """Dense B = 3 (BF16, K = 128): prefill 128 + 72 tokens through the cache equals one
    forward of 200 tokens from the same slots."""
    sf = _sf()
    inp = small_inputs(3, 200, 2, 128, BF16, seed=610, s0=False)
    cache = _cache(2, 128, 4, 611)
    idx = torch.tensor([3, 1, 2], dtype=torch.int32, device="cuda")
    start = cache.clone()
    a = {n: inp[n][:, :128].contiguous() for n in ("q", "k", "v", "gate", "beta")}
    b = {n: inp[n][:, 128:].contiguous() for n in ("q", "k", "v", "gate", "beta")}
    o1 = sf.sf_gdn_paged_chunk_fwd(a["q"], a["k"], a["v"], a["gate"], a["beta"], cache, idx)
    o2 = sf.sf_gdn_paged_chunk_fwd(b["q"], b["k"], b["v"], b["gate"], b["beta"], cache, idx)
    torch.cuda.synchronize()
    s0 = start[idx.long()]
    ref_out, ref_fin = oracle.gdn_fwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]),
                                      f64(inp["gate"]), f64(inp["beta"]), f64(s0))
    got = torch.cat([o1, o2], 1)
    assert rel_err(got, ref_out) <= TOL[BF16]
    assert rel_err(cache[idx.long()], ref_fin) <= TOL[BF16]
    assert torch.equal(cache[0], start[0])
