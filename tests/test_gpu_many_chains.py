"""Forward and backward parity with more (sequence, head) chains than state-chain CTAs
(BF16, K = V = 128), the case where one state-chain CTA walks several chains in turn and
the preparation CTAs claim records across chains of very different lengths.  The FP64
oracle is the reference, element by element, at the BF16 tolerance."""
import numpy as np
import pytest
import torch

from helpers import TOL, active_rows, oracle_bwd, oracle_fwd, rel_err, small_inputs

pytestmark = pytest.mark.gpu
BF16 = torch.bfloat16


def _fwd(inp):
    import chunked_linear_recurrence_gb300 as sf
    from chunked_linear_recurrence_gb300 import _native
    shape = _native.make_shape(inp["q"], inp["v"], inp.get("cu_seqlens"))
    ws = _native.workspace(_native.fwd_workspace_bytes(shape), inp["q"].device)
    out, fin = sf.sf_gdn_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                                   inp.get("initial_state"), cu_seqlens=inp.get("cu_seqlens"),
                                   output_final_state=True, ws=ws)
    _native.sf_workspace_status(ws)     # raises if any wait in the kernel gave up
    torch.cuda.synchronize()
    return out, fin


def test_dense_more_chains_than_chain_ctas():
    """B = 33, H = 2: 66 chains over 64 state-chain CTAs; T = 130 ends in a partial chunk."""
    inp = small_inputs(33, 130, 2, 128, BF16, seed=2024)
    out, fin = _fwd(inp)
    ref_out, ref_fin = oracle_fwd(inp)
    assert rel_err(out, ref_out) <= TOL[BF16]
    assert rel_err(fin, ref_fin) <= TOL[BF16]


def test_packed_uneven_lengths_more_chains_than_chain_ctas():
    """40 packed sequences x 2 heads = 80 chains with lengths from 0 to 450: chain CTAs with
    one or two chains and stream lengths that differ by ~14 chunks."""
    g = torch.Generator().manual_seed(7)
    lengths = torch.randint(0, 451, (40,), generator=g).tolist()
    lengths[3] = 0
    lengths[17] = 450
    lengths[25] = 1
    lengths[31] = 64
    T = sum(lengths) + 19
    inp = small_inputs(1, T, 2, 128, BF16, seed=2025, lengths=lengths)
    out, fin = _fwd(inp)
    ref_out, ref_fin = oracle_fwd(inp)
    rows = active_rows(T, inp["cu_seqlens"])
    assert rel_err(out, ref_out, rows) <= TOL[BF16]
    assert rel_err(fin, ref_fin) <= TOL[BF16]
    assert torch.equal(fin[3], inp["initial_state"][3])     # empty sequence passes S0 through


def test_backward_more_chains_than_chain_ctas():
    """The backward's state replay on the split kernel with 66 chains (two on some chain
    CTAs), checkpoints in its thread order, then every gradient against the oracle."""
    import chunked_linear_recurrence_gb300 as sf
    inp = small_inputs(33, 100, 2, 128, BF16, seed=2026, grads=True)
    got = sf.sf_gdn_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                              inp["initial_state"], inp["d_out"], inp["d_final_state"])
    torch.cuda.synchronize()
    ref = oracle_bwd(inp)
    names = {"dq": "dq", "dk": "dk", "dv": "dv", "dgate": "dg", "dbeta": "dbeta",
             "d_initial_state": "d_initial_state"}
    errs = {n: rel_err(got[n], ref[r]) for n, r in names.items()}
    assert all(e <= TOL[BF16] for e in errs.values()), errs
