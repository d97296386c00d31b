"""Packed sequences under CUDA-graph capture: the forward and backward read cu_seqlens on
the device (the split kernel builds its geometry there, grids depend only on T and N), so
one captured graph serves any lengths with the same N and T.  The graph is captured once
and replayed after rewriting the offsets in place; every replay is checked against the
oracle for the offsets it ran with."""
import pytest
import torch

from helpers import TOL, active_rows, oracle_bwd, oracle_fwd, rel_err, small_inputs

pytestmark = pytest.mark.gpu
BF16 = torch.bfloat16
NAMES = {"dq": "dq", "dk": "dk", "dv": "dv", "dgate": "dg", "dbeta": "dbeta",
         "d_initial_state": "d_initial_state"}


@pytest.mark.parametrize("D", [128, 64])
def test_captured_forward_backward_replays_with_new_lengths(D):
    import chunked_linear_recurrence_gb300 as sf
    from chunked_linear_recurrence_gb300 import _native
    from chunked_linear_recurrence_gb300.workloads import cu_seqlens_of

    T, H = 512, 2
    inp = small_inputs(1, T, H, D, BF16, seed=400 + D, lengths=[100, 200, 150], grads=True)
    cu = inp["cu_seqlens"]
    shape = _native.make_shape(inp["q"], inp["v"], cu)
    wsf = _native.workspace(_native.fwd_workspace_bytes(shape), "cuda")
    wsb = _native.workspace(_native.bwd_workspace_bytes(shape), "cuda")
    out = torch.empty_like(inp["v"])
    fin = torch.empty_like(inp["initial_state"])
    grads = {n: torch.empty_like(inp[src]) for n, src in
             (("dq", "q"), ("dk", "k"), ("dv", "v"), ("dgate", "gate"), ("dbeta", "beta"),
              ("d_initial_state", "initial_state"))}

    def step():
        sf.sf_gdn_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                            inp["initial_state"], cu_seqlens=cu, output_final_state=True,
                            out=out, final_state=fin, ws=wsf)
        sf.sf_gdn_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                            inp["initial_state"], inp["d_out"], inp["d_final_state"],
                            cu_seqlens=cu, grads=grads, ws=wsb)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                                   # eager warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for lengths in ([100, 200, 150], [7, 0, 400], [64, 64, 64], [0, 0, 0]):
        cu.copy_(cu_seqlens_of(lengths).to(cu.device))
        graph.replay()
        torch.cuda.synchronize()
        _native.sf_workspace_status(wsf)
        _native.sf_workspace_status(wsb)
        case = dict(inp, cu_seqlens=cu.clone())
        rows = active_rows(T, case["cu_seqlens"])
        ref_out, ref_fin = oracle_fwd(case)
        if len(rows):
            assert rel_err(out, ref_out, rows) <= TOL[BF16], lengths
        assert rel_err(fin, ref_fin) <= TOL[BF16], lengths
        ref = oracle_bwd(case)
        for n, r in NAMES.items():
            if n == "d_initial_state":
                e = rel_err(grads[n], ref[r])
            elif len(rows):
                e = rel_err(grads[n], ref[r], rows)
            else:
                continue
            assert e <= TOL[BF16], (lengths, n, e)
