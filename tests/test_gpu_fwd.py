"""Forward parity: the CUDA path (through the C ABI) against the FP64 oracle,
element by element, on the same seeded inputs.  Tolerance: max-abs-error /
max|ref| <= 1e-4 for FP32 inputs and <= 2e-2 for BF16 inputs."""
import numpy as np
import pytest
import torch

from helpers import TOL, active_rows, oracle_fwd, rel_err, small_inputs

pytestmark = pytest.mark.gpu


def _lib():
    import chunked_linear_recurrence_gb300 as sf
    return sf


def run_fwd(inp, **kw):
    """Forward through the C ABI; also checks that no kernel reported a timeout."""
    sf = _lib()
    from chunked_linear_recurrence_gb300 import _native
    shape = _native.make_shape(inp["q"], inp["v"], inp.get("cu_seqlens"))
    ws = _native.workspace(_native.fwd_workspace_bytes(shape), inp["q"].device)
    res = sf.sf_gdn_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                              inp.get("initial_state"), cu_seqlens=inp.get("cu_seqlens"),
                              output_final_state=True, ws=ws, **kw)
    _native.sf_workspace_status(ws)
    return res


def check_fwd(inp, tol=None):
    out, fin = run_fwd(inp)
    torch.cuda.synchronize()
    ref_out, ref_fin = oracle_fwd(inp)
    tol = tol or TOL[inp["q"].dtype]
    rows = active_rows(inp["q"].shape[1], inp.get("cu_seqlens"))
    e_out = rel_err(out, ref_out, rows) if len(rows) else 0.0
    e_fin = rel_err(fin, ref_fin)
    assert e_out <= tol and e_fin <= tol, (e_out, e_fin)
    return out, fin, e_out, e_fin


def test_tiny_f32_config():
    """B=1, T=256, H=2, K=V=64, FP32, zero initial state, seed 0."""
    from chunked_linear_recurrence_gb300.workloads import make_inputs, workloads
    inp = make_inputs(workloads()["tiny_f32"], "cuda")
    check_fwd(inp, tol=1e-4)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B,T,H,s0", [(2, 200, 3, True), (1, 1, 2, True), (1, 64, 1, False),
                                      (3, 65, 2, True), (1, 333, 1, True)])
def test_dense_ragged(dtype, D, B, T, H, s0):
    inp = small_inputs(B, T, H, D, dtype, seed=B * 1000 + T + D, s0=s0)
    check_fwd(inp)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("D", [64, 128])
def test_packed_varlen_with_inactive_tail(dtype, D):
    """Empty sequences pass their state through; rows past cu_seqlens[-1]
    (filled with NaN inputs) are neither read into a sequence nor written."""
    lengths = [0, 1, 63, 64, 65, 130, 0, 200]
    T = sum(lengths) + 37
    inp = small_inputs(1, T, 2, D, dtype, seed=77 + D, lengths=lengths)
    tail = sum(lengths)
    for n in ("q", "k", "v"):
        inp[n][:, tail:] = float("nan")
    inp["gate"][:, tail:] = float("nan")
    inp["beta"][:, tail:] = float("nan")
    sf = _lib()
    out = torch.full_like(inp["v"], 7.0)
    out, fin = sf.sf_gdn_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                                   inp["initial_state"], cu_seqlens=inp["cu_seqlens"],
                                   output_final_state=True, out=out)
    torch.cuda.synchronize()
    assert bool((out[:, tail:] == 7.0).all()), "inactive rows were written"
    ref_out, ref_fin = oracle_fwd(inp)
    rows = np.arange(tail)
    assert rel_err(out, ref_out, rows) <= TOL[dtype]
    assert rel_err(fin, ref_fin) <= TOL[dtype]
    # empty sequences: final == initial, bit for bit
    assert torch.equal(fin[0], inp["initial_state"][0])
    assert torch.equal(fin[6], inp["initial_state"][6])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("D", [64, 128])
def test_packed_equals_per_sequence_bitwise(dtype, D):
    """Document-aligned invariant: a packed run is bit-identical to running
    every sequence alone as a dense B=1 call (outputs and final states)."""
    lengths = [40, 192, 152, 0, 77]
    inp = small_inputs(1, sum(lengths), 2, D, dtype, seed=5 + D, lengths=lengths)
    out, fin = run_fwd(inp)
    cu = inp["cu_seqlens"].tolist()
    for n, L in enumerate(lengths):
        s, e = cu[n], cu[n + 1]
        one = {x: inp[x][:, s:e].contiguous() for x in ("q", "k", "v", "gate", "beta")}
        one["initial_state"] = inp["initial_state"][n:n + 1].contiguous()
        if L == 0:
            continue
        o1, f1 = run_fwd(one)
        assert torch.equal(out[:, s:e], o1), n
        assert torch.equal(fin[n:n + 1], f1), n


def test_deterministic_bitwise():
    inp = small_inputs(2, 300, 4, 128, torch.bfloat16, seed=3)
    o1, f1 = run_fwd(inp)
    o2, f2 = run_fwd(inp)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)


def test_page_offset_example_packed():
    """The page's global cu_seqlens (0, 40, 232, 384) as a packed call."""
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "cp_offsets_example.json")) as f:
        cu = json.load(f)["cu_seqlens_global"]
    lengths = [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]
    inp = small_inputs(1, cu[-1], 2, 128, torch.bfloat16, seed=11, lengths=lengths)
    check_fwd(inp)


def test_scale_argument():
    inp = small_inputs(1, 100, 2, 64, torch.float32, seed=9)
    sf = _lib()
    out, fin = sf.sf_gdn_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                                   inp["initial_state"], scale=0.37, output_final_state=True)
    ref_out, ref_fin = oracle_fwd(inp, scale=0.37)
    assert rel_err(out, ref_out) <= 1e-4 and rel_err(fin, ref_fin) <= 1e-4


def test_status_errors_are_reported_before_launch():
    import chunked_linear_recurrence_gb300 as sf
    inp = small_inputs(1, 64, 1, 64, torch.float32, seed=1)
    with pytest.raises(sf.SfError) as ei:
        sf.sf_gdn_chunk_fwd(inp["q"], inp["k"], inp["v"][..., :32].contiguous(), inp["gate"],
                            inp["beta"])
    assert ei.value.status == 2      # SF_ERR_UNSUPPORTED (K != V)
    with pytest.raises(sf.SfError) as ei:
        sf.sf_gdn_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                            ws=torch.zeros(16, dtype=torch.uint8, device="cuda"))
    assert ei.value.status == 3      # SF_ERR_WORKSPACE
