"""Parity at the full sizes of the measured workloads: the CUDA path, called
through the C ABI in the launch configuration the benchmark times, against the
FP64 oracle element by element on the same seeded inputs (Attention Gym,
"Linear Attention", section "Gated Delta Rule": chunking changes only the
decomposition and the floating-point order, so every returned tensor must
match the token-by-token rule).

Tolerance per returned tensor: max |x - ref| / max |ref| <= 2e-2 (BF16 q/k/v).
The oracle runs on the host cores in groups of heads, which bounds its FP64
copies of the inputs at the 262144-token size to a few GB.

Workloads (chunked_linear_recurrence_gb300.workloads):
  * forward B=4, T=4096, H=16, K=V=128, and its low-decay variant;
  * packed varlen, H=32, 8 sequences (one empty, one not a multiple of 64),
    T_phys = 65536 with an inactive tail: outputs, final states, untouched
    inactive rows, and packed == per-sequence bit for bit;
  * state passing, B=1, T=262144, H=16, 16 segments: summaries, the scan,
    the segment forward from the scanned entry states, the single pass and the
    carried-state segment loop, with the default gate (where P underflows to
    zero, so finiteness plus parity) and the low-decay variant (where the
    entry states reach through every segment);
  * forward + backward B=2, T=8192, H=16: out, final state and all six
    gradients.

The state-passing workload also runs with gate x 1e-5 and beta x 0.01 (the
"carry" variant): with the default gate and with the low-decay factors the map
of a 16384-token segment shrinks to zero or about 1e-9, so only this variant
shows that each segment really starts from the state its predecessors left.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL

pytestmark = pytest.mark.gpu
TOLB = TOL[torch.bfloat16]


def _sf():
    import chunked_linear_recurrence_gb300 as sf
    return sf


def _w(name):
    from chunked_linear_recurrence_gb300.workloads import make_inputs, workloads
    w = workloads()[name]
    return w, make_inputs(w, "cuda")


def _np(t, heads=None, axis=2):
    """float64 NumPy copy of a tensor, optionally restricted to a slice of heads."""
    if t is None:
        return None
    if heads is not None:
        t = t.narrow(axis, heads.start, heads.stop - heads.start)
    return t.detach().to("cpu", torch.float64).numpy()


class Err:
    """Accumulates max |x - ref| and max |ref| of one tensor over several parts."""

    def __init__(self):
        self.num = 0.0
        self.den = 0.0

    def add(self, x, ref):
        x = np.asarray(x, np.float64)
        ref = np.asarray(ref, np.float64)
        assert np.isfinite(x).all(), "non-finite GPU values"
        self.num = max(self.num, float(np.abs(x - ref).max()) if x.size else 0.0)
        self.den = max(self.den, float(np.abs(ref).max()) if ref.size else 0.0)

    @property
    def rel(self):
        return self.num / (self.den if self.den > 0 else 1.0)


def _fwd(inp, **kw):
    """Forward through the C ABI with an explicit workspace whose status word is checked."""
    from chunked_linear_recurrence_gb300 import _native
    sf = _sf()
    shape = _native.make_shape(inp["q"], inp["v"], kw.get("cu_seqlens", inp.get("cu_seqlens")))
    ws = _native.workspace(_native.fwd_workspace_bytes(shape), inp["q"].device)
    kw.setdefault("cu_seqlens", inp.get("cu_seqlens"))
    kw.setdefault("initial_state", inp.get("initial_state"))
    res = sf.sf_gdn_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                              output_final_state=True, ws=ws, **kw)
    _native.sf_workspace_status(ws)
    return res


def _oracle_fwd_groups(inp, group, s0=None, cu=None):
    """Oracle forward over groups of `group` heads; yields (heads, out, final)."""
    H = inp["v"].shape[2]
    s0 = inp.get("initial_state") if s0 is None else s0
    for h0 in range(0, H, group):
        hs = slice(h0, min(H, h0 + group))
        ro, rf = oracle.gdn_fwd(_np(inp["q"], hs), _np(inp["k"], hs), _np(inp["v"], hs),
                                _np(inp["gate"], hs), _np(inp["beta"], hs),
                                _np(s0, hs, axis=1), cu_seqlens=cu)
        yield hs, ro, rf


@pytest.mark.parametrize("name", ["fwd_bf16_b4_t4096_h16", "fwd_bf16_b4_t4096_h16_lowdecay"])
def test_forward_b4_t4096_h16(name):
    _, inp = _w(name)
    out, fin = _fwd(inp)
    torch.cuda.synchronize()
    eo, ef = Err(), Err()
    for hs, ro, rf in _oracle_fwd_groups(inp, 16):
        eo.add(_np(out, hs), ro)
        ef.add(_np(fin, hs, axis=1), rf)
    assert eo.rel <= TOLB and ef.rel <= TOLB, (eo.rel, ef.rel)


def test_packed_varlen_h32():
    w, inp = _w("varlen_bf16_h32")
    cu = inp["cu_seqlens"]
    cuh = [int(c) for c in cu]
    tail = cuh[-1]
    assert w.lengths[3] == 0 and w.lengths[5] % 64 != 0 and tail <= inp["q"].shape[1]
    sentinel = 7.0
    out = torch.full_like(inp["v"], sentinel)
    out, fin = _fwd(inp, out=out)
    torch.cuda.synchronize()
    # inactive rows are never written
    assert bool((out[:, tail:] == sentinel).all()), "inactive rows were written"
    eo, ef = Err(), Err()
    for hs, ro, rf in _oracle_fwd_groups(inp, 8, cu=cu.cpu().numpy()):
        eo.add(_np(out, hs)[:, :tail], ro[:, :tail])
        ef.add(_np(fin, hs, axis=1), rf)
    assert eo.rel <= TOLB and ef.rel <= TOLB, (eo.rel, ef.rel)
    # packed == per-sequence dense runs, bit for bit (outputs and final states)
    for n in range(len(w.lengths)):
        a, b = cuh[n], cuh[n + 1]
        one = {x: inp[x][:, a:b].contiguous() for x in ("q", "k", "v", "gate", "beta")}
        o1, f1 = _fwd(one, cu_seqlens=None,
                      initial_state=inp["initial_state"][n:n + 1].contiguous())
        torch.cuda.synchronize()
        assert torch.equal(o1, out[:, a:b]), f"sequence {n}: output differs from the packed run"
        assert torch.equal(f1[0], fin[n]), f"sequence {n}: final state differs"
    # the empty sequence passes its initial state through unchanged
    assert torch.equal(fin[3], inp["initial_state"][3])


@pytest.mark.parametrize("name", ["statepass_bf16_t262144_h16",
                                  "statepass_bf16_t262144_h16_lowdecay",
                                  "statepass_bf16_t262144_h16_carry"])
def test_state_passing_t262144_h16(name):
    from chunked_linear_recurrence_gb300.workloads import segment_bounds
    sf = _sf()
    w, inp = _w(name)
    T, H, R = w.T, w.H, w.segments
    L = T // R
    bounds = segment_bounds(T, R)
    P, E = sf.sf_gdn_segment_summary(inp["k"], inp["v"], inp["gate"], inp["beta"], bounds.cuda())
    s0 = inp.get("initial_state")
    S0 = None if s0 is None else s0[0].contiguous()          # [H,V,K]
    entry, final = sf.sf_state_scan(P, E, S0)
    seg_cu = torch.arange(0, T + 1, L, dtype=torch.int32, device="cuda")
    out_seg, fin_seg = _fwd(inp, cu_seqlens=seg_cu, initial_state=entry.contiguous())
    out_one, fin_one = _fwd(inp)                               # one sequential pass
    # the carried-state loop: each segment run alone from the previous segment's final state
    carried = torch.empty_like(inp["v"])
    cur = s0
    for j in range(R):
        part = {x: inp[x][:, j * L:(j + 1) * L].contiguous()
                for x in ("q", "k", "v", "gate", "beta")}
        o, cur = _fwd(part, cu_seqlens=None, initial_state=cur)
        carried[:, j * L:(j + 1) * L] = o
    torch.cuda.synchronize()
    for t in (P, E, entry, final, out_seg, fin_seg, out_one, fin_one, carried, cur):
        assert bool(torch.isfinite(t).all())

    e = {n: Err() for n in ("P", "E", "entry", "final", "seg_out", "seg_fin", "one_out",
                            "one_fin", "loop_out", "loop_fin")}
    G = 8
    for h0 in range(0, H, G):
        hs = slice(h0, h0 + G)
        Pr, Er = oracle.segment_summary(_np(inp["k"], hs), _np(inp["v"], hs),
                                        _np(inp["gate"], hs), _np(inp["beta"], hs),
                                        bounds.numpy())
        e["P"].add(_np(P, hs, axis=1), Pr)
        e["E"].add(_np(E, hs, axis=1), Er)
        s0h = None if S0 is None else _np(S0, hs, axis=0)
        ent_r, fin_r = oracle.state_scan(Pr, Er, s0h)
        e["entry"].add(_np(entry, hs, axis=1), ent_r)
        e["final"].add(_np(final, hs, axis=0), fin_r)
        ro, rf = oracle.gdn_fwd(_np(inp["q"], hs), _np(inp["k"], hs), _np(inp["v"], hs),
                                _np(inp["gate"], hs), _np(inp["beta"], hs),
                                None if s0 is None else _np(s0, hs, axis=1))
        e["seg_out"].add(_np(out_seg, hs), ro)
        e["seg_fin"].add(_np(fin_seg[R - 1], hs, axis=0), rf[0])
        e["one_out"].add(_np(out_one, hs), ro)
        e["one_fin"].add(_np(fin_one, hs, axis=1), rf)
        e["loop_out"].add(_np(carried, hs), ro)
        e["loop_fin"].add(_np(cur, hs, axis=1), rf)
        del Pr, Er, ro
    bad = {n: x.rel for n, x in e.items() if not x.rel <= TOLB}
    assert not bad, bad
    if w.carry:
        # the entry states must matter here: P keeps a sizeable norm over a whole segment
        assert float(P.abs().max()) > 0.1


def test_forward_backward_b2_t8192_h16():
    sf = _sf()
    from chunked_linear_recurrence_gb300 import _native
    _, inp = _w("fwdbwd_bf16_b2_t8192_h16")
    out, fin = _fwd(inp)
    shape = _native.make_shape(inp["q"], inp["v"])
    ws = _native.workspace(_native.bwd_workspace_bytes(shape), inp["q"].device)
    g = sf.sf_gdn_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                            inp["initial_state"], inp["d_out"], inp["d_final_state"], ws=ws)
    _native.sf_workspace_status(ws)
    torch.cuda.synchronize()
    args = [_np(inp[n]) for n in ("q", "k", "v", "gate", "beta")]
    ro, rf = oracle.gdn_fwd(*args, _np(inp["initial_state"]))
    rg = oracle.gdn_bwd(*args, _np(inp["initial_state"]), _np(inp["d_out"]),
                        _np(inp["d_final_state"]))
    errs = {}
    for n, x, r in (("out", out, ro), ("final_state", fin, rf), ("dq", g["dq"], rg["dq"]),
                    ("dk", g["dk"], rg["dk"]), ("dv", g["dv"], rg["dv"]),
                    ("dgate", g["dgate"], rg["dg"]), ("dbeta", g["dbeta"], rg["dbeta"]),
                    ("d_initial_state", g["d_initial_state"], rg["d_initial_state"])):
        ee = Err()
        ee.add(_np(x), r)
        errs[n] = ee.rel
    bad = {n: v for n, v in errs.items() if not v <= TOLB}
    assert not bad, errs


@pytest.mark.parametrize("D", [64, 128])
def test_empty_token_stream(D):
    """T = 0: the forward passes each initial state through to the final state and the
    backward passes d_final_state through to d_initial_state, launching no token work."""
    sf = _sf()
    from helpers import small_inputs
    inp = small_inputs(2, 0, 2, D, torch.bfloat16, seed=5, grads=True)
    out, fin = sf.sf_gdn_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                                   inp["initial_state"], output_final_state=True)
    g = sf.sf_gdn_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                            inp["initial_state"], inp["d_out"], inp["d_final_state"])
    torch.cuda.synchronize()
    assert torch.equal(fin, inp["initial_state"])
    assert torch.equal(g["d_initial_state"], inp["d_final_state"])
