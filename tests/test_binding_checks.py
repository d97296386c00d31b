"""The Python binding checks the tensor shapes and dtypes that the C ABI takes on trust from
its shape struct, and raises before anything reaches the library (CPU tensors: a call that
passes the checks fails later, on the device check)."""
import pytest
import torch


def _inputs(B=1, T=64, H=2, HK=2, D=64, N=None):
    q = torch.zeros(B, T, HK, D)
    return dict(q=q, k=q.clone(), v=torch.zeros(B, T, H, D), gate=torch.zeros(B, T, H),
                beta=torch.zeros(B, T, H), s0=torch.zeros(N or B, H, D, D),
                d_out=torch.zeros(B, T, H, D))


def _fwd(x, **kw):
    import chunked_linear_recurrence_gb300 as sf
    return sf.sf_gdn_chunk_fwd(x["q"], x["k"], x["v"], x["gate"], x["beta"], x["s0"], **kw)


def _bwd(x, **kw):
    import chunked_linear_recurrence_gb300 as sf
    return sf.sf_gdn_chunk_bwd(x["q"], x["k"], x["v"], x["gate"], x["beta"], x["s0"], x["d_out"],
                               **kw)


def test_consistent_shapes_pass_the_checks():
    with pytest.raises(ValueError, match="CUDA device"):
        _fwd(_inputs())
    with pytest.raises(ValueError, match="CUDA device"):
        _fwd(_inputs(H=4, HK=2))                       # grouped heads
    with pytest.raises(ValueError, match="CUDA device"):
        _bwd(_inputs())


@pytest.mark.parametrize("field,value,msg", [
    ("k", torch.zeros(1, 64, 1, 64), "k "),
    ("gate", torch.zeros(1, 63, 2), "gate must be"),
    ("beta", torch.zeros(1, 64, 3), "beta must be"),
    ("s0", torch.zeros(2, 2, 64, 64), "initial_state must be"),
    ("v", torch.zeros(1, 64, 2, 64, dtype=torch.bfloat16), "one dtype"),
    ("v", torch.zeros(1, 32, 2, 64), "does not match q"),
])
def test_mismatched_inputs_are_rejected(field, value, msg):
    x = _inputs()
    x[field] = value
    with pytest.raises(ValueError, match=msg):
        _fwd(x)


def test_mismatched_outputs_and_cotangents_are_rejected():
    x = _inputs()
    with pytest.raises(ValueError, match="out must be"):
        _fwd(x, out=torch.zeros(1, 64, 2, 32))
    with pytest.raises(ValueError, match="final_state must be"):
        _fwd(x, output_final_state=True, final_state=torch.zeros(1, 2, 64, 32))
    x["d_out"] = torch.zeros(1, 64, 2, 32)
    with pytest.raises(ValueError, match="d_out must be"):
        _bwd(x)
    x = _inputs()
    with pytest.raises(ValueError, match="d_final_state must be"):
        _bwd(x, d_final_state=torch.zeros(3, 2, 64, 64))
    cu = torch.tensor([0, 30, 64], dtype=torch.int32)
    with pytest.raises(ValueError, match="initial_state must be"):
        _bwd(x, cu_seqlens=cu)                         # two sequences, one initial state
    with pytest.raises(ValueError, match="int32"):
        _fwd(x, cu_seqlens=cu.long())
