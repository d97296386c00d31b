"""Failure detection on the device without a fault: a bounded wait that runs out.

The split tensor-core kernel's CTAs hand chunk records to each other through
flags in the workspace, and every wait on a flag or an mbarrier is bounded.
sf_testing_inject_timeout makes the next launch skip publishing one record and
shortens every wait to a few milliseconds: the chain that needs the record
gives up, raises the kernel's abort flag, every CTA leaves once its own copies
and products have completed, and the status word reads SF_ERR_TIMEOUT.  The
context must stay usable: the next, normal launch matches the oracle."""
import pytest
import torch

from helpers import TOL, active_rows, oracle_fwd, rel_err, small_inputs

pytestmark = pytest.mark.gpu
WAIT = 20_000_000          # SM clock cycles (about 10 ms)


def _ws(inp):
    from chunked_linear_recurrence_gb300 import _native
    shape = _native.make_shape(inp["q"], inp["v"], inp.get("cu_seqlens"))
    return _native.workspace(_native.fwd_workspace_bytes(shape), inp["q"].device)


@pytest.mark.parametrize("record", [5, 37])
def test_injected_timeout_is_reported_and_the_next_launch_is_correct(record):
    import chunked_linear_recurrence_gb300 as sf
    from chunked_linear_recurrence_gb300 import _native
    lib = sf.load()
    inp = small_inputs(2, 640, 4, 128, torch.bfloat16, seed=9)    # 8 chains x 10 chunks
    ws = _ws(inp)
    assert lib.sf_testing_inject_timeout(record, WAIT) == 0
    sf.sf_gdn_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                        inp["initial_state"], output_final_state=True, ws=ws)
    with pytest.raises(_native.SfError) as err:
        _native.sf_workspace_status(ws)
    assert err.value.status == _native.SF_ERR_TIMEOUT
    _native.sf_workspace_status(ws)                       # read once, then cleared
    # the same context, the same workspace: a normal launch
    out, fin = sf.sf_gdn_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                                   inp["initial_state"], output_final_state=True, ws=ws)
    _native.sf_workspace_status(ws)
    torch.cuda.synchronize()
    ref_out, ref_fin = oracle_fwd(inp)
    rows = active_rows(inp["q"].shape[1], None)
    assert rel_err(out, ref_out, rows) <= TOL[torch.bfloat16]
    assert rel_err(fin, ref_fin) <= TOL[torch.bfloat16]


def test_injection_rejects_bad_arguments():
    import chunked_linear_recurrence_gb300 as sf
    lib = sf.load()
    assert lib.sf_testing_inject_timeout(-1, WAIT) == 1
    assert lib.sf_testing_inject_timeout(3, 10) == 1
