"""The workspace-free backward (sf_gdn_chunk_bwd_noalloc) against the
workspace backward (sf_gdn_chunk_bwd), called through the C ABI twice in a
row.  It serves callers that cannot allocate device memory where they need
gradients (runtimes whose allocator is frozen after warm-up, embedders that
own all device memory), using a fixed scratch array inside the library
instead.  After every call the array's status word is read back through
sf_gdn_chunk_bwd_noalloc_status: no kernel may have reported a timeout.

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import ctypes

import pytest
import torch

from helpers import TOL, rel_err, small_inputs

pytestmark = pytest.mark.gpu
NAMES = ["dq", "dk", "dv", "dgate", "dbeta", "d_initial_state"]


def _call_noalloc(lib, inp, grads):
    from chunked_linear_recurrence_gb300 import _native
    shape = _native.make_shape(inp["q"], inp["v"], inp.get("cu_seqlens"))
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.sf_gdn_chunk_bwd_noalloc(
        ctypes.byref(shape), p(inp["q"]), p(inp["k"]), p(inp["v"]), p(inp["gate"]),
        p(inp["beta"]), p(inp.get("initial_state")), p(inp.get("cu_seqlens")), p(inp["d_out"]),
        p(inp.get("d_final_state")), p(grads["dq"]), p(grads["dk"]), p(grads["dv"]),
        p(grads["dgate"]), p(grads["dbeta"]), p(grads["d_initial_state"]), stream)


@pytest.mark.parametrize("dtype,D,lengths", [(torch.bfloat16, 128, None),
                                             (torch.float32, 64, [0, 70, 1, 128])])
def test_noalloc_backward_matches_workspace_backward_twice(dtype, D, lengths):
    import chunked_linear_recurrence_gb300 as sf
    lib = sf.load()
    for call in range(2):                       # two calls in a row share the scratch
        if lengths is None:
            inp = small_inputs(2, 150 + 37 * call, 2, D, dtype, seed=40 + call, grads=True)
        else:
            inp = small_inputs(1, sum(lengths) + 9, 2, D, dtype, seed=50 + call,
                               lengths=lengths, grads=True)
        ref = sf.sf_gdn_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                                  inp["initial_state"], inp["d_out"], inp["d_final_state"],
                                  cu_seqlens=inp.get("cu_seqlens"))
        got = {n: torch.full_like(t, float("nan")) for n, t in ref.items()}
        assert _call_noalloc(lib, inp, got) == 0, lib.sf_last_error().decode()
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        assert lib.sf_gdn_chunk_bwd_noalloc_status(stream) == 0, lib.sf_last_error().decode()
        torch.cuda.synchronize()
        T = inp["q"].shape[1]
        rows = torch.arange(T) if lengths is None else torch.arange(sum(lengths))
        for n in NAMES:
            r, g = ref[n], got[n]
            if n != "d_initial_state":
                r, g = r[:, rows], g[:, rows]
            assert rel_err(g, r.double().cpu().numpy()) <= TOL[dtype], (call, n)


def test_noalloc_backward_rejects_shapes_beyond_its_scratch():
    import chunked_linear_recurrence_gb300 as sf
    lib = sf.load()
    # 400 chunk-heads of 115,712 bytes: beyond the 32 MiB scratch
    inp = small_inputs(1, 64 * 400, 1, 128, torch.bfloat16, seed=3, grads=True)
    got = {n: torch.empty_like(inp[n if n != "dgate" else "gate"]) for n in
           ("q", "k", "v", "dgate", "beta")}
    grads = dict(dq=got["q"], dk=got["k"], dv=got["v"], dgate=got["dgate"], dbeta=got["beta"],
                 d_initial_state=None)
    assert _call_noalloc(lib, inp, grads) == 2          # SF_ERR_UNSUPPORTED, nothing launched
    assert b"scratch" in lib.sf_last_error()


def test_noalloc_status_word_reports_an_injected_timeout():
    """A timeout inside the allocation-free backward lands in the built-in array's status
    word, which sf_gdn_chunk_bwd_noalloc_status reads (and clears): the state replay of the
    call below is made to skip one record with a short wait limit.  A normal call follows
    and matches the workspace backward."""
    import chunked_linear_recurrence_gb300 as sf
    lib = sf.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    inp = small_inputs(1, 300, 2, 128, torch.bfloat16, seed=61, grads=True)
    got = {n: torch.empty_like(inp[s]) for n, s in (("dq", "q"), ("dk", "k"), ("dv", "v"),
                                                     ("dgate", "gate"), ("dbeta", "beta"),
                                                     ("d_initial_state", "initial_state"))}
    assert lib.sf_testing_inject_timeout(1, 20_000_000) == 0
    assert _call_noalloc(lib, inp, got) == 0, lib.sf_last_error().decode()
    assert lib.sf_gdn_chunk_bwd_noalloc_status(stream) == 5      # SF_ERR_TIMEOUT
    assert lib.sf_gdn_chunk_bwd_noalloc_status(stream) == 0      # cleared by the read
    ref = sf.sf_gdn_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                              inp["initial_state"], inp["d_out"], inp["d_final_state"])
    assert _call_noalloc(lib, inp, got) == 0, lib.sf_last_error().decode()
    assert lib.sf_gdn_chunk_bwd_noalloc_status(stream) == 0
    torch.cuda.synchronize()
    for n in NAMES:
        assert rel_err(got[n], ref[n].double().cpu().numpy()) <= TOL[torch.bfloat16], n
