"""The C-ABI library loads without a GPU, exports every function include/*.h
declares, and rejects bad arguments on the host before anything launches
(these calls never reach a CUDA API, so they run on the CPU machine)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*(sf_[a-z0-9_]+)\s*\(",
                             src, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    from chunked_linear_recurrence_gb300 import _native
    if not os.path.exists(_native.LIB_PATH):
        from chunked_linear_recurrence_gb300 import build
        build.build()
    return _native.load()


def test_every_declared_symbol_is_exported(lib):
    from chunked_linear_recurrence_gb300 import _native
    names = declared_functions()
    assert len(names) >= 10
    assert names <= set(_native.EXPORTS), names - set(_native.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n
    assert lib.sf_version().decode().startswith("sf_gdn")


def _shape(**kw):
    from chunked_linear_recurrence_gb300._native import sf_gdn_shape
    d = dict(B=1, T=64, H=1, K=128, V=128, N=1, dtype=1, scale=0.0)
    d.update(kw)
    return sf_gdn_shape(**d)


FAKE = ctypes.c_void_p(1 << 20)          # 16-byte aligned, never dereferenced


def _fwd(lib, shape, out_final=0, ws_bytes=4096, ptr=FAKE, cu=None, fin=None):
    return lib.sf_gdn_chunk_fwd(ctypes.byref(shape), ptr, ptr, ptr, ptr, ptr, None, cu, out_final,
                                ptr, fin, FAKE, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(K=96, V=96), 2), (dict(K=128, V=64), 2), (dict(T=-1), 1), (dict(H=0), 1),
    (dict(dtype=7), 1), (dict(N=2), 1), (dict(B=40000, T=40000), 2),
    (dict(H=4, HK=3), 1), (dict(H=4, HK=-1), 1), (dict(H=2, HK=4), 1)])
def test_forward_rejects_bad_shapes(lib, kw, status):
    assert _fwd(lib, _shape(**kw)) == status
    assert len(lib.sf_last_error()) > 0


def test_forward_rejects_bad_pointers_and_workspace(lib):
    assert _fwd(lib, _shape(), ptr=ctypes.c_void_p(0)) == 1
    assert _fwd(lib, _shape(), ptr=ctypes.c_void_p((1 << 20) + 4)) == 1      # misaligned
    assert _fwd(lib, _shape(), out_final=1, fin=None) == 1
    assert _fwd(lib, _shape(), ws_bytes=8) == 3
    # cu_seqlens requires B == 1
    assert _fwd(lib, _shape(B=2, N=3), cu=FAKE) == 1


def test_other_entry_points_reject_bad_arguments(lib):
    s = _shape()
    assert lib.sf_gdn_segment_summary(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, FAKE, -1, FAKE,
                                      FAKE, FAKE, 4096, None) == 1
    assert lib.sf_gdn_segment_summary(ctypes.byref(s), FAKE, None, FAKE, FAKE, FAKE, 2, FAKE,
                                      FAKE, FAKE, 4096, None) == 1
    assert lib.sf_state_scan(2, 1, 96, 96, FAKE, FAKE, None, FAKE, None, None) == 2
    assert lib.sf_state_scan(2, 1, 128, 128, None, FAKE, None, FAKE, None, None) == 1
    s32 = _shape(dtype=0)
    assert lib.sf_gdn_chunk_bwd(ctypes.byref(s32), *([FAKE] * 5), None, None, FAKE, None,
                                *([FAKE] * 5), None, FAKE, 1 << 40, None) == 2
    need = lib.sf_gdn_bwd_workspace(ctypes.byref(s))
    assert need >= 256 + 2 * 128 * 128 * 4      # one chunk: checkpoint + cotangent tape
    assert lib.sf_gdn_chunk_bwd(ctypes.byref(s), *([FAKE] * 5), None, None, FAKE, None,
                                *([FAKE] * 5), None, FAKE, need - 1, None) == 3


def test_grouped_heads_workspace(lib):
    """HK = 0 means HK = H; the backward of grouped heads adds two FP32 [B,T,H,K] areas for
    the per-value-head parts of dq and dk, and nothing else changes."""
    plain = lib.sf_gdn_bwd_workspace(ctypes.byref(_shape(H=4, T=256)))
    assert lib.sf_gdn_bwd_workspace(ctypes.byref(_shape(H=4, HK=4, T=256))) == plain
    grouped = lib.sf_gdn_bwd_workspace(ctypes.byref(_shape(H=4, HK=2, T=256)))
    assert grouped == plain + 2 * 256 * 4 * 128 * 4
    assert (lib.sf_gdn_fwd_workspace(ctypes.byref(_shape(H=4, HK=1, T=256))) ==
            lib.sf_gdn_fwd_workspace(ctypes.byref(_shape(H=4, T=256))))


def test_packed_backward_workspace_scales_with_tokens_not_sequences(lib):
    """Packed inputs (B = 1) need ceil(T/64) + N chunk slots, not N * ceil(T/64): eight
    sequences over T = 4096 at BF16, K = V = 128 cost seven chunk slots per head (115,712
    bytes each: checkpoint, cotangent, factors) and seven more replay-ring streams per head
    (540,672 bytes each: 16 ring slots of 33,792-byte records) beyond one sequence -- not
    eight times as much."""
    one = lib.sf_gdn_bwd_workspace(ctypes.byref(_shape(T=4096, H=2, N=1)))
    eight = lib.sf_gdn_bwd_workspace(ctypes.byref(_shape(T=4096, H=2, N=8)))
    assert eight - one == 7 * 2 * 115712 + 7 * 2 * 540672
    dense = lib.sf_gdn_bwd_workspace(ctypes.byref(_shape(B=8, N=8, T=4096, H=2)))
    assert dense - eight == (8 * 64 - (64 + 8)) * 2 * 115712


def test_reverse_maps_reject_bad_arguments(lib):
    """The reverse summary wants packed offsets (B = 1), C and a large enough workspace;
    the reverse scan the same sizes as the forward scan."""
    s = _shape(T=256, N=2)
    need = lib.sf_gdn_reverse_summary_workspace(ctypes.byref(s))
    args = (FAKE, FAKE, FAKE, FAKE, FAKE)
    assert lib.sf_gdn_segment_reverse_summary(ctypes.byref(s), *args, None, FAKE, FAKE, need,
                                              None) == 1          # no offsets
    assert lib.sf_gdn_segment_reverse_summary(ctypes.byref(s), *args, FAKE, None, FAKE, need,
                                              None) == 1          # no C
    assert lib.sf_gdn_segment_reverse_summary(ctypes.byref(s), *args, FAKE, FAKE, FAKE, need - 1,
                                              None) == 3          # workspace too small
    assert lib.sf_gdn_segment_reverse_summary(ctypes.byref(_shape(B=2, T=256, N=2)), *args, FAKE,
                                              FAKE, FAKE, need, None) == 1   # offsets need B = 1
    assert lib.sf_gdn_segment_reverse_summary(ctypes.byref(_shape(T=256, N=2, dtype=0)), *args,
                                              FAKE, FAKE, FAKE, need, None) == 2   # FP32 at K = 128
    assert lib.sf_state_scan_reverse(2, 1, 128, 64, FAKE, FAKE, None, FAKE, None, None) == 2
    assert lib.sf_state_scan_reverse(-1, 1, 128, 128, FAKE, FAKE, None, FAKE, None, None) == 1
    assert lib.sf_state_scan_reverse(2, 1, 128, 128, None, FAKE, None, FAKE, None, None) == 1


def test_paged_forward_rejects_bad_arguments(lib):
    """The paged forward wants a cache, slot indices, num_slots >= 1 and an aligned cache;
    otherwise it checks exactly what the plain forward checks."""
    s = _shape(T=64, N=1)
    def call(cache=FAKE, nslots=4, idx=FAKE, ws=4 << 20, shape=s):
        return lib.sf_gdn_paged_chunk_fwd(ctypes.byref(shape), FAKE, FAKE, FAKE, FAKE, FAKE, cache,
                                          nslots, idx, None, None, FAKE, FAKE, ws, None)
    assert call(cache=None) == 1
    assert call(idx=None) == 1
    assert call(nslots=0) == 1
    assert call(cache=ctypes.c_void_p((1 << 20) + 4)) == 1    # misaligned cache
    assert call(ws=8) == 3
    assert call(shape=_shape(K=96, V=96)) == 2


_NO_ENCODER_SCRIPT = r'''
import ctypes, sys
sys.path.insert(0, sys.argv[1])
from chunked_linear_recurrence_gb300 import _native
lib = _native.load()
F = ctypes.c_void_p(1 << 20)
sh = _native.sf_gdn_shape(B=1, T=64, H=1, K=128, V=128, N=1, dtype=1, scale=0.0, HK=0)
r = []
ws = lib.sf_gdn_fwd_workspace(ctypes.byref(sh))
r.append(lib.sf_gdn_chunk_fwd(ctypes.byref(sh), F, F, F, F, F, None, None, 0, F, None, F, ws, None))
r.append(lib.sf_last_error())
ws = lib.sf_gdn_summary_workspace(ctypes.byref(sh), 1)
r.append(lib.sf_gdn_segment_summary(ctypes.byref(sh), F, F, F, F, F, 1, F, F, F, ws, None))
r.append(lib.sf_last_error())
ws = lib.sf_gdn_bwd_workspace(ctypes.byref(sh))
r.append(lib.sf_gdn_chunk_bwd(ctypes.byref(sh), F, F, F, F, F, None, None, F, None, F, F, F, F,
                              F, None, F, ws, None))
r.append(lib.sf_last_error())
print(repr(r))
'''


def test_bf16_128_without_tensor_map_encoder_is_unsupported(lib):
    """BF16 with K = V = 128 runs only on the tensor-core kernels: with the driver's TMA
    descriptor encoder reported absent (a host-side switch, set here in a child process),
    the forward, the summary and the backward return SF_ERR_UNSUPPORTED with a message and
    launch nothing -- no CUDA-core kernel stands in for them."""
    import ast
    import subprocess
    import sys
    env = dict(os.environ, SF_GDN_DISABLE_TMA_ENCODER="1")
    res = subprocess.run([sys.executable, "-c", _NO_ENCODER_SCRIPT, ROOT], env=env,
                         capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    r = ast.literal_eval(res.stdout.strip().splitlines()[-1])
    for status, msg in zip(r[0::2], r[1::2]):
        assert status == 2, (status, msg)               # SF_ERR_UNSUPPORTED
        assert b"cuTensorMapEncodeTiled" in msg, msg


def test_noalloc_scratch_capacity_matches_the_header(lib):
    """The allocation-free backward takes shapes whose sf_gdn_bwd_workspace fits its fixed
    scratch (SF_BWD_NOALLOC_SCRATCH_BYTES, 32 MiB); the header states that one sequence of
    2 heads at BF16, K = V = 128 fits up to T = 8896, and no longer."""
    scratch = 32 << 20
    ws = lambda T: lib.sf_gdn_bwd_workspace(ctypes.byref(_shape(T=T, H=2, N=1)))
    assert ws(8896) <= scratch < ws(8897)
