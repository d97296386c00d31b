"""ctypes binding of libsf_gdn.so (include/sf_gdn.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  PyTorch supplies device memory and the current CUDA stream.  If the
library is missing or fails to load, every call raises -- nothing falls back.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libsf_gdn.so")

SF_OK, SF_ERR_INVALID_ARG, SF_ERR_UNSUPPORTED, SF_ERR_WORKSPACE, SF_ERR_CUDA, SF_ERR_TIMEOUT = range(6)
SF_F32, SF_BF16 = 0, 1
STATUS_NAMES = {0: "SF_OK", 1: "SF_ERR_INVALID_ARG", 2: "SF_ERR_UNSUPPORTED",
                3: "SF_ERR_WORKSPACE", 4: "SF_ERR_CUDA", 5: "SF_ERR_TIMEOUT"}

# Every symbol include/sf_gdn.h declares.
EXPORTS = ("sf_last_error", "sf_version", "sf_gdn_fwd_workspace", "sf_gdn_chunk_fwd",
           "sf_gdn_paged_chunk_fwd",
           "sf_gdn_summary_workspace", "sf_gdn_segment_summary", "sf_state_scan",
           "sf_gdn_bwd_workspace", "sf_gdn_chunk_bwd", "sf_gdn_chunk_bwd_noalloc",
           "sf_gdn_chunk_bwd_noalloc_status",
           "sf_gdn_reverse_summary_workspace", "sf_gdn_segment_reverse_summary",
           "sf_state_scan_reverse", "sf_validate_cu_seqlens", "sf_workspace_status",
           "sf_testing_inject_timeout")


class SfError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class sf_gdn_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
                ("K", ctypes.c_int), ("V", ctypes.c_int), ("N", ctypes.c_int),
                ("dtype", ctypes.c_int), ("scale", ctypes.c_float), ("HK", ctypes.c_int)]


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"libsf_gdn.so not built ({path}); run "
                               "`python -m chunked_linear_recurrence_gb300.build`")
        lib = ctypes.CDLL(path)
        vp, sz, st, I = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int
        sp = ctypes.POINTER(sf_gdn_shape)
        lib.sf_last_error.restype = ctypes.c_char_p
        lib.sf_version.restype = ctypes.c_char_p
        lib.sf_gdn_fwd_workspace.argtypes = [sp]
        lib.sf_gdn_fwd_workspace.restype = sz
        lib.sf_gdn_chunk_fwd.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, I, vp, vp, vp, sz, vp]
        lib.sf_gdn_paged_chunk_fwd.argtypes = [sp, vp, vp, vp, vp, vp, vp, I, vp, vp, vp, vp, vp,
                                               sz, vp]
        lib.sf_gdn_summary_workspace.argtypes = [sp, I]
        lib.sf_gdn_summary_workspace.restype = sz
        lib.sf_gdn_segment_summary.argtypes = [sp, vp, vp, vp, vp, vp, I, vp, vp, vp, sz, vp]
        lib.sf_state_scan.argtypes = [I, I, I, I, vp, vp, vp, vp, vp, vp]
        lib.sf_gdn_bwd_workspace.argtypes = [sp]
        lib.sf_gdn_bwd_workspace.restype = sz
        lib.sf_gdn_chunk_bwd.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                         vp, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.sf_gdn_chunk_bwd_noalloc.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                 vp, vp, vp, vp, vp, vp, vp]
        lib.sf_gdn_reverse_summary_workspace.argtypes = [sp]
        lib.sf_gdn_reverse_summary_workspace.restype = sz
        lib.sf_gdn_segment_reverse_summary.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.sf_state_scan_reverse.argtypes = [I, I, I, I, vp, vp, vp, vp, vp, vp]
        lib.sf_validate_cu_seqlens.argtypes = [vp, I, I, vp]
        lib.sf_workspace_status.argtypes = [vp, vp]
        lib.sf_gdn_chunk_bwd_noalloc_status.argtypes = [vp]
        lib.sf_testing_inject_timeout.argtypes = [ctypes.c_longlong, ctypes.c_longlong]
        for f in ("sf_gdn_chunk_fwd", "sf_gdn_paged_chunk_fwd", "sf_gdn_segment_summary",
                  "sf_state_scan",
                  "sf_gdn_chunk_bwd", "sf_gdn_chunk_bwd_noalloc",
                  "sf_gdn_chunk_bwd_noalloc_status", "sf_testing_inject_timeout",
                  "sf_validate_cu_seqlens",
                  "sf_workspace_status", "sf_gdn_segment_reverse_summary",
                  "sf_state_scan_reverse"):
            getattr(lib, f).restype = st
        _lib = lib
        return lib


def _check(rc: int):
    if rc != SF_OK:
        raise SfError(rc, load().sf_last_error().decode())


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(dt):
    if dt == torch.bfloat16:
        return SF_BF16
    if dt == torch.float32:
        return SF_F32
    raise ValueError(f"q/k/v dtype must be bfloat16 or float32, got {dt}")


def make_shape(q, v, cu_seqlens=None, scale=None) -> sf_gdn_shape:
    """Shape of q (or k) [B,T,HK,K] and v [B,T,H,V]: H value heads, HK query/key heads."""
    B, T, HK, K = q.shape
    H, V = v.shape[2], v.shape[-1]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    return sf_gdn_shape(B, T, H, K, V, N, _dtype_code(q.dtype),
                        float(scale) if scale is not None else 0.0, HK)


def _validate(q, v, k=None, gate=None, beta=None, cu_seqlens=None, tensors=(), states=()):
    """The tensor shapes and dtypes that the C ABI takes on trust from the shape struct:
    q, k [B,T,HK,K] of one dtype, v [B,T,H,V] in q's dtype, gate and beta [B,T,H],
    cu_seqlens int32 [N+1] (then B == 1), `tensors` (name, tensor, shape, dtype) entries
    (None tensors are skipped), `states` (name, tensor) pairs [N,H,V,K].  Raises
    ValueError before anything reaches the library (a mismatch there would be read or
    written past its end)."""
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q/k and v must be 4-D: [B,T,HK,K] and [B,T,H,V]")
    B, T, HK, K = q.shape
    H, V = v.shape[2], v.shape[3]
    if tuple(v.shape[:2]) != (B, T):
        raise ValueError(f"v {tuple(v.shape)} does not match q {tuple(q.shape)} in [B,T]")
    if v.dtype != q.dtype:
        raise ValueError("q, k and v must share one dtype")
    if k is not None and (k.shape != q.shape or k.dtype != q.dtype):
        raise ValueError(f"k {tuple(k.shape)} must match q {tuple(q.shape)} in shape and dtype")
    for name, t in (("gate", gate), ("beta", beta)):
        if t is not None and tuple(t.shape) != (B, T, H):
            raise ValueError(f"{name} must be [B,T,H] = {(B, T, H)}, got {tuple(t.shape)}")
    N = B
    if cu_seqlens is not None:
        if cu_seqlens.dim() != 1 or cu_seqlens.dtype != torch.int32:
            raise ValueError("cu_seqlens must be a 1-D int32 tensor")
        N = cu_seqlens.numel() - 1
    for name, t, shp, dt in tensors:
        if t is not None and (tuple(t.shape) != tuple(shp) or t.dtype != dt):
            raise ValueError(f"{name} must be {tuple(shp)} {dt}, got {tuple(t.shape)} {t.dtype}")
    for name, t in states:
        if t is not None and tuple(t.shape) != (N, H, V, K):
            raise ValueError(f"{name} must be [N,H,V,K] = {(N, H, V, K)}, got {tuple(t.shape)}")


def workspace(nbytes: int, device) -> torch.Tensor:
    """Zero-initialised byte buffer (the status word must start at zero)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _f32(t):
    if t is None:
        return None
    if t.dtype != torch.float32:
        raise ValueError("gate, beta and states must be float32")
    return t


def sf_gdn_chunk_fwd(q, k, v, gate, beta, initial_state=None, cu_seqlens=None, scale=None,
                     output_final_state=False, out=None, final_state=None, ws=None, stream=None):
    """chunk_gdn forward.  Returns (out [B,T,H,V], final_state [N,H,V,K] or None)."""
    lib = load()
    _validate(q, v, k, gate, beta, cu_seqlens,
              tensors=[("out", out, v.shape, q.dtype)],
              states=[("initial_state", initial_state), ("final_state", final_state)])
    shape = make_shape(q, v, cu_seqlens, scale)
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise ValueError("cu_seqlens must be int32")
    if out is None:
        out = torch.empty(v.shape, dtype=q.dtype, device=q.device)     # [B,T,H,V]
    if output_final_state and final_state is None:
        final_state = torch.empty(shape.N, shape.H, shape.V, shape.K, dtype=torch.float32,
                                  device=q.device)
    need = lib.sf_gdn_fwd_workspace(ctypes.byref(shape))
    if ws is None:
        ws = workspace(need, q.device)
    _check(lib.sf_gdn_chunk_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(_f32(gate)),
                                _ptr(_f32(beta)), _ptr(_f32(initial_state)), _ptr(cu_seqlens),
                                int(bool(output_final_state)), _ptr(out),
                                _ptr(final_state) if output_final_state else None,
                                _ptr(ws), ws.numel(), _stream(stream)))
    return out, (final_state if output_final_state else None)


def sf_gdn_paged_chunk_fwd(q, k, v, gate, beta, state_cache, state_indices, cu_seqlens=None,
                           has_initial_state=None, scale=None, out=None, ws=None, stream=None):
    """paged_chunk_gdn: the forward advancing state_cache [num_slots,H,V,K] in place at the
    slots state_indices (int32 [N]; <= 0: padding, zero output); has_initial_state (bool
    [N]) False starts from zero.  Returns out [B,T,H,V]."""
    lib = load()
    _validate(q, v, k, gate, beta, cu_seqlens,
              tensors=[("out", out, v.shape, q.dtype)])
    if state_cache.dim() != 4 or tuple(state_cache.shape[1:]) != (v.shape[2], v.shape[3],
                                                                   q.shape[3]):
        raise ValueError("state_cache must be [num_slots,H,V,K]")
    shape = make_shape(q, v, cu_seqlens, scale)
    if state_indices.dtype != torch.int32 or state_indices.numel() != shape.N:
        raise ValueError("state_indices must be int32 [N]")
    if has_initial_state is not None and (has_initial_state.dtype != torch.bool or
                                          has_initial_state.numel() != shape.N):
        raise ValueError("has_initial_state must be bool [N]")
    if out is None:
        out = torch.empty(v.shape, dtype=q.dtype, device=q.device)
    need = lib.sf_gdn_fwd_workspace(ctypes.byref(shape))
    if ws is None:
        ws = workspace(need, q.device)
    _check(lib.sf_gdn_paged_chunk_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v),
                                      _ptr(_f32(gate)), _ptr(_f32(beta)), _ptr(_f32(state_cache)),
                                      state_cache.shape[0], _ptr(state_indices),
                                      _ptr(has_initial_state), _ptr(cu_seqlens), _ptr(out),
                                      _ptr(ws), ws.numel(), _stream(stream)))
    return out


def sf_gdn_segment_summary(k, v, gate, beta, bounds, P=None, S_ext=None, ws=None, stream=None):
    """Affine map of each token range: returns (P [R,H,K,K], S_ext [R,H,V,K])."""
    lib = load()
    _validate(k, v, None, gate, beta)
    if bounds.dim() != 2 or bounds.shape[1] != 2:
        raise ValueError("bounds must be int32 [R,2]")
    shape = make_shape(k, v)
    R = bounds.shape[0]
    if bounds.dtype != torch.int32:
        raise ValueError("bounds must be int32 [R,2]")
    if P is None:
        P = torch.empty(R, shape.H, shape.K, shape.K, dtype=torch.float32, device=k.device)
    if S_ext is None:
        S_ext = torch.empty(R, shape.H, shape.V, shape.K, dtype=torch.float32, device=k.device)
    need = lib.sf_gdn_summary_workspace(ctypes.byref(shape), R)
    if ws is None:
        ws = workspace(need, k.device)
    _check(lib.sf_gdn_segment_summary(ctypes.byref(shape), _ptr(k), _ptr(v), _ptr(_f32(gate)),
                                      _ptr(_f32(beta)), _ptr(bounds), R, _ptr(P), _ptr(S_ext),
                                      _ptr(ws), ws.numel(), _stream(stream)))
    return P, S_ext


def sf_state_scan(P, S_ext, S0=None, entry_states=None, final_state=None, stream=None,
                  want_final=True):
    """Exclusive scan of segment maps: returns (entry_states [R,H,V,K], final [H,V,K])."""
    lib = load()
    R, H, K, _ = P.shape
    V = S_ext.shape[2]
    if entry_states is None:
        entry_states = torch.empty(R, H, V, K, dtype=torch.float32, device=P.device)
    if want_final and final_state is None:
        final_state = torch.empty(H, V, K, dtype=torch.float32, device=P.device)
    _check(lib.sf_state_scan(R, H, K, V, _ptr(_f32(P)), _ptr(_f32(S_ext)), _ptr(_f32(S0)),
                             _ptr(entry_states), _ptr(final_state), _stream(stream)))
    return entry_states, final_state


def sf_gdn_segment_reverse_summary(q, k, gate, beta, d_out, seg_offsets, scale=None, C=None,
                                   ws=None, stream=None):
    """Cotangent map of consecutive segments (offsets [R+1], cu_seqlens convention) of one
    token stream (B = 1): returns C [R,H,V,K], the cotangent each segment's own output
    gradients leave at its start (dS_entry = dS_exit @ P^T + C)."""
    lib = load()
    _validate(q, d_out, k, gate, beta, seg_offsets)
    shape = make_shape(q, d_out, seg_offsets, scale)
    if seg_offsets.dtype != torch.int32:
        raise ValueError("seg_offsets must be int32 [R+1]")
    if C is None:
        C = torch.empty(shape.N, shape.H, shape.V, shape.K, dtype=torch.float32, device=q.device)
    need = lib.sf_gdn_reverse_summary_workspace(ctypes.byref(shape))
    if ws is None:
        ws = workspace(need, q.device)
    _check(lib.sf_gdn_segment_reverse_summary(ctypes.byref(shape), _ptr(q), _ptr(k),
                                              _ptr(_f32(gate)), _ptr(_f32(beta)), _ptr(d_out),
                                              _ptr(seg_offsets), _ptr(C), _ptr(ws), ws.numel(),
                                              _stream(stream)))
    return C


def sf_state_scan_reverse(P, C, dS_final=None, exit_cotangents=None, d_initial=None,
                          stream=None, want_initial=True):
    """Reverse scan of cotangent maps: returns (exit cotangents [R,H,V,K], d_initial [H,V,K])."""
    lib = load()
    R, H, K, _ = P.shape
    V = C.shape[2]
    if exit_cotangents is None:
        exit_cotangents = torch.empty(R, H, V, K, dtype=torch.float32, device=P.device)
    if want_initial and d_initial is None:
        d_initial = torch.empty(H, V, K, dtype=torch.float32, device=P.device)
    _check(lib.sf_state_scan_reverse(R, H, K, V, _ptr(_f32(P)), _ptr(_f32(C)), _ptr(_f32(dS_final)),
                                     _ptr(exit_cotangents), _ptr(d_initial), _stream(stream)))
    return exit_cotangents, d_initial


def reverse_summary_workspace_bytes(shape: sf_gdn_shape) -> int:
    return int(load().sf_gdn_reverse_summary_workspace(ctypes.byref(shape)))


def _validate_bwd(q, k, v, gate, beta, initial_state, d_out, d_final_state, cu_seqlens, grads):
    g = grads or {}
    _validate(q, v, k, gate, beta, cu_seqlens,
              tensors=[("d_out", d_out, v.shape, v.dtype), ("dq", g.get("dq"), q.shape, q.dtype),
                       ("dk", g.get("dk"), k.shape, k.dtype), ("dv", g.get("dv"), v.shape, v.dtype),
                       ("dgate", g.get("dgate"), gate.shape, gate.dtype),
                       ("dbeta", g.get("dbeta"), beta.shape, beta.dtype)],
              states=[("initial_state", initial_state), ("d_final_state", d_final_state),
                      ("d_initial_state", g.get("d_initial_state"))])


def sf_gdn_chunk_bwd(q, k, v, gate, beta, initial_state, d_out, d_final_state=None,
                     cu_seqlens=None, scale=None, want_d_initial_state=True, grads=None, ws=None,
                     stream=None):
    """Backward of sf_gdn_chunk_fwd.  Returns dict dq, dk, dv, dgate, dbeta, d_initial_state."""
    lib = load()
    _validate_bwd(q, k, v, gate, beta, initial_state, d_out, d_final_state, cu_seqlens, grads)
    shape = make_shape(q, v, cu_seqlens, scale)
    dev = q.device
    if grads is None:
        grads = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
                     dgate=torch.empty_like(gate), dbeta=torch.empty_like(beta),
                     d_initial_state=(torch.empty(shape.N, shape.H, shape.V, shape.K,
                                                  dtype=torch.float32, device=dev)
                                      if want_d_initial_state else None))
    need = lib.sf_gdn_bwd_workspace(ctypes.byref(shape))
    if ws is None:
        ws = workspace(need, dev)
    _check(lib.sf_gdn_chunk_bwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(_f32(gate)),
                                _ptr(_f32(beta)), _ptr(_f32(initial_state)), _ptr(cu_seqlens),
                                _ptr(d_out), _ptr(_f32(d_final_state)), _ptr(grads["dq"]),
                                _ptr(grads["dk"]), _ptr(grads["dv"]), _ptr(grads["dgate"]),
                                _ptr(grads["dbeta"]), _ptr(grads["d_initial_state"]),
                                _ptr(ws), ws.numel(), _stream(stream)))
    return grads


def sf_gdn_chunk_bwd_noalloc(q, k, v, gate, beta, initial_state, d_out, d_final_state=None,
                             cu_seqlens=None, scale=None, want_d_initial_state=True, grads=None,
                             stream=None):
    """sf_gdn_chunk_bwd with the library's built-in scratch instead of a workspace
    (for callers that cannot allocate device memory at this point; see
    include/sf_gdn.h for the size limit and the sharing rules)."""
    lib = load()
    _validate_bwd(q, k, v, gate, beta, initial_state, d_out, d_final_state, cu_seqlens, grads)
    shape = make_shape(q, v, cu_seqlens, scale)
    if grads is None:
        grads = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
                     dgate=torch.empty_like(gate), dbeta=torch.empty_like(beta),
                     d_initial_state=(torch.empty(shape.N, shape.H, shape.V, shape.K,
                                                  dtype=torch.float32, device=q.device)
                                      if want_d_initial_state else None))
    _check(lib.sf_gdn_chunk_bwd_noalloc(
        ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(_f32(gate)), _ptr(_f32(beta)),
        _ptr(_f32(initial_state)), _ptr(cu_seqlens), _ptr(d_out), _ptr(_f32(d_final_state)),
        _ptr(grads["dq"]), _ptr(grads["dk"]), _ptr(grads["dv"]), _ptr(grads["dgate"]),
        _ptr(grads["dbeta"]), _ptr(grads["d_initial_state"]), _stream(stream)))
    return grads


def sf_validate_cu_seqlens(cu_seqlens, T, stream=None):
    lib = load()
    _check(lib.sf_validate_cu_seqlens(_ptr(cu_seqlens), cu_seqlens.numel() - 1, int(T),
                                      _stream(stream)))


def sf_gdn_chunk_bwd_noalloc_status(stream=None):
    """Reads and clears the status word of sf_gdn_chunk_bwd_noalloc's built-in scratch on
    the current device; raises SfError (SF_ERR_TIMEOUT) if a kernel reported a timeout."""
    _check(load().sf_gdn_chunk_bwd_noalloc_status(_stream(stream)))


def sf_workspace_status(ws, stream=None):
    _check(load().sf_workspace_status(_ptr(ws), _stream(stream)))


def fwd_workspace_bytes(shape: sf_gdn_shape) -> int:
    return int(load().sf_gdn_fwd_workspace(ctypes.byref(shape)))


def summary_workspace_bytes(shape: sf_gdn_shape, R: int) -> int:
    return int(load().sf_gdn_summary_workspace(ctypes.byref(shape), int(R)))


def bwd_workspace_bytes(shape: sf_gdn_shape) -> int:
    return int(load().sf_gdn_bwd_workspace(ctypes.byref(shape)))
