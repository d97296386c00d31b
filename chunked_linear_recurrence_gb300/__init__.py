"""GB300-native chunk-parallel gated delta rule with boundary-state passing.

The computation lives in ``libsf_gdn.so`` (hand-written sm_103a CUDA behind the
C ABI in ``include/sf_gdn.h``); this package is its thin ctypes binding, with
the same entry-point names:

* ``sf_gdn_chunk_fwd``        -- chunk_gdn forward (output + final state)
* ``sf_gdn_paged_chunk_fwd``  -- the forward advancing a paged state cache in place
* ``sf_gdn_segment_summary``  -- affine map S_out = S_in @ P + S_ext of token ranges
* ``sf_state_scan``           -- exclusive scan of segment maps -> entry states
* ``sf_gdn_chunk_bwd``        -- gradients w.r.t. q, k, v, gate, beta, initial state
* ``sf_gdn_segment_reverse_summary`` -- cotangent map dS_entry = dS_exit @ P^T + C of segments
* ``sf_state_scan_reverse``   -- reverse scan of cotangent maps -> segment exit cotangents

Build the library with ``python -m chunked_linear_recurrence_gb300.build``.
"""
from ._native import (SfError, load, sf_gdn_chunk_bwd, sf_gdn_chunk_fwd,  # noqa: F401
                      sf_gdn_paged_chunk_fwd, sf_gdn_segment_reverse_summary, sf_gdn_segment_summary, sf_state_scan,
                      sf_state_scan_reverse, sf_validate_cu_seqlens, sf_workspace_status)

__all__ = ["SfError", "load", "sf_gdn_chunk_fwd", "sf_gdn_paged_chunk_fwd",
           "sf_gdn_segment_summary", "sf_state_scan",
           "sf_gdn_chunk_bwd", "sf_gdn_segment_reverse_summary", "sf_state_scan_reverse",
           "sf_validate_cu_seqlens", "sf_workspace_status"]
