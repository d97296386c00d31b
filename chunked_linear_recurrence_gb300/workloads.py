"""Seeded synthetic inputs for the chunked gated-delta-rule workloads.

This module draws random inputs and nothing else: it holds none of the
recurrence's arithmetic, so both the CUDA path and the FP64 oracle can be fed
from it.  All draws use a CPU ``torch.Generator`` seeded per workload, in the
fixed order q, k, v, gate, beta, initial state, d_out, d_final_state.

Distributions (the workloads the Attention Gym "Linear Attention" page and the
StateFlow paper train on use L2-normalised q/k, a non-positive natural-log gate
and a sigmoid write gate):

* q, k ~ N(0, 1), then L2-normalised per (token, head) over K in FP32
  (``x / max(||x||, 1e-12)``), then cast to the q/k/v dtype;
* v ~ N(0, 1), cast to the q/k/v dtype;
* gate = -softplus(N(0, 1)) (natural log, <= 0), FP32;
* beta = sigmoid(N(0, 1)), FP32;
* initial state ~ N(0, std) FP32 when requested (std = 0.1 for the BF16
  workloads), else absent (zero);
* d_out ~ N(0, 1) in the q/k/v dtype; d_final_state ~ N(0, 0.01) FP32.

"Low-decay" variants scale the gate by 1e-3 and beta by 0.1 so that the
initial state stays visible over a 4096-token sequence (with the default gate,
exp(sum gate) underflows within a few chunks and split-equals-sequential checks
would be nearly vacuous).  Over a 16384-token segment those factors still shrink
the segment map P to about 1e-9 (exp(sum gate) ~ e^-13, and the delta rule's
write contracts the state by about exp(-T beta / d)); the "carry" variant scales
the gate by 1e-5 and beta by 0.01 instead, which keeps |P| near 0.5 so that the
entry states reach through every segment.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch
import torch.nn.functional as F

CHUNK = 64


@dataclass
class Workload:
    name: str
    B: int
    T: int
    H: int
    K: int
    V: int
    dtype: torch.dtype
    seed: int
    s0_std: float | None = None          # None -> no initial state
    lengths: list[int] | None = None     # packed varlen when set (B == 1)
    lowdecay: bool = False
    carry: bool = False                  # gate x 1e-5, beta x 0.01 (maps carry the state)
    with_grads: bool = False
    segments: int | None = None          # state-passing workload: equal segments
    extra: dict = field(default_factory=dict)

    @property
    def N(self) -> int:
        return self.B if self.lengths is None else len(self.lengths)

    @property
    def tokens(self) -> int:
        """Active tokens (all sequences, one head)."""
        return self.B * self.T if self.lengths is None else int(sum(self.lengths))


def l2norm(x: torch.Tensor) -> torch.Tensor:
    """Per-row L2 normalisation over the last axis, in FP32."""
    n = x.float().pow(2).sum(-1, keepdim=True).sqrt().clamp_min(1e-12)
    return x.float() / n


def cu_seqlens_of(lengths) -> torch.Tensor:
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


def packed_lengths(seed: int, n: int = 8, max_len: int = 16384, total: int = 65536):
    """Varlen lengths: n draws uniform in [0, max_len]; index 3 forced empty;
    index 5 forced to a length that is not a multiple of 64; if the sum
    exceeds ``total`` every length is scaled by total/sum (floor) and both
    forcings are applied again."""
    gen = torch.Generator().manual_seed(seed)
    L = torch.randint(0, max_len + 1, (n,), generator=gen).tolist()

    def force(L):
        if n > 3:
            L[3] = 0
        if n > 5 and L[5] % CHUNK == 0:
            L[5] = L[5] - 1 if L[5] > 0 else 1

    force(L)
    s = sum(L)
    if s > total:
        L = [l * total // s for l in L]
        force(L)
    return L, gen


def make_inputs(w: Workload, device="cpu") -> dict:
    """Draw the workload's tensors.  Returns a dict of torch tensors on ``device``:
    q, k, v, gate, beta, initial_state (or None), cu_seqlens (or None), and for
    gradient workloads d_out, d_final_state."""
    if w.extra.get("lengths_from_seed"):
        _, gen = packed_lengths(w.seed)      # tensors continue the lengths' stream
    else:
        gen = torch.Generator().manual_seed(w.seed)
    B, T, H, K, V = w.B, w.T, w.H, w.K, w.V
    q = l2norm(torch.randn(B, T, H, K, generator=gen)).to(w.dtype)
    k = l2norm(torch.randn(B, T, H, K, generator=gen)).to(w.dtype)
    v = torch.randn(B, T, H, V, generator=gen).to(w.dtype)
    gate = -F.softplus(torch.randn(B, T, H, generator=gen))
    beta = torch.sigmoid(torch.randn(B, T, H, generator=gen))
    if w.lowdecay:
        gate = gate * 1e-3
        beta = beta * 0.1
    if w.carry:
        gate = gate * 1e-5
        beta = beta * 0.01
    s0 = None
    if w.s0_std is not None:
        s0 = torch.randn(w.N, H, V, K, generator=gen) * w.s0_std
    out = dict(q=q, k=k, v=v, gate=gate.float(), beta=beta.float(), initial_state=s0,
               cu_seqlens=None if w.lengths is None else cu_seqlens_of(w.lengths))
    if w.with_grads:
        out["d_out"] = torch.randn(B, T, H, V, generator=gen).to(w.dtype)
        out["d_final_state"] = torch.randn(w.N, H, V, K, generator=gen) * 0.01
    return {n: (t.to(device) if isinstance(t, torch.Tensor) else t) for n, t in out.items()}


def segment_bounds(T: int, segments: int, batch_row: int = 0) -> torch.Tensor:
    """[R,2] int32 flattened token ranges of equal segments of one batch row."""
    L = T // segments
    rows = [(batch_row * T + i * L, batch_row * T + (i + 1) * L) for i in range(segments)]
    return torch.tensor(rows, dtype=torch.int32)


def workloads() -> dict[str, Workload]:
    """The named workloads.  Sizes follow the chunked-GDN configurations this
    library is measured on; ``*_lowdecay`` variants are parity-only."""
    bf16 = torch.bfloat16
    L2, _ = packed_lengths(2)
    ws = [
        Workload("tiny_f32", 1, 256, 2, 64, 64, torch.float32, seed=0),
        Workload("fwd_bf16_b4_t4096_h16", 4, 4096, 16, 128, 128, bf16, seed=1, s0_std=0.1),
        Workload("varlen_bf16_h32", 1, 65536, 32, 128, 128, bf16, seed=2, s0_std=0.1,
                 lengths=L2, extra={"lengths_from_seed": True}),
        Workload("statepass_bf16_t262144_h16", 1, 262144, 16, 128, 128, bf16, seed=3,
                 segments=16),
        Workload("fwdbwd_bf16_b2_t8192_h16", 2, 8192, 16, 128, 128, bf16, seed=4,
                 s0_std=0.1, with_grads=True),
    ]
    d = {w.name: w for w in ws}
    d["fwd_bf16_b4_t4096_h16_lowdecay"] = Workload(
        "fwd_bf16_b4_t4096_h16_lowdecay", 4, 4096, 16, 128, 128, bf16, seed=1, s0_std=0.1,
        lowdecay=True)
    d["statepass_bf16_t262144_h16_lowdecay"] = Workload(
        "statepass_bf16_t262144_h16_lowdecay", 1, 262144, 16, 128, 128, bf16, seed=3,
        segments=16, s0_std=0.1, lowdecay=True)
    d["statepass_bf16_t262144_h16_carry"] = Workload(
        "statepass_bf16_t262144_h16_carry", 1, 262144, 16, 128, 128, bf16, seed=3,
        segments=16, s0_std=0.1, carry=True)
    return d
