"""Throughput of the chunked gated delta rule on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one forward pass (sf_gdn_chunk_fwd) of the headline workload:
B=4, T=4096, H=16, K=V=128, BF16 q/k/v, FP32 gate/beta/state, random initial
state, final state returned.  `value` is tokens/s (B*T tokens per step, all
heads) with inputs resident in HBM; the same line carries the
forward+backward workload (B=2, T=8192, H=16) and the long-context
state-passing workload (T=262144 in 16 segments: summary -> scan -> segment
forward) measured the same way, the end-to-end number through the public
API with host buffers, the roofline of the dominant kernel, and the FP64
oracle timed on the host cores (`cpu_baseline`).

Under torchrun (N > 1) every rank runs its own copy of the workload on its own
GPU (independent problems: weak scaling, no data-path collective); a barrier
brackets the timed region and rank 0 reports the max time over ranks.

`--impl reference` times the FP64 CPU oracle (the reference arm of this
build) on a bounded sample of the same workload; under torchrun only rank 0
runs it.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "chunk_gdn fwd & fwd+bwd tokens/s at K=V=128 BF16; % of roofline"
UNIT = "tokens/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

# Algorithmic traffic / work per token-head at d = 128, chunk 64: the bytes the method must
# move (inputs read once, outputs written once) and its FLOPs with the causal C x C products
# counted as triangles:
FWD_BYTES_PER_TH = 1032          # q,k,v 768 + gate,beta 8 + out 256 (BF16)
FWD_FLOP_PER_TH = 139264         # 6 d^2 + 5 C d
BWD_BYTES_PER_TH = 1808          # read q,k,v,g,beta,dO + write dq,dk,dv,dg,dbeta
SUM_BYTES_PER_TH = 520           # k, v, gate, beta
STATE_BYTES = 128 * 128 * 4      # one [V,K] FP32 state


def fwd_traffic():
    """DRAM bytes per launch of the forward kernel from the committed ncu summary,
    or None when the kernel sources changed since that capture."""
    import hashlib
    csrc = os.path.join(ROOT, "chunked_linear_recurrence_gb300", "csrc")
    h = hashlib.sha256()
    for f in ("fwd_split.cu", "tmap.cu", "tc_ptx.cuh", "solve_tc.cuh", "common.cuh",
              "chunk_record.cuh"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    try:
        rec = {}
        with open(os.path.join(ROOT, "profiles", "gdn_fwd_split_traffic.txt")) as fh:
            for line in fh:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    rec[k.strip()] = v.strip()
        if rec.get("source_sha256") == h.hexdigest():
            return float(rec["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        pass
    return None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


class ClockSampler:
    """nvidia-smi sampled every 100 ms in a background process; samples are
    timestamped so the ones inside the timed window can be selected."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 7:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        window = "timed"
        if not inside:
            inside = [p for (_, p) in self.samples]
            window = "bench"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        reasons = set()
        for p in inside:
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                  "sw_power_cap"), p[3:7]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(inside[0][1]), "reasons": sorted(reasons),
                "samples": len(inside), "window": window}


class NvmlSampler:
    """SM clock and clock-event reasons read through NVML (the driver's libnvidia-ml,
    via ctypes) every few milliseconds in a background thread, so that a timed region of
    a few milliseconds still gets samples.  Read-only: it changes no setting."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid: str | None, index: int, period_s: float = 0.0005):
        import ctypes
        self.samples = []
        self.ok = False
        self.period = period_s
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            rc = 1
            if uuid:
                rc = nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h))
            if rc != 0:
                rc = nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h))
            if rc != 0:
                return
            mx = ctypes.c_uint()
            nv.nvmlDeviceGetMaxClockInfo(h, ctypes.c_int(1), ctypes.byref(mx))   # NVML_CLOCK_SM
            self.max_mhz = float(mx.value)
            self.get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self.nv, self.h, self.ct = nv, h, ctypes
            self.ok = True
        except Exception:
            self.ok = False
        self.run = False

    def start(self):
        if not self.ok:
            return
        self.run = True
        self.th = threading.Thread(target=self._loop, daemon=True)
        self.th.start()

    def _loop(self):
        ct = self.ct
        mhz, rs = ct.c_uint(), ct.c_ulonglong()
        while self.run:
            t = time.time()
            if self.nv.nvmlDeviceGetClockInfo(self.h, ct.c_int(1), ct.byref(mhz)) == 0 and \
                    self.get_reasons(self.h, ct.byref(rs)) == 0:
                self.samples.append((t, float(mhz.value), int(rs.value)))
            time.sleep(self.period)

    def stop(self):
        self.run = False
        if self.ok:
            self.th.join(timeout=2)

    def summary(self, t0, t1):
        inside = [(m, r) for (t, m, r) in self.samples if t0 <= t <= t1]
        if not inside:
            return None
        reasons = sorted({name for (_, r) in inside for bit, name in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(m for m, _ in inside), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(inside), "window": "timed",
                "source": "nvml"}


def device_uuid(dev):
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


def dist_init(backend=None):
    """One process per GPU under torchrun (NCCL); gloo when no GPU is visible (the host-side
    rank logic, which CPU tests drive with world size 2)."""
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = backend or ("nccl" if torch.cuda.is_available() else "gloo")
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def flush_l2(buf):
    buf.add_(1)


def time_loop(fn, steps, warmup, ws, flush=None, stream=None):
    """Returns (ms per step, max over ranks) with CUDA events on `stream`."""
    import torch
    stream = stream or torch.cuda.current_stream()
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    evs = []
    for _ in range(steps):
        if flush is not None:
            flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in evs) / steps
    return max_over_ranks(ms, ws)


def run_ours(args):
    import torch

    import chunked_linear_recurrence_gb300 as sf
    from chunked_linear_recurrence_gb300 import _native
    from chunked_linear_recurrence_gb300.workloads import make_inputs, segment_bounds, workloads

    ws_n, rank, local = dist_init()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sf.load()
    hbm, tflops, peak_src = peaks()
    W = workloads()
    w1 = W["fwd_bf16_b4_t4096_h16"]
    inp = make_inputs(w1, dev)
    out = torch.empty_like(inp["v"])
    fin = torch.empty(w1.N, w1.H, w1.V, w1.K, dtype=torch.float32, device=dev)
    wsb = _native.workspace(_native.fwd_workspace_bytes(_native.make_shape(inp["q"], inp["v"])),
                            dev)
    stream = torch.cuda.current_stream()

    def fwd():
        sf.sf_gdn_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                            inp["initial_state"], output_final_state=True, out=out,
                            final_state=fin, ws=wsb)

    sampler = ClockSampler(local) if rank == 0 else None
    nvml = NvmlSampler(device_uuid(dev), local) if rank == 0 else None
    # about a second of the same step before the timed region, so that it starts at the
    # clocks the GPU holds under this load (these steps are warm-up: not timed)
    for _ in range(args.warmup):
        fwd()
    torch.cuda.synchronize()
    t_load = time.time()
    n_load = 0
    while time.time() - t_load < args.load_s:
        for _ in range(50):
            fwd()
        n_load += 50
        torch.cuda.synchronize()
    if nvml:
        nvml.start()
    t0 = time.time()
    ms = time_loop(fwd, args.steps, 0, ws_n, stream=stream)
    t1 = time.time()
    if nvml:
        nvml.stop()
    _native.sf_workspace_status(wsb)     # raises if a kernel reported a timeout
    clocks = (nvml.summary(t0, t1) if nvml else None) or \
        (sampler.summary(t0, t1) if sampler else None)
    if clocks is not None and sampler:
        smi = sampler.summary(t_load, t1)          # the load phase plus the timed region
        clocks["nvidia_smi_load_window"] = {k: smi.get(k) for k in ("sm_mhz", "reasons", "samples")}
    if sampler:
        sampler.stop()
    tokens = w1.B * w1.T
    value = tokens * ws_n / (ms * 1e-3)
    th = w1.B * w1.T * w1.H
    fwd_bytes = th * FWD_BYTES_PER_TH + 2 * w1.N * w1.H * STATE_BYTES
    achieved = fwd_bytes / (ms * 1e-3) / 1e9
    roofline = {"kernel": "gdn_fwd_split_kernel (one launch per step)", "bound": "hbm",
                "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "peak_source": peak_src,
                "algorithmic_bytes": fwd_bytes,
                "traffic": fwd_traffic(),
                "flops": th * FWD_FLOP_PER_TH,
                "tensor_frac": round(th * FWD_FLOP_PER_TH / (ms * 1e-3) / (tflops * 1e12), 4)}

    # end to end through the public API with pinned host buffers
    host = {n: t.cpu().pin_memory() for n, t in inp.items() if isinstance(t, torch.Tensor)}
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    fin_h = torch.empty(fin.shape, dtype=fin.dtype).pin_memory()
    dev_in = {n: torch.empty_like(t, device=dev) for n, t in host.items()}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size() + fin_h.numel() * fin_h.element_size()

    def e2e_step():
        for n, t in host.items():
            dev_in[n].copy_(t, non_blocking=True)
        sf.sf_gdn_chunk_fwd(dev_in["q"], dev_in["k"], dev_in["v"], dev_in["gate"],
                            dev_in["beta"], dev_in["initial_state"], output_final_state=True,
                            out=out, final_state=fin, ws=wsb)
        out_h.copy_(out, non_blocking=True)
        fin_h.copy_(fin, non_blocking=True)

    e2e_steps = max(3, min(args.steps, 20))
    ms_e2e = time_loop(e2e_step, e2e_steps, 2, ws_n, stream=stream)
    e2e = {"value": tokens * ws_n / (ms_e2e * 1e-3), "unit": UNIT, "ms_per_step": ms_e2e,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    del dev_in, host

    extra = {}
    if not args.fwd_only:
        extra["fwd_bwd"] = bench_fwd_bwd(args, W, dev, ws_n, hbm, peak_src)
        extra["state_passing"] = bench_state_passing(args, W, dev, ws_n, hbm, peak_src)
        extra["varlen"] = bench_varlen(args, W, dev, ws_n, hbm, peak_src)
        extra["tiny_f32"] = bench_tiny(args, W, dev, ws_n)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = oracle_baseline(inp, w1)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_n,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic",
                "config": {"workload": w1.name, "B": w1.B, "T": w1.T, "H": w1.H, "K": w1.K,
                           "V": w1.V, "tokens_per_step": tokens, "l2": "inputs larger than L2",
                           "per_gpu": "each rank runs the full workload (independent problems)"},
                "gpu_launches": args.steps * 1, "clocks": clocks, "e2e": e2e,
                "roofline": roofline, "cpu_baseline": cpu, **extra}
        print(json.dumps(line), flush=True)
    barrier(ws_n)


def bench_fwd_bwd(args, W, dev, ws_n, hbm, peak_src):
    import torch

    import chunked_linear_recurrence_gb300 as sf
    from chunked_linear_recurrence_gb300 import _native
    from chunked_linear_recurrence_gb300.workloads import make_inputs

    w = W["fwdbwd_bf16_b2_t8192_h16"]
    inp = make_inputs(w, dev)
    out = torch.empty_like(inp["v"])
    fin = torch.empty(w.N, w.H, w.V, w.K, dtype=torch.float32, device=dev)
    shape = _native.make_shape(inp["q"], inp["v"])
    wsf = _native.workspace(_native.fwd_workspace_bytes(shape), dev)
    wsb = _native.workspace(_native.bwd_workspace_bytes(shape), dev)
    grads = dict(dq=torch.empty_like(inp["q"]), dk=torch.empty_like(inp["k"]),
                 dv=torch.empty_like(inp["v"]), dgate=torch.empty_like(inp["gate"]),
                 dbeta=torch.empty_like(inp["beta"]),
                 d_initial_state=torch.empty_like(fin))

    def fwd():
        sf.sf_gdn_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                            inp["initial_state"], output_final_state=True, out=out,
                            final_state=fin, ws=wsf)

    def bwd():
        sf.sf_gdn_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                            inp["initial_state"], inp["d_out"], inp["d_final_state"],
                            grads=grads, ws=wsb)

    steps = max(3, min(args.steps, 10))
    ms_f = time_loop(fwd, steps, args.warmup, ws_n)
    ms_b = time_loop(bwd, steps, args.warmup, ws_n)
    _native.sf_workspace_status(wsf)
    _native.sf_workspace_status(wsb)
    tokens = w.B * w.T
    th = tokens * w.H
    bb = th * BWD_BYTES_PER_TH + 4 * w.N * w.H * STATE_BYTES
    fb = th * FWD_BYTES_PER_TH + 2 * w.N * w.H * STATE_BYTES
    return {"workload": w.name, "tokens_per_step": tokens,
            "value": tokens * ws_n / ((ms_f + ms_b) * 1e-3), "unit": UNIT,
            "ms_fwd": ms_f, "ms_bwd": ms_b, "steps": steps,
            "roofline_fwd_bwd": {"bound": "hbm", "achieved": (fb + bb) / ((ms_f + ms_b) * 1e-3) / 1e9,
                                 "peak": hbm, "unit": "GB/s", "peak_source": peak_src,
                                 "frac": (fb + bb) / ((ms_f + ms_b) * 1e-3) / 1e9 / hbm},
            "roofline_bwd": {"bound": "hbm", "achieved": bb / (ms_b * 1e-3) / 1e9, "peak": hbm,
                             "unit": "GB/s", "frac": bb / (ms_b * 1e-3) / 1e9 / hbm}}


def bench_state_passing(args, W, dev, ws_n, hbm, peak_src):
    import torch

    import chunked_linear_recurrence_gb300 as sf
    from chunked_linear_recurrence_gb300 import _native
    from chunked_linear_recurrence_gb300.workloads import make_inputs, segment_bounds

    w = W["statepass_bf16_t262144_h16"]
    inp = make_inputs(w, dev)
    R = w.segments
    L = w.T // R
    bounds = segment_bounds(w.T, R).to(dev)
    cu = torch.arange(0, w.T + 1, L, dtype=torch.int32, device=dev)
    P = torch.empty(R, w.H, w.K, w.K, dtype=torch.float32, device=dev)
    E = torch.empty(R, w.H, w.V, w.K, dtype=torch.float32, device=dev)
    ent = torch.empty_like(E)
    fin = torch.empty(w.H, w.V, w.K, dtype=torch.float32, device=dev)
    out = torch.empty_like(inp["v"])
    seg_fin = torch.empty_like(E)
    wss = _native.workspace(max(_native.fwd_workspace_bytes(_native.make_shape(inp["q"], inp["v"], cu)),
                                _native.summary_workspace_bytes(_native.make_shape(inp["k"], inp["v"]), R)),
                            dev)

    def step():
        sf.sf_gdn_segment_summary(inp["k"], inp["v"], inp["gate"], inp["beta"], bounds, P=P,
                                  S_ext=E, ws=wss)
        sf.sf_state_scan(P, E, None, entry_states=ent, final_state=fin)
        sf.sf_gdn_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"], ent,
                            cu_seqlens=cu, output_final_state=True, out=out,
                            final_state=seg_fin, ws=wss)

    steps = max(3, min(args.steps, 5))
    ms = time_loop(step, steps, min(args.warmup, 3), ws_n)
    _native.sf_workspace_status(wss)
    th = w.T * w.H
    bytes_ = (th * (SUM_BYTES_PER_TH + FWD_BYTES_PER_TH) + 4 * R * w.H * STATE_BYTES)
    return {"workload": w.name, "segments": R, "tokens_per_step": w.T,
            "value": w.T * ws_n / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms, "steps": steps,
            "roofline": {"bound": "hbm", "achieved": bytes_ / (ms * 1e-3) / 1e9, "peak": hbm,
                         "unit": "GB/s", "peak_source": peak_src,
                         "frac": bytes_ / (ms * 1e-3) / 1e9 / hbm}}


def bench_varlen(args, W, dev, ws_n, hbm, peak_src):
    """Packed varlen forward: H = 32, 8 sequences (one empty, one ragged) in a
    T_phys = 65536 stream with an inactive tail; the fraction is on the active tokens."""
    import torch

    import chunked_linear_recurrence_gb300 as sf
    from chunked_linear_recurrence_gb300 import _native
    from chunked_linear_recurrence_gb300.workloads import make_inputs

    w = W["varlen_bf16_h32"]
    inp = make_inputs(w, dev)
    cu = inp["cu_seqlens"]
    out = torch.empty_like(inp["v"])
    fin = torch.empty(w.N, w.H, w.V, w.K, dtype=torch.float32, device=dev)
    wsv = _native.workspace(_native.fwd_workspace_bytes(_native.make_shape(inp["q"], inp["v"], cu)),
                            dev)

    def fwd():
        sf.sf_gdn_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"],
                            inp["initial_state"], cu_seqlens=cu, output_final_state=True,
                            out=out, final_state=fin, ws=wsv)

    steps = max(3, min(args.steps, 20))
    ms = time_loop(fwd, steps, args.warmup, ws_n)
    _native.sf_workspace_status(wsv)
    tokens = w.tokens
    bytes_ = tokens * w.H * FWD_BYTES_PER_TH + 2 * w.N * w.H * STATE_BYTES
    ach = bytes_ / (ms * 1e-3) / 1e9
    return {"workload": w.name, "lengths": w.lengths, "active_tokens": tokens, "T_phys": w.T,
            "value": tokens * ws_n / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms,
            "steps": steps,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                         "peak_source": peak_src, "frac": ach / hbm,
                         "algorithmic_bytes": bytes_}}


def bench_tiny(args, W, dev, ws_n):
    """The small FP32 workload (B=1, T=256, H=2, K=V=64): launch-bound, timed for the
    record (its roofline time is well under a microsecond)."""
    import torch

    import chunked_linear_recurrence_gb300 as sf
    from chunked_linear_recurrence_gb300.workloads import make_inputs

    w = W["tiny_f32"]
    inp = make_inputs(w, dev)
    out = torch.empty_like(inp["v"])
    fin = torch.empty(w.N, w.H, w.V, w.K, dtype=torch.float32, device=dev)

    def fwd():
        sf.sf_gdn_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["gate"], inp["beta"], None,
                            output_final_state=True, out=out, final_state=fin)

    steps = max(3, min(args.steps, 20))
    ms = time_loop(fwd, steps, args.warmup, ws_n)
    return {"workload": w.name, "tokens_per_step": w.B * w.T, "dtype": "f32",
            "value": w.B * w.T * ws_n / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms,
            "steps": steps, "note": "launch-bound (one small kernel launch per step)"}


def oracle_baseline(inp, w, target_s=10.0):
    """The FP64 oracle on a bounded sample of the workload: the whole workload
    (every batch row, head and token) repeated until about `target_s` seconds
    of CPU time have been spent."""
    import oracle

    def f64(t):
        return t.detach().cpu().double().numpy()

    q, k, v, g, b = (f64(inp[n]) for n in ("q", "k", "v", "gate", "beta"))
    s0 = f64(inp["initial_state"])
    reps, el = 0, 0.0
    while el < target_s:
        t0 = time.perf_counter()
        oracle.gdn_fwd(q, k, v, g, b, s0)
        el += time.perf_counter() - t0
        reps += 1
    tokens = reps * w.B * w.T
    return {"value": tokens / el, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"the whole workload (B={w.B}, T={w.T}, H={w.H}) x {reps} passes, "
                      f"{el:.1f} s, FP64 token-by-token, OpenMP over (sequence, head) chains"}


def run_reference(args):
    ws_n = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch

    import oracle
    from chunked_linear_recurrence_gb300.workloads import make_inputs, workloads
    w = workloads()["fwd_bf16_b4_t4096_h16"]
    inp = make_inputs(w, "cpu")

    def f64(t):
        return t.detach().double().numpy()

    # each step: the oracle forward on one batch row (all heads, all tokens) -- a
    # bounded sample, so the whole --steps/--warmup run ends within minutes
    t_tok = min(args.ref_tokens, w.T)
    arrs = [f64(inp[n][:1, :t_tok]) for n in ("q", "k", "v", "gate", "beta")]
    s0 = f64(inp["initial_state"][:1])
    for _ in range(args.warmup):
        oracle.gdn_fwd(*arrs, s0)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.gdn_fwd(*arrs, s0)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = t_tok / (ms * 1e-3)
    sample = (f"one batch row per step: all {w.H} heads, {t_tok} of {w.T} tokens "
              f"(FP64 token-by-token, OpenMP over heads)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_n,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "K": w.K, "V": w.V},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--fwd-only", action="store_true", help="skip the fwd+bwd and state-passing lines")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--load-s", type=float, default=1.0,
                    help="seconds of untimed steps right before the timed region (clock settling)")
    ap.add_argument("--ref-tokens", type=int, default=4096,
                    help="tokens of one batch row the reference arm runs per step")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
