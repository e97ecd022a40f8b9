#!/usr/bin/env python
"""KLA forward (prefill) and decode benchmark on GB300.

Headline: forward tokens/s on the 1B-scale layer (B=4, T=4096, H=16,
dk=dv=128, C=64; bf16 q/k/v/o, fp32 state and gates), one kla_chunk_fwd call
per step over synthetic inputs resident in HBM.  Also reported on the same
line: the decode step (256 sequences x 16 heads, dk=dv=128, fp32 state, 1000
consecutive steps) as steps/s and HBM GB/s, roofline fractions for both, an
end-to-end number through host buffers, and the fp64 CPU oracle timed on the
host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own replica (the work is
independent per sequence and head; no collective on the data path) and rank 0
prints the line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from linear_attention_delta_gb300 import inputs as gen  # noqa: E402
from linear_attention_delta_gb300 import kla  # noqa: E402

METRIC = ("KLA fwd tokens/s (H16,d128,T4096); decode steps/s + HBM GB/s; "
          "% roofline")
L2_FLUSH_BYTES = 512 << 20          # > 2 x the 129 MB L2


# ----------------------------------------------------------------- helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return (float(p["hbm_gbs"]), float(p["bf16_tflops"]),
                float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "measured")
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, 1700.0, "fallback"


def prefill_bytes(w) -> int:
    """Algorithmic HBM bytes of one forward pass: q, k, v read and o written
    once (bf16), log_alpha and eta read once (fp32), h0 read and hT written
    once (fp32 dk x dv per sequence-head)."""
    th = w.B * w.T * w.H
    esz = 2 if w.dtype == "bf16" else 4
    per_th = esz * (2 * w.dk + 2 * w.dv) + 8
    state = 4 * w.dk * w.dv * w.B * w.H
    return th * per_th + 2 * state


def prefill_flops(w) -> int:
    """Algorithmic FLOPs of the chunkwise form per token-head: K K^T and
    Q K^T (2 C dk each), the forward substitution on [B V | B Gamma K]
    ((C-1)(dk+dv)), P U~ (2 C dv) and W S, Q S, K^T U~ (6 dk dv)."""
    C, dk, dv = w.C, w.dk, w.dv
    per = 4 * C * dk + (C - 1) * (dk + dv) + 2 * C * dv + 6 * dk * dv
    return w.B * w.T * w.H * per


def backward_flops(w) -> int:
    """Algorithmic FLOPs of one backward pass, counted as three forward
    passes: the forward recompute that gives the chunk-start states, plus the
    reverse mode, in which every forward contraction C = A B yields two
    (dA = dC B^T, dB = A^T dC)."""
    return 3 * prefill_flops(w)


def fp32_alu_peak_tflops(sm_max_mhz=None) -> tuple:
    """Peak fp32 FMA rate of the CUDA cores: SMs x 128 FP32 lanes x 2 FLOPs
    x the maximum SM clock (NVML's, else 2070 MHz)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    mhz = float(sm_max_mhz) if sm_max_mhz else 2070.0
    return sms * 128 * 2 * mhz * 1e6 / 1e12, sms, mhz


def decode_bytes(w) -> int:
    heads = w.B * w.H
    esz = 2 if w.dtype == "bf16" else 4
    return heads * (2 * 4 * w.dk * w.dv + esz * (2 * w.dk + 2 * w.dv) + 8)


class ClockSampler:
    """SM clock and throttle reasons sampled during the timed region.

    Reads NVML directly through ctypes (every ~1 ms, so that even a timed
    region of a few milliseconds is covered); falls back to `nvidia-smi -lms
    200` when NVML cannot be loaded.  Only reads; changes no GPU setting."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int):
        self.index = index
        self.samples = []           # (sm_mhz, max_mhz, reason_bits)
        self.stop = threading.Event()
        self.nvml = None
        self.proc = None

    def _nvml_handle(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        bus = None
        try:
            pr = torch.cuda.get_device_properties(self.index)
            bus = "%08x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id,
                                        pr.pci_device_id)
        except Exception:
            bus = None
        if bus is None or lib.nvmlDeviceGetHandleByPciBusId_v2(
                bus.encode(), ctypes.byref(h)) != 0:
            if lib.nvmlDeviceGetHandleByIndex_v2(self.index,
                                                 ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
        fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return lib, h, fn

    def _run_nvml(self):
        import ctypes
        lib, h, reasons_fn = self.nvml
        cur, mx = ctypes.c_uint(), ctypes.c_uint()
        bits = ctypes.c_ulonglong()
        while not self.stop.is_set():
            if (lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(cur)) == 0 and
                    lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0
                    and reasons_fn(h, ctypes.byref(bits)) == 0):
                self.samples.append((cur.value, mx.value, bits.value))
            time.sleep(0.001)

    def _run_smi(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 6:
                continue
            try:
                b = 0
                for bit, p in zip((0x8, 0x40, 0x20, 0x4), parts[2:]):
                    if p.lower().startswith("active"):
                        b |= bit
                self.samples.append((float(parts[0]), float(parts[1]), b))
            except ValueError:
                continue

    def __enter__(self):
        try:
            self.nvml = self._nvml_handle()
            self.thread = threading.Thread(target=self._run_nvml, daemon=True)
        except Exception:
            self.nvml = None
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index),
                     "--query-gpu=clocks.sm,clocks.max.sm,"
                     "clocks_event_reasons.hw_slowdown,"
                     "clocks_event_reasons.hw_thermal_slowdown,"
                     "clocks_event_reasons.sw_thermal_slowdown,"
                     "clocks_event_reasons.sw_power_cap",
                     "--format=csv,noheader,nounits", "-lms", "200"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                    text=True)
                self.thread = threading.Thread(target=self._run_smi,
                                               daemon=True)
            except OSError:
                self.thread = None
        if self.thread is not None:
            self.thread.start()
        return self

    def __exit__(self, *exc):
        self.stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0}
        sm = [s[0] for s in self.samples]
        reasons = set()
        for _, _, b in self.samples:
            for bit, name in self.REASONS.items():
                if b & bit:
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)),
                "sm_max_mhz": float(max(s[1] for s in self.samples)),
                "reasons": sorted(reasons), "samples": len(self.samples),
                "source": "nvml" if self.nvml else "nvidia-smi"}


def profiled_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu capture of `kernel`, or
    None when the kernel's sources changed since that capture."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            entry = json.load(f)[kernel]
        h = hashlib.sha256()
        for name in entry["sources"]:
            with open(os.path.join(ROOT, "linear_attention_delta_gb300",
                                   "csrc", name), "rb") as f:
                h.update(f.read())
        if h.hexdigest()[:16] != entry["source_sha16"]:
            return None
        return entry["dram_read_bytes"] + entry["dram_write_bytes"]
    except (OSError, KeyError, ValueError):
        return None


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ our arm

def bench_prefill(w, steps, warmup, world, gpu_index, rule="kaczmarz",
                  inp=None):
    inp = gen.prefill_inputs(w) if inp is None else inp
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
           for k, v in inp.items()}
    o = torch.empty_like(dev["v"])
    hT = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32,
                     device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        kla.chunk_fwd(dev["q"], dev["k"], dev["v"], dev["log_alpha"],
                      dev["eta"], dev["eps"], dev["h0"], C=w.C, o=o, hT=hT,
                      rule=rule)

    for _ in range(warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if kla.device_status() != 0:
        raise RuntimeError("device-side timeout during warm-up")
    ev = [(torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(gpu_index) as clk:
        t0 = time.perf_counter()
        for i in range(steps):
            flush.zero_()                      # L2 flushed between steps
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    barrier(world)
    if kla.device_status() != 0:
        raise RuntimeError("device-side timeout in the timed region")
    per = [a.elapsed_time(b) for a, b in ev]
    ms = max_over_ranks(float(np.mean(per)), world)
    return dict(ms=ms, per_step_ms=per, wall_s=wall, clocks=clk.summary(),
                launches=steps, inputs=inp)


def bench_prefill_e2e(w, inp, steps, warmup):
    """Same forward pass through the host-buffer entry point
    (kla_chunk_fwd_host): every input comes from page-locked host memory and
    o and hT go back to it, all inside the timed region; the library
    overlaps the copies with the kernels segment by segment."""
    names = ("q", "k", "v", "log_alpha", "eta", "h0")
    host = {n: inp[n].pin_memory() for n in names}
    B, T, H, dk, dv = w.B, w.T, w.H, w.dk, w.dv
    o_h = torch.empty((B, T, H, dv), dtype=host["v"].dtype).pin_memory()
    hT_h = torch.empty((B, H, dk, dv), dtype=torch.float32).pin_memory()
    ws = torch.empty(kla.chunk_fwd_host_workspace_size(
        B, T, H, dk, dv, w.C, host["q"].dtype), dtype=torch.uint8,
        device="cuda")
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = o_h.numel() * o_h.element_size() + hT_h.numel() * hT_h.element_size()
    stream = torch.cuda.current_stream()

    def step():
        kla.chunk_fwd_host(host["q"], host["k"], host["v"],
                           host["log_alpha"], host["eta"], inp["eps"],
                           host["h0"], C=w.C, o=o_h, hT=hT_h, workspace=ws)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = (torch.cuda.Event(enable_timing=True),
              torch.cuda.Event(enable_timing=True))
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return ms, h2d, d2h


def bench_decode(w, steps, warmup, distinct=50, gpu_index=0):
    """`steps` consecutive decode steps over the full state; token inputs
    cycle through `distinct` independently drawn steps (the state itself
    evolves through every step).  Returns ms per step and the SM clocks
    sampled over the timed steps."""
    d = gen.decode_inputs(w, steps=distinct)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
           for k, v in d.items()}
    S = dev["S0"].clone()
    o = torch.empty((w.B, w.H, w.dv), dtype=dev["q"].dtype, device="cuda")
    toks = [[dev[n][i] for n in ("q", "k", "v", "log_alpha", "eta")]
            for i in range(distinct)]
    stream = torch.cuda.current_stream()

    def step(i):
        q, k, v, la, eta = toks[i % distinct]
        kla.decode_step(q, k, v, la, eta, S, eps=d["eps"], o=o)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = (torch.cuda.Event(enable_timing=True),
              torch.cuda.Event(enable_timing=True))
    with ClockSampler(gpu_index) as clk:
        e0.record(stream)
        for i in range(steps):
            step(i)
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    if kla.device_status() != 0:
        raise RuntimeError("device-side timeout in decode")
    return ms / steps, clk.summary()


def bench_backward(w, inp, steps, warmup, world):
    """kla_chunk_bwd on the forward's inputs with seeded upstream
    gradients; the workspace is allocated once, outside the timed region;
    L2 is flushed between timed steps."""
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
           for k, v in inp.items()}
    rng = np.random.default_rng(gen.SEEDS[w.name] + 200)
    do = torch.from_numpy(rng.standard_normal(tuple(dev["v"].shape)).astype(
        np.float32)).to(dev["v"].dtype).cuda()
    dhT = torch.from_numpy(rng.standard_normal(
        (w.B, w.H, w.dk, w.dv)).astype(np.float32)).cuda()
    nbytes = kla.chunk_bwd_workspace_size(w.B, w.T, w.H, w.dk, w.dv, w.C)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        kla.chunk_bwd(dev["q"], dev["k"], dev["v"], dev["log_alpha"],
                      dev["eta"], do, dhT, eps=dev["eps"], h0=dev["h0"],
                      C=w.C, workspace=ws)

    for _ in range(warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(steps):
        flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in ev])),
                        world)
    return ms, nbytes


def bench_precond(w, inp, steps, warmup, world):
    """The diagonal-preconditioned variant on the forward's inputs: the
    write-key scan plus the two-key forward (the two-kernel tensor-core
    path's write-key instantiations for bf16 d128 C64, else the CUDA-core
    kernel), beside the plain forward on the same path."""
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
         for k, v in inp.items()}
    o = torch.empty_like(d["v"])
    hT = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32,
                     device="cuda")
    kw = torch.empty_like(d["k"])
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def plain():
        kla.chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["eta"],
                      d["eps"], d["h0"], C=w.C, o=o, hT=hT)

    def keys():
        kla.precond_keys(d["k"], k_write=kw, want_AT=False)

    def fwd_kw():
        kla.chunk_fwd_kw(d["q"], d["k"], kw, d["v"], d["log_alpha"],
                         d["eta"], d["eps"], d["h0"], C=w.C, o=o, hT=hT)

    def timed(fn):
        for _ in range(warmup):
            flush.zero_()
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(steps):
            flush.zero_()
            e0, e1 = (torch.cuda.Event(enable_timing=True),
                      torch.cuda.Event(enable_timing=True))
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return max_over_ranks(float(np.mean(ts)), world)

    t_plain, t_keys, t_fwd = timed(plain), timed(keys), timed(fwd_kw)
    if kla.device_status() != 0:
        raise RuntimeError("device-side timeout in the preconditioned bench")
    return t_plain, t_keys, t_fwd


def seq_segments(w) -> int:
    """The split kla_chunk_fwd_seq picks for segments = 0 (the same rule)."""
    sms = torch.cuda.get_device_properties(
        torch.cuda.current_device()).multi_processor_count
    P = 1
    while (2 * P <= 8 and 4 * w.B * w.H * 2 * P <= sms and
           w.T % (2 * P * w.C) == 0):
        P *= 2
    return P


def bench_seq(w, inp, steps, warmup, world, rule="kaczmarz"):
    """The sequence-split forward (kla_chunk_fwd_seq, segments chosen by the
    library), inputs resident on the device; CUDA events around each call."""
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
         for k, v in inp.items()}
    o = torch.empty_like(d["v"])
    hT = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32,
                     device="cuda")
    ws = torch.empty(max(1, kla.chunk_fwd_seq_workspace_size(
        w.B, w.T, w.H, w.dk, w.dv, w.C, d["q"].dtype, 0)), dtype=torch.uint8,
        device="cuda")

    def call():
        kla.chunk_fwd_seq(d["q"], d["k"], d["v"], d["log_alpha"], d["eta"],
                          d["eps"], d["h0"], C=w.C, segments=0, o=o, hT=hT,
                          workspace=ws, rule=rule)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    ts = []
    for _ in range(steps):
        e0, e1 = (torch.cuda.Event(enable_timing=True),
                  torch.cuda.Event(enable_timing=True))
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    if kla.device_status() != 0:
        raise RuntimeError("device-side timeout in the split prefill")
    return max_over_ranks(float(np.mean(ts)), world), seq_segments(w)


def bench_long_context(world, gpu_index, hbm):
    """The pages' own efficiency points at layer scale: the 131072-token
    prefill (KLA and the learned-step rule on the same kernels), and decode
    steps from the state of a 32768-token prefill."""
    w = gen.LONG_131K
    inp = gen.prefill_inputs(w)
    pf = bench_prefill(w, 3, 3, world, gpu_index, inp=inp)
    gd = bench_prefill(w, 3, 3, world, gpu_index, rule="given", inp=inp)
    split_ms, split_p = bench_seq(w, inp, 3, 3, world)
    split_gd_ms, _ = bench_seq(w, inp, 3, 3, world, rule="given")
    del inp
    gbs = prefill_bytes(w) / (pf["ms"] * 1e-3) / 1e9
    sgbs = prefill_bytes(w) / (split_ms * 1e-3) / 1e9
    prefill = {"workload": w.name, "ms": round(pf["ms"], 4),
               "tokens_per_s": round(world * w.B * w.T / (pf["ms"] * 1e-3), 1),
               "hbm_gbs": round(gbs, 1), "roofline_frac": round(gbs / hbm, 4),
               "gdn_ms": round(gd["ms"], 4),
               "kla_over_gdn_time": round(pf["ms"] / gd["ms"], 4),
               "split": {"entry": "kla_chunk_fwd_seq", "segments": split_p,
                         "ms": round(split_ms, 4),
                         "tokens_per_s": round(world * w.B * w.T /
                                               (split_ms * 1e-3), 1),
                         "hbm_gbs": round(sgbs, 1),
                         "roofline_frac": round(sgbs / hbm, 4),
                         "gdn_ms": round(split_gd_ms, 4),
                         "kla_over_gdn_time": round(split_ms / split_gd_ms,
                                                    4),
                         "speedup_vs_single_launch": round(pf["ms"] /
                                                           split_ms, 3)},
               "timed_steps": 3}

    hw = gen.HANDOFF_32K
    hin = gen.prefill_inputs(hw)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
           for k, v in hin.items()}
    del hin
    S = torch.empty((hw.B, hw.H, hw.dk, hw.dv), dtype=torch.float32,
                    device="cuda")
    o = torch.empty_like(dev["v"])
    e0, e1 = (torch.cuda.Event(enable_timing=True),
              torch.cuda.Event(enable_timing=True))
    kla.chunk_fwd(dev["q"], dev["k"], dev["v"], dev["log_alpha"], dev["eta"],
                  dev["eps"], None, C=hw.C, o=o, hT=S)   # warm-up
    e0.record()
    kla.chunk_fwd(dev["q"], dev["k"], dev["v"], dev["log_alpha"], dev["eta"],
                  dev["eps"], None, C=hw.C, o=o, hT=S)
    e1.record()
    torch.cuda.synchronize()
    prefill_ms = e0.elapsed_time(e1)
    del dev, o
    steps, distinct = 200, 20
    d = gen.decode_inputs(hw, steps=distinct, seed=gen.SEEDS[hw.name] + 100)
    toks = [[d[n][i].cuda() for n in ("q", "k", "v", "log_alpha", "eta")]
            for i in range(distinct)]
    od = torch.empty((hw.B, hw.H, hw.dv), dtype=toks[0][0].dtype,
                     device="cuda")
    for i in range(10):                       # warm-up on a copy
        kla.decode_step(*toks[i % distinct], S.clone(), eps=d["eps"], o=od)
    torch.cuda.synchronize()
    e0.record()
    for i in range(steps):
        kla.decode_step(*toks[i % distinct], S, eps=d["eps"], o=od)
    e1.record()
    torch.cuda.synchronize()
    dms = e0.elapsed_time(e1) / steps
    # the same steps from a CUDA graph: `distinct` decode steps (fixed token
    # buffers) captured once and replayed, one graph launch per `distinct`
    # steps instead of one kernel launch per step
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):               # warm-up off the capture
        kla.decode_step(*toks[0], S.clone(), eps=d["eps"], o=od)
    torch.cuda.current_stream().wait_stream(side)
    with torch.cuda.graph(graph):
        for i in range(distinct):
            kla.decode_step(*toks[i], S, eps=d["eps"], o=od)
    graph.replay()                              # warm-up
    torch.cuda.synchronize()
    e0.record()
    for _ in range(steps // distinct):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    gms = e0.elapsed_time(e1) / (steps // distinct * distinct)
    if kla.device_status() != 0:
        raise RuntimeError("device-side timeout in the long-context points")
    handoff = {"workload": hw.name, "prefill_ms": round(prefill_ms, 4),
               "decode_sequences": hw.B, "decode_steps": steps,
               "decode_steps_per_s": round(1e3 / dms, 1),
               "decode_ms_per_step": round(dms, 5),
               "graph_decode_ms_per_step": round(gms, 5),
               "graph_steps_per_replay": distinct,
               "note": "state carried from the 32768-token prefill; "
                       "4 MiB of state (L2-resident), so launch-bound: "
                       "one kernel launch per step, and the same steps "
                       "replayed from a CUDA graph"}
    return {"prefill_131k": prefill, "decode_after_32k": handoff}


def cpu_baseline_prefill(inp, budget_s=30.0):
    """The fp64 oracle, as it stands, on the host cores: the whole workload,
    repeated until ~10 s have passed (never past the budget)."""
    import oracle
    n = 0
    t0 = time.perf_counter()
    while True:
        oracle.kla_fwd(inp["q"], inp["k"], inp["v"], inp["log_alpha"],
                       inp["eta"], inp["eps"], inp["h0"])
        n += 1
        el = time.perf_counter() - t0
        if el >= 10.0 or el * (n + 1) / n > budget_s:
            break
    w = inp["workload"]
    return dict(value=n * w.B * w.T / el, unit="tokens/s",
                cores=oracle.max_threads(), kind="oracle",
                sample=f"full {w.name} workload x{n} "
                       f"(fp64 C recurrence, OpenMP over batch x head)")


def oracle_rate(fn, units, unit, sample, budget_s=3.0):
    """The oracle call `fn` (a bounded sample of a workload worth `units`
    of `unit`), as it stands, repeated on the host cores until `budget_s`
    have passed (at least once)."""
    import oracle
    n = 0
    t0 = time.perf_counter()
    while True:
        fn()
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return dict(value=n * units / el, unit=unit, cores=oracle.max_threads(),
                kind="oracle", sample=f"{sample} x{n}")


def extra_cpu_baselines(pf_inputs):
    """Oracle timings beside the decode, backward, preconditioned and
    131K-prefill lines, each on a bounded sample of its workload."""
    import oracle
    out = {}
    dw = gen.DECODE
    d = gen.decode_inputs(dw, steps=1)
    args = [d[n][0] for n in ("q", "k", "v", "log_alpha", "eta")]
    S0 = d["S0"].double().numpy()
    out["decode"] = oracle_rate(
        lambda: oracle.kla_decode_step(*args, d["eps"], S0), 1, "steps/s",
        f"one full decode step ({dw.B} x {dw.H} heads, fp64 C)")
    w = gen.LAYER_1B
    sub = {k: (v[:1] if isinstance(v, torch.Tensor) else v)
           for k, v in pf_inputs.items()}
    rng = np.random.default_rng(gen.SEEDS[w.name] + 200)
    do = rng.standard_normal(tuple(sub["v"].shape))
    dhT = rng.standard_normal((1, w.H, w.dk, w.dv))
    out["backward"] = oracle_rate(
        lambda: oracle.kla_bwd(sub["q"], sub["k"], sub["v"],
                               sub["log_alpha"], sub["eta"], sub["eps"],
                               sub["h0"], do, dhT),
        w.T, "tokens/s",
        f"sequence 0 of {w.name} (all {w.H} heads), reverse mode, fp64 C")
    out["preconditioned"] = oracle_rate(
        lambda: oracle.pkla_fwd(sub["q"], sub["k"], sub["v"],
                                sub["log_alpha"], sub["eta"], sub["eps"],
                                sub["h0"]),
        w.T, "tokens/s",
        f"sequence 0 of {w.name} (all {w.H} heads), preconditioned, fp64 C")
    c1w = gen.LAYER_340M
    c1 = gen.prefill_inputs(c1w, B=1)
    out["c1"] = oracle_rate(
        lambda: oracle.kla_fwd(c1["q"], c1["k"], c1["v"], c1["log_alpha"],
                               c1["eta"], c1["eps"], c1["h0"]),
        c1w.T, "tokens/s", f"sequence 0 of {c1w.name} (all heads), fp64 C")
    c3w = gen.LONG_CTX
    c3 = gen.prefill_inputs(c3w, T=4096)
    out["c3"] = oracle_rate(
        lambda: oracle.kla_fwd(c3["q"], c3["k"], c3["v"], c3["log_alpha"],
                               c3["eta"], c3["eps"], c3["h0"]),
        4096, "tokens/s", f"the first 4096 tokens of {c3w.name}, fp64 C")
    lw = gen.LONG_131K
    lt = 8192
    li = gen.prefill_inputs(lw, T=lt)
    out["prefill_131k"] = oracle_rate(
        lambda: oracle.kla_fwd(li["q"], li["k"], li["v"], li["log_alpha"],
                               li["eta"], li["eps"], li["h0"]),
        lt, "tokens/s",
        f"the first {lt} tokens of {lw.name} (all heads; the recurrence "
        f"costs the same per token at any position), fp64 C")
    return out


def run_only(args):
    """A single kernel on its workload, for profiler captures: warm-up
    launches then `--steps` launches, no other GPU work besides input setup
    (and, for the forward pass, the L2 flush between launches)."""
    kla.load_library()
    if args.only == "prefill":
        w = gen.LAYER_1B
        pf = bench_prefill(w, args.steps, args.warmup, 1, 0)
        print(json.dumps({"only": "prefill", "workload": w.name,
                          "ms_per_launch": round(pf["ms"], 5)}))
    else:
        w = gen.DECODE
        ms, _ = bench_decode(w, args.steps, args.warmup)
        print(json.dumps({"only": "decode", "workload": w.name,
                          "ms_per_launch": round(ms, 5)}))


def sig(x, n=4):
    """x rounded to n significant digits (keeps the printed line short)."""
    if x is None or x == 0 or not np.isfinite(x):
        return x
    return float(f"{x:.{n}g}")


def prefill_point(w, world, gpu_index, hbm, steps=5, warmup=3, inp=None,
                  rule="kaczmarz"):
    """Forward pass of workload `w`: ms per call, tokens/s over all ranks and
    the HBM roofline fraction of the path (algorithmic bytes / time)."""
    pf = bench_prefill(w, steps, warmup, world, gpu_index, rule=rule,
                       inp=inp)
    gbs = prefill_bytes(w) / (pf["ms"] * 1e-3) / 1e9
    return pf, {"ms": sig(pf["ms"]),
                "tps": sig(world * w.B * w.T / (pf["ms"] * 1e-3)),
                "frac": sig(gbs / hbm, 3)}


def run_ours(args):
    world, rank, local = dist_setup()
    hbm, tf_burst, tf_sus, peak_src = peaks()
    w = gen.LAYER_1B
    kla.load_library()
    pf = bench_prefill(w, args.steps, args.warmup, world, local)
    ms = pf["ms"]
    tokens = w.B * w.T
    value = world * tokens / (ms * 1e-3)
    nbytes = prefill_bytes(w)
    achieved = nbytes / (ms * 1e-3) / 1e9
    flops = prefill_flops(w)
    path = kla.forward_path(w.B, w.T, w.H, w.dk, w.dv, w.C, torch.bfloat16)
    roofline = {"bound": "hbm", "achieved": sig(achieved, 5), "peak": hbm,
                "unit": "GB/s", "frac": sig(achieved / hbm, 4),
                "traffic": profiled_traffic(path["traffic_key"]),
                "tc_frac": sig(flops / (ms * 1e-3) / 1e12 / tf_burst, 3),
                "src": peak_src}
    inputs = pf["inputs"]

    e2e_ms, h2d, d2h = bench_prefill_e2e(w, inputs, max(3, args.steps // 2),
                                         2)
    e2e = {"value": sig(world * tokens / (e2e_ms * 1e-3), 5),
           "unit": "tokens/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h}

    extra = {}
    # the learned-step (gated DeltaNet) rule on the same kernels and inputs:
    # the pages claim equal prefill latency for the two
    gdn = bench_prefill(w, args.steps, args.warmup, world, local,
                        rule="given", inp=inputs)
    extra["gdn_ratio"] = sig(ms / gdn["ms"], 4)

    if not args.no_decode:
        dw = gen.DECODE
        dms, dclk = bench_decode(dw, args.decode_steps, 20, gpu_index=local)
        gbs = decode_bytes(dw) / (dms * 1e-3) / 1e9
        # the decode section's own clocks: median SM MHz, throttle reasons
        extra["decode"] = {"sps": sig(1e3 / dms, 5), "ms": sig(dms),
                           "gbs": sig(gbs), "frac": sig(gbs / hbm, 3),
                           "mhz": dclk["sm_mhz"], "thr": dclk["reasons"]}

    if not args.no_configs:
        _, extra["c1"] = prefill_point(gen.LAYER_340M, world, local, hbm)
        c3w = gen.LONG_CTX
        c3in = gen.prefill_inputs(c3w)
        _, c3 = prefill_point(c3w, world, local, hbm, steps=3, inp=c3in)
        sms, sp = bench_seq(c3w, c3in, 3, 3, world)
        c3["split_ms"] = sig(sms)
        c3["split_frac"] = sig(prefill_bytes(c3w) / (sms * 1e-3) / 1e9 / hbm,
                               3)
        extra["c3"] = c3
        del c3in

    if not args.no_backward:
        bms, ws_bytes = bench_backward(w, inputs, 3, 3, world)
        bflops = backward_flops(w)
        ach = bflops / (bms * 1e-3) / 1e12
        extra["bwd"] = {"ms": sig(bms), "tps": sig(world * tokens /
                                                    (bms * 1e-3)),
                        "tflops": sig(ach), "frac": sig(ach / tf_sus, 3)}

    if not args.no_precond:
        t_plain, t_keys, t_fwd = bench_precond(w, inputs, 10, 3, world)
        extra["pkla"] = {"keys_ms": sig(t_keys), "fwd_ms": sig(t_fwd),
                         "ratio": sig((t_keys + t_fwd) / t_plain, 3)}

    if not args.no_long:
        lc = bench_long_context(world, local, hbm)
        p131, h32 = lc["prefill_131k"], lc["decode_after_32k"]
        extra["l131k"] = {"ms": p131["ms"], "frac": sig(p131["roofline_frac"],
                                                        3),
                          "split_ms": p131["split"]["ms"],
                          "split_frac": sig(p131["split"]["roofline_frac"],
                                            3),
                          "gdn_ratio": p131["kla_over_gdn_time"]}
        extra["h32k"] = {"prefill_ms": h32["prefill_ms"],
                         "dec_ms": h32["decode_ms_per_step"],
                         "graph_ms": h32["graph_decode_ms_per_step"]}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_prefill(inputs)
        cpu["value"] = sig(cpu["value"], 5)
        ob = extra_cpu_baselines(inputs)
        for key, name in (("decode", "decode"), ("bwd", "backward"),
                          ("pkla", "preconditioned"),
                          ("l131k", "prefill_131k"), ("c1", "c1"),
                          ("c3", "c3")):
            if key in extra and name in ob:
                extra[key]["cpu"] = sig(ob[name]["value"], 4)

    clk = pf["clocks"] or {}
    line = {"metric": METRIC, "value": sig(value, 6), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sig(ms, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": w.name, "l2": "flushed per step",
                       "path": path["name"], "parallelism":
                       f"replicas x{world}"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": pf["launches"] * path["launches"],
            "clocks": {"sm_mhz": clk.get("sm_mhz"),
                       "sm_max_mhz": clk.get("sm_max_mhz"),
                       "reasons": clk.get("reasons", [])}}
    line.update(extra)
    if rank == 0:
        print(json.dumps(line, separators=(",", ":")), flush=True)


# ------------------------------------------------------------ reference arm

def run_reference(args):
    """The oracle as it stands on the host cores: each step runs the fp64
    recurrence over one of the four sequences (all 16 heads, 4096 tokens)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    w = gen.LAYER_1B
    inp = gen.prefill_inputs(w)
    sl = {k: (v[:1] if isinstance(v, torch.Tensor) else v)
          for k, v in inp.items()}

    def step():
        oracle.kla_fwd(sl["q"], sl["k"], sl["v"], sl["log_alpha"],
                       sl["eta"], sl["eps"], sl["h0"])

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    ms = el * 1e3 / args.steps
    value = w.T / (ms * 1e-3)
    sample = f"1 of {w.B} sequences of {w.name} (all heads) per step"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 1),
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded; 1B-layer "
                                    "distributions)",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H,
                       "dk": w.dk, "dv": w.dv, "C": w.C},
            "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s",
                             "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 1), "unit": "tokens/s",
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--decode-steps", type=int, default=1000)
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--no-precond", action="store_true")
    ap.add_argument("--no-long", action="store_true",
                    help="skip the 131K-prefill / 32K-decode points")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the 340M-layer and 65K-context lines")
    ap.add_argument("--only", choices=["prefill", "decode"], default=None,
                    help="run one kernel alone (profiler captures)")
    args = ap.parse_args()
    if args.only:
        run_only(args)
        return
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
