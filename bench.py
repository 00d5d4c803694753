#!/usr/bin/env python3
"""Benchmark of the paged-KV GQA hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
plan + split-KV decode (stage 1 and LSE merge) on the Llama-3-8B-shaped decode
workload (B=64, Hq=32, Hkv=8, D=128, page 16, bf16, L~U[512,8192]), then one
prefix-prefill/extend call on the extend workload (B=8, Hq=32, Hkv=8, D=128,
page 16, ctx~U[0,4096], q~U[1,2048]).

``value`` is the decode KV-read throughput in TB/s: the algorithmic bytes of
one decode call (K and V of min(L, window) keys per request and kv head, plus
q, out, lse and block-table entries) divided by the CUDA-event duration of the
decode call.  Extend TFLOP/s is reported beside it.  Every step streams more
than the 129 MB L2 (1.14 GB of decode KV alone) in a fixed order, so no input
of a step is L2-resident when it starts; L2 is not flushed.

``--impl reference`` times the CPU oracle (the fp64 reference implementation
of the same attention) on the host cores instead, on a bounded sample of the
same decode workload per step.

Multi-GPU (torchrun, one rank per GPU): every rank runs the same per-GPU
workload (weak scaling); there is no collective on the data path.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DECODE_WORKLOAD = "decode_llama3_8b"
EXTEND_WORKLOAD = "prefill"
DECODE_WORKLOADS = ("decode_llama3_8b", "decode_e4m3_window", "decode_softcap_d256", "decode_tiny")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return FALLBACK_PEAKS, "fallback"


# ---- algorithmic work (per call) -------------------------------------------------

def decode_bytes(p) -> int:
    """K+V of the attended keys + q + out + lse + the block-table entries of
    the pages those keys span (a window starting inside a page spans it)."""
    e = 1 if p.kv_dtype == "fp8_e4m3" else 2
    L = p.seq_lens.astype(np.int64)
    n = np.minimum(L, p.window) if p.window > 0 else L
    kv = int(n.sum()) * p.num_kv_heads * p.head_dim * e * 2
    B, Hq, D = p.batch, p.num_q_heads, p.head_dim
    ps = p.page_size
    pages = int(np.where(n > 0, (L - 1) // ps - (L - n) // ps + 1, 0).sum())
    return kv + B * Hq * D * 2 * 2 + B * Hq * 4 + pages * 4


def decode_plan_kw(pb, p, name: str, splits: int = 0) -> dict:
    """pa_plan arguments for a decode workload (the tiny one fixes 4 splits;
    `splits` > 0 fixes the split count, for profiling reduced cases in the
    launch shape of the full workload)."""
    return dict(mode=pb.MODE_DECODE, num_q_heads=p.num_q_heads, num_kv_heads=p.num_kv_heads,
                head_dim=p.head_dim, page_size=p.page_size,
                kv_dtype=pb.KV_FP8_E4M3 if p.kv_dtype == "fp8_e4m3" else pb.KV_BF16, max_batch=p.batch,
                max_pages_per_seq=p.block_table.shape[1], window=p.window, has_sinks=p.sinks is not None,
                soft_cap=p.soft_cap, num_splits=splits if splits > 0 else (4 if name == "decode_tiny" else 0))


def extend_flops(p) -> int:
    """4 * D * Hq per attended (query, key) pair: Q.K^T and P.V, causal pairs only."""
    L = p.seq_lens.astype(np.int64)
    ql = np.diff(p.query_start_loc).astype(np.int64)
    ctx = L - ql
    pairs = 0
    for c, q in zip(ctx, ql):
        if p.window > 0:
            i = np.arange(q)
            pairs += int(np.minimum(c + i + 1, p.window).sum())
        else:
            pairs += int(q * c + q * (q + 1) // 2)
    return 4 * p.head_dim * p.num_q_heads * pairs


def kernel_source_hash(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "paged_kv_gqa_12_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, files):
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    source is unchanged since it was captured."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not t or t.get("source_hash") != kernel_source_hash(files):
        return None
    return t.get("dram_bytes_per_launch")


# ---- multi-rank aggregation ------------------------------------------------------

def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise maximum of per-rank timings (the slowest rank bounds the
    job); identity on one process."""
    import torch
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def weak_scaling_throughput(world: int, steps: int, units_per_step: float, seconds: float) -> float:
    """Whole-job throughput: every rank processed `steps` steps of the same
    per-GPU workload; `seconds` is the max over ranks."""
    return world * steps * units_per_step / max(seconds, 1e-12)


# ---- clocks -----------------------------------------------------------------------

# NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*)
_NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                 0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class ClockSampler:
    """SM clock, power and clock-event reasons sampled every millisecond on a
    background thread through NVML (read-only queries), timestamped on
    arrival, so the timed window -- even a 10 ms one -- can be cut out
    afterwards.  Falls back to ``nvidia-smi -lms 50`` where NVML cannot be
    loaded.  The GPU is found by its PCI bus id, so CUDA_VISIBLE_DEVICES
    renumbering does not matter."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, cuda_index: int, period_s: float = 0.001):
        self.samples = []      # (time, sm_mhz, power_w, [reasons])
        self.max_mhz = None
        self.source = None
        self.proc = None
        self._stop = threading.Event()
        self.period = period_s
        if self._nvml_open(cuda_index):
            self.source = "nvml, 1 ms"
            self.t = threading.Thread(target=self._nvml_loop, daemon=True)
            self.t.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(cuda_index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.source = "nvidia-smi, 50 ms"
        self.t = threading.Thread(target=self._smi_loop, daemon=True)
        self.t.start()

    def _nvml_open(self, cuda_index):
        import ctypes
        try:
            import torch
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return False
            h = ctypes.c_void_p()
            props = torch.cuda.get_device_properties(cuda_index)
            bus = getattr(props, "pci_bus_id", None)
            ok = False
            if bus is not None:
                pci = "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), bus,
                                             getattr(props, "pci_device_id", 0))
                ok = nv.nvmlDeviceGetHandleByPciBusId_v2(pci.encode(), ctypes.byref(h)) == 0
            if not ok:
                ok = nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(cuda_index), ctypes.byref(h)) == 0
            if not ok:
                return False
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:   # NVML_CLOCK_SM
                self.max_mhz = float(mx.value)
            self._nv, self._h = nv, h
            return True
        except (OSError, AttributeError, RuntimeError):
            return False

    def _nvml_loop(self):
        import ctypes
        nv, h = self._nv, self._h
        clk, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            t = time.time()
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                p = pw.value / 1000.0 if nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)) == 0 else None
                rv = rs.value if reasons_fn(h, ctypes.byref(rs)) == 0 else 0
                r = [n for bit, n in _NVML_REASONS.items() if rv & bit]
                self.samples.append((t, float(clk.value), p, r))
            self._stop.wait(self.period)

    def _smi_loop(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            r = [x.strip() for x in line.split(",")]
            if len(r) < 8:
                continue
            try:
                sm, mx = float(r[0]), float(r[1])
            except ValueError:
                continue
            try:
                p = float(r[2])
            except ValueError:
                p = None
            self.max_mhz = mx
            self.samples.append((time.time(), sm, p, [names[i] for i in range(4) if r[4 + i].lower().startswith("active")]))

    def stop(self):
        self._stop.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        """Clock record of the timed window [t0, t1].  If no sample fell inside
        it, the record says so and summarises the whole run instead."""
        rows = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed region"
        if not rows:
            rows = list(self.samples)
            window = "whole run: no sample fell inside the timed region"
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no clock samples"], "samples": 0,
                    "source": self.source}
        sm = [r[1] for r in rows]
        pw = [r[2] for r in rows if r[2] is not None]
        reasons = sorted({n for r in rows for n in r[3]})
        return {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm), "sm_max_mhz": self.max_mhz,
                "power_w_max": max(pw) if pw else None, "reasons": reasons, "samples": len(rows),
                "window": window, "window_ms": round((t1 - t0) * 1e3, 3), "source": self.source}


# ---- our arm ------------------------------------------------------------------------

def run_ours(args):
    import torch
    import torch.distributed as dist

    from paged_kv_gqa_12_gb300 import binding as pb
    from paged_kv_gqa_12_gb300 import workloads as wl

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pb.load()

    def barrier():
        if world > 1:
            dist.barrier()

    def upload(p):
        def t(a):
            if a.dtype == np.uint16:
                return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
            return torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        return dict(q=t(p.q), k=t(p.k_cache), v=t(p.v_cache), bt=t(p.block_table), sl=t(p.seq_lens),
                    qsl=None if p.query_start_loc is None else t(p.query_start_loc),
                    sinks=None if p.sinks is None else t(p.sinks))

    # Weak scaling: each rank holds its own copy of the per-GPU workload.
    dp = wl.workload_problem(args.decode_workload, batch=args.decode_batch)
    ep = wl.workload_problem(EXTEND_WORKLOAD, batch=args.extend_batch)
    dd, ed = upload(dp), upload(ep)
    dplan_kw = decode_plan_kw(pb, dp, args.decode_workload, args.decode_splits)
    dplan = pb.plan(**dplan_kw, host_seq_lens=dp.seq_lens)
    dscr = pb.alloc_scratch(dplan, dev)
    dout = torch.empty(dp.q.shape, dtype=torch.bfloat16, device=dev)
    dlse = torch.empty(dp.q.shape[:2], dtype=torch.float32, device=dev)
    extend_ok = args.only != "decode"
    eplan_kw = dict(mode=pb.MODE_EXTEND, num_q_heads=ep.num_q_heads, num_kv_heads=ep.num_kv_heads,
                    head_dim=ep.head_dim, page_size=ep.page_size, kv_dtype=pb.KV_BF16, max_batch=ep.batch,
                    max_pages_per_seq=ep.block_table.shape[1], max_total_q=ep.num_rows,
                    window=ep.window, has_sinks=ep.sinks is not None, soft_cap=ep.soft_cap)
    try:
        eplan = pb.plan(**eplan_kw)
        escr = pb.alloc_scratch(eplan, dev)
    except pb.PaError:
        extend_ok = False
    decode_on = args.only != "extend"
    eout = torch.empty(ep.q.shape, dtype=torch.bfloat16, device=dev)
    else_ = torch.empty(ep.q.shape[:2], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def decode_call():
        pb.decode(dplan, dd["q"], dd["k"], dd["v"], dd["bt"], dd["sl"], scale=dp.scale, out=dout, lse=dlse,
                  sinks=dd["sinks"], k_scale=dp.k_scale, v_scale=dp.v_scale, scratch=dscr, stream=stream)

    def extend_call():
        pb.extend(eplan, ed["q"], ed["k"], ed["v"], ed["bt"], ed["sl"], ed["qsl"], scale=ep.scale, out=eout,
                  lse=else_, sinks=ed["sinks"], k_scale=ep.k_scale, v_scale=ep.v_scale, scratch=escr,
                  stream=stream)

    K, W = args.steps, args.warmup
    for _ in range(W):
        if decode_on:
            decode_call()
        if extend_ok:
            extend_call()
    torch.cuda.synchronize(dev)
    if pb.check(dscr) != 0 or (extend_ok and pb.check(escr) != 0):
        raise RuntimeError("device error during warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        time.sleep(0.3)
    barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    w0 = time.perf_counter()
    for k in range(K):
        ev[k][0].record(stream)
        if decode_on:
            decode_call()
        ev[k][1].record(stream)
        if extend_ok:
            extend_call()
        ev[k][2].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    loop_s = time.perf_counter() - w0
    t1 = time.time()
    if sampler:
        sampler.stop()
    dec_ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)]
    ext_ms = [ev[k][1].elapsed_time(ev[k][2]) for k in range(K)] if extend_ok else []
    if pb.check(dscr) != 0 or (extend_ok and pb.check(escr) != 0):
        raise RuntimeError("device error during the timed region")

    dec_s, ext_s = sum(dec_ms) / 1e3, sum(ext_ms) / 1e3
    dec_s, ext_s, loop_s = max_over_ranks([dec_s, ext_s, loop_s], dist if world > 1 else None, dev)

    dbytes = decode_bytes(dp)
    eflops = extend_flops(ep) if extend_ok else 0
    # --only extend (profiling runs) times no decode: no decode value
    value_tbs = weak_scaling_throughput(world, K, dbytes, dec_s) / 1e12 if decode_on else None

    # ---- end to end through the public API with host buffers ---------------------
    # Every step copies its inputs from pinned host memory, plans, runs the
    # call and copies its results back; the copies of neighbouring steps
    # overlap the kernels on two copy streams (e2e_pipelined), and the timed
    # region holds every copy of every step.
    copy_streams = (torch.cuda.Stream(dev), torch.cuda.Stream(dev))   # host to device, device to host

    def pinned(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()
        return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()

    Ke = min(K, 200)
    d_host_in = [pinned(dp.q), pinned(dp.block_table), pinned(dp.seq_lens)]
    d_dev_in = [[torch.empty_like(x, device=dev) for x in d_host_in] for _ in range(2)]
    d_dev_out = [[torch.empty_like(dout), torch.empty_like(dlse)] for _ in range(2)]
    d_host_out = [[torch.empty(dout.shape, dtype=dout.dtype).pin_memory(),
                   torch.empty(dlse.shape, dtype=dlse.dtype).pin_memory()] for _ in range(2)]

    def d_compute(ins, outs):
        plan = pb.plan(**dplan_kw, host_seq_lens=dp.seq_lens)
        pb.decode(plan, ins[0], dd["k"], dd["v"], ins[1], ins[2], scale=dp.scale, out=outs[0], lse=outs[1],
                  sinks=dd["sinks"], k_scale=dp.k_scale, v_scale=dp.v_scale, scratch=dscr, stream=stream)

    e2e_s = None
    if decode_on:
        e2e_pipelined(torch, stream, copy_streams, d_host_in, d_dev_in, d_compute, d_dev_out, d_host_out, 3)
        torch.cuda.synchronize(dev)
        barrier()
        e2e_s = e2e_pipelined(torch, stream, copy_streams, d_host_in, d_dev_in, d_compute, d_dev_out, d_host_out, Ke)
        e2e_s = max_over_ranks([e2e_s], dist if world > 1 else None, dev)[0]
        if pb.check(dscr) != 0:
            raise RuntimeError("device error during the decode end-to-end loop")
    h2d = sum(x.numel() * x.element_size() for x in d_host_in)
    d2h = sum(x.numel() * x.element_size() for x in d_host_out[0])

    e2e_ext = None
    if extend_ok:
        x_host_in = [pinned(ep.q), pinned(ep.block_table), pinned(ep.seq_lens), pinned(ep.query_start_loc)]
        x_dev_in = [[torch.empty_like(x, device=dev) for x in x_host_in] for _ in range(2)]
        x_dev_out = [[torch.empty_like(eout), torch.empty_like(else_)] for _ in range(2)]
        x_host_out = [[torch.empty(eout.shape, dtype=eout.dtype).pin_memory(),
                       torch.empty(else_.shape, dtype=else_.dtype).pin_memory()] for _ in range(2)]

        def x_compute(ins, outs):
            plan = pb.plan(**eplan_kw)
            pb.extend(plan, ins[0], ed["k"], ed["v"], ins[1], ins[2], ins[3], scale=ep.scale, out=outs[0],
                      lse=outs[1], sinks=ed["sinks"], k_scale=ep.k_scale, v_scale=ep.v_scale, scratch=escr,
                      stream=stream)

        Kx = min(K, 50)
        e2e_pipelined(torch, stream, copy_streams, x_host_in, x_dev_in, x_compute, x_dev_out, x_host_out, 3)
        torch.cuda.synchronize(dev)
        barrier()
        xs = e2e_pipelined(torch, stream, copy_streams, x_host_in, x_dev_in, x_compute, x_dev_out, x_host_out, Kx)
        xs = max_over_ranks([xs], dist if world > 1 else None, dev)[0]
        e2e_ext = {"value": round(weak_scaling_throughput(world, Kx, extend_flops(ep), xs) / 1e12, 2),
                   "unit": "TFLOP/s", "steps": Kx,
                   "h2d_bytes_per_step": int(sum(x.numel() * x.element_size() for x in x_host_in)),
                   "d2h_bytes_per_step": int(sum(x.numel() * x.element_size() for x in x_host_out[0])),
                   "what": "extend through the C ABI: pinned-host q/block_table/seq_lens/query_start_loc H2D, "
                           "pa_plan, pa_extend, out/lse D2H, every step; the copies of neighbouring steps "
                           "overlap the kernels on two copy streams"}
        if pb.check(escr) != 0:
            raise RuntimeError("device error during the extend end-to-end loop")

    # the extras are stated for the default decode workload's sequences
    extras = None if args.no_extras or args.decode_workload != DECODE_WORKLOAD or args.decode_splits else \
        measure_extras(pb, wl, dp, dd, dev, stream)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peaks, peak_src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    bf16 = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    kernels = {}
    if decode_on:
        dec_mean = statistics.mean(dec_ms) / 1e3
        dec_ach = dbytes / dec_mean / 1e9
        kernels["decode"] = {"bound": "hbm", "achieved": round(dec_ach, 1), "peak": hbm, "unit": "GB/s",
                             "frac": round(dec_ach / hbm, 4),
                             # the record is per launch of the full default workload
                             "traffic": recorded_traffic("decode_split_kernel", ["decode.cu", "ptx.cuh", "pa_internal.h"])
                             if (args.decode_workload == DECODE_WORKLOAD and args.decode_batch is None
                                 and args.decode_splits == 0) else None,
                             "timed": "pa_decode call (split kernel; the last split of each request and kv head merges), CUDA events, mean over steps",
                             "algorithmic_bytes_per_launch": dbytes, "peak_source": f"{peak_src} hbm_gbs"}
    if extend_ok:
        ext_mean = statistics.mean(ext_ms) / 1e3
        ext_ach = eflops / ext_mean / 1e12
        kernels["extend"] = {"bound": "tensor", "achieved": round(ext_ach, 2), "peak": bf16, "unit": "TFLOP/s",
                             "frac": round(ext_ach / bf16, 4),
                             "traffic": recorded_traffic("extend_attn_kernel", ["extend.cu", "ptx.cuh", "tcgen05.cuh", "pa_internal.h"])
                             if args.extend_batch is None else None,
                             "timed": "pa_extend call (scheduler + attention kernel), CUDA events, mean over steps",
                             "algorithmic_flops_per_launch": eflops, "peak_source": f"{peak_src} bf16_tflops (burst)"}
    dominant = "decode" if decode_on else "extend"
    if decode_on and extend_ok and statistics.mean(ext_ms) > statistics.mean(dec_ms):
        dominant = "extend"
    roof = {k: v for k, v in kernels[dominant].items() if k in ("bound", "achieved", "peak", "unit", "frac", "traffic")}
    roof["kernel"] = dominant

    cpu = cpu_baseline(dp, ep if extend_ok else None, args.cpu_sample) \
        if (world == 1 and not args.no_cpu_baseline) else None
    clocks = sampler.summary(t0, t1) if sampler else None
    line = {
        "metric": "paged decode KV-read TB/s (% of HBM peak); extend TFLOP/s (% bf16 peak)",
        "value": round(value_tbs, 4) if value_tbs is not None else None,
        "unit": "TB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(loop_s / K * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; N(0,1) values, shuffled page pools)",
        "config": {"workload": "decode " + wl.WORKLOADS[args.decode_workload] + " + extend " + wl.WORKLOADS[EXTEND_WORKLOAD],
                   "decode_batch": dp.batch, "decode_tokens": int(dp.seq_lens.sum()),
                   "extend_batch": ep.batch, "extend_q_rows": ep.num_rows,
                   "l2": "not flushed: each step streams > 1.2 GB (L2 129 MB) in a fixed order",
                   "decode_plan": {"tile_tokens": dplan.tile_tokens, "split_tiles": dplan.split_tiles,
                                   "max_splits": dplan.max_splits, "stages": dplan.stages}},
        "decode_ms": round(statistics.mean(dec_ms), 4) if decode_on else None,
        "extend_ms": round(statistics.mean(ext_ms), 4) if extend_ok else None,
        "extend_tflops": round(weak_scaling_throughput(world, K, eflops, ext_s) / 1e12, 2) if extend_ok else None,
        "roofline": roof,
        "kernels": kernels,
        "e2e": {"value": round(weak_scaling_throughput(world, Ke, dbytes, e2e_s) / 1e12, 4), "unit": "TB/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "what": "decode through the C ABI: pinned-host q/block_table/seq_lens H2D, pa_plan, pa_decode, "
                        "out/lse D2H, every step; the copies of neighbouring steps overlap the kernels on two "
                        "copy streams",
                "extend": e2e_ext}
               if e2e_s is not None else None,
        "gpu_launches": K * ((dplan.launches if decode_on else 0) + (eplan.launches if extend_ok else 0)),
        "extras": extras,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


# ---- end to end ---------------------------------------------------------------------

def e2e_pipelined(torch, stream, copy_streams, host_in, dev_in, compute, dev_out, host_out, steps):
    """`steps` end-to-end steps through the public API; returns seconds.

    Step k copies `host_in` (pinned) into device slot k % 2 on the first copy
    stream, runs compute(dev_in[slot], dev_out[slot]) on `stream` once its
    inputs have landed, and copies dev_out[slot] back into host_out[slot] on
    the second copy stream once it is done.  So the inputs of step k+1 go in
    while step k computes and its results come back meanwhile, both
    directions at once.  A slot's inputs are overwritten once the step that
    used them two steps before has computed, its outputs once that step's
    results have been copied back.  The CUDA events bracket all of it: the
    first input copy to the last result copy."""
    h2d, d2h = copy_streams
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    freed = [torch.cuda.Event() for _ in range(2)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def copy_in(k):
        i = k % 2
        with torch.cuda.stream(h2d):
            if k >= 2:
                h2d.wait_event(done[i])   # step k - 2 has read its inputs
            for d, h in zip(dev_in[i], host_in):
                d.copy_(h, non_blocking=True)
            in_ready[i].record(h2d)

    e0.record(stream)
    h2d.wait_event(e0)
    copy_in(0)
    for k in range(steps):
        i = k % 2
        stream.wait_event(in_ready[i])
        if k >= 2:
            stream.wait_event(freed[i])   # step k - 2's results are back on the host
        with torch.cuda.stream(stream):
            compute(dev_in[i], dev_out[i])
        done[i].record(stream)
        if k + 1 < steps:
            copy_in(k + 1)
        with torch.cuda.stream(d2h):
            d2h.wait_event(done[i])
            for h, d in zip(host_out[i], dev_out[i]):
                h.copy_(d, non_blocking=True)
            freed[i].record(d2h)
    stream.wait_event(freed[(steps - 1) % 2])
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / 1e3


# ---- further hot-path modes, timed apart from the step -------------------------------

def _time_calls(torch, fn, stream, n=50, warm=5):
    for _ in range(warm):
        fn()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(n):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n / 1e3


def measure_extras(pb, wl, dp, dd, dev, stream):
    """Verify mode on the decode workload's sequences (3 speculative tokens per
    request, K/V of the new tokens already in the pages) and extend with an
    e4m3 KV cache on the extend workload."""
    import dataclasses
    import torch
    peaks, _ = load_peaks()
    res = {}
    # verify: q_len = 4 per request over the decode workload's cache
    q_len = 4
    B, Hq, D = dp.batch, dp.num_q_heads, dp.head_dim
    g = torch.Generator(device="cpu").manual_seed(4242)
    qv = torch.randn(B * q_len, Hq, D, generator=g).to(torch.bfloat16).to(dev)
    qsl = torch.arange(0, B * q_len + 1, q_len, dtype=torch.int32, device=dev)
    vplan = pb.plan(mode=pb.MODE_VERIFY, num_q_heads=Hq, num_kv_heads=dp.num_kv_heads, head_dim=D,
                    page_size=dp.page_size, max_batch=B, max_pages_per_seq=dp.block_table.shape[1],
                    max_total_q=B * q_len, q_len=q_len, host_seq_lens=dp.seq_lens)
    vscr = pb.alloc_scratch(vplan, dev)
    vout = torch.empty_like(qv)
    vlse = torch.empty(qv.shape[:2], dtype=torch.float32, device=dev)
    t = _time_calls(torch, lambda: pb.extend(vplan, qv, dd["k"], dd["v"], dd["bt"], dd["sl"], qsl, scale=dp.scale,
                                             out=vout, lse=vlse, scratch=vscr, stream=stream), stream)
    vb = decode_bytes(dp) + B * Hq * D * 2 * 2 * (q_len - 1)
    res["verify"] = {"workload": "decode workload's sequences, q_len 4 per request (3 speculative tokens)",
                     "ms": round(t * 1e3, 4), "kv_read_tbs": round(vb / t / 1e12, 4),
                     "frac_of_hbm": round(vb / t / 1e9 / float(peaks.get("hbm_gbs", 6800.0)), 4),
                     "device_error": pb.check(vscr)}
    # extend with an e4m3 cache
    ep8 = wl.workload_problem(EXTEND_WORKLOAD, kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.05)

    def t8(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    e8 = {k: t8(getattr(ep8, a)) for k, a in (("q", "q"), ("k", "k_cache"), ("v", "v_cache"), ("bt", "block_table"),
                                             ("sl", "seq_lens"), ("qsl", "query_start_loc"))}
    eplan8 = pb.plan(mode=pb.MODE_EXTEND, num_q_heads=ep8.num_q_heads, num_kv_heads=ep8.num_kv_heads,
                     head_dim=ep8.head_dim, page_size=ep8.page_size, kv_dtype=pb.KV_FP8_E4M3, max_batch=ep8.batch,
                     max_pages_per_seq=ep8.block_table.shape[1], max_total_q=ep8.num_rows)
    escr8 = pb.alloc_scratch(eplan8, dev)
    eout8 = torch.empty_like(e8["q"])
    t = _time_calls(torch, lambda: pb.extend(eplan8, e8["q"], e8["k"], e8["v"], e8["bt"], e8["sl"], e8["qsl"],
                                             scale=ep8.scale, out=eout8, k_scale=ep8.k_scale, v_scale=ep8.v_scale,
                                             scratch=escr8, stream=stream), stream)
    fl = extend_flops(ep8)
    res["extend_fp8"] = {"workload": "extend workload with an e4m3 KV cache (scales 0.05)", "ms": round(t * 1e3, 4),
                         "tflops": round(fl / t / 1e12, 2),
                         "frac_of_bf16_peak": round(fl / t / 1e12 / float(peaks.get("bf16_tflops", 1900.0)), 4),
                         "device_error": pb.check(escr8)}
    # the other decode workloads: each call timed alone, L2 flushed before it
    # by writing a 256 MB buffer and then reading another 256 MB: the read
    # evicts the written lines, so their write-back to DRAM happens before
    # the timed call instead of inside it (with the write alone, about 129 MB
    # of dirty lines were written back during the call: ~5 us of the e4m3
    # window workload's 52).  The write-only figure is reported beside it.
    peak_hbm = float(peaks.get("hbm_gbs", 6800.0))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    for name in DECODE_WORKLOADS[1:]:
        p = wl.workload_problem(name)

        def t8(a):
            if a.dtype == np.uint16:
                return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
            return torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        g = {k: t8(getattr(p, a)) for k, a in (("q", "q"), ("k", "k_cache"), ("v", "v_cache"),
                                              ("bt", "block_table"), ("sl", "seq_lens"))}
        g["sinks"] = None if p.sinks is None else t8(p.sinks)
        plan = pb.plan(**decode_plan_kw(pb, p, name), host_seq_lens=p.seq_lens)
        scr = pb.alloc_scratch(plan, dev)
        out = torch.empty(p.q.shape, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(p.q.shape[:2], dtype=torch.float32, device=dev)

        def call():
            pb.decode(plan, g["q"], g["k"], g["v"], g["bt"], g["sl"], scale=p.scale, out=out, lse=lse,
                      sinks=g["sinks"], k_scale=p.k_scale, v_scale=p.v_scale, scratch=scr, stream=stream)
        for _ in range(5):
            call()

        def timed(read_after_write):
            ms = []
            for i in range(30):
                flush.fill_(i & 255)
                if read_after_write:
                    flush_rd.sum()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                call()
                e1.record(stream)
                e1.synchronize()
                ms.append(e0.elapsed_time(e1))
            return statistics.median(ms)
        ms = [timed(True)]
        ms_write_only = timed(False)
        t = statistics.median(ms) / 1e3
        nb = decode_bytes(p)
        res[name] = {"workload": wl.WORKLOADS[name], "ms": round(t * 1e3, 4), "kv_read_tbs": round(nb / t / 1e12, 4),
                     "frac_of_hbm": round(nb / t / 1e9 / peak_hbm, 4), "algorithmic_bytes": nb,
                     "max_splits": int(plan.max_splits),
                     "timing": "median of 30 calls; before each, 256 MB written then another 256 MB read (L2 holds "
                               "neither the inputs nor dirty lines)",
                     "ms_write_only_flush": round(ms_write_only, 4),
                     "device_error": pb.check(scr)}
        del g, scr, out, lse
    # extend at other head dims / group sizes on the extend workload's
    # lengths (same flush, median of 30): the kernel configurations the
    # benchmark step does not launch
    base = wl.workload_problem("prefill")
    ql = np.diff(base.query_start_loc)
    for (Hq, Hkv, D) in ((32, 8, 64), (16, 8, 256), (64, 8, 128)):
        p = wl.build_problem("extend", num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=16,
                             seq_lens=base.seq_lens, query_lens=ql, seed=1004, poison=False)

        def t8(a):
            if a.dtype == np.uint16:
                return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
            return torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        g = {k: t8(getattr(p, a)) for k, a in (("q", "q"), ("k", "k_cache"), ("v", "v_cache"), ("bt", "block_table"),
                                              ("sl", "seq_lens"), ("qsl", "query_start_loc"))}
        plan = pb.plan(mode=pb.MODE_EXTEND, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=16,
                       max_batch=p.batch, max_pages_per_seq=p.block_table.shape[1], max_total_q=p.num_rows)
        scr = pb.alloc_scratch(plan, dev)
        out = torch.empty(p.q.shape, dtype=torch.bfloat16, device=dev)

        def call():
            pb.extend(plan, g["q"], g["k"], g["v"], g["bt"], g["sl"], g["qsl"], scale=p.scale, out=out, scratch=scr,
                      stream=stream)
        for _ in range(5):
            call()
        ms = []
        for i in range(30):
            flush.fill_(i & 255)
            flush_rd.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call()
            e1.record(stream)
            e1.synchronize()
            ms.append(e0.elapsed_time(e1))
        t = statistics.median(ms) / 1e3
        fl = extend_flops(p)
        res[f"extend_hq{Hq}_hkv{Hkv}_d{D}"] = {
            "workload": f"extend workload's lengths, Hq {Hq}, Hkv {Hkv}, D {D}, page 16, bf16",
            "ms": round(t * 1e3, 4), "tflops": round(fl / t / 1e12, 2),
            "frac_of_bf16_peak": round(fl / t / 1e12 / float(peaks.get("bf16_tflops", 1900.0)), 4),
            "timing": "median of 30 calls; L2 flushed before each as above", "device_error": pb.check(scr)}
        del g, scr, out
    # KV append: the extend workload's new tokens written into their slots of
    # a cache shaped like the workload's (bf16 copy; e4m3 quantisation into an
    # e4m3 cache).  Bytes: the new K and V read, the slot mapping, the rows
    # written; HBM-bound.
    T, Hkv, D = base.num_rows, base.num_kv_heads, base.head_dim
    ps = base.page_size
    slots = np.empty(T, np.int64)
    for b in range(base.batch):
        q0, q1 = int(base.query_start_loc[b]), int(base.query_start_loc[b + 1])
        L = int(base.seq_lens[b])
        pos = np.arange(L - (q1 - q0), L)
        slots[q0:q1] = base.block_table[b, pos // ps].astype(np.int64) * ps + pos % ps
    g2 = torch.Generator(device="cpu").manual_seed(4243)
    kn = torch.randn(T, Hkv, D, generator=g2).to(torch.bfloat16).to(dev)
    vn = torch.randn(T, Hkv, D, generator=g2).to(torch.bfloat16).to(dev)
    slot_t = torch.from_numpy(slots).to(dev)
    for name, kvd, cdt, esz in (("append_bf16", pb.KV_BF16, torch.bfloat16, 2),
                                ("append_e4m3", pb.KV_FP8_E4M3, torch.uint8, 1)):
        kc = torch.zeros(base.k_cache.shape, dtype=cdt, device=dev)
        vc = torch.zeros(base.v_cache.shape, dtype=cdt, device=dev)
        ascr = torch.zeros(65536, dtype=torch.uint8, device=dev)

        def call():
            pb.append_kv(kn, vn, kc, vc, slot_t, kv_dtype=kvd, k_scale=0.05, v_scale=0.05, scratch=ascr,
                         stream=stream)
        for _ in range(5):
            call()
        ms = []
        for i in range(30):
            flush.fill_(i & 255)
            flush_rd.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call()
            e1.record(stream)
            e1.synchronize()
            ms.append(e0.elapsed_time(e1))
        t = statistics.median(ms) / 1e3
        nb = T * Hkv * D * (2 * 2 + 2 * esz) + T * 8
        res[name] = {"workload": f"the extend workload's {T} new tokens x {Hkv} kv heads x {D} dims into their "
                                 f"slots ({'bf16' if esz == 2 else 'e4m3'} cache)",
                     "ms": round(t * 1e3, 4), "gbs": round(nb / t / 1e9, 1),
                     "frac_of_hbm": round(nb / t / 1e9 / peak_hbm, 4), "algorithmic_bytes": nb,
                     "timing": "median of 30 calls; L2 flushed before each as above",
                     "device_error": pb.check(ascr)}
        del kc, vc
    # CUDA-graph replay: the decode call with a capacity plan (no host
    # lengths), captured once and replayed (inputs > L2, no flush)
    gplan = pb.plan(**decode_plan_kw(pb, dp, "decode_llama3_8b"))
    gscr = pb.alloc_scratch(gplan, dev)
    gout = torch.empty(dp.q.shape, dtype=torch.bfloat16, device=dev)
    glse = torch.empty(dp.q.shape[:2], dtype=torch.float32, device=dev)

    def gcall():
        pb.decode(gplan, dd["q"], dd["k"], dd["v"], dd["bt"], dd["sl"], scale=dp.scale, out=gout, lse=glse,
                  sinks=dd["sinks"], k_scale=dp.k_scale, v_scale=dp.v_scale, scratch=gscr)
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        gcall()
    torch.cuda.current_stream().wait_stream(cs)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gcall()
    t = _time_calls(torch, graph.replay, torch.cuda.current_stream())
    nb = decode_bytes(dp)
    res["decode_graph_replay"] = {"workload": "the decode workload through a captured CUDA graph (capacity plan)",
                                  "ms": round(t * 1e3, 4), "kv_read_tbs": round(nb / t / 1e12, 4),
                                  "frac_of_hbm": round(nb / t / 1e9 / peak_hbm, 4),
                                  "max_splits": int(gplan.max_splits), "device_error": pb.check(gscr)}
    return res


# ---- CPU oracle legs --------------------------------------------------------------

def cpu_baseline(p, ep, n_requests: int, min_seconds: float = 6.0):
    """The oracle, as it stands, on bounded samples of the step's workloads,
    on the host cores: the decode batch (its first n_requests requests, all
    heads; all cores, repeated until about min_seconds have been timed, at
    least 3 passes), whole requests of the extend workload (all cores; the
    shortest requests in batch order until about a fifth of the workload's
    FLOPs), one pass over each other decode workload (all cores), and the
    tiny decode workload on one core.  ``value`` is the decode figure, in
    the unit of the benchmark's metric."""
    import oracle
    from paged_kv_gqa_12_gb300 import workloads as wl
    rows = np.arange(min(n_requests, p.batch), dtype=np.int32)
    cores = os.cpu_count() or 1
    oracle.attention(p, rows=rows[:1], num_threads=cores)  # load + warm
    passes, dt = 0, 0.0
    while passes < 3 or dt < min_seconds:
        t = time.perf_counter()
        oracle.attention(p, rows=rows, num_threads=cores)
        dt += time.perf_counter() - t
        passes += 1
    sub = sample_bytes(p, rows) * passes
    res = {"value": round(sub / dt / 1e12, 9), "unit": "TB/s", "cores": cores, "kind": "oracle",
           "seconds": round(dt, 3),
           "sample": f"decode requests 0..{len(rows) - 1} of the same workload (all {p.num_q_heads} heads), "
                     f"{sub // passes} algorithmic bytes per pass, {passes} passes"}
    if ep is not None:
        # extend: whole requests, smallest first, until a fifth of the FLOPs
        import dataclasses
        qsl = ep.query_start_loc
        per_req = [extend_flops(dataclasses.replace(ep, seq_lens=ep.seq_lens[b:b + 1],
                                                    query_start_loc=np.array([0, qsl[b + 1] - qsl[b]], np.int32)))
                   for b in range(ep.batch)]
        total = sum(per_req)
        chosen, fl = [], 0
        for b in sorted(range(ep.batch), key=lambda b: per_req[b]):
            if fl >= total / 5:
                break
            chosen.append(b)
            fl += per_req[b]
        chosen.sort()
        erows = np.concatenate([np.arange(qsl[b], qsl[b + 1]) for b in chosen]).astype(np.int32)
        t = time.perf_counter()
        oracle.attention(ep, rows=erows, num_threads=cores)
        et = time.perf_counter() - t
        res["extend"] = {"value": round(fl / et / 1e12, 9), "unit": "TFLOP/s", "gflops": round(fl / et / 1e9, 3),
                         "cores": cores, "kind": "oracle", "seconds": round(et, 3),
                         "sample": f"extend requests {chosen} of the extend workload (whole requests, all "
                                   f"{ep.num_q_heads} heads), {fl} algorithmic FLOPs ({fl / total:.1%} of the call)"}
    # the other decode workloads: one pass over the whole batch each, all cores
    for name in ("decode_e4m3_window", "decode_softcap_d256"):
        op = wl.workload_problem(name)
        t = time.perf_counter()
        oracle.attention(op, num_threads=cores)
        ot = time.perf_counter() - t
        ob = decode_bytes(op)
        res[name] = {"value": round(ob / ot / 1e12, 9), "unit": "TB/s", "cores": cores, "kind": "oracle",
                     "seconds": round(ot, 3), "sample": f"the whole {name} batch ({ob} algorithmic bytes), one pass"}
    tp = wl.workload_problem("decode_tiny")
    passes, dt = 0, 0.0
    while passes < 3 or dt < 2.0:
        t = time.perf_counter()
        oracle.attention(tp, num_threads=1)
        dt += time.perf_counter() - t
        passes += 1
    tb = decode_bytes(tp)
    res["decode_tiny_one_core"] = {"value": round(tb * passes / dt / 1e12, 9), "unit": "TB/s", "cores": 1,
                                   "kind": "oracle", "ms_per_call": round(dt / passes * 1e3, 4),
                                   "sample": f"the whole tiny decode workload ({tb} algorithmic bytes), "
                                             f"{passes} passes"}
    return res


def sample_bytes(p, rows):
    import dataclasses
    sub = dataclasses.replace(p, q=p.q[rows], seq_lens=p.seq_lens[rows], block_table=p.block_table[rows])
    return decode_bytes(sub)


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from paged_kv_gqa_12_gb300 import workloads as wl
    p = wl.workload_problem(DECODE_WORKLOAD)
    cores = os.cpu_count() or 1
    K, W = args.steps, args.warmup
    # bounded per-step sample: one request (all heads) per step, cycling
    times, nbytes = [], 0
    for k in range(W + K):
        r = np.array([k % p.batch], np.int32)
        t = time.perf_counter()
        oracle.attention(p, rows=r, num_threads=cores)
        dt = time.perf_counter() - t
        if k >= W:
            times.append(dt)
            nbytes += sample_bytes(p, r)
    tot = sum(times)
    value = nbytes / tot / 1e12
    line = {"impl": "reference", "metric": "paged decode KV-read TB/s (% of HBM peak); extend TFLOP/s (% bf16 peak)",
            "value": value, "unit": "TB/s", "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": K,
            "warmup": W, "ms_per_step": tot / K * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": "decode " + wl.WORKLOADS[DECODE_WORKLOAD]},
            "cpu_baseline": {"value": value, "unit": "TB/s", "cores": cores, "kind": "oracle",
                             "sample": "one decode request (all heads) per step, cycling through the batch"},
            "e2e": {"value": value, "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-sample", type=int, default=64, help="decode requests in the CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the verify / fp8-extend measurements")
    ap.add_argument("--only", choices=["decode", "extend"], default=None,
                    help="run one of the two calls per step (profiling of reduced cases)")
    ap.add_argument("--decode-batch", type=int, default=None, help="keep the first N decode requests")
    ap.add_argument("--decode-workload", choices=DECODE_WORKLOADS, default=DECODE_WORKLOAD,
                    help="decode workload of the step (profiling runs of the other decode workloads)")
    ap.add_argument("--decode-splits", type=int, default=0,
                    help="fixed KV splits per request (profiling a reduced batch in the full plan's shape)")
    ap.add_argument("--extend-batch", type=int, default=None, help="keep the first N extend requests")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
