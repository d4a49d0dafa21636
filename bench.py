"""Benchmark of one canvas refinement step on B300.

A step is one pass of the whole hot path over one batch of synthetic input:
canvas_attention on the global-layer workload (batch 1, canvas 256, committed
prefix 32768 in a paged bf16 cache, d_model 2816, 16 query / 2 KV heads,
head_dim 512, shared W_v = W_k, partial RoPE) followed by canvas_sample on the
full-vocab workload (256 positions x vocab 262144 bf16 logits, E 262144 x 2816
bf16).  All inputs are seeded synthetic draws (canvas_workloads); no dataset or
trained weights are involved.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
    python bench.py --workload loop --prefix P [--steps K] [--warmup W]
    python bench.py --workload sliding [--steps K] [--warmup W]
    python bench.py --workload moe [--steps K] [--warmup W]

Prints ONE JSON line (rank 0).  ``--workload loop`` times instead the batched
denoising loop (4 canvases x 256, 5 sliding + 1 global layers, vocab 262144,
committed prefix P), one line per run; ``--workload sliding`` times one
sliding-window layer call (batch 1, canvas 256, prefix 4096, 16/8 heads,
head_dim 256, window 1024).  Under torchrun every rank runs its own step on
its own GPU (canvases are independent: weak scaling, no data-path
collective); times are the max over ranks.  ``--impl reference`` times the
fp64 CPU oracle (the reference arm of this tier) on bounded samples.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import canvas_workloads as wl  # noqa: E402

METRIC = "canvas steps/sec (attn+sampler), attention TFLOP/s, sampler HBM GB/s"
WORKLOAD = ("global-layer canvas step: canvas_attention B=1 C=256 prefix=32768 D=2816 Hq=16 Hkv=2 d=512 "
            "(shared W_v=W_k, partial RoPE, paged bf16 cache, page 64) + canvas_sample rows=256 V=262144 "
            "E=262144x2816 bf16")
L2_BYTES = 126 * 1024 * 1024


def attn_flops(cfg: wl.AttnConfig) -> float:
    """Algorithmic attention FLOPs: 4 * d per visible (query, key) pair per head
    (2d for Q.K, 2d for P.V); masked pairs and split-combine work not counted."""
    pairs = 0
    for P in cfg.prefix:
        for i in range(cfg.C):
            lo = 0 if (cfg.layer == "global" or cfg.window <= 0) else max(0, P + i - cfg.window)
            pairs += (P - lo) + cfg.C
    return 4.0 * cfg.d * cfg.Hq * pairs


def sampler_bytes(s: wl.SampleConfig) -> float:
    """Algorithmic bytes of the vocab reduction: read logits once, write the
    bf16 probabilities once (plus per-row outputs)."""
    return s.rows * s.V * 2 + s.rows * s.V * 2 + s.rows * 17


def soft_emb_bytes(s: wl.SampleConfig) -> float:
    """Algorithmic bytes of P.E: read E and P once, write fp32 soft_emb once."""
    return s.V * s.D * 2 + s.rows * s.V * 2 + s.rows * s.D * 4


def soft_emb_flops(s: wl.SampleConfig) -> float:
    return 2.0 * s.rows * s.V * s.D


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d.get("hbm_gbs", 6400.0), d.get("bf16_tflops", 1800.0), "measured"
    return 6400.0, 1800.0, "fallback"


class ClockSampler:
    """SM clock, power and clock-event (throttle) reasons sampled through NVML
    every few milliseconds on a background thread during the timed region."""

    REASONS = (("hw_slowdown", "nvmlClocksEventReasonHwSlowdown", 0x8),
               ("sw_thermal_slowdown", "nvmlClocksEventReasonSwThermalSlowdown", 0x20),
               ("hw_thermal_slowdown", "nvmlClocksEventReasonHwThermalSlowdown", 0x40),
               ("hw_power_brake_slowdown", "nvmlClocksEventReasonHwPowerBrakeSlowdown", 0x80),
               ("sw_power_cap", "nvmlClocksEventReasonSwPowerCap", 0x4))

    def __init__(self, gpu_index: int, period_s: float = 0.004):
        self.gpu, self.period = gpu_index, period_s
        self.samples, self.thread, self.nv = [], None, None

    def start(self):
        import threading
        try:
            import pynvml as nv
            nv.nvmlInit()
            self.nv = nv
            self.h = nv.nvmlDeviceGetHandleByIndex(self.gpu)
            self.max_mhz = nv.nvmlDeviceGetMaxClockInfo(self.h, nv.NVML_CLOCK_SM)
        except Exception as e:  # no NVML binding: sample through nvidia-smi instead
            self.err = repr(e)
            self._start_smi()
            return
        self.stop_flag = threading.Event()

        def loop():
            nv = self.nv
            get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            while not self.stop_flag.is_set():
                try:
                    self.samples.append((nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM),
                                         nv.nvmlDeviceGetPowerUsage(self.h) / 1000.0, int(get_reasons(self.h))))
                except Exception:
                    pass
                self.stop_flag.wait(self.period)

        self.thread = threading.Thread(target=loop, daemon=True)
        self.thread.start()

    SMI_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.hw_power_brake_slowdown,clocks_event_reasons.sw_power_cap")

    def _start_smi(self):
        import subprocess
        import tempfile
        self.smi_file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.smi = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.SMI_FIELDS}",
                                         "--format=csv,noheader,nounits", "-lms", "10"], stdout=self.smi_file,
                                        stderr=subprocess.DEVNULL)
        except Exception as e:
            self.smi, self.err = None, self.err + "; " + repr(e)
            return
        # nvidia-smi takes a moment to start: begin timing once it samples
        t0 = time.time()
        while time.time() - t0 < 5.0 and os.path.getsize(self.smi_file.name) == 0:
            time.sleep(0.05)

    def _stop_smi(self):
        self.smi.terminate()
        try:
            self.smi.wait(timeout=5)
        except Exception:
            self.smi.kill()
        self.smi_file.seek(0)
        sm, mx, pw, reasons = [], [], [], set()
        for line in self.smi_file:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
                pw.append(float(parts[2]))
            except ValueError:
                continue
            for (name, _, _), v in zip(self.REASONS, parts[3:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        self.smi_file.close()
        os.unlink(self.smi_file.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm), "power_w_max": max(pw) if pw else None,
                "source": "nvidia-smi -lms 10"}

    def stop(self):
        if self.thread is None:
            if getattr(self, "smi", None) is not None:
                return self._stop_smi()
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [f"no clock source: {getattr(self, 'err', '')}"]}
        self.stop_flag.set()
        self.thread.join()
        reasons = set()
        for _, _, bits in self.samples:
            for name, const, default in self.REASONS:
                if bits & getattr(self.nv, const, default):
                    reasons.add(name)
        sm = [c for c, _, _ in self.samples]
        pw = [w for _, w, _ in self.samples]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": round(max(pw), 1) if pw else None, "source": "nvml"}


def max_over_ranks(values, device=None):
    """Elementwise maximum of a list of floats over every rank of the process
    group (the step time of a multi-GPU run is its slowest rank's); a plain
    copy when there is one process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


# --------------------------------------------------------------------------- our arm
class Step:
    """Device state of one canvas step (attention + sampler)."""

    def __init__(self, device):
        import torch
        import canvas_denoising_step_03_b300 as cv
        self.cv, self.torch = cv, torch
        self.acfg, self.scfg = wl.GLOBAL, wl.FULL_SAMPLE
        a = wl.make_attention_inputs(self.acfg)
        s = wl.make_sample_inputs(self.scfg)
        self.a_in, self.s_in = a, s
        dev = device

        def d16(x):
            return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev).view(torch.bfloat16)

        c = self.acfg
        self.x = d16(a.x)
        self.W_q, self.W_k = d16(a.W_q), d16(a.W_k)
        self.gq = torch.from_numpy(a.gamma_q).to(dev)
        self.gk = torch.from_numpy(a.gamma_k).to(dev)
        self.freq = torch.from_numpy(a.freq).to(dev)
        table, npages = wl.page_layout(c)
        self.table = torch.from_numpy(table).to(dev)
        self.pool = d16(wl.scatter_pages(a.cache_k, table, npages, c.page_tokens))
        self.kv = cv.make_kv_cache(self.pool, None, self.table, c.page_tokens)
        self.prefix = torch.from_numpy(a.prefix_len).to(dev)
        self.out = torch.empty((c.B, c.C, c.Hq * c.d), dtype=torch.bfloat16, device=dev)
        self.aws = cv.workspace(cv.canvas_attention_workspace_size(cv.CANVAS_BF16, c.B, c.C, c.D, c.Hq, c.Hkv, c.d,
                                                                   c.max_prefix, cv.CANVAS_LAYER_GLOBAL), dev)
        sc = self.scfg
        self.logits = d16(s.logits)
        self.E = d16(s.E)
        R = sc.rows
        self.tokens = torch.empty(R, dtype=torch.int32, device=dev)
        self.mask = torch.empty(R, dtype=torch.uint8, device=dev)
        self.ent = torch.empty(R, dtype=torch.float32, device=dev)
        self.conf = torch.empty(R, dtype=torch.float32, device=dev)
        self.soft = torch.empty((R, sc.D), dtype=torch.float32, device=dev)
        self.sws = cv.workspace(cv.canvas_sample_workspace_size(cv.CANVAS_BF16, R, sc.V, sc.D), dev)
        self.flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def run(self, step_idx: int = 0, x=None, logits=None):
        cv, c, sc = self.cv, self.acfg, self.scfg
        cv.canvas_attention(self.x if x is None else x, self.W_q, self.W_k, None, c.Hq, c.Hkv, c.d, self.gq,
                            self.gk, c.eps, self.freq, cv.CANVAS_LAYER_GLOBAL, self.kv, self.prefix, c.max_prefix,
                            0, 1.0, 0, self.out, None, self.aws)
        cv.canvas_sample(self.logits if logits is None else logits, self.E, sc.bound, sc.seed, step_idx, 1.0, 0,
                         sc.C, None, None, self.tokens, self.mask, self.ent, self.conf, None, None, cv.CANVAS_BF16,
                         self.soft, self.sws)

    def flush_l2(self):
        self.flush.fill_(1.0)


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    if rank == 0:
        import __graft_entry__
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    import canvas_denoising_step_03_b300 as cv
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    st = Step(dev)
    stream = torch.cuda.current_stream()
    ids = [cv.CANVAS_KERNEL_PREP, cv.CANVAS_KERNEL_ATTENTION, cv.CANVAS_KERNEL_SAMPLER, cv.CANVAS_KERNEL_SOFT_EMB]
    names = {cv.CANVAS_KERNEL_PREP: "attention_prep", cv.CANVAS_KERNEL_ATTENTION: "attention_core",
             cv.CANVAS_KERNEL_SAMPLER: "sampler", cv.CANVAS_KERNEL_SOFT_EMB: "soft_emb_gemm"}

    for w in range(args.warmup):
        st.flush_l2()
        st.run(w)
    assert cv.canvas_device_status() == cv.CANVAS_OK, cv.canvas_last_error()

    # per-step, per-kernel events
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in ids]
          for _ in range(args.steps)]
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for row in ev:  # materialise the event handles
        for a, b in row:
            a.record(); b.record()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    launches0 = cv.canvas_kernel_launches()
    t0 = time.perf_counter()
    for k in range(args.steps):
        st.flush_l2()  # outside the step's events
        for kid, (a, b) in zip(ids, ev[k]):
            cv.canvas_profile_events(kid, a, b)
        step_ev[k][0].record(stream)
        st.run(args.warmup + k)
        step_ev[k][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    launches = cv.canvas_kernel_launches() - launches0
    clk = clocks.stop()
    for kid in ids:
        cv.canvas_profile_events(kid, None, None)
    if world > 1:
        dist.barrier()
    status = cv.canvas_device_status()
    assert status == cv.CANVAS_OK, cv.canvas_last_error()
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    kern_ms = {names[kid]: statistics.median(ev[k][j][0].elapsed_time(ev[k][j][1]) for k in range(args.steps))
               for j, kid in enumerate(ids)}
    ms = max_over_ranks([statistics.median(step_ms)], dev)[0]

    # ---- end to end: host inputs (pinned) -> device, results -> host, every step
    x_h = torch.empty(st.x.shape, dtype=torch.bfloat16).pin_memory()
    lg_h = torch.empty(st.logits.shape, dtype=torch.bfloat16).pin_memory()
    x_h.copy_(st.x.cpu())
    lg_h.copy_(st.logits.cpu())
    x_d = torch.empty_like(st.x)
    lg_d = torch.empty_like(st.logits)
    outs = [st.out, st.tokens, st.mask, st.ent, st.conf, st.soft]
    outs_h = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    h2d = x_h.numel() * 2 + lg_h.numel() * 2
    d2h = sum(o.numel() * o.element_size() for o in outs)
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for w in range(2):
        x_d.copy_(x_h, non_blocking=True)
        lg_d.copy_(lg_h, non_blocking=True)
        st.run(w, x_d, lg_d)
        for o, oh in zip(outs, outs_h):
            oh.copy_(o, non_blocking=True)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    for k in range(args.steps):
        st.flush_l2()
        e2e_ev[k][0].record(stream)
        x_d.copy_(x_h, non_blocking=True)
        lg_d.copy_(lg_h, non_blocking=True)
        st.run(k, x_d, lg_d)
        for o, oh in zip(outs, outs_h):
            oh.copy_(o, non_blocking=True)
        e2e_ev[k][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks([statistics.median(a.elapsed_time(b) for a, b in e2e_ev)], dev)[0]
    assert cv.canvas_device_status() == cv.CANVAS_OK

    if rank != 0:
        return None
    hbm, bf16, peak_src = measured_peaks()
    af = attn_flops(st.acfg)
    att_tflops = af / (kern_ms["attention_core"] * 1e-3) / 1e12
    samp_gbs = sampler_bytes(st.scfg) / (kern_ms["sampler"] * 1e-3) / 1e9
    se_gbs = soft_emb_bytes(st.scfg) / (kern_ms["soft_emb_gemm"] * 1e-3) / 1e9
    dominant = max(("attention_core", "soft_emb_gemm", "sampler"), key=lambda n: kern_ms[n])
    if dominant == "attention_core":
        roof = {"kernel": "attention_core", "bound": "tensor", "achieved": round(att_tflops, 2), "peak": bf16,
                "unit": "TFLOP/s", "frac": round(att_tflops / bf16, 4),
                "algorithmic": f"{af:.4g} FLOP per launch (4*d per visible query-key pair per head)"}
    elif dominant == "soft_emb_gemm":
        roof = {"kernel": "soft_emb_gemm", "bound": "hbm", "achieved": round(se_gbs, 1), "peak": hbm,
                "unit": "GB/s", "frac": round(se_gbs / hbm, 4),
                "algorithmic": f"{soft_emb_bytes(st.scfg):.4g} B per launch (E + P read once, soft_emb written)"}
    else:
        roof = {"kernel": "sampler", "bound": "hbm", "achieved": round(samp_gbs, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(samp_gbs / hbm, 4),
                "algorithmic": f"{sampler_bytes(st.scfg):.4g} B per launch (logits read, bf16 probs written)"}
    roof["peak_source"] = f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'recipe fallback'}, burst)"
    roof["traffic"] = load_traffic(roof["kernel"])
    line = {
        "metric": METRIC,
        "value": round(world * 1000.0 / ms, 3),
        "unit": "canvas steps/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded draws; random weights and caches; no dataset)",
        "config": {"workload": WORKLOAD, "l2": "flushed between timed steps (252 MB write, outside the step events)",
                   "parallelism": f"replicas x{world} (independent canvases per GPU)"},
        "attention_tflops": round(att_tflops, 2),
        "sampler_hbm_gbs": round(samp_gbs, 1),
        "soft_emb_hbm_gbs": round(se_gbs, 1),
        "kernel_ms": {k: round(v, 4) for k, v in kern_ms.items()},
        "roofline": roof,
        "e2e": {"value": round(world * 1000.0 / e2e_ms, 3), "unit": "canvas steps/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": int(launches),
        "clocks": clk,
        "wall_s_timed_region": round(wall, 4),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(st.a_in, st.s_in)
    return line


# --------------------------------------------------------------------------- one sliding-window layer
SLIDING_WORKLOAD = ("sliding-window layer: canvas_attention B=1 C=256 prefix=4096 D=2816 Hq=16 Hkv=8 d=256 "
                    "window 1024 (full RoPE theta 1e4, paged bf16 cache of final keys and values, page 64)")


def run_sliding(args, rank, world, local_rank):
    """canvas_attention on the sliding-window layer workload: the call's rate,
    and the attention core (kernel + KV-split combine) against the bf16 peak."""
    import torch
    import torch.distributed as dist
    if rank == 0:
        import __graft_entry__
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    import canvas_denoising_step_03_b300 as cv
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    c = wl.SLIDING
    a = wl.make_attention_inputs(c)

    def d16(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev).view(torch.bfloat16)

    x, W_q, W_k, W_v = d16(a.x), d16(a.W_q), d16(a.W_k), d16(a.W_v)
    gq, gk, freq = (torch.from_numpy(t).to(dev) for t in (a.gamma_q, a.gamma_k, a.freq))
    table, npages = wl.page_layout(c)
    bt = torch.from_numpy(table).to(dev)
    kp = d16(wl.scatter_pages(a.cache_k, table, npages, c.page_tokens))
    vp = d16(wl.scatter_pages(a.cache_v, table, npages, c.page_tokens))
    kv = cv.make_kv_cache(kp, vp, bt, c.page_tokens)
    prefix = torch.from_numpy(a.prefix_len).to(dev)
    out = torch.empty((c.B, c.C, c.Hq * c.d), dtype=torch.bfloat16, device=dev)
    ws = cv.workspace(cv.canvas_attention_workspace_size(cv.CANVAS_BF16, c.B, c.C, c.D, c.Hq, c.Hkv, c.d,
                                                         c.max_prefix, cv.CANVAS_LAYER_SLIDING), dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def call(xin):
        cv.canvas_attention(xin, W_q, W_k, W_v, c.Hq, c.Hkv, c.d, gq, gk, c.eps, freq, cv.CANVAS_LAYER_SLIDING, kv,
                            prefix, c.max_prefix, c.window, 1.0, 0, out, None, ws)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        call(x)
    assert cv.canvas_device_status() == cv.CANVAS_OK, cv.canvas_last_error()
    ids = [cv.CANVAS_KERNEL_PREP, cv.CANVAS_KERNEL_ATTENTION]
    names = {cv.CANVAS_KERNEL_PREP: "attention_prep", cv.CANVAS_KERNEL_ATTENTION: "attention_core"}
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in ids]
          for _ in range(args.steps)]
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for row in ev:  # materialise the event handles (a torch event exists once recorded)
        for e0, e1 in row:
            e0.record()
            e1.record()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    launches0 = cv.canvas_kernel_launches()
    for k in range(args.steps):
        flush.fill_(1.0)
        for kid, (e0, e1) in zip(ids, ev[k]):
            cv.canvas_profile_events(kid, e0, e1)
        step_ev[k][0].record(stream)
        call(x)
        step_ev[k][1].record(stream)
    torch.cuda.synchronize()
    launches = cv.canvas_kernel_launches() - launches0
    clk = clocks.stop()
    for kid in ids:
        cv.canvas_profile_events(kid, None, None)
    assert cv.canvas_device_status() == cv.CANVAS_OK, cv.canvas_last_error()
    kern_ms = {names[kid]: statistics.median(ev[k][j][0].elapsed_time(ev[k][j][1]) for k in range(args.steps))
               for j, kid in enumerate(ids)}
    ms = max_over_ranks([statistics.median(e0.elapsed_time(e1) for e0, e1 in step_ev)], dev)[0]
    # end to end: x from pinned host memory in, the layer output out, every step
    x_h = torch.empty(x.shape, dtype=torch.bfloat16).pin_memory()
    x_h.copy_(x.cpu())
    out_h = torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()
    x_d = torch.empty_like(x)
    e2e = []
    for k in range(args.warmup + args.steps):
        flush.fill_(1.0)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        x_d.copy_(x_h, non_blocking=True)
        call(x_d)
        out_h.copy_(out, non_blocking=True)
        e1.record(stream)
        if k >= args.warmup:
            e2e.append((e0, e1))
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks([statistics.median(e0.elapsed_time(e1) for e0, e1 in e2e)], dev)[0]
    if rank != 0:
        return None
    hbm, bf16, peak_src = measured_peaks()
    af = attn_flops(c)
    tfl = af / (kern_ms["attention_core"] * 1e-3) / 1e12
    return {
        "metric": METRIC, "value": round(world * 1000.0 / ms, 3), "unit": "sliding-layer canvas_attention calls/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded draws; random weights and caches; no dataset)",
        "config": {"workload": SLIDING_WORKLOAD,
                   "l2": "flushed between timed calls (252 MB write, outside the call's events)",
                   "parallelism": f"replicas x{world}"},
        "attention_tflops": round(tfl, 2),
        "kernel_ms": {k: round(v, 4) for k, v in kern_ms.items()},
        "roofline": {"kernel": "attention_core", "bound": "tensor", "achieved": round(tfl, 2), "peak": bf16,
                     "unit": "TFLOP/s", "frac": round(tfl / bf16, 4), "traffic": None,
                     "algorithmic": f"{af:.4g} FLOP per launch (4*d per visible query-key pair per head)",
                     "peak_source": f"{peak_src} (burst)"},
        "e2e": {"value": round(world * 1000.0 / e2e_ms, 3), "unit": "sliding-layer canvas_attention calls/s",
                "h2d_bytes_per_step": int(x_h.numel() * 2), "d2h_bytes_per_step": int(out_h.numel() * 2)},
        "gpu_launches": int(launches),
        "clocks": clk,
        "cpu_baseline": None,
    }


# --------------------------------------------------------------------------- mixture of experts
MOE_WORKLOAD = ("mixture-of-experts block: canvas_moe R=1024 tokens (4 canvases x 256) D=2816, 128 experts "
                "(top-8) of width 704 + 1 shared expert of width 704, gated GELU, random bf16 weights")


def run_moe(args, rank, world, local_rank):
    """canvas_moe on R = 1024 tokens with the pages' routing shape (128 experts,
    8 active + 1 shared): calls/s, the GEMM rate, and weight streaming against
    HBM (each expert's weights are read once per call for the few dozen tokens
    routed to it, so the call is bound by memory, not the tensor cores)."""
    import torch
    import torch.distributed as dist
    if rank == 0:
        import __graft_entry__
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    import canvas_denoising_step_03_b300 as cv
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    R, D, E, F, k, Fs = 1024, 2816, 128, 704, 8, 704
    gen = torch.Generator(device=dev).manual_seed(17)

    def w(*shape, std):
        return (torch.randn(*shape, device=dev, generator=gen) * std).to(torch.bfloat16)

    x = w(R, D, std=1.0)
    router = w(E, D, std=D ** -0.5)
    Wg, Wu = w(E * F, D, std=D ** -0.5), w(E * F, D, std=D ** -0.5)
    Wd = w(E * D, F, std=F ** -0.5)
    Sg, Su, Sd = w(Fs, D, std=D ** -0.5), w(Fs, D, std=D ** -0.5), w(D, Fs, std=Fs ** -0.5)
    out = torch.empty((R, D), device=dev)
    ws = cv.workspace(cv.canvas_moe_workspace_size(R, D, E, F, k, Fs), dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def call(xin):
        cv.canvas_moe(xin, router, k, None, Wg, Wu, Wd, Sg, Su, Sd, out, None, None, ws)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        call(x)
    assert cv.canvas_device_status() == cv.CANVAS_OK, cv.canvas_last_error()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    launches0 = cv.canvas_kernel_launches()
    for e0, e1 in evs:
        flush.fill_(1.0)
        e0.record(stream)
        call(x)
        e1.record(stream)
    torch.cuda.synchronize()
    launches = cv.canvas_kernel_launches() - launches0
    clk = clocks.stop()
    assert cv.canvas_device_status() == cv.CANVAS_OK, cv.canvas_last_error()
    ms = max_over_ranks([statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)], dev)[0]
    # end to end: tokens from pinned host memory in, the block's output out
    x_h = torch.empty(x.shape, dtype=torch.bfloat16).pin_memory()
    x_h.copy_(x.cpu())
    out_h = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    x_d = torch.empty_like(x)
    e2e = []
    for i in range(args.warmup + args.steps):
        flush.fill_(1.0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        x_d.copy_(x_h, non_blocking=True)
        call(x_d)
        out_h.copy_(out, non_blocking=True)
        e1.record(stream)
        if i >= args.warmup:
            e2e.append((e0, e1))
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks([statistics.median(e0.elapsed_time(e1) for e0, e1 in e2e)], dev)[0]
    if rank != 0:
        return None
    hbm, bf16, peak_src = measured_peaks()
    flops = 2.0 * R * D * E + 3 * 2.0 * R * k * D * F + 3 * 2.0 * R * D * Fs
    wbytes = 2.0 * (E * D + 3 * E * F * D + 3 * Fs * D)
    gbs = wbytes / (ms * 1e-3) / 1e9
    return {
        "metric": METRIC, "value": round(world * 1000.0 / ms, 3), "unit": "moe block calls/s (1024 tokens)",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded random weights and tokens; no dataset)",
        "config": {"workload": MOE_WORKLOAD, "l2": "flushed between timed calls (252 MB write)",
                   "parallelism": f"replicas x{world}"},
        "tflops": round(flops / (ms * 1e-3) / 1e12, 2),
        "roofline": {"kernel": "canvas_moe call (router, grouped expert GEMMs, shared expert)", "bound": "hbm",
                     "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4),
                     "traffic": None, "algorithmic": f"{wbytes:.4g} B of weights per call, each read once",
                     "peak_source": f"{peak_src}"},
        "e2e": {"value": round(world * 1000.0 / e2e_ms, 3), "unit": "moe block calls/s (1024 tokens)",
                "h2d_bytes_per_step": int(x_h.numel() * 2), "d2h_bytes_per_step": int(out_h.numel() * 4)},
        "gpu_launches": int(launches),
        "clocks": clk,
        "cpu_baseline": None,
    }


# --------------------------------------------------------------------------- the batched loop
def run_loop(args, rank, world, local_rank):
    """Steps of the batched denoising loop (canvas_denoising_step_03_b300.loop):
    per step, 6 attention layers + the sampler (the metric's attn+sampler
    time, from CUDA events around those calls) and the whole step with its
    glue (embedding, W_o, LM head)."""
    import torch
    import torch.distributed as dist
    if rank == 0:
        import __graft_entry__
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    import canvas_denoising_step_03_b300 as cv
    from canvas_denoising_step_03_b300.loop import CanvasLoop
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    cfg = wl.loop_config(args.prefix, steps=args.warmup + args.steps)
    run = CanvasLoop(wl.make_loop_inputs(cfg), device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        run.step()
    torch.cuda.synchronize()
    assert cv.canvas_device_status() == cv.CANVAS_OK, cv.canvas_last_error()
    nl = len(run.layers)

    def new_ev():
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        return e
    rec = []
    clocks = ClockSampler(local_rank)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    launches0 = cv.canvas_kernel_launches()
    for k in range(args.steps):
        marks = []
        t0 = new_ev()
        run.step(mark=lambda name: marks.append((name, new_ev())))
        rec.append((t0, new_ev(), marks))
    torch.cuda.synchronize()
    launches = cv.canvas_kernel_launches() - launches0
    clk = clocks.stop()
    assert cv.canvas_device_status() == cv.CANVAS_OK, cv.canvas_last_error()
    step_ms, attn_ms, samp_ms, layer_ms = [], [], [], [[] for _ in range(nl)]
    for t0, t1, marks in rec:
        step_ms.append(t0.elapsed_time(t1))
        a = [m for m in marks if m[0].startswith("attention")]
        per = [a[2 * j][1].elapsed_time(a[2 * j + 1][1]) for j in range(nl)]
        for j in range(nl):
            layer_ms[j].append(per[j])
        attn_ms.append(sum(per))
        sm = {n: e for n, e in marks if n.startswith("sample")}
        samp_ms.append(sm["sample_begin"].elapsed_time(sm["sample_end"]))
    ms_core, ms_step = max_over_ranks([statistics.median(a + s_ for a, s_ in zip(attn_ms, samp_ms)),
                                       statistics.median(step_ms)], dev)
    # end to end: the step's result (tokens, commit mask) read back to pinned
    # host memory inside every timed step
    tok_h = torch.empty(run.tokens.shape, dtype=run.tokens.dtype).pin_memory()
    mask_h = torch.empty(run.mask.shape, dtype=run.mask.dtype).pin_memory()
    e2e = []
    for k in range(args.steps):
        t0 = new_ev()
        run.step()
        tok_h.copy_(run.tokens, non_blocking=True)
        mask_h.copy_(run.mask, non_blocking=True)
        e2e.append((t0, new_ev()))
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks([statistics.median(a.elapsed_time(b) for a, b in e2e)], dev)[0]
    if rank != 0:
        return None
    lcs = cfg.layer_cfgs()
    flops = [attn_flops(lc) for lc in lcs]
    layer_mean = [statistics.median(v) for v in layer_ms]
    g = nl - 1  # the global layer
    hbm, bf16, peak_src = measured_peaks()
    g_tflops = flops[g] / (layer_mean[g] * 1e-3) / 1e12
    return {
        "metric": METRIC, "value": round(world * 1000.0 / ms_core, 3), "unit": "canvas steps/s (attn+sampler)",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_core, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded draws; random weights and caches; no dataset)",
        "config": {"workload": f"batched loop: B={cfg.B} canvases x C={cfg.C}, committed prefix {cfg.prefix}, "
                               f"{cfg.n_sliding} sliding (d=256, window 1024) + {cfg.n_global} global (d=512) "
                               f"layers, D={cfg.D}, V={cfg.V}, tied LM head, self-conditioning input",
                   "l2": "not flushed: every step reads E (1.48 GB) and 1024 x 262144 logits, far above L2",
                   "parallelism": f"replicas x{world}"},
        "loop_steps_per_s": round(world * 1000.0 / ms_step, 3),
        "loop_ms_per_step": round(ms_step, 4),
        "attention_ms_per_layer": [round(v, 4) for v in layer_mean],
        "attention_tflops_per_layer": [round(f / (m * 1e-3) / 1e12, 1) for f, m in zip(flops, layer_mean)],
        "sampler_ms": round(statistics.median(samp_ms), 4),
        "roofline": {"kernel": "global-layer canvas_attention call (projections, key preparation, attention)",
                     "bound": "tensor", "achieved": round(g_tflops, 2), "peak": bf16, "unit": "TFLOP/s",
                     "frac": round(g_tflops / bf16, 4), "traffic": None,
                     "algorithmic": f"{flops[g]:.4g} FLOP per call (4*d per visible query-key pair per head)",
                     "peak_source": f"{peak_src}, burst"},
        "e2e": {"value": round(world * 1000.0 / e2e_ms, 3), "unit": "loop steps/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": int(tok_h.numel() * 4 + mask_h.numel()),
                "note": "the loop's inputs are the previous step's device state; tokens and commit mask read back "
                        "every step"},
        "gpu_launches": int(launches),
        "clocks": clk,
        "cpu_baseline": None,
    }


def load_traffic(kernel: str):
    """dram bytes per launch from the committed ncu summary of this kernel, if any."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh)
    return d.get(kernel)


# --------------------------------------------------------------------------- oracle timings
def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        return max((i.get("num_threads", 1) for i in info), default=1)
    except Exception:
        return os.cpu_count()


def cpu_baseline(a_in, s_in):
    """The oracle's whole step, extrapolated from one timing of every piece
    (OracleClock), on this host's cores."""
    clock = OracleClock(a_in, s_in)
    t0 = time.perf_counter()
    for i, piece in enumerate(clock.pieces):
        clock.run(piece, i)
    spent = time.perf_counter() - t0
    return {"value": round(1.0 / clock.estimate(), 6), "unit": "canvas steps/s", "cores": blas_threads(),
            "kind": "oracle", "sample": clock.describe(rotating=False), "cpu_seconds_spent": round(spent, 2),
            "host_cpus": len(os.sched_getaffinity(0))}


class OracleClock:
    """Times the fp64 oracle's step in bounded pieces and extrapolates the
    whole step from the latest time of each piece: the attention call for one
    query row (it includes the projections and every key transform) and for
    1 + R rows (the difference is R rows' cost), the sampler statistics and
    decision of one position, and that position's soft embedding over one
    16384-entry slice of E.  Inputs are converted to fp64 outside every
    timed piece; only the oracle's own arithmetic is timed."""

    CHUNK = 16384
    R = 16

    def __init__(self, a_in, s_in):
        c = a_in.cfg
        f = lambda x: None if x is None else wl.as_f64(x, c.dtype)  # noqa: E731
        self.a_in, self.s_in, self.c, self.sc = a_in, s_in, c, s_in.cfg
        self.args = (f(a_in.x), f(a_in.W_q), f(a_in.W_k), f(a_in.W_v), c.Hq, c.Hkv, c.d,
                     a_in.gamma_q.astype(np.float64), a_in.gamma_k.astype(np.float64), c.eps,
                     a_in.freq.astype(np.float64), c.layer, f(a_in.cache_k), f(a_in.cache_v), a_in.prefix_len, c.window)
        self.n_chunks = (self.sc.V + self.CHUNK - 1) // self.CHUNK
        self.t = {}
        self.probs = None
        self.pieces = ["attn1", "attnR", "stats"] + [f"chunk{j}" for j in range(self.n_chunks)]

    def _rows(self, k, n):
        return [(0, (k + j) % self.c.Hq, (37 * (k + j)) % self.c.C) for j in range(n)]

    def run(self, piece, k):
        """Run one piece (k picks the rows / position); returns its seconds."""
        from oracle import attention as oatt
        from oracle import sampler as osamp
        if piece.startswith("attn"):
            rows = self._rows(k, 1 if piece == "attn1" else 1 + self.R)
            t0 = time.perf_counter()
            oatt.canvas_attention(*self.args, storage=self.c.dtype if self.c.dtype == "bf16" else "fp64", rows=rows)
            dt = time.perf_counter() - t0
        elif piece == "stats":
            lg = wl.as_f64(self.s_in.logits[[k % self.sc.rows]], self.sc.dtype)
            t0 = time.perf_counter()
            res = osamp.canvas_sample(lg, None, self.sc.bound, self.sc.seed, 0, canvas_len=self.sc.C,
                                      probs_storage="bf16" if self.sc.dtype == "bf16" else "fp64")
            dt = time.perf_counter() - t0
            self.probs = res["probs"]
        else:
            if self.probs is None:
                self.run("stats", k)
            v0 = int(piece[5:]) * self.CHUNK
            E64 = wl.as_f64(self.s_in.E[v0:v0 + self.CHUNK], self.sc.dtype)
            t0 = time.perf_counter()
            _ = self.probs[:, v0:v0 + self.CHUNK] @ E64
            dt = time.perf_counter() - t0
        self.t[piece] = dt
        return dt

    def estimate(self):
        """Seconds of one whole step from the latest piece times."""
        per_row = max(self.t["attnR"] - self.t["attn1"], 0.0) / self.R
        fixed = max(self.t["attn1"] - per_row, 0.0)
        rows = self.c.B * self.c.C * self.c.Hq
        per_pos = self.t["stats"] + sum(self.t[f"chunk{j}"] for j in range(self.n_chunks))
        return fixed + per_row * rows + per_pos * self.sc.rows

    def describe(self, rotating=True):
        how = "one piece per step in rotation" if rotating else "every piece once"
        return (f"fp64 numpy oracle timed in pieces ({how}): attention with 1 and "
                f"{1 + self.R} query rows (projections and every key transform included), the sampler of one "
                f"position, its soft embedding over one of {self.n_chunks} slices of E; whole step extrapolated "
                f"linearly in query rows ({self.c.B * self.c.C * self.c.Hq}) and positions ({self.sc.rows}) from "
                f"the latest time of every piece")


def run_reference(args, rank, world):
    if rank != 0:
        return None
    clock = OracleClock(wl.make_attention_inputs(wl.GLOBAL), wl.make_sample_inputs(wl.FULL_SAMPLE))
    for i, piece in enumerate(clock.pieces):  # every piece measured once before the first estimate
        clock.run(piece, i)
    npieces = len(clock.pieces)
    times = []
    for k in range(args.warmup + args.steps):
        clock.run(clock.pieces[k % npieces], k)
        if k >= args.warmup:
            times.append(clock.estimate())
    ms = statistics.median(times) * 1000.0
    v = round(1000.0 / ms, 6)
    cores = blas_threads()
    desc = clock.describe()
    return {"metric": METRIC, "value": v, "unit": "canvas steps/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded draws)", "impl": "reference",
            "config": {"workload": WORKLOAD, "l2": "flushed between timed steps (252 MB write, outside the step events)",
                       "parallelism": f"replicas x{world} (independent canvases per GPU)"},
            "cpu_baseline": {"value": v, "unit": "canvas steps/s", "cores": cores,
                                                              "kind": "oracle", "sample": desc},
            "e2e": {"value": v, "unit": "canvas steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="step", choices=["step", "loop", "sliding", "moe"])
    ap.add_argument("--prefix", type=int, default=1024, help="committed prefix of the loop workload")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    elif args.workload == "loop":
        line = run_loop(args, rank, world, local_rank)
    elif args.workload == "sliding":
        line = run_sliding(args, rank, world, local_rank)
    elif args.workload == "moe":
        line = run_moe(args, rank, world, local_rank)
    else:
        line = run_ours(args, rank, world, local_rank)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
