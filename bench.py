"""Benchmark: quantized KV-cache decode step on GB300.

One step = for every layer of the workload: kvq_append_decode_attn, i.e. the
append of one new token per sequence (quantize / stage / seal) and the split-K
attention over the packed cache, in one launch (the format's fused decode
specialisation; formats without one run kvq_append then kvq_decode_attn).
The default workload is the Llama-2-13B-shaped MHA cache (40 layers, batch
16, 40 heads, head_dim 128, 4096 + 17 cached tokens fp16, keys with 4 fixed
outlier channels per head x15), K 2-bit per-channel G=32 / V 2-bit per-token
G=32 with a 17-token fp16 key tail: the largest workload that fits one GPU.
`--workload` takes any registered workload (every variant of the five
configurations, bit_quantized_kv_02_gb300.synth.WORKLOADS), an alias, a group
(gpt2_sweep, llama2_13b_axes, wide_gqa_all, all) or a comma-separated list;
one JSON line is printed per workload.

The step is captured once as a CUDA graph of the public calls (planned for the
full capacity, so one graph stays valid as the cache grows) and replayed.
Between timed steps a 256 MB buffer is written to flush the 126 MB L2.

  value : algorithmic decode bytes (packed codes + metadata + fp16 tail + q,
          from kvq_decode_traffic) per step / device time of the step, inputs
          already resident in HBM (the step's new tokens and queries are copied
          device-to-device into the graph's input buffers inside the timed region)
  e2e   : same metric with every step's inputs copied from pinned host memory
          and its outputs copied back to pinned host memory inside the timed
          region (the steps enqueued back to back)
  roofline : decode kernel alone; CUDA events on the launching stream around a
          graph of the step's decode launches.  `traffic` is null: the DRAM
          byte counts come from separate ncu captures (see profiles/).
  config.cta_warps : the CTA shape of each graph (four-warp CTAs, or one-warp
          CTAs where the format has them), the faster of the two timed first.
`--phase prefill` times kvq_prefill_quantize instead (fp16 keys and values of
every layer in HBM -> packed codes, metadata and fp16 tails): bytes = fp16
input read + codes, metadata and tail written.
Under torchrun each rank runs its own shard of sequences (weak scaling, no
data-path collective); rank 0 prints the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_quantized_kv_02_gb300 import build as kbuild  # noqa: E402
from bit_quantized_kv_02_gb300 import dist as kdist  # noqa: E402
from bit_quantized_kv_02_gb300 import kvq, synth  # noqa: E402

METRIC = "decode-attn achieved HBM GB/s (% of peak) and cached tokens/s on 1 GB300"
L2_FLUSH_BYTES = 256 << 20
# kvq_set_decode_kernel values of the two CTA shapes the bench chooses between
# (0: four-warp CTAs; 4: one-warp CTAs where the format has them)
CTA_SHAPES = (0, 4)
TUNE_REPS = 2


def workload(name: str, tokens: int = 0) -> synth.Workload:
    wl = synth.workload(name)
    if tokens:
        wl.lens = [min(int(x), tokens) for x in wl.lens]
        wl.name += f"_t{tokens}"
    return wl


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class _Nvml:
    """Read-only NVML queries through ctypes (SM clock, max SM clock, clock
    event reasons) for the clock sampler."""
    SM = 1
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, dev: torch.device):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        ok = False
        try:
            pr = torch.cuda.get_device_properties(dev)
            bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0".encode()
            ok = self.lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(self.h)) == 0
        except Exception:
            ok = False
        if not ok and self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(dev.index or 0), ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle")
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = fn if fn is not None else self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sample(self):
        c = self.c
        sm, mx, rs = c.c_uint(), c.c_uint(), c.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.SM, c.byref(sm)) != 0:
            return None
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.SM, c.byref(mx))
        self.reasons_fn(self.h, c.byref(rs))
        return float(sm.value), float(mx.value), [n for bit, n in self.REASONS.items() if rs.value & bit]


class Clocks:
    """SM clock / clock-event-reason sampler for the timed region: one NVML
    sample from the calling thread once a step is enqueued, while the GPU runs
    it (no sampler thread competing with the host while it enqueues a step
    between its timing events, and no back-to-back driver queries while the
    GPU works), else nvidia-smi every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, dev: torch.device):
        self.proc = None
        self.samples = []
        self.nv = None
        try:
            self.nv = _Nvml(dev)
            self.source = "nvml, one sample while each timed step runs"
            return
        except Exception:
            self.nv = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={dev.index or 0}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi 200 ms"
        except Exception:
            self.proc = None

    def poll(self):
        """One sample from the calling thread (called while the GPU runs a step)."""
        if self.nv is None:
            return
        r = self.nv.sample()
        if r is not None:
            self.samples.append(r)

    def stop(self):
        if self.nv is None and not self.proc:
            return None
        if self.nv is None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in out.strip().splitlines():
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    self.samples.append((float(f[1]), float(f[2]),
                                         [n for n, v in zip(names, f[5:9]) if v.lower().startswith("active")]))
                except ValueError:
                    continue
        if not self.samples:
            return None
        sm = [x[0] for x in self.samples]
        reasons = sorted({r for x in self.samples for r in x[2]})
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(x[1] for x in self.samples)),
                "reasons": reasons, "samples": len(sm), "source": self.source}


def run_ours(args, rank, world, name):
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    wl = workload(name, args.tokens)
    # weak scaling: each rank owns `batch` sequences of its own (its shard of the job)
    B = wl.batch
    L = wl.layers
    steps, warm = args.steps, args.warmup
    e2e_steps = min(steps, max(3, steps // 2))
    tune_steps = 2 * len(CTA_SHAPES) * TUNE_REPS  # fused steps the CTA-shape choice replays
    cap = wl.max_tokens + warm + steps + 2 * e2e_steps + tune_steps + 2
    cfg = kvq.make_config(L, B, wl.q_heads, wl.kv_heads, wl.head_dim, cap, wl.k, wl.v, recent_window=args.window,
                          rope_theta=args.rope)
    cache = kvq.KVQCache(cfg, device=dev)
    cache.kvq_set_decode_plan(cap)
    # prefill every layer from GPU-generated synthetic data (layer by layer)
    for l in range(L):
        k, v = wl.layer_kv(l, dev, T=wl.max_tokens)
        cache.kvq_prefill_quantize(l, k, v, wl.lens)
        del k, v
    torch.cuda.synchronize()
    Hq, H, D = wl.q_heads, wl.kv_heads, wl.head_dim
    nsteps = warm + steps
    # per-step inputs, resident on the device; pinned host copies for e2e
    # a step's inputs (new keys / values of every layer, then the queries) are
    # one contiguous buffer, so each step moves them with one copy
    nk, nq = L * 2 * B * H * D, L * B * Hq * D
    kin_all = torch.stack([torch.stack(wl.step_kv(l, s, dev)) for s in range(nsteps) for l in range(L)])
    q_all = torch.stack([wl.layer_query(l, s, dev) for s in range(nsteps) for l in range(L)])
    inp_all = torch.cat([kin_all.reshape(nsteps, nk), q_all.reshape(nsteps, nq)], dim=1).contiguous()
    del kin_all, q_all
    inp_host = inp_all.cpu().pin_memory()
    # static graph buffers (views of one input buffer; the queries start at a
    # multiple of 128 bytes)
    inp = torch.empty(nk + nq, dtype=wl.dtype, device=dev)
    kin = inp[:nk].view(L, 2, B, H, D)
    qin = inp[nk:].view(L, B, Hq, D)
    out = torch.empty((L, B, Hq, D), dtype=torch.float32, device=dev)
    # pinned host buffers for the end-to-end steps' outputs (one per step)
    out_host = torch.empty((max(e2e_steps, 1),) + tuple(out.shape), dtype=torch.float32).pin_memory()
    scale = float(np.float32(1.0 / np.sqrt(D)))
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())
    inp.copy_(inp_all[0])
    torch.cuda.synchronize()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = None

    def capture(shape):
        """The step graph (per layer the append fused into the decode launch;
        consecutive launches overlap their launch latency through programmatic
        dependent launch, so the graph holds no timing events between them) and
        the decode kernel alone (the step's L decode launches back to back, same
        inputs and cache state), both captured in one CTA shape."""
        cache.kvq_set_decode_kernel(shape)
        g = torch.cuda.CUDAGraph()
        n = 0
        with torch.cuda.graph(g, stream=stream):
            for l in range(L):
                cache.kvq_append_decode_attn(l, kin[l, 0], kin[l, 1], qin[l], out[l], scale, stream=stream)
                n += cache.kvq_last_launches()
        cache.kvq_refresh_lens(stream)  # capturing launched nothing
        gd = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gd, stream=stream):
            for l in range(L):
                cache.kvq_decode_attn(l, qin[l], out[l], scale, stream=stream)
        return g, gd, n

    def timed_replay(g):
        with torch.cuda.stream(stream):
            flush.zero_()
            e0.record(stream)
            g.replay()
            e1.record(stream)
        stream.synchronize()
        return e0.elapsed_time(e1)

    # CTA shape of the decode launches: four-warp CTAs (the library's default)
    # or one-warp CTAs (kvq_set_decode_kernel bit 2, where the format has that
    # specialisation).  Which is faster depends on how the (sequence, head)
    # ranges divide over the SMs, so each graph is timed in both shapes first
    # (after the L2 flush, best of TUNE_REPS) and captured in the faster one.
    # (a shape whose kernels are the default's is not timed twice)
    tuned = {}
    seen = set()
    for shape in CTA_SHAPES:
        cache.kvq_set_decode_kernel(shape)
        warps = (cache.kvq_decode_cta_warps(False), cache.kvq_decode_cta_warps(True))
        if warps in seen:
            continue
        seen.add(warps)
        g, gd, n = capture(shape)
        ts = min(timed_replay(g) for _ in range(TUNE_REPS))
        td = min(timed_replay(gd) for _ in range(TUNE_REPS))
        tuned[shape] = (ts, td, warps)
        del g, gd
    step_shape = min(tuned, key=lambda x: tuned[x][0])
    dec_shape = min(tuned, key=lambda x: tuned[x][1])
    graph, _, launches_per_step = capture(step_shape)
    step_warps = cache.kvq_decode_cta_warps(True) or cache.kvq_decode_cta_warps(False)
    _, graph_dec, _ = capture(dec_shape)
    dec_warps = cache.kvq_decode_cta_warps(False)
    cache.kvq_refresh_lens(stream)

    def traffic():
        cache.kvq_refresh_lens(stream)
        return sum(cache.kvq_decode_traffic(l, kvq.F16) for l in range(L)), \
            sum(sum(cache.kvq_get_lens(l)) for l in range(L))

    def one_step(s):
        with torch.cuda.stream(stream):
            flush.zero_()
            e0.record(stream)
            inp.copy_(inp_all[s], non_blocking=True)
            graph.replay()
            e1.record(stream)
        if clocks:
            clocks.poll()  # the GPU is running the step now
        stream.synchronize()
        return e0.elapsed_time(e1)

    def decode_pass():
        with torch.cuda.stream(stream):
            flush.zero_()
            e0.record(stream)
            graph_dec.replay()
            e1.record(stream)
        if clocks:
            clocks.poll()
        stream.synchronize()
        return e0.elapsed_time(e1)

    # warm-up (untimed)
    for s in range(warm):
        one_step(s)
        decode_pass()
    kdist.barrier()
    clocks = Clocks(dev) if rank == 0 else None
    t_steps, t_decode, tot_bytes, tot_tokens = 0.0, 0.0, 0.0, 0.0
    for s in range(warm, nsteps):
        t_steps += one_step(s)
        by, tk = traffic()
        tot_bytes += by
        tot_tokens += tk
        t_decode += decode_pass()
    clk = clocks.stop() if clocks else None
    clocks = None
    kdist.barrier()
    # materialised baseline (optional): per layer kvq_dequantize into fp16 rows,
    # then decode attention over those rows; timed like the fused decode graph
    mat = None
    if args.materialized:
        shape = (B, H, cache.tcap, D)
        k16 = torch.zeros(shape, dtype=torch.float16, device=dev)
        v16 = torch.zeros(shape, dtype=torch.float16, device=dev)
        out_m = torch.empty_like(out)
        graph_mat = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_mat, stream=stream):
            for l in range(L):
                cache.kvq_dequantize(l, k16, v16, stream=stream)
                cache.kvq_decode_attn_materialized(l, k16, v16, qin[l], out_m[l], scale, stream=stream)
        t_mat = []
        for r in range(warm + steps):
            with torch.cuda.stream(stream):
                flush.zero_()
                e0.record(stream)
                graph_mat.replay()
                e1.record(stream)
            stream.synchronize()
            if r >= warm:
                t_mat.append(e0.elapsed_time(e1))
        fused_ms = t_decode / steps
        mat_ms = float(np.mean(t_mat))
        diff = (out_m - out).abs().max().item() / max(out.abs().max().item(), 1e-30)
        mat = {"ms_per_step": round(mat_ms, 4), "fused_decode_ms_per_step": round(fused_ms, 4),
               "fused_speedup": round(mat_ms / fused_ms, 2), "max_rel_diff_vs_fused": diff,
               "path": "per layer: kvq_dequantize (packed -> fp16 rows) + kvq_decode_attn_materialized",
               "fp16_bytes_written_and_read_per_layer": 2 * 2 * sum(wl.lens) * H * D * 2}
        del k16, v16
    # End to end: every step copies its inputs from pinned host memory to the
    # device, replays the step graph and copies its outputs back into a pinned
    # host buffer of its own.  The steps are enqueued back to back between one
    # pair of events, so the GPU runs them in order while the host enqueues the
    # next one: a host-side stall while a copy is being enqueued (measured: now
    # and then 1.5 ms, when each step sat between its own events) does not
    # count as GPU time.  The cache is far larger than L2, so no flush between
    # the steps.  The sequence runs once untimed first (the first copies from
    # and to pinned buffers in a process cost extra).
    t_e2e, by_e2e = 0.0, 0.0
    if e2e_steps:
        for timed in (False, True):
            by0 = traffic()[0]
            with torch.cuda.stream(stream):
                flush.zero_()
                e0.record(stream)
                for s in range(e2e_steps):
                    inp.copy_(inp_host[warm + s], non_blocking=True)
                    graph.replay()
                    out_host[s].copy_(out, non_blocking=True)
                e1.record(stream)
            stream.synchronize()
            t_e2e = e0.elapsed_time(e1)
            by_e2e = 0.5 * (by0 + traffic()[0]) * e2e_steps
    # correctness guard: the device reported no timed-out wait
    st = cache.kvq_device_status(stream)
    if st != 0:
        raise SystemExit(f"device status {kvq.STATUS.get(st, st)}")

    t_max = kdist.max_over_ranks(t_steps, device=dev)
    bytes_all = kdist.sum_over_ranks(tot_bytes, device=dev)
    tokens_all = kdist.sum_over_ranks(tot_tokens, device=dev)
    t_e2e_max = kdist.max_over_ranks(t_e2e, device=dev)
    bytes_e2e_all = kdist.sum_over_ranks(by_e2e, device=dev)
    peak, peak_kind = measured_peaks()
    res = None
    if rank == 0:
        value = bytes_all / (t_max * 1e-3) / 1e9
        dec_bytes_per_launch = tot_bytes / (steps * L)
        dec_ms_per_launch = t_decode / (steps * L)
        achieved = dec_bytes_per_launch / (dec_ms_per_launch * 1e-3) / 1e9
        h2d = inp.numel() * inp.element_size()
        d2h = out.numel() * out.element_size()
        res = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": steps, "warmup": warm,
            "ms_per_step": round(t_max / steps, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp16 in, 2..8-bit codes, fp32 accumulate", "data": "synthetic",
            "pct_of_peak": round(100.0 * value / peak, 2),
            "cached_tokens_per_s": round(tokens_all / (t_max * 1e-3), 1),
            "config": {"workload": wl.name + (f"_w{args.window}" if args.window else "") +
                       (f"_rope{args.rope:g}" if args.rope else ""), "layers": L, "rope_theta": args.rope,
                       "batch_per_gpu": B, "q_heads": Hq, "kv_heads": H, "recent_window": args.window,
                       "head_dim": D, "cached_tokens": wl.lens[0], "k": list(wl.k), "v": list(wl.v),
                       "k_format": "bits,group,axis(0 per-token,1 per-channel),mode(0 asym,1 sym)",
                       "step": "per layer: kvq_append_decode_attn (append fused into the decode launch; CUDA graph)",
                       "l2": "256 MB buffer written before every timed step (L2 flushed)",
                       "cta_warps": {"step": step_warps, "decode": dec_warps,
                                     "choice": "each graph timed in every CTA shape the format has (best of "
                                               f"{TUNE_REPS} after an L2 flush) before the warm-up; "
                                               "the faster captured",
                                     "ms_step": {tuned[x][2][1] or tuned[x][2][0]: round(tuned[x][0], 4)
                                                 for x in tuned},
                                     "ms_decode": {tuned[x][2][0]: round(tuned[x][1], 4) for x in tuned}},
                       "parallelism": f"dp{world} (sequences sharded, no collective)"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": None,
                         "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                         else "fallback",
                         "kernel": "decode_kernel", "bytes_per_launch": round(dec_bytes_per_launch),
                         "us_per_launch": round(dec_ms_per_launch * 1e3, 3),
                         "timing": "CUDA events on the launching stream around a graph of the step's "
                                   f"{L} decode launches (after an L2 flush), once per timed step",
                         "decode_launches_timed": L * steps},
            "gpu_launches": launches_per_step * steps,
            "e2e": {"value": round(bytes_e2e_all / (t_e2e_max * 1e-3) / 1e9, 2) if e2e_steps else None,
                    "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "path": "per step: pinned host -> device copy of the inputs, graph of kvq_append_decode_attn, "
                            "device -> pinned host copy of the outputs; steps enqueued back to back"},
            "clocks": clk,
        }
        if mat is not None:
            res["materialized"] = mat
    return res, wl


def run_prefill(args, rank, world, name):
    """kvq_prefill_quantize of every layer: fp16 keys and values resident in
    HBM (a few distinct input buffers, each far larger than L2, cycled over
    the layers) -> packed codes, metadata and fp16 tails."""
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    wl = workload(name, args.tokens)
    B, L, H, D = wl.batch, wl.layers, wl.kv_heads, wl.head_dim
    steps, warm = args.steps, args.warmup
    cfg = kvq.make_config(L, B, wl.q_heads, H, D, wl.max_tokens, wl.k, wl.v)
    cache = kvq.KVQCache(cfg, device=dev)
    nin = min(L, 3)
    inputs = [wl.layer_kv(l, dev, T=wl.max_tokens) for l in range(nin)]
    bt = kvq.kvq_cache_bytes(cfg, wl.lens)
    read = 2.0 * sum(wl.lens) * H * D * 2  # fp16 keys and values of every valid token
    written = (bt.packed + bt.metadata + bt.tail) / L
    per_call = read + written
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = 0

    def one_step():
        nonlocal launches
        launches = 0
        with torch.cuda.stream(stream):
            e0.record(stream)
            for l in range(L):
                k, v = inputs[l % nin]
                cache.kvq_prefill_quantize(l, k, v, wl.lens, stream=stream)
                launches += cache.kvq_last_launches()
            e1.record(stream)
        if clocks:
            clocks.poll()  # the GPU is running the layers now
        stream.synchronize()
        return e0.elapsed_time(e1)

    clocks = None
    for _ in range(warm):
        one_step()
    kdist.barrier()
    clocks = Clocks(dev) if rank == 0 else None
    t = 0.0
    for _ in range(steps):
        t += one_step()
    clk = clocks.stop() if clocks else None
    kdist.barrier()
    # end to end: the layer's fp16 inputs copied from pinned host memory inside the timed region
    k_host = [x.cpu().pin_memory() for x in inputs[0]]
    kd, vd = torch.empty_like(inputs[0][0]), torch.empty_like(inputs[0][1])
    e2e_layers = min(L, 4)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for l in range(e2e_layers):
            kd.copy_(k_host[0], non_blocking=True)
            vd.copy_(k_host[1], non_blocking=True)
            cache.kvq_prefill_quantize(l, kd, vd, wl.lens, stream=stream)
        e1.record(stream)
    stream.synchronize()
    t_e2e = e0.elapsed_time(e1)
    t_max = kdist.max_over_ranks(t, device=dev)
    peak, peak_kind = measured_peaks()
    res = None
    if rank == 0:
        value = per_call * L * steps * world / (t_max * 1e-3) / 1e9
        achieved = per_call * L * steps / (t * 1e-3) / 1e9
        res = {
            "metric": "prefill quantize-and-pack achieved HBM GB/s (% of peak) on 1 GB300", "phase": "prefill",
            "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": steps, "warmup": warm,
            "ms_per_step": round(t_max / steps, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp16 in, 2..8-bit codes + fp16 metadata out", "data": "synthetic",
            "pct_of_peak": round(100.0 * value / peak, 2),
            "tokens_per_s": round(sum(wl.lens) * L * steps * world / (t_max * 1e-3), 1),
            "config": {"workload": wl.name, "layers": L, "batch_per_gpu": B, "kv_heads": H, "head_dim": D,
                       "cached_tokens": wl.lens[0], "k": list(wl.k), "v": list(wl.v),
                       "step": "kvq_prefill_quantize of every layer (inputs cycled over "
                               f"{nin} resident buffers of {2 * B * wl.max_tokens * H * D * 2 / 1e9:.2f} GB)",
                       "l2": "inputs larger than L2"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": None,
                         "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                         else "fallback",
                         "kernel": "kvq_prefill_quantize (prefill_channel_kernel / prefill_token_kernel per tensor)",
                         "bytes_per_launch": round(per_call), "read_bytes": round(read),
                         "written_bytes": round(written), "us_per_call": round(t / (steps * L) * 1e3, 3)},
            "gpu_launches": launches * steps,
            "e2e": {"value": round(per_call * e2e_layers / (t_e2e * 1e-3) / 1e9, 2), "unit": "GB/s",
                    "h2d_bytes_per_step": 2 * inputs[0][0].numel() * 2 * e2e_layers, "d2h_bytes_per_step": 0,
                    "layers": e2e_layers, "path": "pinned host -> device copy of the layer's keys and values, "
                                                  "kvq_prefill_quantize"},
            "clocks": clk,
        }
    return res, wl


def cpu_quantize_sample(wl, seconds=5.0):
    """The oracle's quantizer on one (layer, sequence) sample, repeated for
    about `seconds`: GB/s of the prefill path's algorithmic bytes."""
    import oracle

    D, H = wl.head_dim, wl.kv_heads
    n = wl.lens[0]
    k, v = wl.layer_kv(0, "cpu", T=n)
    k, v = k[:1].float().numpy(), v[:1].float().numpy()
    lens = np.array([n], np.int32)
    pk, mk, tk = oracle.tensor_bytes(1, H, D, lens, wl.k[0], wl.k[1], wl.k[2], bool(wl.k[3]))
    pv, mv, tv = oracle.tensor_bytes(1, H, D, lens, wl.v[0], wl.v[1], wl.v[2], bool(wl.v[3]))
    sample_bytes = 2.0 * n * H * D * 2 + pk + mk + tk + pv + mv + tv
    t0 = time.perf_counter()
    count = 0
    while True:
        oracle.quantize_tensor(k, lens, n + (-n) % 128, *wl.k[:3], sym=bool(wl.k[3]))
        oracle.quantize_tensor(v, lens, n + (-n) % 128, *wl.v[:3], sym=bool(wl.v[3]))
        count += 1
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    return {"value": round(sample_bytes * count / el / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{count} x (one layer, one sequence: {n} tokens x {H} kv heads x {D}; quantize keys and "
                      f"values), 1 thread, {el:.1f} s"}


def cpu_oracle_sample(wl, seconds=10.0, max_samples=64, threads=1):
    """Time the CPU oracle (dequantize + fp64 attention) on (layer, sequence)
    samples of the workload until `seconds` have elapsed, on `threads` host
    threads (each runs whole samples; the oracle's C routines release the GIL).
    Returns (GB/s of the path's algorithmic decode bytes, description, seconds
    per sample per thread)."""
    import concurrent.futures as cf

    import oracle

    D, H, Hq = wl.head_dim, wl.kv_heads, wl.q_heads
    n = wl.lens[0]
    k, v = wl.layer_kv(0, "cpu", T=n)
    k, v = k[:1].contiguous(), v[:1].contiguous()
    lens = np.array([n], np.int32)
    q = wl.layer_query(0)[:1].float().numpy()
    ok = oracle.quantize_tensor(k.float().numpy(), lens, n + (-n) % 128, *wl.k[:3], sym=bool(wl.k[3]))
    ov = oracle.quantize_tensor(v.float().numpy(), lens, n + (-n) % 128, *wl.v[:3], sym=bool(wl.v[3]))
    pk, mk, tk = oracle.tensor_bytes(1, H, D, lens, wl.k[0], wl.k[1], wl.k[2], bool(wl.k[3]))
    pv, mv, tv = oracle.tensor_bytes(1, H, D, lens, wl.v[0], wl.v[1], wl.v[2], bool(wl.v[3]))
    sample_bytes = pk + mk + tk + pv + mv + tv + Hq * D * 2
    scale = np.float32(1.0 / np.sqrt(D))
    per_thread = max(1, max_samples // threads) if threads > 1 else max_samples

    def worker():
        t0 = time.perf_counter()
        count = 0
        while True:
            kh = oracle.dequant_tensor(ok, lens, *wl.k[:3], sym=bool(wl.k[3]))
            vh = oracle.dequant_tensor(ov, lens, *wl.v[:3], sym=bool(wl.v[3]))
            oracle.attention(kh, vh, q, lens, scale)
            count += 1
            if time.perf_counter() - t0 >= seconds or count >= per_thread:
                return count

    t0 = time.perf_counter()
    if threads > 1:
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            count = sum(ex.map(lambda _: worker(), range(threads)))
    else:
        count = worker()
    el = time.perf_counter() - t0
    gbs = sample_bytes * count / el / 1e9
    desc = (f"{count} x (one layer, one sequence: {n} tokens x {H} kv heads x {D}; dequantize + fp64 attention "
            f"for {Hq} query heads), {threads} thread{'s' if threads > 1 else ''}, {el:.1f} s")
    return gbs, desc, el * threads / count


def host_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def cpu_baseline(wl, seconds):
    """The oracle on every host core (the reported baseline) and on one thread."""
    nt = host_threads()
    gbs1, desc1, per1 = cpu_oracle_sample(wl, seconds=seconds / 2, max_samples=1 << 30, threads=1)
    gbs, desc, _ = cpu_oracle_sample(wl, seconds=seconds / 2, max_samples=1 << 30, threads=nt)
    return ({"value": round(gbs, 4), "unit": "GB/s", "cores": nt, "kind": "oracle", "sample": desc,
             "single_thread": {"value": round(gbs1, 4), "unit": "GB/s", "cores": 1, "sample": desc1}}, per1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama2_13b",
                    help="registered workload, alias, group or comma-separated list (one JSON line each)")
    ap.add_argument("--phase", default="decode", choices=["decode", "prefill"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--tokens", type=int, default=0, help="cap the cached tokens per sequence (profiling runs)")
    ap.add_argument("--window", type=int, default=0,
                    help="full-precision recent window of both tensors (multiple of 16; 0 = none)")
    ap.add_argument("--rope", type=float, default=0.0,
                    help="pre-RoPE key cache: rotary base applied to the dequantized keys at decode (0 = none)")
    ap.add_argument("--materialized", action="store_true",
                    help="also time the materialised baseline (dequantize to fp16, then decode) beside the fused path")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, _ = kdist.rank_env()
    if args.impl == "reference":
        # the reference arm is the CPU oracle; under torchrun only rank 0 works
        if rank != 0:
            return
        wl = workload(synth.workload_names(args.workload)[0], args.tokens)
        import oracle
        oracle.build()
        cb, per = cpu_baseline(wl, seconds=max(2.0, min(40.0, args.cpu_seconds * (args.steps + args.warmup) / 25)))
        gbs = cb["value"]
        line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": 1,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per * 1e3, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp64 oracle",
                "data": "synthetic", "config": {"workload": wl.name},
                "cpu_baseline": cb,
                "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return
    kbuild.build()
    kvq.lib()
    if world > 1:
        kdist.init("nccl")
    for name in synth.workload_names(args.workload):
        if args.phase == "prefill":
            res, wl = run_prefill(args, rank, world, name)
        else:
            res, wl = run_ours(args, rank, world, name)
        if rank == 0:
            import oracle
            oracle.build()
            if args.phase == "prefill":
                res["cpu_baseline"] = cpu_quantize_sample(wl, seconds=args.cpu_seconds)
            else:
                res["cpu_baseline"], _ = cpu_baseline(wl, seconds=args.cpu_seconds)
            print(json.dumps(res), flush=True)
        torch.cuda.empty_cache()
    if world > 1:
        kdist.barrier()
        torch.distributed.destroy_process_group()

if __name__ == "__main__":
    main()
