"""Benchmark: paged GQA decode KV GB/s (and varlen prefill TFLOP/s) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one fw_paged_decode call (split-KV attention kernel + combine
kernel) over the Qwen3-14B-shaped workload: batch 64, 40 Q / 8 KV heads,
head_dim 128, 128-token pages, seq_lens uniform in [512, 32768], BF16 ~N(0,1)
in shuffled physical pages.  The KV cache (4.4 GB) is far larger than L2, so
no flush is needed between steps.  `value` is KV bytes read per step divided
by the step time (CUDA events on the launching stream, inputs resident).
The prefill object times fw_varlen_prefill on the causal varlen GQA workload
(16 sequences, lengths uniform in [256, 8192], 32 Q / 8 KV heads, hd 128).

With N > 1 (torchrun, one rank per GPU) every rank runs its own replica of
the workload (no collective on the data path: decode units are independent),
so scaling is weak; the reported time is the max over ranks.

--impl reference times the fp64 CPU oracle (the only other implementation of
this method in the repository) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode KV GB/s (% of HBM peak); prefill TFLOP/s (% of BF16 peak)"
DECODE_WL = "qwen3_14b_paged_decode"
PREFILL_WL = "varlen_gqa_prefill"
PREFILL_HD256_WL = "dense_causal_mha_hd256"
LATENT_WL = "latent_paged_decode"
DECODE_FP8_WL = "qwen3_14b_paged_decode_fp8"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": pk["hbm_gbs"], "bf16_tflops": pk["bf16_tflops"],
                "bf16_tflops_sustained": pk.get("bf16_tflops_sustained", pk["bf16_tflops"]),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def max_over_ranks(dist, values, device):
    """Element-wise maximum of `values` over all ranks (the slowest rank sets
    the time); `dist` is torch.distributed with an initialised group, or None."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(bytes_per_step_per_rank, steps, world, elapsed_ms):
    """Aggregate GB/s over all ranks: every rank processes the same per-step
    bytes (weak scaling), over the slowest rank's time."""
    if not (elapsed_ms == elapsed_ms) or elapsed_ms <= 0:
        return None
    return bytes_per_step_per_rank * steps * world / (elapsed_ms * 1e-3) / 1e9


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during a timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.device = device_index

    def __enter__(self):
        import torch
        target = None
        try:
            uuid = str(torch.cuda.get_device_properties(self.device).uuid)
            target = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            target = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if target:
            cmd += ["-i", target]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        self.samples = []
        if self.proc is None:
            return False
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                self.samples.append({"sm": float(parts[1]), "max": float(parts[2]), "power": float(parts[3]),
                                     "hw_slowdown": parts[5], "hw_thermal": parts[6],
                                     "sw_thermal": parts[7], "sw_power_cap": parts[8]})
            except ValueError:
                continue
        return False

    def summary(self):
        s = getattr(self, "samples", [])
        if not s:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        reasons = set()
        for x in s:
            for key, name in (("hw_slowdown", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power_cap", "sw_power_cap")):
                if x[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(x["sm"] for x in s), "sm_max_mhz": max(x["max"] for x in s),
                "reasons": sorted(reasons), "samples": len(s),
                "power_w_max": max(x["power"] for x in s)}


def source_sha(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "ragged_softmax_attention_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


# Files whose bytes decide each profiled kernel and its launch: a committed ncu
# summary counts only while their hash still matches.
DECODE_SOURCES = ["decode_kernel.cu", "decode_common.cuh", "fw_ptx.cuh", "fw_internal.h", "abi.cu"]
FP8_SOURCES = ["decode_fp8_kernel.cu", "decode_common.cuh", "fw_ptx.cuh", "fw_internal.h", "abi.cu"]
PREFILL_SOURCES = ["prefill_kernel.cu", "fw_pair.cuh", "fw_ptx.cuh", "fw_internal.h", "abi.cu"]
LATENT_SOURCES = ["latent_pair_kernel.cu", "fw_pair.cuh", "fw_ptx.cuh", "decode_common.cuh", "fw_internal.h", "abi.cu"]


def ncu_traffic(profile_name, sources, units):
    """DRAM bytes per launch from a committed ncu summary, scaled to `units`
    of work; None when the kernel source changed since the capture."""
    path = os.path.join(ROOT, "profiles", profile_name)
    try:
        with open(path) as f:
            prof = json.load(f)
    except Exception:
        return None
    if prof.get("source_sha256") != source_sha(*sources):
        return None
    per_unit = prof["dram_bytes_per_launch"] / prof["units_per_launch"]
    return per_unit * units


def timed_calls(torch, stream, call, n):
    """n back-to-back calls between CUDA events on `stream`, nvidia-smi clocks
    sampled meanwhile; returns (ms per call, clock summary)."""
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(n):
            call()
        stop.record(stream)
        torch.cuda.synchronize()
    return start.elapsed_time(stop) / n, clk.summary()


def e2e_calls(torch, device, stream, dev_inputs, call, outputs, n):
    """End to end through the public call: every step copies the call's inputs
    from pinned host memory to the device, runs `call(inputs)` (which returns
    its device outputs) and copies the outputs back to pinned host memory, all
    inside the timed region.  Returns (ms per step, H2D bytes, D2H bytes)."""
    host = {k: (v.cpu().pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in dev_inputs.items()}
    dev = {k: (torch.empty_like(v, device=device) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    outs_h = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outputs]
    h2d = sum(v.numel() * v.element_size() for v in host.values() if isinstance(v, torch.Tensor))
    d2h = sum(o.numel() * o.element_size() for o in outs_h)

    def step():
        for k, v in host.items():
            if isinstance(v, torch.Tensor):
                dev[k].copy_(v, non_blocking=True)
        for oh, od in zip(outs_h, call(dev)):
            oh.copy_(od, non_blocking=True)

    step()
    ms, _ = timed_calls(torch, stream, step, n)
    del dev, host
    return ms, h2d, d2h


# ----------------------------------------------------------------- decode

def decode_work(inp, wl):
    lens = inp["seq_lens"].long().cpu()
    kv = int(lens.sum()) * wl.num_kv_heads * (wl.head_dim_qk + wl.head_dim_v) * 2
    rows = wl.batch * wl.q_len * wl.num_q_heads
    pages = int(((lens + wl.page_size - 1) // wl.page_size).sum())
    other = rows * wl.head_dim_qk * 2 + rows * wl.head_dim_v * 2 + rows * 4 + pages * 4 + wl.batch * 4
    return kv, kv + other, int(lens.sum())


def bench_decode(fw, torch, steps, warmup, device, peaks, batch=None, do_e2e=True, barrier=lambda: None):
    import dataclasses
    from ragged_softmax_attention_gb300.workloads import WORKLOADS, make_decode_inputs, workload_seq_lens
    wl = WORKLOADS[DECODE_WL]
    if batch:   # a prefix of the same batch (profiling captures on a smaller case)
        lens = workload_seq_lens(wl)[:batch]
        wl = dataclasses.replace(wl, batch=batch, seq_len_range=None, seq_lens=tuple(lens))
    d = make_decode_inputs(wl, device)
    kv_bytes, alg_bytes, tokens = decode_work(d, wl)
    out, lse = fw.paged_decode(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["scale"])
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def step():
        fw.paged_decode(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["scale"],
                        out=out, lse=lse)

    for _ in range(max(3, warmup)):
        step()
    torch.cuda.synchronize()
    fw.set_option(fw.FW_OPT_KERNEL_TIMING, 1)
    fw.kernel_timing_read()
    launches0 = fw.launch_count()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(steps):
            step()
        stop.record(stream)
        torch.cuda.synchronize()
        barrier()
    elapsed_ms = start.elapsed_time(stop)
    launches = fw.launch_count() - launches0
    kernel_ms, kernel_n = fw.kernel_timing_read()
    fw.set_option(fw.FW_OPT_KERNEL_TIMING, 0)
    status = fw.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} during the decode benchmark")
    per_launch_ms = kernel_ms / max(1, kernel_n)
    achieved = alg_bytes / (per_launch_ms * 1e-3) / 1e9
    traffic = ncu_traffic("paged_decode_qwen3_14b_ncu.json", DECODE_SOURCES,
                          tokens)
    roof = {"kernel": "paged_decode_kernel<128,16>", "bound": "hbm", "achieved": round(achieved, 1),
            "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": traffic, "peak_source": peaks["source"],
            "algorithmic_bytes_per_launch": alg_bytes, "kernel_ms_per_launch": round(per_launch_ms, 4)}

    cfg = {"workload": DECODE_WL, "batch": wl.batch, "q_len": wl.q_len, "num_q_heads": wl.num_q_heads,
           "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim_qk, "page_size": wl.page_size,
           "seq_len_range": [512, 32768], "total_kv_tokens": tokens,
           "kv_bytes_per_step": kv_bytes, "l2": "inputs larger than L2 (KV cache 4.4 GB), no flush",
           "scale": wl.scale}
    res = {"elapsed_ms": elapsed_ms, "kv_bytes": kv_bytes, "launches": launches, "roofline": roof,
           "clocks": clk.summary(), "config": cfg, "inputs": d, "wl": wl,
           "e2e_ms": float("nan"), "h2d": 0, "d2h": 0, "e2e_steps": 0}
    if not do_e2e:
        return res

    # End to end through the public API from pinned host buffers.
    host = {k: (v.cpu().pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    dev = {k: (torch.empty_like(v, device=device) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    if wl.latent:
        raise RuntimeError("latent workload not expected here")
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values() if isinstance(v, torch.Tensor))
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()
    e2e_steps = max(3, min(steps, 10))

    def e2e_step():
        for k, v in host.items():
            if isinstance(v, torch.Tensor):
                dev[k].copy_(v, non_blocking=True)
        o, l_ = fw.paged_decode(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"], dev["seq_lens"],
                                dev["scale"], out=out, lse=lse)
        out_h.copy_(o, non_blocking=True)
        lse_h.copy_(l_, non_blocking=True)

    e2e_step()
    barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    stop.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = start.elapsed_time(stop) / e2e_steps
    del dev, host
    res.update(e2e_ms=e2e_ms, h2d=h2d, d2h=d2h, e2e_steps=e2e_steps)
    return res


# ---------------------------------------------------------------- prefill

def prefill_flops(cu_q, cu_k, hq, dk, dv, causal):
    total = 0
    for i in range(len(cu_q) - 1):
        lq = cu_q[i + 1] - cu_q[i]
        lk = cu_k[i + 1] - cu_k[i]
        if causal:
            pairs = sum(max(0, min(lk, r + lk - lq + 1)) for r in range(lq)) if lq != lk else lq * (lq + 1) // 2
        else:
            pairs = lq * lk
        total += pairs
    return total * hq * 2 * (dk + dv)


def bench_prefill(fw, torch, steps, warmup, device, peaks, name=None, softmax="static", do_e2e=True,
                  do_cpu=False):
    name = name or PREFILL_WL
    fw.set_option(fw.FW_OPT_PREFILL_SOFTMAX, 1 if softmax == "online" else 0)
    try:
        return _bench_prefill(fw, torch, steps, warmup, device, peaks, name, softmax, do_e2e, do_cpu)
    finally:
        fw.set_option(fw.FW_OPT_PREFILL_SOFTMAX, 0)


def _bench_prefill(fw, torch, steps, warmup, device, peaks, name, softmax, do_e2e, do_cpu):
    from ragged_softmax_attention_gb300.workloads import WORKLOADS, make_prefill_inputs
    wl = WORKLOADS[name]
    d = make_prefill_inputs(wl, device)
    cu_q = d["cu_seqlens_q"].cpu().tolist()
    cu_k = d["cu_seqlens_k"].cpu().tolist()
    flops = prefill_flops(cu_q, cu_k, wl.num_q_heads, wl.head_dim_qk, wl.head_dim_v, wl.causal)
    try:
        out, lse = fw.varlen_prefill(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], wl.causal,
                                     wl.scale)
    except fw.FwError as e:
        if e.status == 2:
            return {"workload": name, "value": None, "unit": "TFLOP/s", "unavailable": str(e)}
        raise
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    for _ in range(max(3, warmup)):
        fw.varlen_prefill(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], wl.causal, wl.scale,
                          out=out, lse=lse)
    torch.cuda.synchronize()
    fw.set_option(fw.FW_OPT_KERNEL_TIMING, 1)
    fw.kernel_timing_read()
    fw.read_counters()
    n = max(3, min(steps, 50))
    l0 = fw.launch_count()
    ms, clocks = timed_calls(torch, stream, lambda: fw.varlen_prefill(
        d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], wl.causal, wl.scale, out=out, lse=lse), n)
    launches = fw.launch_count() - l0
    kms, kn = fw.kernel_timing_read()
    fw.set_option(fw.FW_OPT_KERNEL_TIMING, 0)
    replays = fw.read_counters()["prefill_replays"]
    if fw.device_status() != 0:
        raise RuntimeError("device status nonzero during the prefill benchmark")
    per = kms / max(1, kn)
    e2e = None
    if do_e2e:
        e_ms, h2d, d2h = e2e_calls(
            torch, device, stream, {k: d[k] for k in ("q", "k", "v", "cu_seqlens_q", "cu_seqlens_k")},
            lambda x: fw.varlen_prefill(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_k"], wl.causal,
                                        wl.scale, out=out, lse=lse), [out, lse], max(3, min(steps, 10)))
        e2e = {"value": round(flops / (e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": round(e_ms, 4),
               "note": "q, k, v and cu_seqlens copied from pinned host memory and out + lse copied back every "
                       "step, through fw_varlen_prefill"}
    cpu = None
    if do_cpu:
        try:
            cpu = prefill_cpu_baseline(torch, d, wl)
        except Exception as e:   # the baseline is context; report why it is missing
            cpu = {"value": None, "unit": "TFLOP/s", "kind": "oracle", "error": str(e)}
    ach = flops / (per * 1e-3) / 1e12
    profile = {PREFILL_WL: "varlen_prefill_gqa_ncu.json", PREFILL_HD256_WL: "varlen_prefill_hd256_ncu.json"}[name]
    traffic = ncu_traffic(profile, PREFILL_SOURCES, flops)
    return {"workload": name, "value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "steps": n, "flops_per_step": flops,
            "gpu_launches": launches, "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu,
            "anchor_replays_per_call": round(replays / n, 2),
            "config": {"num_seqs": wl.num_seqs, "num_q_heads": wl.num_q_heads, "num_kv_heads": wl.num_kv_heads,
                       "head_dim": wl.head_dim_qk, "causal": wl.causal, "total_tokens": cu_q[-1],
                       "seq_len_range": list(wl.seq_len_range) if wl.seq_len_range else None,
                       "seq_lens": list(wl.seq_lens) if wl.seq_lens else None, "scale": wl.scale,
                       "softmax": "static anchor, check and replay" if softmax == "static"
                       else "online, conditional rescale (8 log2 units)"},
            "roofline": {"kernel": "varlen_prefill_kernel" if wl.head_dim_qk == 128 else "varlen_prefill_pair_kernel", "bound": "tensor", "achieved": round(ach, 1),
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(ach / peaks["bf16_tflops"], 4),
                         "frac_of_sustained": round(ach / peaks["bf16_tflops_sustained"], 4),
                         "traffic": traffic, "peak_source": peaks["source"], "kernel_ms_per_launch": round(per, 4)}}


# ------------------------------------------------------ FP8 KV decode

def bench_decode_fp8(fw, torch, steps, warmup, device, peaks, batch=None):
    import dataclasses
    from ragged_softmax_attention_gb300.workloads import WORKLOADS, make_decode_inputs, workload_seq_lens
    wl = WORKLOADS[DECODE_FP8_WL]
    if batch:   # a prefix of the same batch (profiling captures on a smaller case)
        lens = workload_seq_lens(wl)[:batch]
        wl = dataclasses.replace(wl, batch=batch, seq_len_range=None, seq_lens=tuple(lens))
    d = make_decode_inputs(wl, device)
    lens = d["seq_lens"].long().cpu()
    tokens = int(lens.sum())
    kv = tokens * wl.num_kv_heads * (wl.head_dim_qk + wl.head_dim_v)          # one byte per value
    rows = wl.batch * wl.q_len * wl.num_q_heads
    pages = int(((lens + wl.page_size - 1) // wl.page_size).sum())
    alg = kv + rows * wl.head_dim_qk * 2 + rows * wl.head_dim_v * 2 + rows * 4 + pages * 4 + wl.batch * 4
    args = (d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["scale"], d["k_scale"],
            d["v_scale"])
    out, lse = fw.paged_decode_fp8(*args)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    for _ in range(max(3, warmup)):
        fw.paged_decode_fp8(*args, out=out, lse=lse)
    torch.cuda.synchronize()
    fw.set_option(fw.FW_OPT_KERNEL_TIMING, 1)
    fw.kernel_timing_read()
    n = max(3, min(steps, 100))
    l0 = fw.launch_count()
    ms, clocks = timed_calls(torch, stream, lambda: fw.paged_decode_fp8(*args, out=out, lse=lse), n)
    kms, kn = fw.kernel_timing_read()
    fw.set_option(fw.FW_OPT_KERNEL_TIMING, 0)
    if fw.device_status() != 0:
        raise RuntimeError("device status nonzero during the FP8 decode benchmark")
    per = kms / max(1, kn)
    ach = alg / (per * 1e-3) / 1e9
    return {"workload": DECODE_FP8_WL, "value": round(kv / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "kv_tokens_per_s": round(tokens / (ms * 1e-3), 1), "ms_per_step": round(ms, 4), "steps": n,
            "kv_bytes_per_step": kv, "gpu_launches": fw.launch_count() - l0, "clocks": clocks,
            "config": {"batch": wl.batch, "q_len": wl.q_len, "num_q_heads": wl.num_q_heads,
                       "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim_qk, "page_size": wl.page_size,
                       "kv_dtype": "fp8_e4m3, one scale per cache", "total_kv_tokens": tokens},
            "roofline": {"kernel": "paged_decode_fp8_kernel<16,8>", "bound": "hbm", "achieved": round(ach, 1),
                         "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4),
                         "traffic": ncu_traffic("paged_decode_fp8_ncu.json", FP8_SOURCES, tokens),
                         "peak_source": peaks["source"], "algorithmic_bytes_per_launch": alg,
                         "kernel_ms_per_launch": round(per, 4)}}


def bench_decode_window(fw, torch, steps, warmup, device, peaks, fp8=False, window=4096):
    """Sliding-window decode ("TokenSpeed-MLA 2.0.1", window_left) on the
    Qwen3-14B-shaped workload: each row reads only its last window + q_len keys.
    The metric counts those keys' bytes (the window's own KV), so it compares
    directly with the full-row decode's GB/s."""
    from ragged_softmax_attention_gb300.workloads import WORKLOADS, make_decode_inputs
    wl = WORKLOADS[DECODE_FP8_WL if fp8 else DECODE_WL]
    d = make_decode_inputs(wl, device)
    lens = d["seq_lens"].long().cpu()
    first = (lens - wl.q_len - window).clamp(min=0)
    tokens = int((lens - first).sum())
    esz = 1 if fp8 else 2
    kv = tokens * wl.num_kv_heads * (wl.head_dim_qk + wl.head_dim_v) * esz
    rows = wl.batch * wl.q_len * wl.num_q_heads
    pages = int((((lens + wl.page_size - 1) // wl.page_size) - first // wl.page_size).sum())
    alg = kv + rows * wl.head_dim_qk * 2 + rows * wl.head_dim_v * 2 + rows * 4 + pages * 4 + wl.batch * 4
    ks, vs = (d["k_scale"], d["v_scale"]) if fp8 else (1.0, 1.0)
    args = (d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["scale"], window)
    out, lse = fw.paged_decode_window(*args, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    for _ in range(max(3, warmup)):
        fw.paged_decode_window(*args, k_scale=ks, v_scale=vs, out=out, lse=lse)
    torch.cuda.synchronize()
    fw.set_option(fw.FW_OPT_KERNEL_TIMING, 1)
    fw.kernel_timing_read()
    n = max(3, min(steps, 100))
    l0 = fw.launch_count()
    ms, clocks = timed_calls(torch, stream, lambda: fw.paged_decode_window(*args, k_scale=ks, v_scale=vs, out=out,
                                                                           lse=lse), n)
    kms, kn = fw.kernel_timing_read()
    fw.set_option(fw.FW_OPT_KERNEL_TIMING, 0)
    if fw.device_status() != 0:
        raise RuntimeError("device status nonzero during the sliding-window decode benchmark")
    per = kms / max(1, kn)
    ach = alg / (per * 1e-3) / 1e9
    kernel = "paged_decode_fp8_kernel<16,8>" if fp8 else "paged_decode_kernel<128,16>"
    return {"workload": (DECODE_FP8_WL if fp8 else DECODE_WL) + f", window_left {window}",
            "value": round(kv / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "kv_tokens_per_s": round(tokens / (ms * 1e-3), 1), "ms_per_step": round(ms, 4), "steps": n,
            "kv_bytes_per_step": kv, "window_kv_tokens": tokens, "gpu_launches": fw.launch_count() - l0,
            "clocks": clocks,
            "roofline": {"kernel": kernel, "bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4), "traffic": None,
                         "peak_source": peaks["source"], "algorithmic_bytes_per_launch": alg,
                         "kernel_ms_per_launch": round(per, 4)}}


def bench_decode_append(fw, torch, steps, warmup, device, peaks):
    """The Qwen3-14B-shaped decode with each row's new token appended in the
    same call (fw_paged_decode_append, the append folded into the plan
    launch): same metric as the plain decode line, so the difference is the
    append's cost."""
    from ragged_softmax_attention_gb300.workloads import WORKLOADS, make_decode_inputs
    wl = WORKLOADS[DECODE_WL]
    d = make_decode_inputs(wl, device)
    lens = d["seq_lens"].long().cpu()
    bt = d["block_table"].cpu()
    ps = wl.page_size
    slots = torch.tensor([int(bt[b, (int(lens[b]) - 1) // ps]) * ps + (int(lens[b]) - 1) % ps
                          for b in range(wl.batch)], dtype=torch.int32, device=device)
    g = torch.Generator(device="cpu").manual_seed(17)
    k_new = torch.randn(wl.batch, 1, wl.num_kv_heads, wl.head_dim_qk, generator=g).to(torch.bfloat16).to(device)
    v_new = torch.randn(wl.batch, 1, wl.num_kv_heads, wl.head_dim_v, generator=g).to(torch.bfloat16).to(device)
    kv = int(lens.sum()) * wl.num_kv_heads * (wl.head_dim_qk + wl.head_dim_v) * 2
    args = (d["q"], k_new, v_new, slots, 0, d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["scale"])
    out, lse = fw.paged_decode_append(*args)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    for _ in range(max(3, warmup)):
        fw.paged_decode_append(*args, out=out, lse=lse)
    torch.cuda.synchronize()
    n = max(3, min(steps, 100))
    l0 = fw.launch_count()
    ms, clocks = timed_calls(torch, stream, lambda: fw.paged_decode_append(*args, out=out, lse=lse), n)
    if fw.device_status() != 0:
        raise RuntimeError("device status nonzero during the append + decode benchmark")
    appended = wl.batch * wl.num_kv_heads * (wl.head_dim_qk + wl.head_dim_v) * 2
    return {"workload": DECODE_WL + ", new token appended in the call", "value": round(kv / (ms * 1e-3) / 1e9, 1),
            "unit": "GB/s", "ms_per_step": round(ms, 4), "steps": n, "kv_bytes_per_step": kv,
            "appended_bytes_per_step": appended, "gpu_launches": fw.launch_count() - l0, "clocks": clocks}


# ------------------------------------------------------- latent decode

def latent_work(lens, wl):
    """FLOPs (each query token t of a row with n keys sees n - q_len + t + 1)
    and KV bytes (the 576-wide key rows; values are a view of them)."""
    flops = 0
    for n in lens:
        for t in range(wl.q_len):
            flops += max(0, min(n, n - wl.q_len + t + 1)) * wl.num_q_heads * 2 * (wl.head_dim_qk + wl.head_dim_v)
    kv = sum(lens) * wl.num_kv_heads * wl.head_dim_qk * 2
    return flops, kv


# 128 query heads per KV head: the CTA-pair kernel serves the latent workload.
LATENT_KERNEL = "latent_pair_decode_kernel"


def bench_latent(fw, torch, steps, warmup, device, peaks, batch=None, do_e2e=True, do_cpu=False):
    import dataclasses
    from ragged_softmax_attention_gb300.workloads import WORKLOADS, make_decode_inputs
    wl = WORKLOADS[LATENT_WL]
    if batch:   # a prefix of the same batch (profiling captures on a smaller case)
        wl = dataclasses.replace(wl, batch=batch, seq_lens=wl.seq_lens[:batch])
    d = make_decode_inputs(wl, device)
    lens = d["seq_lens"].cpu().tolist()
    flops, kv = latent_work(lens, wl)
    args = (d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["scale"])
    out, lse = fw.paged_decode(*args)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    for _ in range(max(3, warmup)):
        fw.paged_decode(*args, out=out, lse=lse)
    torch.cuda.synchronize()
    fw.set_option(fw.FW_OPT_KERNEL_TIMING, 1)
    fw.kernel_timing_read()
    fw.read_counters()
    n = max(3, min(steps, 50))
    l0 = fw.launch_count()
    ms, clocks = timed_calls(torch, stream, lambda: fw.paged_decode(*args, out=out, lse=lse), n)
    launches = fw.launch_count() - l0
    kms, kn = fw.kernel_timing_read()
    fw.set_option(fw.FW_OPT_KERNEL_TIMING, 0)
    rescales = fw.read_counters()["latent_rescales"]
    if fw.device_status() != 0:
        raise RuntimeError("device status nonzero during the latent decode benchmark")
    per = kms / max(1, kn)
    ach = flops / (per * 1e-3) / 1e12
    e2e = None
    if do_e2e:
        # The values are a view of the key cache: only the 576-wide cache crosses the link.
        e_ms, h2d, d2h = e2e_calls(
            torch, device, stream, {k: d[k] for k in ("q", "k_cache", "block_table", "seq_lens")},
            lambda x: fw.paged_decode(x["q"], x["k_cache"], x["k_cache"][..., :wl.head_dim_v], x["block_table"],
                                      x["seq_lens"], d["scale"], out=out, lse=lse), [out, lse], 3)
        e2e = {"value": round(flops / (e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": round(e_ms, 4),
               "note": "q, the key cache (values are its first 512 columns), block table and seq_lens copied "
                       "from pinned host memory and out + lse copied back every step, through fw_paged_decode"}
    cpu = None
    if do_cpu:
        try:
            cpu = latent_cpu_baseline(torch, d, wl)
        except Exception as e:   # the baseline is context; report why it is missing
            cpu = {"value": None, "unit": "TFLOP/s", "kind": "oracle", "error": str(e)}
    return {"workload": LATENT_WL, "value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "kv_gbs": round(kv / (ms * 1e-3) / 1e9, 1), "ms_per_step": round(ms, 4), "steps": n,
            "flops_per_step": flops, "kv_bytes_per_step": kv, "gpu_launches": launches,
            "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu,
            "anchor_rescales_per_call": round(rescales / n, 2),
            "config": {"batch": wl.batch, "q_len": wl.q_len, "num_q_heads": wl.num_q_heads,
                       "num_kv_heads": wl.num_kv_heads, "head_dim_qk": wl.head_dim_qk,
                       "head_dim_v": wl.head_dim_v, "page_size": wl.page_size, "seq_lens": "81920 each",
                       "scale": wl.scale, "v": "first 512 columns of the key cache"},
            "roofline": {"kernel": LATENT_KERNEL, "bound": "tensor", "achieved": round(ach, 1),
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(ach / peaks["bf16_tflops"], 4),
                         "frac_of_sustained": round(ach / peaks["bf16_tflops_sustained"], 4),
                         "traffic": ncu_traffic("latent_pair_decode_ncu.json", LATENT_SOURCES,
                                                sum(lens)), "peak_source": peaks["source"], "kernel_ms_per_launch": round(per, 4)}}


# ------------------------------------------------------------ CPU oracle

def oracle_sample_rate(torch, inp, wl, rows_b, heads, threads):
    """Run the fp64 oracle on batch rows `rows_b` x query heads `heads`;
    returns (KV bytes those rows read, seconds)."""
    import oracle
    lens = inp["seq_lens"].cpu()
    bt = inp["block_table"].cpu()
    G = wl.num_q_heads // wl.num_kv_heads
    total_bytes = 0
    total_s = 0.0
    for b in rows_b:
        npg = -(-int(lens[b]) // wl.page_size)
        pages = bt[b, :npg].long()
        k = inp["k_cache"][pages.to(inp["k_cache"].device)].cpu()
        v = inp["v_cache"][pages.to(inp["v_cache"].device)].cpu()
        sub_bt = torch.arange(npg, dtype=torch.int32).unsqueeze(0)
        q = inp["q"][b:b + 1].cpu()
        t0 = time.perf_counter()
        oracle.paged_decode(q, k, v, sub_bt, lens[b:b + 1], wl.scale, rows=list(heads), threads=threads)
        total_s += time.perf_counter() - t0
        kv_heads = sorted({h // G for h in heads})
        total_bytes += int(lens[b]) * len(kv_heads) * (wl.head_dim_qk + wl.head_dim_v) * 2
    return total_bytes, total_s


def cpu_baseline(torch, inp, wl, budget_s=12.0):
    """The oracle, as it stands, on the host cores: whole batch rows (all query
    heads) in batch order, cycling through the batch until about `budget_s`
    seconds of oracle time have accumulated."""
    threads = max(1, os.cpu_count() or 1)
    heads = list(range(wl.num_q_heads))
    by, s, n = 0, 0.0, 0
    while s < budget_s and n < 64 * wl.batch:
        b_by, b_s = oracle_sample_rate(torch, inp, wl, [n % wl.batch], heads, threads)
        by, s, n = by + b_by, s + b_s, n + 1
    return {"value": round(by / s / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} batch rows in batch order ({n / wl.batch:.1f} passes over the {wl.batch}-row batch), "
                      f"all {wl.num_q_heads} query heads ({s:.1f} s of fp64 CPU work, {threads} threads)"}


def prefill_cpu_baseline(torch, d, wl, budget_s=8.0):
    """The oracle, as it stands, on the host cores over a fixed sample of the
    prefill's (query row, head) units: evenly spaced rows of the flattened
    [total_q, Hq] list, doubling the sample until about `budget_s` seconds of
    oracle time.  The rate is the sample's algorithmic FLOPs over its time;
    the whole workload's time is extrapolated from it."""
    import numpy as np
    import oracle
    threads = max(1, os.cpu_count() or 1)
    q, k, v = d["q"].cpu(), d["k"].cpu(), d["v"].cpu()
    cq, ck = d["cu_seqlens_q"].cpu(), d["cu_seqlens_k"].cpu()
    cql, ckl = cq.tolist(), ck.tolist()
    total = q.shape[0] * wl.num_q_heads
    seq_of = np.searchsorted(np.asarray(cql), np.arange(q.shape[0]), side="right") - 1

    def row_flops(rows):
        tok = rows // wl.num_q_heads
        sq = seq_of[tok]
        lq = np.asarray(cql)[sq + 1] - np.asarray(cql)[sq]
        lk = np.asarray(ckl)[sq + 1] - np.asarray(ckl)[sq]
        r = tok - np.asarray(cql)[sq]
        vis = np.clip(r + lk - lq + 1, 0, lk) if wl.causal else lk
        return int(vis.sum()) * 2 * (wl.head_dim_qk + wl.head_dim_v)

    n = 1024
    while True:
        rows = np.linspace(0, total - 1, num=min(n, total)).astype(np.int64)
        t0 = time.perf_counter()
        oracle.varlen_prefill(q, k, v, cq, ck, wl.causal, wl.scale, rows=rows, threads=threads)
        sec = time.perf_counter() - t0
        if sec >= budget_s / 2 or n >= total:
            break
        n *= 2
    f = row_flops(rows)
    rate = f / sec
    whole = prefill_flops(cql, ckl, wl.num_q_heads, wl.head_dim_qk, wl.head_dim_v, wl.causal)
    return {"value": round(rate / 1e12, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{rows.size} evenly spaced (query row, head) units of {total} ({f / 1e9:.1f} GFLOP, "
                      f"{sec:.1f} s of fp64 CPU work, {threads} threads)",
            "extrapolated": True, "whole_workload_s": round(whole / rate, 1)}


def latent_cpu_baseline(torch, d, wl, budget_s=8.0):
    """The oracle, as it stands, on the host cores over whole requests (all
    query tokens and heads) in batch order until about `budget_s` seconds of
    oracle time; the rate is their algorithmic FLOPs over that time and the
    whole workload's time is extrapolated from it."""
    import oracle
    threads = max(1, os.cpu_count() or 1)
    lens = d["seq_lens"].cpu()
    bt = d["block_table"].cpu()
    f, sec, nb = 0, 0.0, 0
    while sec < budget_s and nb < wl.batch:
        b = nb
        npg = -(-int(lens[b]) // wl.page_size)
        pages = bt[b, :npg].long().to(d["k_cache"].device)
        kc = d["k_cache"][pages].cpu()
        sub_bt = torch.arange(npg, dtype=torch.int32).unsqueeze(0)
        t0 = time.perf_counter()
        oracle.paged_decode(d["q"][b:b + 1].cpu(), kc, kc[..., :wl.head_dim_v], sub_bt, lens[b:b + 1], wl.scale,
                            threads=threads)
        sec += time.perf_counter() - t0
        f += latent_work([int(lens[b])], wl)[0]
        nb += 1
    rate = f / sec
    whole = latent_work(lens.tolist(), wl)[0]
    return {"value": round(rate / 1e12, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{nb} of {wl.batch} requests, all {wl.q_len} tokens x {wl.num_q_heads} heads "
                      f"({f / 1e9:.1f} GFLOP, {sec:.1f} s of fp64 CPU work, {threads} threads)",
            "extrapolated": True, "whole_workload_s": round(whole / rate, 1)}


def run_reference(args):
    import torch
    world, rank, local = dist_env()
    if rank != 0:
        return 0
    from ragged_softmax_attention_gb300.workloads import WORKLOADS, make_decode_inputs
    wl = WORKLOADS[DECODE_WL]
    # Inputs are drawn where they are cheapest to draw (the GPU when present);
    # only the oracle call itself is timed, on the host cores.
    inp = make_decode_inputs(wl, "cuda" if torch.cuda.is_available() else "cpu")
    threads = max(1, os.cpu_count() or 1)
    G = wl.num_q_heads // wl.num_kv_heads
    total_bytes, total_s = 0, 0.0
    for i in range(args.warmup + args.steps):
        b = i % wl.batch
        g = (i // wl.batch) % wl.num_kv_heads
        by, s = oracle_sample_rate(torch, inp, wl, [b], range(g * G, (g + 1) * G), threads)
        if i >= args.warmup:
            total_bytes += by
            total_s += s
    value = total_bytes / total_s / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_s / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": DECODE_WL, "batch": wl.batch,
                                            "num_q_heads": wl.num_q_heads, "num_kv_heads": wl.num_kv_heads,
                                            "head_dim": wl.head_dim_qk, "page_size": wl.page_size},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": "each step: one (batch row, KV head group) of the workload, "
                                       "cycling through rows"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--only", choices=["all", "decode", "decode_fp8", "decode_window", "decode_append", "prefill",
                                       "prefill256", "latent"],
                    default="all",
                    help="profiling runs: time one path only")
    ap.add_argument("--decode-batch", type=int, default=0,
                    help="profiling runs: a prefix of the decode batch (smaller capture)")
    ap.add_argument("--latent-batch", type=int, default=0,
                    help="profiling runs: a prefix of the latent decode batch (smaller capture)")
    ap.add_argument("--prefill-softmax", choices=["static", "online"], default="static",
                    help="with --only prefill/prefill256: the prefill softmax mode to time")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import ragged_softmax_attention_gb300 as fw
    from ragged_softmax_attention_gb300 import build as fwbuild

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        pg = dist
    if rank == 0:
        fwbuild.build()
    if pg:
        pg.barrier()
    fw.load_library()
    peaks = load_peaks()

    if pg:
        pg.barrier()
    if args.only in ("prefill", "prefill256"):
        key = "prefill" if args.only == "prefill" else "prefill_hd256"
        pre = bench_prefill(fw, torch, args.steps, args.warmup, device, peaks,
                            name=PREFILL_WL if args.only == "prefill" else PREFILL_HD256_WL,
                            softmax=args.prefill_softmax)
        if rank == 0:
            print(json.dumps({key: pre}), flush=True)
        return 0
    if args.only == "decode_fp8":
        f8 = bench_decode_fp8(fw, torch, args.steps, args.warmup, device, peaks, batch=args.decode_batch or None)
        if rank == 0:
            print(json.dumps({"decode_fp8": f8}), flush=True)
        return 0
    if args.only == "decode_window":
        w16 = bench_decode_window(fw, torch, args.steps, args.warmup, device, peaks, fp8=False)
        w8 = bench_decode_window(fw, torch, args.steps, args.warmup, device, peaks, fp8=True)
        if rank == 0:
            print(json.dumps({"decode_window": w16, "decode_fp8_window": w8}), flush=True)
        return 0
    if args.only == "decode_append":
        app = bench_decode_append(fw, torch, args.steps, args.warmup, device, peaks)
        if rank == 0:
            print(json.dumps({"decode_append": app}), flush=True)
        return 0
    if args.only == "latent":
        lat = bench_latent(fw, torch, args.steps, args.warmup, device, peaks, batch=args.latent_batch or None)
        if rank == 0:
            print(json.dumps({"latent_decode": lat}), flush=True)
        return 0
    dec = bench_decode(fw, torch, args.steps, args.warmup, device, peaks, batch=args.decode_batch or None,
                       do_e2e=not args.no_e2e, barrier=(pg.barrier if pg else (lambda: None)))
    # CPU baselines on rank 0 of a single-GPU run only (they hold no GPU work).
    do_cpu = world == 1 and not args.no_cpu_baseline and not args.decode_batch
    pre = None if args.only == "decode" else bench_prefill(fw, torch, args.steps, args.warmup, device, peaks,
                                                           do_e2e=not args.no_e2e, do_cpu=do_cpu)
    pre256 = (None if args.only == "decode" else
              bench_prefill(fw, torch, args.steps, args.warmup, device, peaks, name=PREFILL_HD256_WL,
                            do_e2e=not args.no_e2e, do_cpu=do_cpu))
    lat = None if args.only == "decode" else bench_latent(fw, torch, args.steps, args.warmup, device, peaks,
                                                         do_e2e=not args.no_e2e, do_cpu=do_cpu)
    f8 = None if args.only == "decode" else bench_decode_fp8(fw, torch, args.steps, args.warmup, device, peaks)
    w16 = (None if args.only == "decode" else
           bench_decode_window(fw, torch, args.steps, args.warmup, device, peaks, fp8=False))
    w8 = (None if args.only == "decode" else
          bench_decode_window(fw, torch, args.steps, args.warmup, device, peaks, fp8=True))
    app = None if args.only == "decode" else bench_decode_append(fw, torch, args.steps, args.warmup, device, peaks)
    elapsed_ms, e2e_ms = max_over_ranks(pg, [dec["elapsed_ms"], dec["e2e_ms"]], device)
    value = whole_job_rate(dec["kv_bytes"], args.steps, world, elapsed_ms)
    e2e_value = whole_job_rate(dec["kv_bytes"], 1, world, e2e_ms)
    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return 0
    line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(elapsed_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(dec["config"], parallelism=f"replicas{world}" if world > 1 else "single"),
            "frac_of_hbm_peak": round(value / world / peaks["hbm_gbs"], 4),
            "roofline": dec["roofline"], "clocks": dec["clocks"], "gpu_launches": dec["launches"],
            "e2e": {"value": round(e2e_value, 1) if e2e_value else None, "unit": "GB/s", "h2d_bytes_per_step": dec["h2d"],
                    "d2h_bytes_per_step": dec["d2h"], "steps": dec["e2e_steps"],
                    "note": "inputs (incl. the KV cache) copied from pinned host memory every step"},
            "prefill": pre, "prefill_hd256": pre256, "latent_decode": lat, "decode_fp8": f8,
            "decode_window": w16, "decode_fp8_window": w8, "decode_append": app}
    if do_cpu:
        try:
            line["cpu_baseline"] = cpu_baseline(torch, dec["inputs"], dec["wl"])
        except Exception as e:   # the baseline is context; report why it is missing
            line["cpu_baseline"] = {"value": None, "unit": "GB/s", "kind": "oracle", "error": str(e)}
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
