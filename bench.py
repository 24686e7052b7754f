#!/usr/bin/env python
"""Benchmark of the batch-invariant forward hot path on GB300.

One step = one pass of every kernel of the path over one synthetic batch:
  1. bi_rmsnorm            16384 rows x 4096 (eps 1e-6, 1% outliers x100)
  2. bi_gemm               Qwen3-8B-shaped linear layers at M = 4096 tokens:
                           qkv [4096->6144], o [4096->4096],
                           gate|up [4096->24576], down [12288->4096]
  3. bi_decode_attention   256 sequences, GQA 32/8 heads, head_dim 128, 16-token
                           pages, lengths uniform on [1, 8192]
Every input is seeded synthetic data of those shapes, resident in HBM before
the timed region.  The per-step working set (about 5.5 GB, mostly the KV
cache) is far larger than L2, so every step starts from a cold L2.

Headline `value`: bi_gemm TFLOP/s = GEMM FLOPs of the timed steps / GEMM
device time (CUDA events on the launching stream).  The other parts of the
metric go alongside: decode-attention and RMSNorm GB/s of algorithmic bytes
with their HBM-roofline fractions, the same-run cost of the non-invariant
cuBLAS / F.rms_norm references, and bitwise batch-invariance checks.

`--impl reference` times the fp64 CPU oracle on the host cores instead, on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

RMS_ROWS, HIDDEN, EPS = 16384, 4096, 1e-6
GEMM_M = 4096
LAYERS = [("qkv", 6144, 4096), ("o", 4096, 4096), ("gate_up", 24576, 4096), ("down", 4096, 12288)]
ATT_B, HQ, HKV, HD, MAX_LEN = 256, 32, 8, 128, 8192
METRIC = "bi_gemm TFLOP/s; split-KV decode attn GB/s (% roofline); bitwise batch-invariant"
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal (about 8 TB/s)

CONFIG = {
    "workload": ("qwen3-8b-shaped hot path: rmsnorm 16384x4096 + bi_gemm qkv/o/gate_up/down at "
                 "M=4096 + paged decode attention B=256 (GQA 32/8, d128, L~U[1,8192])"),
    "rmsnorm": {"rows": RMS_ROWS, "hidden": HIDDEN, "eps": EPS},
    "gemm": {"M": GEMM_M, "layers": {n: {"N": N, "K": K} for n, N, K in LAYERS}},
    "attention": {"B": ATT_B, "Hq": HQ, "Hkv": HKV, "D": HD, "page": 16, "chunk": 256,
                  "seq_len": f"U[1,{MAX_LEN}]"},
    "l2": "per-step working set ~5.5 GB >> 129 MB L2 (inputs larger than L2)",
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-next-rows", action="store_true",
                    help="skip the cold-L2 timings of the kernels beyond the bench step")
    ap.add_argument("--no-c5", action="store_true",
                    help="skip the C5 decoder run (36 layers, 1000 requests) of the default line")
    ap.add_argument("--case", choices=["gemm_gate_up", "gemm_qkv", "gemm_layers", "attention",
                                       "rmsnorm", "decoder", "prefill", "add_rmsnorm",
                                       "logprobs", "qk_norm_rope_append", "silu_mul",
                                       "gemm_swiglu", "decode_latency"],
                    help="time one kernel of the path alone (for profiling); prints its own line")
    ap.add_argument("--requests", type=int, default=1000, help="C5 decoder (--case decoder and the default line): requests")
    ap.add_argument("--layers", type=int, default=36, help="--case decoder: decoder layers")
    ap.add_argument("--new-tokens", type=int, default=100, help="--case decoder: tokens per request")
    ap.add_argument("--budget", type=int, default=8192,
                    help="--case decoder: tokens per step (decode rows + prompt chunks)")
    ap.add_argument("--track", type=int, default=16,
                    help="--case decoder: requests re-run alone for the bitwise check")
    ap.add_argument("--batch", type=int, default=ATT_B,
                    help="sequences for --case attention (a smaller case for ncu captures)")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


KERNEL_SOURCES = {"bi_gemm": "gemm.cu", "bi_decode_attention": "decode_attention.cu",
                  "bi_rmsnorm": "rmsnorm.cu", "bi_add_rmsnorm": "rmsnorm.cu",
                  "bi_prefill_attention": "prefill_attention.cu", "bi_logprobs": "logprobs.cu",
                  "bi_qk_norm_rope_append": "decoder_ops.cu", "bi_silu_mul": "decoder_ops.cu",
                  "bi_gemm_swiglu": "gemm.cu"}


def kernel_source_sha(src: str) -> str:
    """sha256[:16] of a kernel's .cu file followed by every header of the
    package it includes (transitively, each once, in first-include order)."""
    import re
    csrc = os.path.join(ROOT, "invariant_bi_rmsnorm_gb300", "csrc")
    inc = os.path.join(ROOT, "include")
    h = hashlib.sha256()
    seen, todo = set(), [os.path.join(csrc, src)]
    while todo:
        path = todo.pop(0)
        if path in seen:
            continue
        seen.add(path)
        text = open(path, "rb").read()
        h.update(text)
        for name in re.findall(rb'#include "([^"]+)"', text):
            for d in (os.path.dirname(path), csrc, inc):
                cand = os.path.join(d, name.decode())
                if os.path.exists(cand):
                    todo.append(os.path.normpath(cand))
                    break
    return h.hexdigest()[:16]


def traffic_record(kernel: str):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current source of that kernel (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    sha = kernel_source_sha(KERNEL_SOURCES[kernel])
    if not os.path.exists(p):
        return None
    for line in open(p):
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel and parts[1] == sha:
            return float(parts[2])
    return None


# ----------------------------------------------------------------- clocks ---
class ClockSampler:
    """nvidia-smi samples of SM clock, power and throttle reasons, every 100 ms,
    read by a thread and stamped with the host clock, so the samples that
    fall inside a measurement window can be picked out."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.device_index = device_index
        self.lines = []
        self.thread = None

    def start(self, wait_s: float = 3.0):
        """Start sampling; returns once the first sample has arrived (or after wait_s)."""
        try:
            pci = torch.cuda.get_device_properties(self.device_index)
            sel = ["-i", str(self.device_index)]
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
            if len(vis) > self.device_index and vis[self.device_index].strip().isdigit():
                sel = ["-i", vis[self.device_index].strip()]
            bus = getattr(pci, "pci_bus_id", None)
            if bus is not None:
                dom = getattr(pci, "pci_domain_id", 0)
                dev = getattr(pci, "pci_device_id", 0)
                sel = ["-i", f"{dom:08x}:{bus:02x}:{dev:02x}.0"]
            self.proc = subprocess.Popen(
                ["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        import threading

        def reader():
            for line in self.proc.stdout:
                self.lines.append((time.perf_counter(), line))
        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        t0 = time.perf_counter()
        while not self.lines and time.perf_counter() - t0 < wait_s:
            time.sleep(0.01)

    def stop(self, window=None):
        """Summary of the samples stamped inside window = (t0, t1) (host
        perf_counter seconds), or of all samples."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, line in self.lines:
            if window is not None and not (window[0] <= t <= window[1]):
                continue
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
                power.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w": round(statistics.median(power), 1) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------- multi-rank -----
def reduce_max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise max of `values` over all ranks (each rank's timings; the
    slowest rank sets the job time).  Identity without a process group."""
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist is not None and dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def weak_scaling_rate(units_per_rank: float, world: int, steps: int, max_ms: float) -> float:
    """Whole-job throughput: every rank processed the same per-rank work."""
    return world * units_per_rank * steps / (max_ms * 1e-3)


# ------------------------------------------------------------ our arm -------
class Workload:
    def __init__(self, dev):
        import invariant_bi_rmsnorm_gb300 as bi
        from invariant_bi_rmsnorm_gb300 import inputs
        self.bi = bi
        self.dev = dev
        torch.cuda.set_device(dev)
        self.stream = torch.cuda.current_stream(dev)
        # RMSNorm
        self.rx = inputs.rmsnorm_rows(RMS_ROWS, HIDDEN, seed=3, device=dev)
        self.rw = inputs.rmsnorm_weight(HIDDEN, seed=4, device=dev)
        self.ry = torch.empty_like(self.rx)
        # GEMM
        self.W = {n: inputs.gemm_weight(N, K, seed=40 + i, device=dev)
                  for i, (n, N, K) in enumerate(LAYERS)}
        self.gx = {K: inputs.gemm_rows(GEMM_M, K, seed=50 + K, device=dev)
                   for K in sorted({K for _, _, K in LAYERS})}
        self.gy = {n: torch.empty(GEMM_M, N, dtype=torch.bfloat16, device=dev) for n, N, _ in LAYERS}
        # attention
        p = inputs.decode_problem(ATT_B, Hq=HQ, Hkv=HKV, D=HD, max_len=MAX_LEN, seed=270, device=dev)
        self.att = {k: v.to(dev) for k, v in p.items()}
        self.att_out = torch.empty(ATT_B, HQ, HD, dtype=torch.bfloat16, device=dev)
        self.ws = torch.zeros(bi.decode_attention_workspace_size(ATT_B, HQ, HD, MAX_LEN),
                              dtype=torch.uint8, device=dev)
        lens = p["seq_lens"].to(torch.int64)
        self.att_lens = lens
        # algorithmic work
        self.gemm_flops = sum(2.0 * GEMM_M * N * K for _, N, K in LAYERS)
        self.rms_bytes = 2.0 * RMS_ROWS * HIDDEN * 2 + HIDDEN * 2
        pages = (lens + 15) // 16
        self.att_bytes = float((lens * HKV * HD * 2 * 2).sum() + ATT_B * HQ * HD * 2 * 2
                               + 4 * pages.sum() + 4 * ATT_B)
        self.att_flops = float((4.0 * HQ * HD * lens).sum())
        self.launches_per_step = 1 + len(LAYERS) + int(
            bi._lib.load().bi_decode_attention_launches(ATT_B, HKV, MAX_LEN))
        torch.cuda.synchronize(dev)

    def rmsnorm(self):
        self.bi.rmsnorm(self.rx, self.rw, EPS, out=self.ry)

    def gemms(self):
        for n, N, K in LAYERS:
            self.bi.gemm(self.gx[K], self.W[n], out=self.gy[n])

    def attention(self):
        a = self.att
        self.bi.decode_attention(a["q"], a["k_cache"], a["v_cache"], a["block_table"],
                                 a["seq_lens"], max_seq_len=MAX_LEN, out=self.att_out,
                                 workspace=self.ws)

    def step(self, ev=None):
        if ev is not None:
            ev[0].record(self.stream)
        self.rmsnorm()
        if ev is not None:
            ev[1].record(self.stream)
        self.gemms()
        if ev is not None:
            ev[2].record(self.stream)
        self.attention()
        if ev is not None:
            ev[3].record(self.stream)

    # bitwise batch-invariance spot checks (outside the timed region)
    def invariance(self):
        bi = self.bi
        ok = {}
        self.step()
        full = self.ry.clone()
        ok["rmsnorm_row0_alone_vs_16384"] = bool(torch.equal(bi.rmsnorm(self.rx[:1], self.rw, EPS), full[:1]))
        x = self.gx[4096]
        W = self.W["qkv"]
        big = bi.gemm(x, W)
        small = bi.gemm(x[:64].contiguous(), W)
        ok["gemm_rows0_64_at_M64_vs_M4096"] = bool(torch.equal(small, big[:64]))
        one = bi.gemm(x[4000:4001].contiguous(), W)
        ok["gemm_row4000_alone"] = bool(torch.equal(one[0], big[4000]))
        a = self.att
        outs = self.att_out.clone()
        s = 17
        alone = bi.decode_attention(a["q"][s:s + 1], a["k_cache"], a["v_cache"],
                                    a["block_table"][s:s + 1].contiguous(), a["seq_lens"][s:s + 1],
                                    max_seq_len=MAX_LEN)
        ok["attention_seq17_alone_vs_batch256"] = bool(torch.equal(alone[0], outs[s]))
        torch.cuda.synchronize()
        bi.get_device_error()
        return ok

    def negative_controls(self):
        """The same checks on the non-invariant library ops: how many rows of
        the first 64 change bits between a batch of 64 and a batch of 4096
        (informative counts; not a pass/fail condition)."""
        import torch.nn.functional as F
        x, W = self.gx[4096], self.W["qkv"]
        big = torch.matmul(x, W.t())
        small = torch.matmul(x[:64].contiguous(), W.t())
        ours_big, ours_small = self.bi.gemm(x, W), self.bi.gemm(x[:64].contiguous(), W)
        r_big = F.rms_norm(self.rx[:4096], (HIDDEN,), self.rw, EPS)
        r_small = F.rms_norm(self.rx[:1], (HIDDEN,), self.rw, EPS)
        rows = lambda a, b: int((a != b).any(dim=-1).sum())  # noqa: E731
        return {"cublas_rows_differing_M64_vs_M4096_of_64": rows(small, big[:64]),
                "bi_gemm_rows_differing_M64_vs_M4096_of_64": rows(ours_small, ours_big[:64]),
                "torch_rms_norm_row0_differs_B1_vs_B4096": bool(rows(r_small, r_big[:1]))}

    def next_rows(self, reps: int = 10):
        """Cold-L2 timings (outside the timed steps) of the decode-attention
        batch sweep and of the kernels beyond the step: prefill attention, the
        fused residual add + RMSNorm, log-probabilities, and the decoder's
        per-token ops.  Each with its roofline fraction and, for attention, the
        same-batch fixed-split-count reference."""
        from invariant_bi_rmsnorm_gb300 import inputs
        hbm, bf16 = load_peaks()[:2]
        flush = torch.ones(64 << 20, dtype=torch.int32, device=self.dev)
        res = {"l2": "a 256 MB buffer is read before every launch (L2 left clean and cold); "
                     f"mean of {reps} launches"}
        a = self.att
        by_b = {}
        for B in (1, 16, 128):
            lens = self.att_lens[:B]
            nbytes = float((lens * HKV * HD * 4).sum() + B * HQ * HD * 4 + 4 * ((lens + 15) // 16).sum() + 4 * B)
            q, bt, sl = a["q"][:B], a["block_table"][:B], a["seq_lens"][:B]
            out = torch.empty(B, HQ, HD, dtype=torch.bfloat16, device=self.dev)
            t = time_cold(lambda: self.bi.decode_attention(
                q, a["k_cache"], a["v_cache"], bt, sl, max_seq_len=MAX_LEN, out=out,
                workspace=self.ws), reps, flush)
            ns = max(1, min(32, -(-2 * 152 // (B * HKV))))
            ws = torch.zeros(self.bi.decode_attention_workspace_size(B, HQ, HD, ns * 256),
                             dtype=torch.uint8, device=self.dev)
            t_fc = time_cold(lambda: self.bi.decode_attention_fixed_splits(
                q, a["k_cache"], a["v_cache"], bt, sl, MAX_LEN, ns, out=out, workspace=ws),
                reps, flush)
            by_b[str(B)] = {"ms": round(t, 4), "gbs": round(nbytes / t / 1e6, 1),
                            "frac_of_measured_hbm": round(nbytes / t / 1e6 / hbm, 4),
                            "kv_tokens": int(lens.sum()),
                            "fixed_split_count": ns, "fixed_split_count_ms": round(t_fc, 4),
                            "cost_vs_fixed_split_count": round(t / t_fc, 4),
                            "launches": int(self.bi._lib.load().bi_decode_attention_launches(
                                B, HKV, MAX_LEN))}
        res["bi_decode_attention_by_batch"] = by_b
        for name in NEXT_CASES:
            fn, work, unit, info = build_next_case(name, self.dev, self.bi, inputs)
            t = time_cold(fn, reps, flush)
            rate = work / (t * 1e-3) / (1e12 if unit == "TFLOP/s" else 1e9)
            entry = {"ms": round(t, 4), ("tflops" if unit == "TFLOP/s" else "gbs"): round(rate, 2)}
            if unit == "TFLOP/s":
                entry["frac_of_measured_bf16_burst"] = round(rate / bf16, 4)
                entry["gbs"] = round(info.pop("bytes") / t / 1e6, 1)
                entry["bound"] = "tensor (tcgen05)"
            else:
                entry["frac_of_measured_hbm"] = round(rate / hbm, 4)
                entry["bound"] = "hbm"
            kname = "bi_" + name if name != "prefill" else "bi_prefill_attention"
            entry["traffic"] = traffic_record(kname)
            entry.update(info)
            res[kname] = entry
            del fn
        torch.cuda.synchronize()
        self.bi.get_device_error()
        return res

    def references(self, reps: int = 5):
        """Same-run timings of the non-invariant library references."""
        import torch.nn.functional as F
        res = {}

        def timeit(fn):
            fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                fn()
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / reps  # ms

        def cublas():
            for n, N, K in LAYERS:
                torch.matmul(self.gx[K], self.W[n].t(), out=self.gy[n])
        t = timeit(cublas)
        res["cublas_tflops"] = self.gemm_flops / (t * 1e-3) / 1e12
        res["cublas_ms"] = t
        # bi_gemm over the C3 batch sizes: tensor roofline at large M, weight
        # streaming (HBM) at small M; cuBLAS on the same shapes beside it
        by_m = {}
        hbm = load_peaks()[0]
        for M in (1, 8, 64, 256, 1024, 4096):
            xs = {K: self.gx[K][:M] for K in self.gx}
            outs = {n: self.gy[n][:M] for n in self.gy}

            def ours():
                for n, N, K in LAYERS:
                    self.bi.gemm(xs[K], self.W[n], out=outs[n])

            def theirs():
                for n, N, K in LAYERS:
                    torch.matmul(xs[K], self.W[n].t(), out=outs[n])
            t_ours, t_cub = timeit(ours), timeit(theirs)
            flops = sum(2.0 * M * N * K for _, N, K in LAYERS)
            wbytes = sum(2.0 * (N * K + M * K + M * N) for _, N, K in LAYERS)
            by_m[str(M)] = {"ms": round(t_ours, 4), "tflops": round(flops / t_ours / 1e9, 2),
                            "gbs": round(wbytes / t_ours / 1e6, 1),
                            "frac_of_measured_hbm": round(wbytes / t_ours / 1e6 / hbm, 4),
                            "cublas_ms": round(t_cub, 4), "cost_vs_cublas": round(t_ours / t_cub, 4)}
        res["gemm_by_m"] = by_m
        # fixed split COUNT attention (not batch-invariant), with the split
        # count a split-KV kernel would pick to fill 152 SMs at this batch
        ns = max(1, min(32, -(-2 * 152 // (ATT_B * HKV))))
        a = self.att
        ws_fc = torch.zeros(self.bi.decode_attention_workspace_size(ATT_B, HQ, HD, ns * 256),
                            dtype=torch.uint8, device=self.dev)
        t = timeit(lambda: self.bi.decode_attention_fixed_splits(
            a["q"], a["k_cache"], a["v_cache"], a["block_table"], a["seq_lens"], MAX_LEN, ns,
            out=self.att_out, workspace=ws_fc))
        res["fixed_split_count_attention_gbs"] = self.att_bytes / (t * 1e-3) / 1e9
        res["fixed_split_count"] = ns
        if hasattr(F, "rms_norm"):
            t = timeit(lambda: F.rms_norm(self.rx, (HIDDEN,), self.rw, EPS))
            res["torch_rms_norm_gbs"] = self.rms_bytes / (t * 1e-3) / 1e9
            res["torch_rms_norm_ms"] = t
        return res


def run_ours(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    hbm, bf16, bf16_sus, peak_src = load_peaks()

    import __graft_entry__
    __graft_entry__.build()
    wl = Workload(dev)
    invariant = wl.invariance()
    controls = wl.negative_controls()
    refs = wl.references()
    extra = wl.next_rows() if not args.no_next_rows else None

    def barrier():
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier(device_ids=[local])

    for _ in range(max(args.warmup, 0)):
        wl.step()
    barrier()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    h0 = time.perf_counter()
    # After the barrier the GPU is idle, so the first timed kernel would wait
    # for the host to launch it and that wait would be charged to its events.
    # A short device-side spin, queued before the timed region opens, lets the
    # host queue the first steps while it runs.
    if hasattr(torch.cuda, "_sleep"):
        with torch.cuda.stream(wl.stream):
            torch.cuda._sleep(HEAD_START_CYCLES)
    t_start.record(wl.stream)
    for i in range(args.steps):
        wl.step(evs[i])
    t_end.record(wl.stream)
    barrier()
    # The timed steps can be shorter than the sampling interval. So the same step keeps
    # running, untimed, for SOAK_S more seconds. The clocks are taken over the timed steps
    # and that continuation.
    while time.perf_counter() - h0 < SOAK_S:
        for _ in range(20):
            wl.step()
        torch.cuda.synchronize(dev)
    h1 = time.perf_counter()
    barrier()
    clk = clocks.stop(window=(h0, h1))
    clk["window_s"] = round(h1 - h0, 3)
    clk["window"] = "the timed steps plus an untimed continuation of the same step"
    if "sw_power_cap" in clk.get("reasons", []):
        clk["note"] = "software power cap active under the dense GEMMs"
    total_ms = t_start.elapsed_time(t_end)
    rms_ms = sum(e[0].elapsed_time(e[1]) for e in evs)
    gemm_ms = sum(e[1].elapsed_time(e[2]) for e in evs)
    att_ms = sum(e[2].elapsed_time(e[3]) for e in evs)
    total_ms, rms_ms, gemm_ms, att_ms = reduce_max_over_ranks(
        [total_ms, rms_ms, gemm_ms, att_ms], dist, device=dev)
    K = args.steps
    gemm_tflops = weak_scaling_rate(wl.gemm_flops, world, K, gemm_ms) / 1e12
    att_gbs = weak_scaling_rate(wl.att_bytes, world, K, att_ms) / 1e9
    rms_gbs = weak_scaling_rate(wl.rms_bytes, world, K, rms_ms) / 1e9
    per_gpu_gemm = gemm_tflops / world

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(wl, args, dev, barrier, dist, world)
    c5 = None
    if world == 1 and not args.no_c5:
        # the end-to-end C5 run, after every timed region of the line
        torch.cuda.empty_cache()
        c5 = decoder_c5(args.requests, args.layers, args.new_tokens, args.budget, args.track)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    gemm_traffic = traffic_record("bi_gemm")
    line = {
        "metric": METRIC,
        "value": round(gemm_tflops, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / K, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; random-init weights; no dataset)",
        "config": dict(CONFIG, parallelism=f"replicas x{world}"),
        "roofline": {
            "bound": "tensor",
            "achieved": round(per_gpu_gemm, 2),
            "peak": bf16,
            "unit": "TFLOP/s",
            "frac": round(per_gpu_gemm / bf16, 4),
            "traffic": gemm_traffic,
            "peak_source": f"{peak_src} bf16 dense burst (MEASURED_PEAKS.json)" if peak_src == "measured"
                           else "fallback 1.9 PFLOP/s",
            "kernel": "bi_gemm (gemm_tcgen05_pair_kernel), 4 launches per step",
        },
        "components": {
            "bi_gemm": {"tflops": round(per_gpu_gemm, 2), "ms_per_step": round(gemm_ms / K, 4),
                        "frac_of_measured_bf16_burst": round(per_gpu_gemm / bf16, 4),
                        "frac_of_measured_bf16_sustained": round(per_gpu_gemm / bf16_sus, 4),
                        "flops_per_step": wl.gemm_flops,
                        "cublas_tflops_same_run": round(refs["cublas_tflops"], 2),
                        "cost_vs_cublas": round(refs["cublas_tflops"] / per_gpu_gemm, 4)},
            "bi_gemm_by_m": refs["gemm_by_m"],
            "bi_decode_attention": {
                "gbs": round(att_gbs / world, 1), "ms_per_step": round(att_ms / K, 4),
                "frac_of_measured_hbm": round(att_gbs / world / hbm, 4),
                "frac_of_8tbs": round(att_gbs / world / NOMINAL_HBM_GBS, 4),
                "algorithmic_bytes_per_step": wl.att_bytes,
                "fixed_split_count_gbs_same_run": round(refs["fixed_split_count_attention_gbs"], 1),
                "fixed_split_count": refs["fixed_split_count"],
                "cost_vs_fixed_split_count": round(refs["fixed_split_count_attention_gbs"] / (att_gbs / world), 4),
                "traffic": traffic_record("bi_decode_attention")},
            "bi_rmsnorm": {
                "gbs": round(rms_gbs / world, 1), "ms_per_step": round(rms_ms / K, 4),
                "frac_of_measured_hbm": round(rms_gbs / world / hbm, 4),
                "frac_of_8tbs": round(rms_gbs / world / NOMINAL_HBM_GBS, 4),
                "algorithmic_bytes_per_step": wl.rms_bytes,
                "torch_rms_norm_gbs_same_run": round(refs.get("torch_rms_norm_gbs", float("nan")), 1),
                "traffic": traffic_record("bi_rmsnorm")},
        },
        # the components' headline fractions, repeated at the top level
        "cost_vs_cublas": round(refs["cublas_tflops"] / per_gpu_gemm, 4),
        "attention_frac_of_measured_hbm": round(att_gbs / world / hbm, 4),
        "rmsnorm_frac_of_measured_hbm": round(rms_gbs / world / hbm, 4),
        **({"attention_small_batch_frac_of_measured_hbm": {
            b: extra["bi_decode_attention_by_batch"][b]["frac_of_measured_hbm"]
            for b in ("1", "16")}} if extra is not None else {}),
        "bitwise_invariant": all(invariant.values()) and (c5 is None or c5["bitwise_invariant"]),
        **({"next_rows": extra} if extra is not None else {}),
        "invariance_checks": invariant,
        "negative_controls": controls,
        "clocks": clk,
        "gpu_launches": wl.launches_per_step * K,
        # which kernel sources this line measured (the box has no git metadata)
        "kernel_sources_sha256_16": {k: kernel_source_sha(v) for k, v in KERNEL_SOURCES.items()},
    }
    if e2e is not None:
        line["e2e"] = e2e
    if c5 is not None:
        line["c5"] = c5
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


SOAK_S = 0.6  # seconds of the bench step under the clock sampler (timed steps included)
HEAD_START_CYCLES = 1_000_000  # about 0.5 ms of GPU spin before the timed steps
E2E_BUFFER_SETS = 2  # 3 or 4 sets measured the same: the copy engines are the bound
E2E_RUNS = 3  # timed e2e runs; the median is reported


def run_e2e(wl, args, dev, barrier, dist, world):
    """The same step through the Python API with every step's inputs copied
    in from pinned host memory and every output copied back out, pipelined the
    way a serving loop would run it: while step i computes, later steps'
    inputs are copied in and step i-1's outputs copied out (E2E_BUFFER_SETS
    device buffer sets, three streams, event dependencies).  Every step's
    copies are inside the timed region."""
    bi = wl.bi
    host_in = {"rx": wl.rx.cpu().pin_memory(), "q": wl.att["q"].cpu().pin_memory()}
    for K in wl.gx:
        host_in[f"gx{K}"] = wl.gx[K].cpu().pin_memory()
    host_out = {"ry": torch.empty_like(wl.ry, device="cpu").pin_memory(),
                "att": torch.empty_like(wl.att_out, device="cpu").pin_memory()}
    for n in wl.gy:
        host_out[n] = torch.empty_like(wl.gy[n], device="cpu").pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())

    def buffers():
        b = {"rx": torch.empty_like(wl.rx), "q": torch.empty_like(wl.att["q"]),
             "ry": torch.empty_like(wl.ry), "att": torch.empty_like(wl.att_out)}
        for K in wl.gx:
            b[f"gx{K}"] = torch.empty_like(wl.gx[K])
        for n in wl.gy:
            b[n] = torch.empty_like(wl.gy[n])
        return b
    nsets = E2E_BUFFER_SETS
    sets = [buffers() for _ in range(nsets)]
    comp = wl.stream
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_done, comp_done, out_done = ([ev() for _ in range(nsets)] for _ in range(3))
    a = wl.att

    def copy_in(i):
        b = sets[i % nsets]
        with torch.cuda.stream(s_in):
            s_in.wait_event(comp_done[i % nsets])  # step i-nsets finished reading this set
            b["rx"].copy_(host_in["rx"], non_blocking=True)
            b["q"].copy_(host_in["q"], non_blocking=True)
            for K in wl.gx:
                b[f"gx{K}"].copy_(host_in[f"gx{K}"], non_blocking=True)
            in_done[i % nsets].record(s_in)

    def compute(i):
        b = sets[i % nsets]
        comp.wait_event(in_done[i % nsets])
        comp.wait_event(out_done[i % nsets])  # step i-nsets's outputs already copied out
        with torch.cuda.stream(comp):
            bi.rmsnorm(b["rx"], wl.rw, EPS, out=b["ry"])
            for n, N, K in LAYERS:
                bi.gemm(b[f"gx{K}"], wl.W[n], out=b[n])
            bi.decode_attention(b["q"], a["k_cache"], a["v_cache"], a["block_table"],
                                a["seq_lens"], max_seq_len=MAX_LEN, out=b["att"],
                                workspace=wl.ws)
        comp_done[i % nsets].record(comp)

    def copy_out(i):
        b = sets[i % nsets]
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[i % nsets])
            host_out["ry"].copy_(b["ry"], non_blocking=True)
            host_out["att"].copy_(b["att"], non_blocking=True)
            for n in wl.gy:
                host_out[n].copy_(b[n], non_blocking=True)
            out_done[i % nsets].record(s_out)

    def run(n):
        ahead = nsets - 1  # steps whose inputs are copied in ahead of the compute
        for i in range(min(ahead, n)):
            copy_in(i)
        for i in range(n):
            if i + ahead < n:
                copy_in(i + ahead)
            compute(i)
            copy_out(i)

    for e in comp_done + out_done:  # first use: nothing to wait for
        e.record(comp)
    run(max(args.warmup, 1))
    torch.cuda.synchronize(dev)
    # three timed runs of `steps` steps each; the median run is reported (all
    # three are in the line), so one host hiccup does not set the figure
    runs_ms = []
    for _ in range(E2E_RUNS):
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        run(args.steps)
        e1.record(s_out)
        torch.cuda.synchronize(dev)
        barrier()
        runs_ms.append(reduce_max_over_ranks([e0.elapsed_time(e1)], dist, device=dev)[0])
    ms = sorted(runs_ms)[len(runs_ms) // 2]
    # the pipelined outputs equal the device-resident run's
    ok = bool(torch.equal(host_out["down"], wl.gy["down"].cpu()))
    # this box's copy-engine rates, for the floor the step's copies impose
    probe_h = torch.empty(256 << 20, dtype=torch.uint8).pin_memory()
    probe_d = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def copy_ms(fn):
        fn()
        torch.cuda.synchronize(dev)
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record()
        for _ in range(3):
            fn()
        c1.record()
        torch.cuda.synchronize(dev)
        return c0.elapsed_time(c1) / 3
    h2d_gbs = probe_h.numel() / copy_ms(lambda: probe_d.copy_(probe_h, non_blocking=True)) / 1e6
    d2h_gbs = probe_h.numel() / copy_ms(lambda: probe_h.copy_(probe_d, non_blocking=True)) / 1e6
    del probe_h, probe_d
    return {"value": round(weak_scaling_rate(wl.gemm_flops, world, args.steps, ms) / 1e12, 2),
            "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(ms / args.steps, 4),
            "ms_per_step_runs": [round(r / args.steps, 4) for r in runs_ms],
            "outputs_match_device_run": ok,
            "copy_engines_gbs": {"h2d": round(h2d_gbs, 1), "d2h": round(d2h_gbs, 1)},
            "copy_only_ms_per_step": round(h2d / h2d_gbs / 1e6 + d2h / d2h_gbs / 1e6, 4),
            "what": ("GEMM FLOPs of one step / wall time per step through the Python API with "
                     "every step's inputs copied in from pinned memory and all outputs copied "
                     "out, copies of neighbouring steps overlapping the step's kernels; "
                     "median of three timed runs of `steps` steps")}


# ------------------------------------------------------------ CPU oracle ----
def _oracle_sample(x_rows: dict, Ws: dict, att, rms_x, rms_w):
    """Time the oracle on a sample; returns dict of timings and work."""
    import oracle
    res = {}
    t = time.perf_counter()
    flops = 0.0
    for n, N, K in LAYERS:
        oracle.gemm(x_rows[K], Ws[n])
        flops += 2.0 * x_rows[K].shape[0] * N * K
    res["gemm_s"] = time.perf_counter() - t
    res["gemm_flops"] = flops
    t = time.perf_counter()
    oracle.decode_attention(**att)
    res["att_s"] = time.perf_counter() - t
    lens = att["seq_lens"].to(torch.int64)
    res["att_bytes"] = float((lens * HKV * HD * 4).sum() + lens.numel() * HQ * HD * 4)
    t = time.perf_counter()
    oracle.rmsnorm(rms_x, rms_w, EPS)
    res["rms_s"] = time.perf_counter() - t
    res["rms_bytes"] = 4.0 * rms_x.numel()
    return res


def _compact_sequences(a, pick):
    """The listed sequences with only their own pages copied to the host
    (block table renumbered), so the oracle never touches the full cache."""
    bt = a["block_table"][pick].cpu()
    used = bt[bt >= 0].unique()
    remap = torch.full((int(a["k_cache"].shape[0]),), -1, dtype=torch.int32)
    remap[used.long()] = torch.arange(used.numel(), dtype=torch.int32)
    nbt = torch.where(bt >= 0, remap[bt.clamp(min=0).long()], bt)
    idx = used.long().to(a["k_cache"].device)
    return {"q": a["q"][pick].cpu(), "k_cache": a["k_cache"][idx].cpu(),
            "v_cache": a["v_cache"][idx].cpu(), "block_table": nbt.contiguous(),
            "seq_lens": a["seq_lens"][pick].cpu()}


def cpu_baseline(wl):
    """The oracle as it stands, on the host cores, on a bounded sample of the
    same workload (about 10-30 s of CPU work)."""
    import oracle
    Ws = {n: W.cpu() for n, W in wl.W.items()}
    att = _compact_sequences(wl.att, [0, 1])
    # calibrate the GEMM sample (rows per layer) to ~12 s
    rows = 4
    probe = _oracle_sample({K: wl.gx[K][:rows].cpu() for K in wl.gx}, Ws, att,
                           wl.rx[:64].cpu(), wl.rw.cpu())
    rows = int(max(4, min(2048, rows * 12.0 / max(probe["gemm_s"], 1e-3))))
    r = _oracle_sample({K: wl.gx[K][:rows].cpu() for K in wl.gx}, Ws, att,
                       wl.rx[:256].cpu(), wl.rw.cpu())
    return {"value": round(r["gemm_flops"] / r["gemm_s"] / 1e12, 6), "unit": "TFLOP/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": (f"fp64 oracle GEMM on the first {rows} rows of each of the 4 layers "
                       f"({r['gemm_flops'] / 1e9:.1f} GFLOP in {r['gemm_s']:.1f} s); attention on 2 "
                       f"sequences: {r['att_bytes'] / r['att_s'] / 1e9:.3f} GB/s; rmsnorm 256 rows: "
                       f"{r['rms_bytes'] / r['rms_s'] / 1e9:.3f} GB/s")}


def run_reference(args):
    """The fp64 oracle, as it stands, timed on the host cores: each step is a
    bounded sample of the same workload (8 GEMM rows per layer, 2 attention
    sequences, 64 RMSNorm rows)."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    import oracle
    from invariant_bi_rmsnorm_gb300 import inputs
    oracle.build_oracle()
    Ws = {n: inputs.gemm_weight(N, K, seed=40 + i) for i, (n, N, K) in enumerate(LAYERS)}
    xs = {K: inputs.gemm_rows(8, K, seed=50 + K) for K in sorted({K for _, _, K in LAYERS})}
    att = inputs.decode_problem(2, Hq=HQ, Hkv=HKV, D=HD, seq_lens=[4096, 4097], seed=270)
    rx = inputs.rmsnorm_rows(64, HIDDEN, seed=3)
    rw = inputs.rmsnorm_weight(HIDDEN, seed=4)
    for _ in range(max(args.warmup, 0)):
        _oracle_sample(xs, Ws, att, rx, rw)
    t0 = time.perf_counter()
    gemm_s = flops = 0.0
    for _ in range(args.steps):
        r = _oracle_sample(xs, Ws, att, rx, rw)
        gemm_s += r["gemm_s"]
        flops += r["gemm_flops"]
    wall = time.perf_counter() - t0
    value = flops / gemm_s / 1e12
    sample = "fp64 oracle: 8 GEMM rows per layer, 2 attention sequences (L=4096,4097), 64 RMSNorm rows per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(wall / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": CONFIG,
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


PREFILL_BUDGET = 8192  # tokens of one prefill step
LOGPROB_ROWS, VOCAB = 1024, 151936
OPS_TOKENS = 8192


def build_next_case(name: str, dev, bi, inputs):
    """Full-size input of one kernel beyond the bench step, as (fn, work, unit,
    info).  `work` is the algorithmic bytes (GB/s cases) or FLOPs (TFLOP/s)
    of one launch.  Shared by the default line's cold-L2 measurements and by
    `--case` (the command the ncu captures use)."""
    if name == "prefill":
        # one step of whole-prompt prefill: prompts of U[32, 512] tokens until
        # the 8192-token budget is full, causal attention over each prompt
        lens_all = inputs.seq_lens_uniform(64, 512, seed=610, min_len=32).tolist()
        lens, tot = [], 0
        for L in lens_all:
            if tot + L > PREFILL_BUDGET:
                break
            lens.append(L)
            tot += L
        p = inputs.decode_problem(len(lens), Hq=HQ, Hkv=HKV, D=HD, seq_lens=lens, seed=611,
                                  device=dev)
        q = inputs.normal_bf16((tot, HQ, HD), 612, device=dev)
        a = {k: v.to(dev) for k, v in p.items() if k != "q"}
        indptr = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device=dev)
        out = torch.empty(tot, HQ, HD, dtype=torch.bfloat16, device=dev)
        pws = torch.empty(max(1, bi.prefill_attention_workspace_size(tot, HQ, HD, max(lens))),
                          dtype=torch.uint8, device=dev)
        fn = lambda: bi.prefill_attention(q, a["k_cache"], a["v_cache"], a["block_table"],  # noqa: E731
                                          a["seq_lens"], indptr, max_q_len=max(lens),
                                          max_seq_len=max(lens), out=out, workspace=pws)
        flops = float(sum(4.0 * HD * HQ * L * (L + 1) / 2 for L in lens))
        nbytes = float(2 * tot * HQ * HD * 2 + sum(L * HKV * HD * 4 for L in lens))
        return fn, flops, "TFLOP/s", {"sequences": len(lens), "tokens": tot,
                                      "prompt_len": "U[32,512]", "bytes": nbytes}
    if name == "add_rmsnorm":
        x = inputs.rmsnorm_rows(RMS_ROWS, HIDDEN, seed=3, device=dev)
        res = inputs.rmsnorm_rows(RMS_ROWS, HIDDEN, seed=13, device=dev)
        w = inputs.rmsnorm_weight(HIDDEN, seed=4, device=dev)
        y = torch.empty_like(x)
        fn = lambda: bi.add_rmsnorm(x, res, w, EPS, out=y)  # noqa: E731
        return fn, 4.0 * 2 * RMS_ROWS * HIDDEN + 2 * HIDDEN, "GB/s", {
            "rows": RMS_ROWS, "hidden": HIDDEN,
            "bytes_per_row": "x read, residual read + write, y write"}
    if name == "logprobs":
        logits = inputs.normal_bf16((LOGPROB_ROWS, VOCAB), 620, device=dev)
        tgt = torch.randint(0, VOCAB, (LOGPROB_ROWS,), generator=torch.Generator().manual_seed(621),
                            dtype=torch.int64).to(torch.int32).to(dev)
        fn = lambda: bi.logprobs(logits, tgt)  # noqa: E731
        return fn, float(LOGPROB_ROWS * VOCAB * 2 + LOGPROB_ROWS * 12), "GB/s", {
            "rows": LOGPROB_ROWS, "vocab": VOCAB}
    if name == "qk_norm_rope_append":
        T = OPS_TOKENS
        qkv = inputs.normal_bf16((T, (HQ + 2 * HKV) * HD), 630, device=dev)
        npages = T // 16
        kc = torch.empty(npages, HKV, 16, HD, dtype=torch.bfloat16, device=dev)
        vc = torch.empty_like(kc)
        g = torch.Generator().manual_seed(631)
        pos = torch.randint(0, 8192, (T,), generator=g, dtype=torch.int64).to(torch.int32).to(dev)
        slots = torch.randperm(npages * 16, generator=g).to(torch.int32).to(dev)
        from invariant_bi_rmsnorm_gb300.qwen3 import rope_table
        rope = rope_table(8192, 1e6, HD, device=dev)
        ones = torch.ones(HD, dtype=torch.bfloat16, device=dev)
        qo = torch.empty(T, HQ, HD, dtype=torch.bfloat16, device=dev)
        fn = lambda: bi.qk_norm_rope_append(qkv, HQ, HKV, pos, slots, rope, ones, ones,  # noqa: E731
                                            kc, vc, EPS, q_out=qo)
        per_tok = (HQ + 2 * HKV) * HD * 2 + HQ * HD * 2 + 2 * HKV * HD * 2 + HD * 4 + 8
        return fn, float(T * per_tok), "GB/s", {
            "tokens": T, "bytes_per_token": "qkv read, q write, k/v cache write, rope row, "
                                           "position and slot"}
    if name == "gemm_swiglu":
        # the decoder MLP's gate|up projection fused with SwiGLU, M = 4096 tokens
        F, K = 12288, HIDDEN
        x = inputs.gemm_rows(GEMM_M, K, seed=50 + K, device=dev)
        W = bi.interleave_gate_up(inputs.gemm_weight(2 * F, K, seed=42, device=dev))
        h = torch.empty(GEMM_M, F, dtype=torch.bfloat16, device=dev)
        fn = lambda: bi.gemm_swiglu(x, W, out=h)  # noqa: E731
        return fn, 2.0 * GEMM_M * 2 * F * K, "TFLOP/s", {
            "M": GEMM_M, "F": F, "K": K,
            "bytes": float(2 * (GEMM_M * K + 2 * F * K + GEMM_M * F))}
    if name == "silu_mul":
        T, F = OPS_TOKENS, 12288
        gu = inputs.normal_bf16((T, 2 * F), 640, device=dev)
        h = torch.empty(T, F, dtype=torch.bfloat16, device=dev)
        fn = lambda: bi.silu_mul(gu, out=h)  # noqa: E731
        return fn, float(T * 3 * F * 2), "GB/s", {"tokens": T, "ffn": F}
    raise ValueError(name)


NEXT_CASES = ("prefill", "add_rmsnorm", "logprobs", "qk_norm_rope_append", "silu_mul",
              "gemm_swiglu")


def time_cold(fn, reps: int, flush: torch.Tensor) -> float:
    """Mean device time (ms) of fn over reps launches, L2 flushed before each
    by reading a buffer twice the size of L2 (outside the timed events).  A
    read leaves clean lines behind; overwriting the buffer instead would leave
    L2 full of dirty lines whose write-back the timed kernel would pay for."""
    fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    for e0, e1 in evs:
        torch.sum(flush)
        e0.record()
        fn()
        e1.record()
    torch.cuda.synchronize()
    return sum(e0.elapsed_time(e1) for e0, e1 in evs) / reps


def run_case(args):
    """One kernel of the path, launched steps + warmup times on its full-size
    input: the small, self-contained command the ncu captures use."""
    import __graft_entry__
    import invariant_bi_rmsnorm_gb300 as bi
    from invariant_bi_rmsnorm_gb300 import inputs
    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if args.case == "gemm_layers":
        # the bench step's four GEMM launches (qkv, o, gate_up, down at M = 4096)
        xs = {K: inputs.gemm_rows(GEMM_M, K, seed=50 + K, device=dev) for _, _, K in LAYERS}
        Ws = [inputs.gemm_weight(N, K, seed=40 + i, device=dev) for i, (_, N, K) in enumerate(LAYERS)]
        ys = [torch.empty(GEMM_M, N, dtype=torch.bfloat16, device=dev) for _, N, _ in LAYERS]

        def fn():
            for (_, N, K), W, y in zip(LAYERS, Ws, ys):
                bi.gemm(xs[K], W, out=y)
        work, unit = sum(2.0 * GEMM_M * N * K for _, N, K in LAYERS), "TFLOP/s"
    elif args.case in NEXT_CASES:
        fn, work, unit, _ = build_next_case(args.case, dev, bi, inputs)
    elif args.case.startswith("gemm"):
        n, N, K = {"gemm_gate_up": LAYERS[2], "gemm_qkv": LAYERS[0]}[args.case]
        x = inputs.gemm_rows(GEMM_M, K, seed=50 + K, device=dev)
        W = inputs.gemm_weight(N, K, seed=42, device=dev)
        y = torch.empty(GEMM_M, N, dtype=torch.bfloat16, device=dev)
        fn, work, unit = (lambda: bi.gemm(x, W, out=y)), 2.0 * GEMM_M * N * K, "TFLOP/s"
    elif args.case == "attention":
        B = args.batch
        p = inputs.decode_problem(B, max_len=MAX_LEN, seed=270, device=dev)
        a = {k: v.to(dev) for k, v in p.items()}
        out = torch.empty(B, HQ, HD, dtype=torch.bfloat16, device=dev)
        ws = torch.zeros(bi.decode_attention_workspace_size(B, HQ, HD, MAX_LEN),
                         dtype=torch.uint8, device=dev)
        lens = p["seq_lens"].to(torch.int64)
        work = float((lens * HKV * HD * 4).sum() + B * HQ * HD * 4 + 4 * ((lens + 15) // 16).sum())
        fn = lambda: bi.decode_attention(a["q"], a["k_cache"], a["v_cache"], a["block_table"],  # noqa: E731
                                         a["seq_lens"], max_seq_len=MAX_LEN, out=out, workspace=ws)
        unit = "GB/s"
    else:
        x = inputs.rmsnorm_rows(RMS_ROWS, HIDDEN, seed=3, device=dev)
        w = inputs.rmsnorm_weight(HIDDEN, seed=4, device=dev)
        y = torch.empty_like(x)
        fn, work, unit = (lambda: bi.rmsnorm(x, w, EPS, out=y)), 4.0 * RMS_ROWS * HIDDEN, "GB/s"
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    bi.get_device_error()
    ms = e0.elapsed_time(e1) / max(args.steps, 1)
    scale = 1e12 if unit == "TFLOP/s" else 1e9
    print(json.dumps({"case": args.case, "ms_per_launch": round(ms, 4),
                      "value": round(work / (ms * 1e-3) / scale, 2), "unit": unit}), flush=True)


TORCH_ARM_SWAPS = ("GEMMs -> torch.matmul (cuBLAS, unfused gate|up then bi_silu_mul) and RMSNorms "
                   "-> torch.nn.functional.rms_norm; attention, q/k norm + RoPE + KV append and "
                   "SwiGLU stay on this library, so the bi arm's fused gate|up+SwiGLU GEMM is "
                   "part of the wall-time difference, not only the cost of invariance")


def decoder_c5(requests: int = 1000, layers: int = 36, new_tokens: int = 100,
               budget: int = 8192, track: int = 16) -> dict:
    """The random-init Qwen3-8B-shaped decoder served with continuous batching:
    `requests` prompts of U[32, 512] random tokens, `new_tokens` greedy tokens
    each, at most `budget` tokens per step (prompts split across steps as
    needed).  Timed: the whole batched run (wall clock, host scheduling
    included).  Then `track` requests are re-run alone and their logits
    compared bit for bit with the batched run at every generated token; the
    same batched run with torch/cuBLAS GEMMs and torch RMSNorms swapped in is
    timed and checked the same way, as the non-invariant comparison."""
    import __graft_entry__
    from invariant_bi_rmsnorm_gb300 import qwen3
    __graft_entry__.build()
    cfg = qwen3.Qwen3Config(layers=layers)
    w = qwen3.Qwen3Weights(cfg, seed=1000)

    def make_requests():
        return qwen3.random_requests(requests, cfg.vocab, 32, 512, new_tokens, seed=7)

    reqs = make_requests()
    pages = sum(-(-(len(r.prompt) + new_tokens) // 16) for r in reqs) + 64
    tracked = sorted({int(i) for i in np.linspace(0, requests - 1, track)})
    result = {"requests": requests, "layers": layers,
              "prompt_len": "U[32,512]", "new_tokens": new_tokens,
              "max_tokens_per_step": budget, "model": "random-init Qwen3-8B-shaped "
              "(hidden 4096, FFN 12288, 32/8 heads, d128, vocab 151936, RoPE 1e6)",
              "prompt_tokens": int(sum(len(r.prompt) for r in reqs)),
              "torch_arm_swaps": TORCH_ARM_SWAPS}
    for ops in ("bi", "torch"):
        eng = qwen3.Engine(w, num_pages=pages, max_tokens_per_step=budget, ops=ops)
        warm = qwen3.random_requests(4, cfg.vocab, 32, 64, 2, seed=99)
        eng.generate(warm)
        eng.reset()
        reqs = make_requests()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        logs = eng.generate(reqs, record=set(tracked))
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        steps = eng.steps
        mism_logits = mism_tokens = 0
        for sid in tracked:
            eng.reset()
            one = qwen3.Sequence(sid=sid, prompt=list(reqs[sid].prompt), max_new=new_tokens)
            alone = eng.generate([one], record={sid})
            mism_tokens += int(one.generated != reqs[sid].generated)
            mism_logits += sum(int(not torch.equal(a, b)) for a, b in zip(alone[sid], logs[sid]))
        toks = result["prompt_tokens"] + requests * new_tokens
        result[ops] = {"wall_s": round(wall, 3), "steps": steps,
                       "tokens_per_s": round(toks / wall, 1),
                       "tracked_requests": len(tracked),
                       "logit_rows_compared": len(tracked) * new_tokens,
                       "logit_rows_differing_alone_vs_batched": mism_logits,
                       "requests_whose_tokens_differ": mism_tokens}
        del eng
        torch.cuda.empty_cache()
    del w
    torch.cuda.empty_cache()
    result["bitwise_invariant"] = result["bi"]["logit_rows_differing_alone_vs_batched"] == 0
    result["cost_vs_torch_ops"] = round(result["bi"]["wall_s"] / result["torch"]["wall_s"], 4)
    return result


def run_decoder(args):
    """`--case decoder`: the C5 decoder run alone, its own JSON line."""
    torch.cuda.set_device(0)
    res = decoder_c5(args.requests, args.layers, args.new_tokens, args.budget, args.track)
    print(json.dumps({"case": "decoder", **res}), flush=True)


def run_decode_latency(args):
    """Small-batch decode on the random-init Qwen3-8B-shaped decoder: B
    requests of 128 prompt tokens each generate 64 tokens; ms per decode step
    with eager launches and with CUDA-graph steps (bit-identical logits; the
    graphs remove per-launch host work).  Wall clock of the whole generate
    call divided by its steps, after a warm-up run that captures the graphs."""
    import __graft_entry__
    from invariant_bi_rmsnorm_gb300 import qwen3
    __graft_entry__.build()
    torch.cuda.set_device(0)
    cfg = qwen3.Qwen3Config(layers=args.layers)
    w = qwen3.Qwen3Weights(cfg, seed=1000)
    out = {"case": "decode_latency", "layers": args.layers, "prompt_len": 128,
           "new_tokens": 64, "unit": "ms per step"}
    for B in (1, 8, 64, 256):
        row = {}
        for graphs in (False, True):
            eng = qwen3.Engine(w, num_pages=B * 16 + 64, max_tokens_per_step=8192,
                               cuda_graphs=graphs)
            eng.generate(qwen3.random_requests(B, cfg.vocab, 128, 128, 4, seed=6))
            eng.reset()
            reqs = qwen3.random_requests(B, cfg.vocab, 128, 128, 64, seed=5)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            eng.generate(reqs)
            torch.cuda.synchronize()
            row["graphs" if graphs else "eager"] = round((time.perf_counter() - t0) / eng.steps * 1e3, 3)
            del eng
            torch.cuda.empty_cache()
        out[str(B)] = row
    print(json.dumps(out), flush=True)


def main():
    args = parse_args()
    if args.case == "decoder":
        run_decoder(args)
    elif args.case == "decode_latency":
        run_decode_latency(args)
    elif args.case:
        run_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
