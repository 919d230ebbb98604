#!/usr/bin/env python
"""Throughput of the fused Q4_K SwiGLU feed-forward block on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Default workload: one 4096 -> 11008 -> 4096 Q4_K SwiGLU layer at T=2048 tokens
(bf16 activations with 1% outlier rows x20, weights N(0, 0.02) quantised with
the min/max quantiser; seed 2).  A step is one call of the block over the
whole batch, inputs resident in HBM, L2 flushed (512 MB write) between steps
outside the timed events.  The single-token dense workload instead rotates over
twelve copies of its weights (913 MB, more than six L2s) and runs its steps
back to back, as consecutive layers of a decode step do: every step still streams its
weights from HBM.  Under torchrun each rank runs its own replica of
the workload on its own GPU (no collective on the data path: tokens are
independent), so the scaling is weak and `value` is the tokens of all ranks
divided by the slowest rank's time.

The JSON line carries: the device-timed throughput (`value`, tok/s) and
TFLOP/s, the end-to-end throughput with host buffers through the library's
host pipeline (`e2e`: each step's x uploaded from and y downloaded to pinned
host memory, overlapped with the neighbouring steps' blocks, wall clock), the
roofline of the dominant kernel (the fused tensor-core kernel, timed alone
through the residual entry point), the CPU oracle timed on this host's cores
on a bounded sample (`cpu_baseline`), SM clocks sampled during the timed
region, and the number of this library's kernels launched.  Dense lines add
the RMSNorm in front of the block (`rmsnorm`), routed lines the device router
(`router`), single-token lines the block with W_down in the other block
formats (`down_formats`), each timed on its own.

--impl reference times the CPU oracle itself (the only reference this
build has: the source pages publish no code) on the same workload and metric.
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
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused Q4_K SwiGLU-MLP tok/s & TFLOP/s at T=2048; % of BF16 TC / HBM roof"
L2_FLUSH_BYTES = 512 << 20

WORKLOADS = {
    # name: (kind, T, H, I, seed, outlier_frac, E, top_k)
    "prefill_T2048": ("dense", 2048, 4096, 11008, 2, 0.01, 1, 1),
    "prefill_T256": ("dense", 256, 4096, 11008, 1, 0.0, 1, 1),
    "decode_T1": ("dense", 1, 4096, 11008, 3, 0.0, 1, 1),
    "moe_T256": ("moe", 256, 2048, 768, 4, 0.0, 128, 8),
    "moe_T1": ("moe", 1, 2048, 768, 4, 0.0, 128, 8),
}
DESCR = {
    "prefill_T2048": "Q4_K SwiGLU layer H=4096 I=11008, T=2048 prefill, 1% outlier rows x20 (seed 2)",
    "prefill_T256": "Q4_K SwiGLU layer H=4096 I=11008, T=256 prefill (seed 1)",
    "decode_T1": "Q4_K SwiGLU layer H=4096 I=11008, T=1 decode, one token per step (seed 3)",
    "moe_T256": "Q4_K MoE layer E=128 H=2048 I=768 top-8, T=256 (seed 4)",
    "moe_T1": "Q4_K MoE layer E=128 H=2048 I=768 top-8, T=1 (seed 4)",
}


def row_bytes(cols):
    return ((cols + 255) // 256) * 144


def algorithmic(kind, T, H, I, E, k):
    """FLOP and HBM bytes the method must move once (Q4_K weights read once at
    4.5 bits/weight, x read once in bf16, y written once in fp32)."""
    if kind == "dense":
        flop = 6.0 * T * H * I
        wbytes = 2 * I * row_bytes(H) + H * row_bytes(I)
    else:
        flop = 6.0 * T * k * H * I
        per_expert = 2 * I * row_bytes(H) + H * row_bytes(I)
        touched = E if T * k >= E else min(E, T * k)
        wbytes = touched * per_expert
    return flop, wbytes + T * H * 2 + T * H * 4


def max_over_ranks(values, dist, device):
    """Each value's maximum over the ranks: the slowest replica's times."""
    import torch
    t = torch.tensor(list(values), device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_rates(tokens_per_rank, flop_per_rank, world, ms):
    """Whole-job tokens/s and TFLOP/s of `world` replicas, each doing the same
    work, timed by the slowest (ms per step)."""
    return (tokens_per_rank * world / (ms * 1e-3),
            flop_per_rank * world / (ms * 1e-3) / 1e12)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# Source files that define the dominant kernel of each workload: a committed
# ncu traffic figure stays valid while these files are unchanged.
KERNEL_SOURCES = {
    "prefill": ("ffn_tc.cu", "zffn_internal.cuh"),
    "moe": ("moe_tc.cu", "moe_route.cu", "zffn_internal.cuh"),
    "decode": ("ffn_matvec.cu", "zffn_internal.cuh"),
}


def kernel_source_hash(workload=None):
    """sha256 (16 hex digits) over the kernel sources of `workload` (all of
    csrc when None)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_ffn_gb300", "csrc")
    names = sorted(os.listdir(csrc))
    if workload is not None:
        kind = "moe" if workload.startswith("moe") else (
            "decode" if workload.startswith("decode") else "prefill")
        if workload == "moe_T1":
            kind = "decode"
        names = sorted(KERNEL_SOURCES[kind])
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", f"ncu_{workload}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256_16") != kernel_source_hash(workload):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


THROTTLE_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clocks_rejected(clocks):
    """Why a timed region's clock record rejects its numbers, or None if they
    stand: a hardware or thermal slowdown, or a median SM clock under load
    well below the maximum with no reason reported (a clock lock left
    behind).  A power cap is normal under a dense load and is kept."""
    reasons = clocks.get("reasons") or []
    bad = [r for r in reasons if r in THROTTLE_REASONS]
    if bad:
        return ",".join(bad)
    sm, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    if sm and mx and sm < 0.85 * mx and "sw_power_cap" not in reasons:
        return "SM clock %.0f of %.0f MHz with no reason reported" % (sm, mx)
    return None


class ClockSampler:
    """nvidia-smi samples every 100 ms while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        except Exception:
            pass
        finally:
            if self.path and os.path.exists(self.path):
                os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[5 + i]
                          and "Not" not in r[5 + i]})
        loaded = [s for s in sm if s >= 0.5 * max(sm)] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "samples": len(rows), "reasons": reasons}


# ---------------------------------------------------------------------------
# inputs
# ---------------------------------------------------------------------------

def make_host_inputs(name):
    from quantized_ffn_gb300 import synth
    kind, T, H, I, seed, outl, E, k = WORKLOADS[name]
    if kind == "dense":
        if name == "decode_T1":
            d = synth.decode(n_tokens=1000, seed=seed, H=H, I=I)
        else:
            d = synth.prefill(T, seed, H, I, outl)
        return d
    return synth.MoE(T, seed=seed, E=E, H=H, I=I, top_k=k)


def quantize_on_gpu(w_f32, torch, zffn):
    t = torch.from_numpy(w_f32).cuda()
    q = zffn.q4k_quantize(t)
    del t
    return q


# ---------------------------------------------------------------------------
# GPU leg
# ---------------------------------------------------------------------------

def run_gpu(args):
    import torch
    import torch.distributed as dist

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from quantized_ffn_gb300 import build as zbuild
    zbuild.build()
    from quantized_ffn_gb300 import zffn

    name = args.workload
    kind, T, H, I, seed, outl, E, k = WORKLOADS[name]
    flop, abytes = algorithmic(kind, T, H, I, E, k)
    peaks = load_peaks()

    host = make_host_inputs(name)
    dev = torch.device("cuda", local)
    if kind == "dense":
        W = [quantize_on_gpu(host[n], torch, zffn) for n in ("Wg_f32", "Wu_f32", "Wd_f32")]
        x_all = torch.from_numpy(host["x"].view(np.int16)).to(dev).view(torch.bfloat16)
        ids = wts = None
    else:
        Wg = torch.empty((E, I, row_bytes(H)), dtype=torch.uint8, device=dev)
        Wu = torch.empty_like(Wg)
        Wd = torch.empty((E, H, row_bytes(I)), dtype=torch.uint8, device=dev)
        for e in range(E):
            g, u, d = host.expert_f32(e)
            Wg[e] = quantize_on_gpu(g, torch, zffn)
            Wu[e] = quantize_on_gpu(u, torch, zffn)
            Wd[e] = quantize_on_gpu(d, torch, zffn)
        W = [Wg, Wu, Wd]
        x_all = torch.from_numpy(host.x.view(np.int16)).to(dev).view(torch.bfloat16)
        # the layer's router turns the logits into ids and weights on the
        # device, once, before the timed steps (the block reads them as inputs)
        logits_dev = torch.from_numpy(host.logits).to(dev)
        ids, wts = zffn.moe_router_topk(logits_dev, k)
    torch.cuda.synchronize()
    # Decode reads 76 MB per token, less than the L2: rotate over copies of the
    # weights at different addresses so that every step streams from HBM.
    wbytes = sum(w.numel() for w in W)
    n_sets = 1
    if name == "decode_T1" or name == "moe_T1":
        # between two uses of a copy at least six L2s' worth of other copies
        # stream through, so (whatever the replacement policy) next to none
        # of it is still in L2
        n_sets = max(1, math.ceil(6 * 129e6 / wbytes) + 1)
    sets = [W] + [[w.clone() for w in W] for _ in range(n_sets - 1)]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    # Dense decode touches all of a copy every step, and the copies together
    # exceed the L2, so its steps need no flush.  (The routed layer touches
    # only the token's experts, which could stay in L2 across copies: it is
    # flushed.)
    flush_between = name != "decode_T1"

    def maybe_flush():
        if flush_between:
            flush.zero_()
    y = torch.empty((T, H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    zffn.reserve(max(T, 1), H, I, E, k)

    def x_for(step):
        if name == "decode_T1":
            r = step % x_all.shape[0]
            return x_all[r:r + 1]
        return x_all

    def call(step, residual=False):
        Wg_, Wu_, Wd_ = sets[step % n_sets]
        if kind == "dense":
            zffn.swiglu_q4k(x_for(step), Wg_, Wu_, Wd_, I, y=y, residual=residual)
        else:
            zffn.moe_swiglu_q4k(x_for(step), ids, wts, Wg_, Wu_, Wd_, I, E, y=y, residual=residual)

    launches_per_call = 2                          # x conversion (+ zero fill) + fused kernel, or gate/up + down
    if kind == "moe" and T == 1:
        launches_per_call = zffn.single_token_launches(H, I, E, k)   # one cooperative launch, or the pair
    if kind == "moe" and T > 1:
        launches_per_call = 3                      # route, gather (+ fp16, + zero fill of y), grouped kernel

    def barrier():
        if world > 1:
            dist.barrier()

    for s in range(args.warmup):
        maybe_flush()
        call(s)
    torch.cuda.synchronize()
    assert zffn.get_device_error() == zffn.OK

    def timed(step_fn):
        """Mean device time of one step over args.steps steps: events around
        each step when the L2 is flushed between steps (outside the events),
        else one pair of events around the back-to-back steps."""
        if flush_between:
            st = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
            en = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
            for s in range(args.steps):
                maybe_flush()
                st[s].record(stream)
                step_fn(s)
                en[s].record(stream)
            torch.cuda.synchronize()
            return statistics.mean(a.elapsed_time(b) for a, b in zip(st, en))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for s in range(args.steps):
            step_fn(s)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    def measure():
        barrier()
        torch.cuda.synchronize()
        with ClockSampler(local) as clk:
            wall0 = time.perf_counter()
            ms = timed(lambda s: call(s))
            wall = time.perf_counter() - wall0
            barrier()
            # the dominant kernel alone: the residual entry skips the zero fill
            kms = timed(lambda s: call(s, residual=True))
        return ms, wall, kms, clk.summary()

    ms, wall, kms, clocks = measure()
    why = clocks_rejected(clocks)
    # every rank re-measures if any rank's clock record rejects its number
    redo = bool(why) if world == 1 else max_over_ranks([1.0 if why else 0.0], dist, dev)[0] > 0
    if redo:
        first = dict(clocks, rejected=why or "another rank's clock record")
        ms, wall, kms, clocks = measure()
        clocks["first_run"] = first
    assert zffn.get_device_error() == zffn.OK

    # End to end through the library's host pipeline: every step uploads its
    # x from pinned host memory and downloads its y into pinned host memory,
    # overlapped with the neighbouring steps' blocks; wall clock from the
    # first submission to the final sync.
    n_rows = x_all.shape[0]
    x_rows = torch.empty(tuple(x_all.shape), dtype=torch.bfloat16, pin_memory=True)
    x_rows.copy_(x_all)
    y_bufs = [torch.empty((T, H), dtype=torch.float32, pin_memory=True) for _ in range(2)]
    pipe = zffn.Pipeline(T, H, I, 2)

    def host_x(step):
        if name == "decode_T1":
            r = step % n_rows
            return x_rows[r:r + 1]
        return x_rows

    # The routed single-token steps run back to back here, without the L2
    # flush of the device-timed loop: so that they do not keep reusing the
    # same 8 experts' weights from L2, each step takes the route of another
    # token (64 extra seeded logit rows through the device router).
    routes = [(ids, wts)]
    if kind == "moe" and T == 1:
        more = np.random.default_rng(seed + 1000).standard_normal((64, E)).astype(np.float32)
        r_ids, r_wts = zffn.moe_router_topk(torch.from_numpy(more).to(dev), k)
        routes = [(r_ids[i:i + 1], r_wts[i:i + 1]) for i in range(64)]
        torch.cuda.synchronize()

    def submit_all(n):
        for s in range(n):
            Wg_, Wu_, Wd_ = sets[s % n_sets]
            if kind == "dense":
                pipe.submit(host_x(s), Wg_, Wu_, Wd_, y_bufs[s % 2])
            else:
                r_ids, r_wts = routes[s % len(routes)]
                pipe.submit_moe(host_x(s), r_ids, r_wts, Wg_, Wu_, Wd_, E, y_bufs[s % 2])
        pipe.sync()
    submit_all(args.warmup)
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    submit_all(args.steps)
    e2e_ms = (time.perf_counter() - t0) * 1e3 / args.steps
    pipe.close()
    assert zffn.get_device_error() == zffn.OK
    e2e_in, e2e_out = int(host_x(0).numel() * 2), int(y_bufs[0].numel() * 4)
    e2e_how = ("zffn_pipeline (host buffers, upload / block / download on three streams, "
               "overlapped across steps), wall clock")

    # the normalisation in front of the dense block (fp32 residual stream ->
    # bf16 block input), timed on its own over the workload's rows
    norm = None
    if kind == "dense":
        h_res = x_all[:T].float().contiguous()
        gamma = torch.ones(H, dtype=torch.float32, device=dev)
        xn = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        # (one call between events after an L2 flush, whatever the workload:
        # back to back, a one-row call would time the host, not the kernel)
        n_st = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        n_en = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for s in range(args.steps):
            flush.zero_()
            n_st[s].record(stream)
            zffn.rmsnorm_bf16(h_res, gamma, 1e-6, out=xn)
            n_en[s].record(stream)
        torch.cuda.synchronize()
        n_ms = statistics.mean(a.elapsed_time(b) for a, b in zip(n_st, n_en))
        n_bytes = T * H * 6 + H * 4
        n_gbs = n_bytes / (n_ms * 1e-3) / 1e9
        norm = {"kernel": "rmsnorm_bf16_kernel", "ms": round(n_ms, 5), "hbm_bytes": n_bytes,
                "achieved_gbs": round(n_gbs, 2), "frac_of_hbm_peak": round(n_gbs / peaks["hbm"], 4)}
        if T == 1:
            # one token: the pre-norm residual block folds the normalisation
            # into the gate/up kernel (two launches); the block alone, same
            # setting, beside it
            h_row = h_res.clone()
            p_ms, b_ms = [], []
            for s in range(args.steps):
                for fn, acc in ((lambda: zffn.swiglu_q4k_prenorm_residual(h_row, gamma, 1e-6, W[0], W[1], W[2], I),
                                 p_ms),
                                (lambda: zffn.swiglu_q4k(x_for(0), W[0], W[1], W[2], I, y=y), b_ms)):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    flush.zero_()
                    e0.record(stream)
                    fn()
                    e1.record(stream)
                    acc.append((e0, e1))
            torch.cuda.synchronize()
            assert zffn.get_device_error() == zffn.OK
            norm["prenorm_block_ms"] = round(statistics.mean(a.elapsed_time(b) for a, b in p_ms), 5)
            norm["block_ms"] = round(statistics.mean(a.elapsed_time(b) for a, b in b_ms), 5)
            norm["prenorm_block_launches"] = 2
            norm["prenorm_timing"] = "one isolated call after an L2 flush, each"

    # The staged pipeline the fusion replaces ("Fused SwiGLU MLP...", sections
    # "Counting the bytes the intermediate actually moves" and "What it is
    # worth"): dequantise each matrix to a 16-bit scratch copy, then the gate
    # and up GEMMs, the SwiGLU as its own pass, the down GEMM -- four
    # dispatches with the intermediate crossing device memory six times.
    # Benchmark-only: the library's dequantisation kernel, cuBLAS (torch.matmul)
    # and torch's elementwise kernels; nothing of it is in the library.
    staged = None
    if kind == "dense" and T > 1:
        import torch.nn.functional as F
        wf = [torch.empty((I, H), dtype=torch.float32, device=dev), torch.empty((I, H), dtype=torch.float32, device=dev),
              torch.empty((H, I), dtype=torch.float32, device=dev)]
        wb = [torch.empty_like(w, dtype=torch.bfloat16) for w in wf]
        gs = torch.empty((T, I), dtype=torch.bfloat16, device=dev)
        us = torch.empty_like(gs)
        hs = torch.empty_like(gs)
        ys = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        xs = x_for(0)

        def dequant_all():
            for q, (r_, c_), f, b in zip(W, ((I, H), (I, H), (H, I)), wf, wb):
                zffn.q4k_dequant(q, r_, c_, out=f)
                b.copy_(f)

        def gemms():
            torch.matmul(xs, wb[0].t(), out=gs)
            torch.matmul(xs, wb[1].t(), out=us)
            torch.mul(F.silu(gs), us, out=hs)
            torch.matmul(hs, wb[2].t(), out=ys)

        def staged_call():
            dequant_all()
            gemms()

        for _ in range(args.warmup):          # first calls carry library set-up
            staged_call()
        torch.cuda.synchronize()
        s_ms = timed(lambda s: staged_call())
        g_ms = timed(lambda s: gemms())
        torch.cuda.synchronize()
        y_f = zffn.swiglu_q4k(xs, W[0], W[1], W[2], I)
        rel = float(torch.linalg.vector_norm(ys.float() - y_f) / torch.linalg.vector_norm(y_f))
        staged = {"what": "dequant (library kernel) to fp32 and bf16 scratch, cuBLAS gate and up "
                          "GEMMs, SwiGLU (torch elementwise), cuBLAS down GEMM; bf16 operands, "
                          "timed like the fused call",
                  "ms": round(s_ms, 4), "ms_gemms_only": round(g_ms, 4),
                  "ms_dequant_to_scratch": round(s_ms - g_ms, 4),
                  "fused_ms": round(ms, 4), "fused_speedup": round(s_ms / ms, 3),
                  "fused_speedup_vs_gemms_only": round(g_ms / ms, 3),
                  "intermediate_dram_bytes": {"staged_model": 6 * T * I * 2, "fused_measured": 0,
                                              "how": "staged: g and u written, read by the SwiGLU, "
                                                     "h written and read by the down GEMM (bf16); "
                                                     "fused: ncu DRAM writes of the fused kernel "
                                                     "are y only"},
                  "rel_l2_vs_fused": round(rel, 5)}
        del wf, wb, gs, us, hs, ys

    # blocks with W_down in the other block formats (W_gate and W_up the
    # workload's Q4_K matrices, W_down seeded random blocks of the format),
    # one call between events after an L2 flush: the single-token workloads,
    # and the routed layer at T > 1 (the grouped tensor-core kernel)
    down_formats = None
    if T == 1 or kind == "moe":
        from quantized_ffn_gb300 import synth as _synth
        down_formats = {}
        rng_f = np.random.default_rng(seed + 2000)
        for fname, fmt in (("Q5_K", zffn.FMT_Q5_K), ("Q6_K", zffn.FMT_Q6_K), ("Q5_1", zffn.FMT_Q5_1)):
            Wd_f = torch.from_numpy(np.stack([_synth.random_blocks(rng_f, fmt, H, I, 1e-3)
                                              for _ in range(E)])).to(dev)
            f_st = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
            f_en = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
            for s in range(args.steps + 2):
                flush.zero_()
                if s >= 2:
                    f_st[s - 2].record(stream)
                if kind == "dense":
                    zffn.swiglu_q4k_wd(x_for(0), W[0], W[1], Wd_f, fmt, I, y=y)
                else:
                    zffn.moe_swiglu_q4k_wd(x_for(0), ids, wts, W[0], W[1], Wd_f, fmt, I, E, y=y)
                if s >= 2:
                    f_en[s - 2].record(stream)
            torch.cuda.synchronize()
            assert zffn.get_device_error() == zffn.OK
            f_ms = statistics.mean(a.elapsed_time(b) for a, b in zip(f_st, f_en))
            touched = 1 if kind == "dense" else (k if T == 1 else int(torch.unique(ids[ids >= 0]).numel()))
            f_bytes = touched * (2 * I * row_bytes(H) + H * zffn.row_bytes_fmt(fmt, I)) + T * H * 2 + T * H * 4
            f_gbs = f_bytes / (f_ms * 1e-3) / 1e9
            down_formats[fname] = {"ms": round(f_ms, 5), "hbm_bytes": f_bytes,
                                   "achieved_gbs": round(f_gbs, 1),
                                   "frac_of_hbm_peak": round(f_gbs / peaks["hbm"], 4)}
            del Wd_f

    # the router of the routed layer (logits -> ids, weights), timed on its own
    router = None
    if kind == "moe":
        ids_r, wts_r = torch.empty_like(ids), torch.empty_like(wts)
        r_ms = timed(lambda s: zffn.moe_router_topk(logits_dev, k, ids_r, wts_r))
        assert torch.equal(ids_r, ids) and torch.equal(wts_r, wts)
        r_bytes = T * E * 4 + T * k * 8
        router = {"kernel": "moe_router_kernel", "ms": round(r_ms, 5),
                  "hbm_bytes": r_bytes, "achieved_gbs": round(r_bytes / (r_ms * 1e-3) / 1e9, 2),
                  "frac_of_hbm_peak": round(r_bytes / (r_ms * 1e-3) / 1e9 / peaks["hbm"], 5)}

    if world > 1:
        ms, kms, e2e_ms = max_over_ranks([ms, kms, e2e_ms], dist, dev)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    value, tflops = job_rates(T, flop, world, ms)
    # prefill is a dense contraction; decode and the routed layer stream weights
    bound = "tensor" if name.startswith("prefill") else "hbm"
    if bound == "tensor":
        achieved = flop / (kms * 1e-3) / 1e12
        peak, unit = peaks["bf16"], "TFLOP/s"
    else:
        achieved = abytes / (kms * 1e-3) / 1e9
        peak, unit = peaks["hbm"], "GB/s"
    traffic = profiled_traffic(name)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(name, host, seconds=args.cpu_seconds)
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tok/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": DESCR[name],
            "name": name, "T": T, "H": H, "I": I,
            **({"E": E, "top_k": k} if kind == "moe" else {}),
            "parallelism": "replicas" if world > 1 else "single-gpu",
            "l2": ("flushed between steps (512 MB write outside the timed events)"
                   + (f"; weights rotated over {n_sets} copies" if n_sets > 1 else ""))
                  if flush_between else
                  (f"inputs larger than L2: weights rotated over {n_sets} copies "
                   f"({n_sets * wbytes / 1e6:.0f} MB), steps back to back, no flush"),
        },
        "tflops": round(tflops, 2),
        "roofline": {
            "bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "kernel": "x_to_f16_kernel+ffn_tc_kernel" if bound == "tensor" else
                      (("ffn_token_fused_kernel" if kind == "moe" and launches_per_call == 1 else
                        "ffn_gu_kernel+ffn_down_kernel") if T == 1 else
                       "moe_route_kernel+moe_gather_kernel+moe_group_kernel"),
            "kernel_ms": round(kms, 4),
            "peak_source": f"{peaks['source']} (burst)",
            "algorithmic": {"flop": flop, "hbm_bytes": abytes},
        },
        "e2e": {"value": round(T * world / (e2e_ms * 1e-3), 1), "unit": "tok/s",
                "h2d_bytes_per_step": e2e_in,
                "d2h_bytes_per_step": e2e_out,
                "ms_per_step": round(e2e_ms, 4), "how": e2e_how},
        "cpu_baseline": cpu,
        **({"router": router} if router is not None else {}),
        **({"rmsnorm": norm} if norm is not None else {}),
        **({"staged": staged} if staged is not None else {}),
        **({"down_formats": {"kernels": ("ffn_gu_kernel + down_fmt_kernel" if T == 1 else
                                         "moe_route_kernel + moe_gather_kernel + moe_group_kernel<F>"),
                             "timing": "one isolated call after an L2 flush", **down_formats}}
           if down_formats is not None else {}),
        "clocks": clocks,
        "gpu_launches": launches_per_call * args.steps,
        "wall_s_timed_loop": round(wall, 4),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and --impl reference)
# ---------------------------------------------------------------------------

def oracle_layer(name, host):
    from oracle import oracle as orc
    kind = WORKLOADS[name][0]
    if kind == "dense":
        return dict(Wg=orc.q4k_quantize(host["Wg_f32"]), Wu=orc.q4k_quantize(host["Wu_f32"]),
                    Wd=orc.q4k_quantize(host["Wd_f32"]))
    E = host.E
    Wg = np.empty((E, host.I, row_bytes(host.H)), np.uint8)
    Wu = np.empty_like(Wg)
    Wd = np.empty((E, host.H, row_bytes(host.I)), np.uint8)
    for e in range(E):
        g, u, d = host.expert_f32(e)
        Wg[e], Wu[e], Wd[e] = orc.q4k_quantize(g), orc.q4k_quantize(u), orc.q4k_quantize(d)
    return dict(Wg=Wg, Wu=Wu, Wd=Wd)


def oracle_tokens(name, host, layer, rows):
    from oracle import oracle as orc
    kind, T, H, I, seed, outl, E, k = WORKLOADS[name]
    if kind == "dense":
        x = host["x"][rows].copy()
        return orc.swiglu_ffn(x, layer["Wg"], layer["Wu"], layer["Wd"], len(rows), H, I)
    ids, w = orc.route_top_k(host.logits[rows].copy(), k)
    return orc.moe_swiglu_ffn(host.x[rows].copy(), ids, w, layer["Wg"], layer["Wu"], layer["Wd"],
                              len(rows), H, I, E, k)


def _oracle_rate(name, host, layer, seconds, per_call):
    """Tokens per second of the oracle on consecutive tokens of the workload,
    calls of per_call tokens, for about `seconds`."""
    n_rows = host["x"].shape[0] if isinstance(host, dict) else host.x.shape[0]
    done, t0, r = 0, time.perf_counter(), 0
    while time.perf_counter() - t0 < seconds:
        rows = [(r + i) % n_rows for i in range(per_call)]
        oracle_tokens(name, host, layer, rows)
        done += per_call
        r += per_call
    return done, time.perf_counter() - t0


def cpu_baseline(name, host, seconds=10.0):
    """The oracle timed on this host's cores: its source built with OpenMP on
    all cores (the row loops in parallel) and the plain single-threaded
    build, each on a bounded sample of the workload's tokens; plus the
    dequantisation of one weight matrix on its own (the part of every call
    that does not depend on the tokens)."""
    from oracle import oracle as orc
    layer = oracle_layer(name, host)
    T = WORKLOADS[name][1]
    kind = WORKLOADS[name][0]
    per_call = 4 if T > 1 else 1
    ncores = os.cpu_count() or 1
    try:
        ncores = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        pass
    Wg = layer["Wg"] if kind == "dense" else layer["Wg"][0]
    rows, cols = Wg.shape[0], WORKLOADS[name][2]

    def dequant_s():
        t0 = time.perf_counter()
        orc.q4k_dequant(Wg, rows, cols)
        return time.perf_counter() - t0

    d1 = dequant_s()
    n1, t1 = _oracle_rate(name, host, layer, seconds * 0.5, per_call)
    out = {"value": round(n1 / t1, 3), "unit": "tok/s", "cores": 1, "kind": "oracle",
           "sample": f"{n1} tokens of the workload in calls of {per_call} (full weights; the "
                     f"oracle dequantises every weight row once per call)",
           "dequant_s_one_matrix": {"rows": rows, "cols": cols, "1_core": round(d1, 4)}}
    omp = orc.build_omp()
    if omp is not None:
        prev = orc.use_library(omp)
        try:
            dn = dequant_s()
            per_n = max(per_call, ncores) if T > 1 else 1
            nn, tn = _oracle_rate(name, host, layer, seconds * 0.5, per_n)
        finally:
            orc.use_library(prev)
        out["dequant_s_one_matrix"]["all_cores"] = round(dn, 4)
        # the all-cores build is the headline baseline; the plain build stays beside it
        single = {k: out[k] for k in ("value", "cores", "sample")}
        out.update({"value": round(nn / tn, 3), "cores": ncores,
                    "sample": f"{nn} tokens in calls of {per_n}, oracle built with OpenMP "
                              f"(row loops over {ncores} cores)",
                    "single_core": single})
    return out


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    name = args.workload
    kind, T, H, I, seed, outl, E, k = WORKLOADS[name]
    host = make_host_inputs(name)
    layer = oracle_layer(name, host)
    n_rows = host["x"].shape[0] if isinstance(host, dict) else host.x.shape[0]
    per_step = 2 if T > 1 else 1
    for s in range(args.warmup):
        oracle_tokens(name, host, layer, [(s * per_step + i) % n_rows for i in range(per_step)])
    times = []
    for s in range(args.steps):
        rows = [((s + args.warmup) * per_step + i) % n_rows for i in range(per_step)]
        t0 = time.perf_counter()
        oracle_tokens(name, host, layer, rows)
        times.append(time.perf_counter() - t0)
    mean = statistics.mean(times)
    value = per_step / mean
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "tok/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(mean * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": DESCR[name], "name": name, "T": T, "H": H, "I": I},
        "cpu_baseline": {"value": round(value, 3), "unit": "tok/s", "cores": 1, "kind": "oracle",
                         "sample": f"{per_step} token(s) of the workload per step"},
        "e2e": {"value": round(value, 3), "unit": "tok/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="prefill_T2048", choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
