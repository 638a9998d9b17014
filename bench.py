#!/usr/bin/env python3
"""Benchmark of the ring-attention hot path on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one pass of the whole path over one batch of synthetic input resident in
HBM: natural -> rank-major permutation of Q, K and V, the fused ring-attention
kernel (every virtual rank's queries against the KV blocks in ring order), and the
inverse permutation of the output and its log-sum-exp.  The metric is
causal-adjusted attention TFLOP/s: 4*B*Hq*d*S^2 per step, halved when causal.

Several GPUs run independent replicas of the same workload (the c virtual ranks of
the ring all live on one GPU; there is no data-path collective).  --impl reference
times the float64 CPU oracle on the host cores on a bounded sample of the workload.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from online_softmax_attention_zigzag_gb300.configs import (  # noqa: E402
    CAUSAL_GQA_S32K, CAUSAL_MHA_S4K, WORKLOADS, with_layout)
from online_softmax_attention_zigzag_gb300.inputs import doc_ids, make_qkv, sample_rows  # noqa: E402

METRIC = "causal-adjusted attention TFLOP/s and % of GB300 bf16 tensor peak, 1 GPU"
# GB300 dense bf16 tensor rate: NVIDIA's HGX B300 datasheet lists 36 PFLOPS FP16/BF16 for
# eight GPUs with 2:4 sparsity, i.e. 4.5 PFLOPS sparse and 2.25 PFLOPS dense per GPU.
NOMINAL_BF16_TFLOPS = 2250.0
UNIT = "TFLOP/s"
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
# the attention kernel's source and the headers it includes (its device code lives in all three)
KERNEL_SRCS = tuple(os.path.join(ROOT, "online_softmax_attention_zigzag_gb300", "csrc", f)
                    for f in ("attn_bf16.cu", "ptx.cuh", "internal.h"))


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=CAUSAL_GQA_S32K.name, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU-oracle sample budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the 128k workload and the natural-order step measured beside the headline")
    ap.add_argument("--per-hop-sweep", action="store_true",
                    help="instead of the headline: fused vs per-hop + merge over the workload's kv_block sweep")
    ap.add_argument("--backward", action="store_true",
                    help="instead of the headline: the backward pass (ringattn_bwd) on the workload")
    ap.add_argument("--ulysses", action="store_true",
                    help="instead of the headline: Ulysses on one GPU (relayouts + attention) on the workload")
    ap.add_argument("--attention-only", action="store_true",
                    help="instead of the headline: the attention kernel alone on the workload, --steps launches")
    ap.add_argument("--per-rank", action="store_true",
                    help="instead of the headline: one launch per virtual rank, both layouts (4k MHA and the workload)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return j.get("bf16_tflops"), j.get("bf16_tflops_sustained"), j.get("hbm_gbs"), "measured"
    return FALLBACK_BF16_TFLOPS, None, FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln.strip())


def src_hash() -> str:
    """Fingerprint of the attention kernel's code: SHA-256 of its source file and the
    headers it includes, each with the comments and blank lines taken out, so that a
    comment edit keeps a recorded traffic figure and any code edit drops it."""
    h = hashlib.sha256()
    for path in KERNEL_SRCS:
        with open(path, encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
        h.update(b"\0")
    return h.hexdigest()[:16]


def traffic_for(workload: str):
    """DRAM bytes per launch of the attention kernel from the committed ncu summary, or
    None when there is none for this workload or the kernel changed since."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        j = json.load(f)
    e = j.get(workload)
    if not e or e.get("attn_kernel_code_sha256_16") != src_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            ident = str(device_index)
        self.cmd = ["nvidia-smi", "-i", ident, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", "200"]

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(self.cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle baseline
CPU_UNIT_ROWS = 4096  # query rows per timed unit of the CPU oracle (one full_attention_rows call)


def cpu_oracle_units(w, qkv, budget_s: float, first_unit: int = 0, min_units: int = 1, check=None):
    """Time the float64 oracle on units of CPU_UNIT_ROWS seeded random query rows of
    workload ``w`` (unit i draws its rows with seed 7000 + i), until ``budget_s`` seconds
    of oracle time and at least ``min_units`` units are spent.  Returns a list of
    (flop, seconds) per unit.  Input generation is not timed.  The GPU arm's cpu_baseline
    and the reference arm both time these units, so they report the same quantity.
    ``check(heads, positions, out, lse)``, if given, receives each unit's oracle rows
    after its timing."""
    from oracle.attention import full_attention_rows
    q, k, v = qkv
    res, spent, i = [], 0.0, first_unit
    while spent < budget_s or len(res) < min_units:
        hs, ps = sample_rows(w.bhq, w.seq, CPU_UNIT_ROWS, seed=7000 + i)
        hs, ps = hs.numpy(), ps.numpy()
        keys = (ps + 1) if w.causal else np.full_like(ps, w.seq)
        flop = float(np.sum(4.0 * w.d * keys))
        t0 = time.perf_counter()
        o, l = full_attention_rows(q, k, v, hs, ps, bool(w.causal))
        dt = time.perf_counter() - t0
        res.append((flop, dt))
        spent += dt
        i += 1
        if check is not None:
            check(hs, ps, o, l)
    return res


# bf16 tolerances on the output and the natural-log lse (max abs error)
TOL_OUT, TOL_LSE = 2e-2, 1e-3


class RowParity:
    """Max abs error of a natural-order GPU result held in host memory (out [BH, S, d],
    lse [BH, S]) against the oracle rows that the cpu_baseline leg computes anyway.  A
    failure inside the comparison is recorded, never raised, so that it cannot cost the
    bench its line."""

    def __init__(self, out_h: torch.Tensor, lse_h: torch.Tensor, source: str):
        self.out_h, self.lse_h, self.source = out_h, lse_h, source
        self.rows, self.nonfinite = 0, 0
        self.err_out, self.err_lse = 0.0, 0.0
        self.error = None

    def __call__(self, hs, ps, o, l):
        try:
            h = torch.from_numpy(np.asarray(hs, dtype=np.int64))
            pos = torch.from_numpy(np.asarray(ps, dtype=np.int64))
            go = self.out_h[h, pos].to(torch.float64).numpy()
            gl = self.lse_h[h, pos].to(torch.float64).numpy()
            finite = np.isfinite(go).all(axis=1) & np.isfinite(gl)
            self.nonfinite += int(np.count_nonzero(~finite))
            if finite.any():
                self.err_out = max(self.err_out, float(np.max(np.abs(go[finite] - o[finite]))))
                self.err_lse = max(self.err_lse, float(np.max(np.abs(gl[finite] - l[finite]))))
            self.rows += len(h)
        except Exception as e:  # recorded in the line instead
            self.error = f"{type(e).__name__}: {e}"

    def summary(self) -> dict:
        ok = (self.error is None and self.rows > 0 and self.nonfinite == 0
              and self.err_out <= TOL_OUT and self.err_lse <= TOL_LSE)
        return {"output_of": self.source, "rows": self.rows,
                "sample": "the cpu_baseline leg's seeded random query rows",
                "max_abs_err_out": self.err_out, "max_abs_err_lse": self.err_lse,
                "nonfinite_rows": self.nonfinite, "tolerance": {"out": TOL_OUT, "lse": TOL_LSE},
                "within_tolerance": ok, "error": self.error}


def cpu_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        if info:
            return max(i.get("num_threads", 1) for i in info)
    except Exception:
        pass
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def run_reference(args, w, rank):
    """The reference arm: the float64 CPU oracle as it stands, one unit of
    CPU_UNIT_ROWS sampled query rows per step, rank 0 only."""
    if rank != 0:
        return
    qkv = make_qkv(w)
    units = cpu_oracle_units(w, qkv, 0.0, first_unit=0, min_units=args.warmup + args.steps)[args.warmup:]
    flop = sum(f for f, _ in units)
    secs = sum(t for _, t in units)
    value = flop / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1))",
        "config": {"workload": w.name, "S": w.seq, "Hq": w.hq, "Hkv": w.hkv, "d": w.d, "c": w.c,
                   "causal": w.causal, "layout": "zigzag" if w.layout else "contiguous", "batch": w.batch},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                         "sample": f"{args.steps} units of {CPU_UNIT_ROWS} seeded random query rows "
                                   f"({secs:.1f} s), float64 numpy"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ multi-GPU helpers
def max_over_ranks(values, dist, device):
    """Element-wise max of per-rank timings (the slowest replica sets the step time)."""
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


# Dense bf16 tensor work per SM per clock: one 128x128x16 tcgen05.mma (2*128*128*16 FLOP)
# every 64 cycles, measured on this GPU with a single-SM stream of MMAs.
TENSOR_FLOP_PER_CLK_PER_SM = 8192


def clock_ceiling(achieved_tflops, clk, device):
    """The kernel's fraction of the tensor ceiling at the SM clock seen during the timed
    region (SMs x 8192 FLOP/clk x median SM MHz), beside the cuBLAS-burst fraction."""
    mhz = clk.get("sm_mhz") if clk else None
    if not mhz:
        return {"clock_ceiling": None, "frac_of_clock_ceiling": None}
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    ceil_tf = sms * TENSOR_FLOP_PER_CLK_PER_SM * mhz * 1e6 / 1e12
    return {"clock_ceiling": ceil_tf, "frac_of_clock_ceiling": achieved_tflops / ceil_tf,
            "clock_ceiling_how": f"{sms} SMs x {TENSOR_FLOP_PER_CLK_PER_SM} FLOP/clk x {mhz:.0f} MHz (median SM clock "
                                 "in the timed region)"}


def whole_job_value(flop_per_step: float, world: int, ms_per_step: float) -> float:
    """TFLOP/s of all replicas together: every rank runs one step of the workload."""
    return world * flop_per_step / (ms_per_step * 1e-3) / 1e12


# ------------------------------------------------------------------ GPU arm
def time_events(fn, reps, stream):
    """Mean device time (ms) of fn() over reps calls, CUDA events on `stream`."""
    fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def doc_flops(w, doc) -> float:
    """Attention FLOP of the visible pairs under the document mask: 4*d per pair, per head;
    a document of L tokens holds L(L+1)/2 causal pairs."""
    lens = torch.bincount(doc.to(torch.int64)).to(torch.float64)
    return 4.0 * w.d * w.bhq * float((lens * (lens + 1) / 2).sum())


def attention_only(ra, w, dev, stream, reps, peak):
    """Fused kernel on rank-major device inputs of workload w: TFLOP/s and fraction of peak.
    A workload with packed documents runs the document-masked all-gather kernel."""
    q_h, k_h, v_h = make_qkv(w)
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    del q_h, k_h, v_h
    qr, kr, vr = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    for src, dst in ((q, qr), (k, kr), (v, vr)):
        ra.permute(src, dst, c=w.c, layout=w.layout, inverse=0)
    del q, k, v
    o = torch.empty((w.bhq, w.seq, w.d), dtype=torch.float32, device=dev)
    l = torch.empty((w.bhq, w.seq), dtype=torch.float32, device=dev)
    if w.doc_len:
        doc = doc_ids(w.seq, *w.doc_len)
        doc_d = doc.to(dev)
        ds = torch.empty_like(doc_d)
        ms = time_events(lambda: ra.fwd_docmask(qr, kr, vr, o, l, doc_d, ds, c=w.c, layout=w.layout), reps, stream)
        flop = doc_flops(w, doc)
        what = {"kernel": "doc_start_kernel + attn_bf16_kernel<%d, true>" % w.d,
                "documents": int(doc[-1]) + 1, "flop": "visible pairs only (causal inside each document)"}
    else:
        kw = dict(c=w.c, causal=w.causal, layout=w.layout, kv_block=w.kv_block)
        ms = time_events(lambda: ra.fwd(qr, kr, vr, o, l, **kw), reps, stream)
        flop = w.flops()
        what = {"kernel": "attn_bf16_kernel<%d, false>" % w.d}
    if ra.sync_status() != ra.RA_OK:
        raise SystemExit("device wait timed out")
    tf = flop / (ms * 1e-3) / 1e12
    return {"workload": w.name, "kernel_ms": ms, "achieved": tf, "unit": "TFLOP/s", "peak": peak,
            "frac": tf / peak, "launches": reps + 1, **what}


def ulysses_only(ra, w, dev, stream, reps, peak, hbm_peak):
    """Ulysses on one GPU for workload w: the all-to-all relayout of q, k, v to head
    shards, attention of every rank's heads over the whole sequence, relayout of out and
    lse back.  TFLOP/s of the whole call, and GB/s of the q relayout alone."""
    q_h, k_h, v_h = make_qkv(w)
    seq = []
    for x in (q_h, k_h, v_h):
        xd = x.to(dev)
        xs = torch.empty((w.seq, xd.shape[0], w.d), dtype=xd.dtype, device=dev)
        ra.relayout(xd, xs, c=w.c, layout=w.layout, to_heads=0)   # natural heads -> sequence shards
        seq.append(xs)
        del xd
    del q_h, k_h, v_h
    qs, ks, vs = seq
    o = torch.empty((w.seq, w.bhq, w.d), dtype=torch.float32, device=dev)
    l = torch.empty((w.seq, w.bhq), dtype=torch.float32, device=dev)
    ws = torch.empty(ra.host_workspace_bytes(w.seq, w.bhq, w.bhkv, w.d), dtype=torch.uint8, device=dev)
    ms = time_events(lambda: ra.ulysses_fwd(qs, ks, vs, o, l, ws, c=w.c, causal=w.causal, layout=w.layout),
                     reps, stream)
    qh = torch.empty((w.bhq, w.seq, w.d), dtype=qs.dtype, device=dev)
    ms_q = time_events(lambda: ra.relayout(qs, qh, c=w.c, layout=w.layout, to_heads=1), reps, stream)
    if ra.sync_status() != ra.RA_OK:
        raise SystemExit("device wait timed out")
    tf = w.flops() / (ms * 1e-3) / 1e12
    qbytes = 2 * qs.numel() * qs.element_size()
    return {"workload": w.name, "mode": "Ulysses (relayout q, k, v; attention per head group; relayout out, lse)",
            "ms": ms, "achieved": tf, "unit": "TFLOP/s", "peak": peak, "frac": tf / peak,
            "relayout_q": {"kernel": "relayout_kernel<uint4>", "ms": ms_q, "bytes": qbytes,
                           "GB/s": qbytes / (ms_q * 1e-3) / 1e9, "frac": qbytes / (ms_q * 1e-3) / 1e9 / hbm_peak}}


def backward_only(ra, w, dev, stream, reps, peak):
    """ringattn_bwd on workload w (rank-major device tensors, the forward's out and lse):
    TFLOP/s of the whole call (delta, dq and dk/dv kernels) with the backward counted as
    2.5 forward passes (five tile products of 2*d FLOP per visible pair against two)."""
    q_h, k_h, v_h = make_qkv(w)
    g = torch.Generator().manual_seed(221)
    do_h = torch.randn((w.bhq, w.seq, w.d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    t = []
    for x in (q_h, k_h, v_h, do_h):
        xd = x.to(dev)
        xr = torch.empty_like(xd)
        ra.permute(xd, xr, c=w.c, layout=w.layout, inverse=0)
        t.append(xr)
        del xd
    qr, kr, vr, dor = t
    o = torch.empty((w.bhq, w.seq, w.d), dtype=torch.float32, device=dev)
    l = torch.empty((w.bhq, w.seq), dtype=torch.float32, device=dev)
    kw = dict(c=w.c, causal=w.causal, layout=w.layout, kv_block=w.kv_block)
    ra.fwd(qr, kr, vr, o, l, **kw)
    dq = torch.empty_like(o)
    dk = torch.empty((w.bhkv, w.seq, w.d), dtype=torch.float32, device=dev)
    dv = torch.empty_like(dk)
    delta = torch.empty_like(l)
    ms = time_events(lambda: ra.bwd(qr, kr, vr, o, l, dor, dq, dk, dv, delta, **kw), reps, stream)
    if ra.sync_status() != ra.RA_OK:
        raise SystemExit("device wait timed out")
    flop = 2.5 * w.flops()
    tf = flop / (ms * 1e-3) / 1e12
    return {"workload": w.name, "mode": "backward (ringattn_bwd: delta, dq, dk/dv kernels)", "ms": ms,
            "achieved": tf, "unit": "TFLOP/s", "peak": peak, "frac": tf / peak,
            "flop": "2.5 x the causal-adjusted forward FLOP"}


def per_hop_sweep(ra, w, dev, stream, reps=3):
    """Fused kernel vs the ring-faithful per-hop path (one partial per message, folded in
    with the merge kernel) for each kv_block of the workload's sweep."""
    q_h, k_h, v_h = make_qkv(w)
    qr, kr, vr = (torch.empty(x.shape, dtype=x.dtype, device=dev) for x in (q_h, k_h, v_h))
    for src, dst in ((q_h, qr), (k_h, kr), (v_h, vr)):
        ra.permute(src.to(dev), dst, c=w.c, layout=w.layout, inverse=0)
    o = torch.empty((w.bhq, w.seq, w.d), dtype=torch.float32, device=dev)
    l = torch.empty((w.bhq, w.seq), dtype=torch.float32, device=dev)
    op, lp = torch.empty_like(o), torch.empty_like(l)
    rows = w.bhq * w.seq
    out = []
    for kvb in (w.kv_sweep or (w.kv_block,)):
        kw = dict(c=w.c, causal=w.causal, layout=w.layout, kv_block=kvb)
        fused_ms = time_events(lambda: ra.fwd(qr, kr, vr, o, l, **kw), reps, stream)
        n_msg = (w.seq // w.c) // kvb

        def ring():
            o.zero_()
            l.fill_(-float("inf"))
            for hop in range(w.c):
                for sub in range(n_msg):
                    ra.fwd_hop(qr, kr, vr, op, lp, hop=hop, sub=sub, **kw)
                    ra.merge(o, l, op, lp)
        ring_ms = time_events(ring, 1, stream)
        merge_ms = time_events(lambda: ra.merge(o, l, op, lp), reps, stream)
        mbytes = rows * (12 * w.d + 12)
        out.append({"kv_block": kvb, "messages": w.c * n_msg, "fused_ms": fused_ms,
                    "fused_tflops": w.flops() / (fused_ms * 1e-3) / 1e12, "per_hop_ms": ring_ms,
                    "per_hop_tflops": w.flops() / (ring_ms * 1e-3) / 1e12, "merge_ms": merge_ms,
                    "merge_gbs": mbytes / (merge_ms * 1e-3) / 1e9,
                    "merge_traffic_gib": w.c * n_msg * mbytes / 2**30})
    if ra.sync_status() != ra.RA_OK:
        raise SystemExit("device wait timed out")
    return out


def per_rank(ra, workloads, dev, stream, reps=5):
    """One ringattn_fwd_rank launch per virtual rank, contiguous and zigzag: device time,
    128x128 tiles and visible (query, key) pairs of each rank.  The time of a ring step is
    the slowest rank's; zigzag evens the ranks out."""
    out = []
    for w0 in workloads:
        for layout in (0, 1):
            w = with_layout(w0, layout)
            q_h, k_h, v_h = make_qkv(w)
            qr, kr, vr = (torch.empty(x.shape, dtype=x.dtype, device=dev) for x in (q_h, k_h, v_h))
            for src, dst in ((q_h, qr), (k_h, kr), (v_h, vr)):
                ra.permute(src.to(dev), dst, c=w.c, layout=w.layout, inverse=0)
            o = torch.empty((w.bhq, w.seq, w.d), dtype=torch.float32, device=dev)
            l = torch.empty((w.bhq, w.seq), dtype=torch.float32, device=dev)
            kw = dict(c=w.c, causal=w.causal, layout=w.layout, kv_block=w.kv_block)
            units, pairs, tiles = ra.rank_work(w.seq, w.c, w.causal, w.layout, 128)
            ranks = []
            for r in range(w.c):
                ms = time_events(lambda: ra.fwd_rank(qr, kr, vr, o, l, rank=r, **kw), reps, stream)
                fl = 4.0 * w.d * w.bhq * float(pairs[r])
                ranks.append({"rank": r, "kernel_ms": ms, "units": int(units[r]), "tiles_per_head": int(tiles[r]),
                              "pairs_per_head": int(pairs[r]), "tflops": fl / (ms * 1e-3) / 1e12})
            full_ms = time_events(lambda: ra.fwd(qr, kr, vr, o, l, **kw), reps, stream)
            t = [x["kernel_ms"] for x in ranks]
            out.append({"workload": w.name, "layout": "zigzag" if layout else "contiguous", "ranks": ranks,
                        "max_over_min_ms": max(t) / min(t), "sum_ms": sum(t), "all_ranks_one_launch_ms": full_ms})
            del qr, kr, vr, o, l
            torch.cuda.empty_cache()
    if ra.sync_status() != ra.RA_OK:
        raise SystemExit("device wait timed out")
    return out


def main():
    args = parse()
    w = WORKLOADS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, w, rank)
        return
    if w.dtype != "bf16":
        raise SystemExit("the bench times the bf16 tensor-core path; pick a bf16 workload")

    from online_softmax_attention_zigzag_gb300 import ringattn as ra
    ra.lib()
    torch.cuda.set_device(local)
    if args.per_hop_sweep:
        dev = torch.device("cuda", local)
        res = per_hop_sweep(ra, w, dev, torch.cuda.current_stream(dev))
        if rank == 0:
            print(json.dumps({"metric": METRIC, "unit": UNIT, "mode": "per-hop sweep", "workload": w.name,
                              "sweep": res}), flush=True)
        return
    if args.backward:
        dev = torch.device("cuda", local)
        res = backward_only(ra, w, dev, torch.cuda.current_stream(dev), max(1, args.steps), peaks()[0])
        if rank == 0:
            print(json.dumps({"metric": METRIC, "unit": UNIT, **res}), flush=True)
        return
    if args.ulysses:
        dev = torch.device("cuda", local)
        res = ulysses_only(ra, w, dev, torch.cuda.current_stream(dev), max(1, args.steps), peaks()[0], peaks()[2])
        if rank == 0:
            print(json.dumps({"metric": METRIC, "unit": UNIT, **res}), flush=True)
        return
    if args.attention_only:
        dev = torch.device("cuda", local)
        res = attention_only(ra, w, dev, torch.cuda.current_stream(dev), max(1, args.steps), peaks()[0])
        if rank == 0:
            print(json.dumps({"metric": METRIC, "unit": UNIT, "mode": "attention kernel only", **res}), flush=True)
        return
    if w.doc_len:
        raise SystemExit("packed-document workloads are timed with --attention-only")
    if args.per_rank:
        dev = torch.device("cuda", local)
        res = per_rank(ra, [CAUSAL_MHA_S4K, w], dev, torch.cuda.current_stream(dev))
        if rank == 0:
            print(json.dumps({"metric": METRIC, "unit": UNIT, "mode": "per-rank launches", "per_rank": res}),
                  flush=True)
        return
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier()

    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    S, c, L = w.seq, w.c, w.layout
    q_h, k_h, v_h = make_qkv(w)
    q_h, k_h, v_h = q_h.pin_memory(), k_h.pin_memory(), v_h.pin_memory()
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    qr, kr, vr = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    o_r = torch.empty((w.bhq, S, w.d), dtype=torch.float32, device=dev)
    l_r = torch.empty((w.bhq, S), dtype=torch.float32, device=dev)
    out = torch.empty_like(o_r)
    lse = torch.empty_like(l_r)
    out_h = torch.empty(out.shape, dtype=torch.float32, pin_memory=True)
    lse_h = torch.empty(lse.shape, dtype=torch.float32, pin_memory=True)
    kw = dict(c=c, causal=w.causal, layout=L, kv_block=w.kv_block)
    attn_ev = []

    def step(record=False):
        ra.permute(q, qr, c=c, layout=L, inverse=0)
        ra.permute(k, kr, c=c, layout=L, inverse=0)
        ra.permute(v, vr, c=c, layout=L, inverse=0)
        if record:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
        ra.fwd(qr, kr, vr, o_r, l_r, **kw)
        if record:
            e1.record(stream)
            attn_ev.append((e0, e1))
        ra.permute(o_r, out, c=c, layout=L, inverse=1)
        ra.permute(l_r, lse, c=c, layout=L, inverse=1)

    launches_per_step = 6
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if ra.sync_status() != ra.RA_OK:
        raise SystemExit("device wait timed out during warm-up")

    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step(record=True)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms_total = t0.elapsed_time(t1)
    if ra.sync_status() != ra.RA_OK:
        raise SystemExit("device wait timed out in the timed region")
    attn_ms = float(np.mean([a.elapsed_time(b) for a, b in attn_ev]))

    # end to end through the C-ABI call on host buffers (ringattn_fwd_host): H2D of Q/K/V
    # from pinned memory, the attention, D2H of out and lse, every step inside the timed
    # region; the library overlaps the copies with the attention by KV-head groups.  Each call
    # is timed on its own and the median is the figure: the host link stalls now and then for
    # tens of milliseconds whatever runs over it, so the mean (reported beside it) mostly
    # measures how many stalls fell into the window.
    e2e_steps = max(1, min(args.steps, 20))
    ws = torch.empty(ra.host_workspace_bytes(S, w.bhq, w.bhkv, w.d), dtype=torch.uint8, device=dev)
    for _ in range(3):   # the first call creates the copy streams; all touch every host page
        ra.fwd_host(q_h, k_h, v_h, out_h, lse_h, ws, **kw)
    torch.cuda.synchronize()
    e2e_ev = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps + 1)]
    e2e_ev[0].record(stream)
    for i in range(e2e_steps):
        ra.fwd_host(q_h, k_h, v_h, out_h, lse_h, ws, **kw)
        e2e_ev[i + 1].record(stream)
    torch.cuda.synchronize()
    e2e_mean_ms = e2e_ev[0].elapsed_time(e2e_ev[-1]) / e2e_steps
    e2e_each = [e2e_ev[i].elapsed_time(e2e_ev[i + 1]) for i in range(e2e_steps)]
    e2e_ms = float(np.median(e2e_each))
    del ws
    if ra.sync_status() != ra.RA_OK:
        raise SystemExit("device wait timed out in the end-to-end region")

    # secondary HBM-bound kernels: the merge (per-hop path) and one permutation
    def time_ms(fn, reps=5):
        fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    # the same path with the chunk map folded into the kernel's tile addressing: no
    # permutation passes (natural-order inputs and outputs)
    nat_ms = time_ms(lambda: ra.fwd_natural(q, k, v, out, lse, **kw))
    rows = w.bhq * S
    merge_ms = time_ms(lambda: ra.merge(o_r, l_r, out, lse))
    merge_bytes = rows * (12 * w.d + 12)
    perm_ms = time_ms(lambda: ra.permute(q, qr, c=c, layout=L, inverse=0))
    perm_bytes = 2 * q.numel() * q.element_size()
    torch.cuda.synchronize()

    ms_step = ms_total / args.steps
    if dist is not None:
        ms_step, e2e_ms = max_over_ranks([ms_step, e2e_ms], dist, dev)
    flop = w.flops()
    value = whole_job_value(flop, world, ms_step)
    e2e_value = whole_job_value(flop, world, e2e_ms)
    bf16_peak, bf16_sust, hbm_peak, peak_src = peaks()
    achieved = flop / (attn_ms * 1e-3) / 1e12
    traffic = traffic_for(w.name)
    h2d = sum(x.numel() * x.element_size() for x in (q_h, k_h, v_h))
    d2h = out_h.numel() * 4 + lse_h.numel() * 4

    extra = None
    if not args.no_extra and w.name == CAUSAL_GQA_S32K.name:
        del qr, kr, vr, o_r, l_r
        torch.cuda.empty_cache()
        extra = [attention_only(ra, WORKLOADS[name], dev, stream, 5, peaks()[0])
                 for name in ("causal_gqa_S131072_h32x8_d128_c16_zigzag", "docmask_gqa_S32768_h64x8_d128_c8_zigzag")]
        extra.append(ulysses_only(ra, w, dev, stream, 5, peaks()[0], peaks()[2]))
        torch.cuda.empty_cache()
        extra.append(backward_only(ra, w, dev, stream, 3, peaks()[0]))
        torch.cuda.empty_cache()
        # the non-causal B=2 S=65536 outlier workload: fused kernel against the per-hop
        # path (one partial per ring message + merge) at every message size of its sweep
        w5 = WORKLOADS["noncausal_mha_B2_S65536_h16_d128_c8_contig"]
        extra.append({"mode": "per-hop sweep (fused kernel vs one partial per message + merge)",
                      "workload": w5.name, "sweep": per_hop_sweep(ra, w5, dev, stream, reps=2)})
        torch.cuda.empty_cache()
        # per-rank work of the 4096-token MHA workload, contiguous and zigzag: one launch
        # restricted to each virtual rank's rows
        extra.append({"mode": "per-rank launches", "per_rank": per_rank(ra, [CAUSAL_MHA_S4K], dev, stream)})

    cpu = None
    parity = None
    if rank == 0 and not args.no_cpu_baseline:
        # the last end-to-end call left its natural-order result in out_h, lse_h
        check = RowParity(out_h, lse_h, "ringattn_fwd_host (the last end-to-end call)")
        units = cpu_oracle_units(w, (q_h, k_h, v_h), args.cpu_seconds, check=check)
        parity = check.summary()
        secs = sum(t for _, t in units)
        cpu = {"value": sum(f for f, _ in units) / secs / 1e12, "unit": UNIT, "cores": cpu_threads(),
               "kind": "oracle",
               "sample": f"{len(units)} units of {CPU_UNIT_ROWS} seeded random query rows ({secs:.1f} s), "
                         "float64 numpy, same inputs (the reference arm times the same units)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1), see inputs.py)",
            "config": {"workload": w.name, "S": S, "Hq": w.hq, "Hkv": w.hkv, "d": w.d, "c": c,
                       "causal": w.causal, "layout": "zigzag" if L else "contiguous", "kv_block": w.kv_block,
                       "batch": w.batch, "step": "permute QKV + fused ring attention + inverse permute O, LSE",
                       "l2": "inputs larger than L2 (Q+K+V %.2f GiB per step)" % (h2d / 2**30),
                       "replicas": "one independent replica per GPU"},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": achieved / bf16_peak, "traffic": traffic,
                         "kernel": "attn_bf16_kernel<%d, false>" % w.d, "kernel_ms": attn_ms,
                         "peak_source": f"{peak_src} bf16 burst (MEASURED_PEAKS.json bf16_tflops)",
                         "frac_of_sustained": (achieved / bf16_sust) if bf16_sust else None,
                         "nominal_peak": NOMINAL_BF16_TFLOPS, "frac_of_nominal": achieved / NOMINAL_BF16_TFLOPS,
                         **clock_ceiling(achieved, clk, dev)},
            "natural_step": {"ms_per_step": nat_ms, "value": flop / (nat_ms * 1e-3) / 1e12, "unit": UNIT,
                             "what": "ringattn_fwd_natural: chunk map in TMA addressing, no permutation passes"},
            "also_measured": extra,
            "secondary": {
                "merge": {"bound": "hbm", "achieved": merge_bytes / (merge_ms * 1e-3) / 1e9, "peak": hbm_peak,
                          "unit": "GB/s", "frac": merge_bytes / (merge_ms * 1e-3) / 1e9 / hbm_peak,
                          "kernel_ms": merge_ms, "bytes": merge_bytes},
                "permute_q": {"bound": "hbm", "achieved": perm_bytes / (perm_ms * 1e-3) / 1e9, "peak": hbm_peak,
                              "unit": "GB/s", "frac": perm_bytes / (perm_ms * 1e-3) / 1e9 / hbm_peak,
                              "kernel_ms": perm_ms, "bytes": perm_bytes},
            },
            "cpu_baseline": cpu,
            "parity": parity,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms, "steps": e2e_steps, "statistic": "median of the calls' times",
                    "ms_per_step_mean": e2e_mean_ms, "ms_per_step_min": min(e2e_each),
                    "ms_per_step_max": max(e2e_each),
                    "call": "ringattn_fwd_host (natural order; copies overlapped with attention by KV-head groups)"},
            "context": {"overlap_condition_tokens_per_block": {
                "pages_H100_989TFLOPs_over_450GBs_NVLink": 2198,
                "GB300_nominal_2250TFLOPs_over_900GBs_NVLink5": 2500,
                "GB300_at_this_kernel_rate": round(achieved * 1e12 / 900e9)}},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
