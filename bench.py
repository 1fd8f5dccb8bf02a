#!/usr/bin/env python3
"""Benchmark of the sparse FP8 MLA attention hot path on GB300.

One step = one pass of the hot path over one batch of the chosen workload:
the fused BF16 -> FP8 KV writer stores the batch's new latent rows, then the
sparse attention call (index translation, row gather, dequantisation, QK^T,
softmax, PV, split-K merge) produces O and LSE for every query token.
The prefill workload also quantises its queries to FP8 on the GPU first.

Default workload: decode_raw512 (64 query tokens, 16 heads, top-k 2048 over
a 131072-row raw FP8 pool, page size 64).  L2 is flushed (a 2x-L2 buffer is
written) before every timed step; steps are timed with CUDA events on the
launching stream at the step boundaries, and the attention call alone (for the
roofline) in a second loop with the same flush.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference   # the CPU oracle timed on the host cores
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sparse_mla_attention_page_gb300 import workloads as W  # noqa: E402

METRIC = "sparse-attn query-tokens/s and KV-gather HBM GB/s (fraction of GB300 roofline)"
UNIT = "query-tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
ATTN_SOURCES = ["sparse_mla_attention_page_gb300/csrc/sparse_attn_tc.cu",
                "sparse_mla_attention_page_gb300/csrc/tc_ptx.cuh",
                "sparse_mla_attention_page_gb300/csrc/combine.cu"]
ATTN_KERNEL = "sparse_attn_tc_kernel + combine_kernel (the attention call)"
COMPUTE_DTYPE = "e4m3"         # tcgen05 kind::f8f6f4 MMAs (E4M3 operands, FP32 accumulation)


ROW_BYTES = {"raw512": 512, "scaled528": 528, "rope656": 656}
WRITERS = {"raw512": lambda b: b.dsa_kv_write_raw, "scaled528": lambda b: b.dsa_kv_write_scaled,
           "rope656": lambda b: b.dsa_kv_write_rope656}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=list(W.WORKLOADS), default="decode_raw512")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=300)
    p.add_argument("--op", choices=["attention", "gather_dequant", "kv_write"], default="attention",
                   help="gather_dequant times the BF16 reader over the workload's top-k lists instead; "
                        "kv_write times one KV writer on 16384 new rows into a 262144-row pool")
    p.add_argument("--layout", choices=["raw512", "scaled528", "rope656"], default="raw512",
                   help="row layout of --op kv_write and of --workload writer_sweep (raw512, scaled528)")
    p.add_argument("--heads", type=int, default=16, help="head count of --workload writer_sweep")
    p.add_argument("--warm", action="store_true",
                   help="informational: no L2 flush between steps (inputs may stay in L2); "
                        "the default run flushes before every step")
    return p.parse_args()


# ----------------------------------------------------------------- workloads

def make_workload(name: str, heads: int = 16, layout: str = "raw512") -> dict:
    if name == "writer_sweep":   # decode over freshly written rows: --heads, --layout
        if layout not in ("raw512", "scaled528"):
            raise SystemExit("writer_sweep takes --layout raw512 or scaled528")
        return W.writer_sweep(H=heads, layout=layout)
    return W.make(name)


def step_rows(w: dict) -> tuple[np.ndarray, np.ndarray]:
    """The batch's new latent rows (one per query token) and their slots: the
    last T physical rows of the pool (re-written with the same bytes each step)."""
    rng = W.rng_for(9000 + w["T"])
    width = 576 if w["layout"] == "rope656" else 512
    x = W.f32_to_bf16_bits(rng.standard_normal((w["T"], width), dtype=np.float32))
    slots = np.arange(w["pool_rows"] - w["T"], w["pool_rows"], dtype=np.int64)
    return x, slots


def algorithmic_bytes(w: dict) -> int:
    """Bytes the attention call must move: each valid entry's row once, plus the
    query, q_scale, top-k list, O and LSE."""
    T, H, K = w["T"], w["H"], w["K"]
    R = ROW_BYTES[w["layout"]]
    valid = W.valid_entry_count(w["topk"])
    q8 = w["name"].startswith("prefill_q8")
    q_width = 576 if w["layout"] == "rope656" else 512
    q_bytes = T * H * q_width * (1 if q8 else 2) + (T * H * 4 if q8 else 0)
    return valid * R + q_bytes + T * K * 4 + T * H * 512 * 2 + T * H * 4


def attn_flops(w: dict) -> int:
    """QK^T over the key width (576 with RoPE) and PV over the 512 latent dims."""
    dk = 576 if w["layout"] == "rope656" else 512
    return 2 * w["H"] * (dk + 512) * W.valid_entry_count(w["topk"])


def run_gather(args) -> dict:
    """The gather/dequantise reader over the workload's pool and top-k lists:
    CUDA events around each call, L2 flushed before every call."""
    import torch

    from sparse_mla_attention_page_gb300 import binding
    dev = torch.device("cuda", 0)
    w = make_workload(args.workload, args.heads, args.layout)
    T, K, layout = w["T"], w["K"], w["layout"]
    R = 512 if layout == "raw512" else 528
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)  # noqa: E731
    pool = torch.zeros(w["pool_rows"], R, dtype=torch.uint8, device=dev)
    (binding.dsa_kv_write_raw if layout == "raw512" else binding.dsa_kv_write_scaled)(
        bf(w["kv_src"]), torch.from_numpy(w["kv_slots"]).to(dev), pool)
    topk = torch.from_numpy(w["topk"]).to(dev)
    pt = None if w["page_table"] is None else torch.from_numpy(w["page_table"]).to(dev)
    out = torch.empty(T * K, 512, dtype=torch.bfloat16, device=dev)
    idx = torch.empty(T, K, dtype=torch.int32, device=dev)
    flush = torch.empty(max(2 * torch.cuda.get_device_properties(dev).L2_cache_size, 256 << 20),
                        dtype=torch.uint8, device=dev)
    call = lambda: binding.dsa_gather_dequant(pool, layout, topk, out, idx, page_table=pt,  # noqa: E731
                                              page_size=w["page_size"])
    for _ in range(args.warmup):
        flush.zero_()
        call()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record()
        call()
        ev[i][1].record()
    torch.cuda.synchronize(dev)
    us = float(np.mean([e[0].elapsed_time(e[1]) for e in ev])) * 1e3
    valid = W.valid_entry_count(w["topk"])
    abytes = valid * R + valid * 1024 + T * K * 8
    peak = float(measured_peaks().get("hbm_gbs", FALLBACK_HBM_GBS))
    achieved = abytes / (us * 1e-6) / 1e9
    return {"metric": "gather-dequant selected rows/s and HBM GB/s (fraction of GB300 roofline)",
            "value": round(valid / (us * 1e-6), 1), "unit": "rows/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "us_per_call": round(us, 3), "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.workload, "op": "gather_dequant", "T": T, "K": K, "layout": layout,
                       "valid_entries": valid, "l2": "flushed before every call"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "algorithmic_bytes_per_call": abytes}}


def run_kv_write(args) -> dict:
    """One fused BF16 -> FP8 KV writer on 16384 new rows (N(0,1) x U(0.1, 8)) into
    distinct random slots of a 262144-row pool: CUDA events around each call,
    L2 flushed before every call."""
    import torch

    from sparse_mla_attention_page_gb300 import binding
    dev = torch.device("cuda", 0)
    w = W.writer_rows()
    layout, n = args.layout, w["n_rows"]
    x = w["x_bf16"]
    if layout == "rope656":   # 576-wide input rows: 512 latent dims + 64 RoPE dims
        rope = W.f32_to_bf16_bits(W.rng_for(8).standard_normal((n, W.D_ROPE), dtype=np.float32))
        x = np.concatenate([x, rope], axis=1)
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(dev)
    slots = torch.from_numpy(w["slots"]).to(dev)
    pool = torch.zeros(w["pool_rows"], ROW_BYTES[layout], dtype=torch.uint8, device=dev)
    write = WRITERS[layout](binding)
    flush = torch.empty(max(2 * torch.cuda.get_device_properties(dev).L2_cache_size, 256 << 20),
                        dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        flush.zero_()
        write(xd, slots, pool)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record()
        write(xd, slots, pool)
        ev[i][1].record()
    torch.cuda.synchronize(dev)
    us = float(np.mean([e[0].elapsed_time(e[1]) for e in ev])) * 1e3
    abytes = n * (x.shape[1] * 2 + ROW_BYTES[layout] + 8)     # BF16 row in, FP8 row out, slot
    peak = float(measured_peaks().get("hbm_gbs", FALLBACK_HBM_GBS))
    achieved = abytes / (us * 1e-6) / 1e9
    return {"metric": "KV writer rows/s and HBM GB/s (fraction of GB300 roofline)",
            "value": round(n / (us * 1e-6), 1), "unit": "rows/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "us_per_call": round(us, 3), "higher_is_better": True,
            "dtype": "e4m3", "data": "synthetic",
            "config": {"op": "kv_write", "layout": layout, "n_rows": n, "pool_rows": w["pool_rows"],
                       "slots": "distinct, uniform over the pool", "l2": "flushed before every call"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "algorithmic_bytes_per_call": abytes}}


def max_over_ranks(x: float, dist, device) -> float:
    """The largest of every rank's x (x itself with no process group): a job is
    as slow as its slowest rank."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f)
    return {}


def kernel_source_sha() -> str:
    """Hash of the attention kernels' code with comments and blank lines removed, so
    that recorded ncu counters stay valid across comment-only edits."""
    h = hashlib.sha256()
    for rel in ATTN_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        code = "\n".join(ln.rstrip() for ln in src.splitlines() if ln.strip())
        h.update(code.encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per attention call from a committed ncu summary, only while the
    kernel source is the one that was profiled."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    e = rec.get(workload)
    if not e or e.get("source_sha") != kernel_source_sha():
        return None
    return e.get("dram_bytes_per_call")


# -------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.samples = []
        self.proc = None
        self.gpu_id = gpu_id

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if self.gpu_id is not None:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if not self.samples:
            return None
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        used = inside or [min(self.samples, key=lambda ts: min(abs(ts[0] - t0), abs(ts[0] - t1)))[1]]
        sm = [float(s[0]) for s in used if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in used if s[1].replace(".", "").isdigit()]
        reasons = sorted({name for s in used for name, v in zip(self.REASONS, s[4:8]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples_in_window": len(inside)}


# ---------------------------------------------------------------- our arm

def run_ours(args, rank: int, world: int, local_rank: int, dist):
    import torch

    from sparse_mla_attention_page_gb300 import binding

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = make_workload(args.workload, args.heads, args.layout)
    T, H, K = w["T"], w["H"], w["K"]
    layout = w["layout"]
    prefill = w["name"].startswith("prefill_q8")

    def to_dev(a, dtype=None):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return (t.view(dtype) if dtype is not None else t).to(dev)

    def bf16(a):
        return to_dev(a.view(np.int16), torch.bfloat16)

    write = WRITERS[layout](binding)
    pool = torch.zeros(w["pool_rows"], ROW_BYTES[layout], dtype=torch.uint8, device=dev)
    kv_src = bf16(w["kv_src"])
    write(kv_src, to_dev(w["kv_slots"]), pool)
    del kv_src
    x_new_h, slots_h = step_rows(w)
    x_new, slots = bf16(x_new_h), to_dev(slots_h)
    q = bf16(w["q_bf16"])
    topk = to_dev(w["topk"])
    pt = None if w["page_table"] is None else to_dev(w["page_table"])
    o = torch.empty(T, H, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(T, H, dtype=torch.float32, device=dev)
    ws = binding.workspace_for(T, H, K, device=dev)
    q8 = torch.empty(T, H, 512, dtype=torch.uint8, device=dev) if prefill else None
    qs = torch.empty(T, H, dtype=torch.float32, device=dev) if prefill else None
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush():
        if not args.warm:
            flush_buf.zero_()

    def step_write():
        write(x_new, slots, pool)
        if prefill:
            binding.dsa_quantize_q8(q, q8, qs)

    def step_attn():
        if prefill:
            binding.dsa_sparse_attn_prefill_q8(q8, qs, pool, layout, topk, w["sm_scale"], o, lse, ws,
                                               page_table=pt, page_size=w["page_size"])
        else:
            binding.dsa_sparse_attn_decode(q, pool, layout, topk, w["sm_scale"], o, lse, ws,
                                           page_table=pt, page_size=w["page_size"])

    # writer, [q8 quantiser], attention, [split-unit merge when a unit spans CTAs]
    launches_per_step = 1 + (1 if prefill else 0) + 1 + (1 if ws is not None else 0)

    for _ in range(args.warmup):
        flush()
        step_write()
        step_attn()
    torch.cuda.synchronize(dev)

    props = torch.cuda.get_device_properties(dev)
    gpu_id = None
    if all(hasattr(props, f) for f in ("pci_domain_id", "pci_bus_id", "pci_device_id")):
        gpu_id = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)
    # whole steps, events at the step boundaries only: the attention kernel is a
    # programmatic dependent launch and may start its set-up while the writer runs
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    for i in range(args.steps):
        flush()
        ev[i][0].record(stream)
        step_write()
        step_attn()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    # the attention call alone (its kernels' duration, for the roofline): same
    # L2 flush before every call, the inputs of the last step
    ev_a = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush()
        ev_a[i][0].record(stream)
        step_attn()
        ev_a[i][1].record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    time.sleep(0.2)
    sampler.stop()
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    attn_ms = [e[0].elapsed_time(e[1]) for e in ev_a]
    total_ms = max_over_ranks(float(sum(step_ms)), dist, dev)

    # end to end through the public API: the step's inputs from one pinned host
    # buffer (one H2D copy), the results back in one D2H copy
    def packed(parts):
        """Byte offsets of 256-byte-aligned parts in one buffer, and its size."""
        offs, n = [], 0
        for a in parts:
            offs.append(n)
            n += (a.nbytes + 255) // 256 * 256
        return offs, n

    in_parts = [np.ascontiguousarray(w["q_bf16"]), np.ascontiguousarray(w["topk"]),
                np.ascontiguousarray(x_new_h), np.ascontiguousarray(slots_h)]
    if w["page_table"] is not None:
        in_parts.append(np.ascontiguousarray(w["page_table"]))
    in_offs, in_n = packed(in_parts)
    h_in = torch.empty(in_n, dtype=torch.uint8).pin_memory()
    for a, off in zip(in_parts, in_offs):
        h_in[off:off + a.nbytes].copy_(torch.from_numpy(a.view(np.uint8).reshape(-1)))
    d_in = torch.empty(in_n, dtype=torch.uint8, device=dev)

    def view(buf, off, a_shape, dtype):
        n = int(np.prod(a_shape)) * torch.empty(0, dtype=dtype).element_size()
        return buf[off:off + n].view(dtype).view(*a_shape)

    q_e = view(d_in, in_offs[0], w["q_bf16"].shape, torch.bfloat16)
    topk_e = view(d_in, in_offs[1], w["topk"].shape, torch.int32)
    x_e = view(d_in, in_offs[2], x_new_h.shape, torch.bfloat16)
    slots_e = view(d_in, in_offs[3], slots_h.shape, torch.int64)
    pt_e = None if w["page_table"] is None else view(d_in, in_offs[4], w["page_table"].shape, torch.int32)
    (o_off, lse_off), out_n = packed([np.empty((T, H, 512), np.uint16), np.empty((T, H), np.float32)])
    d_out = torch.empty(out_n, dtype=torch.uint8, device=dev)
    h_out = torch.empty(out_n, dtype=torch.uint8).pin_memory()
    o_e = view(d_out, o_off, (T, H, 512), torch.bfloat16)
    lse_e = view(d_out, lse_off, (T, H), torch.float32)
    if prefill:
        q8_e = torch.empty(T, H, 512, dtype=torch.uint8, device=dev)
        qs_e = torch.empty(T, H, dtype=torch.float32, device=dev)
    h2d, d2h = in_n, out_n
    n_e2e = max(1, min(args.e2e_steps, args.steps))
    e2e_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_e2e)]
    for i in range(n_e2e + 3):
        flush()
        if i >= 3:
            e2e_ev[i - 3][0].record(stream)
        d_in.copy_(h_in, non_blocking=True)
        write(x_e, slots_e, pool)
        if prefill:
            binding.dsa_quantize_q8(q_e, q8_e, qs_e)
            binding.dsa_sparse_attn_prefill_q8(q8_e, qs_e, pool, layout, topk_e, w["sm_scale"], o_e, lse_e, ws,
                                               page_table=pt_e, page_size=w["page_size"])
        else:
            binding.dsa_sparse_attn_decode(q_e, pool, layout, topk_e, w["sm_scale"], o_e, lse_e, ws,
                                           page_table=pt_e, page_size=w["page_size"])
        h_out.copy_(d_out, non_blocking=True)
        if i >= 3:
            e2e_ev[i - 3][1].record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(float(sum(e[0].elapsed_time(e[1]) for e in e2e_ev)), dist, dev)

    if rank != 0:
        return None
    peaks = measured_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    attn_mean_s = statistics.mean(attn_ms) / 1e3
    abytes = algorithmic_bytes(w)
    achieved = abytes / attn_mean_s / 1e9
    traffic = recorded_traffic(args.workload)
    value = world * T * args.steps / (total_ms / 1e3)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": COMPUTE_DTYPE,
        "data": "synthetic (seeded generators; no dataset, no weights)",
        "config": {"workload": args.workload, "T": T, "H": H, "K": K, "layout": layout,
                   "pool_rows": w["pool_rows"], "page_size": w["page_size"],
                   "valid_entries": W.valid_entry_count(w["topk"]),
                   "step": ("quantize_q8 + " if prefill else "") + f"kv_write_{layout[:3]} of {T} new rows + sparse attention",
                   "l2": ("not flushed (warm; informational)" if args.warm
                          else f"flushed before every step ({flush_buf.numel() >> 20} MiB write)"),
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": ATTN_KERNEL, "algorithmic_bytes_per_call": abytes,
                     "attn_us_per_call": round(attn_mean_s * 1e6, 3),
                     "peak_source": "measured" if "hbm_gbs" in peaks else "fallback",
                     "tensor_tflops": round(attn_flops(w) / attn_mean_s / 1e12, 2),
                     # FP8 dense peak = measured BF16 burst x the nominal FP8/BF16 ratio (2)
                     "tensor_peak_tflops": round(2.0 * float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS)), 1),
                     "tensor_frac": round(attn_flops(w) / attn_mean_s / 1e12
                                          / (2.0 * float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))), 4)},
        "e2e": {"value": round(world * T * n_e2e / (e2e_ms / 1e3), 1), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": sampler.summary(t_wall0, t_wall1),
    }
    return line, w


# ------------------------------------------------------------------- oracle

def oracle_pass(w: dict, pool: np.ndarray, tokens, n_threads: int, q8=None, qs=None):
    import oracle
    if q8 is not None:
        oracle.sparse_attn(pool, w["layout"], w["topk"], w["sm_scale"], q8=q8, q_scale=qs,
                           page_table=w["page_table"], page_size=w["page_size"],
                           tokens=tokens, n_threads=n_threads)
    else:
        oracle.sparse_attn(pool, w["layout"], w["topk"], w["sm_scale"], q_bf16=w["q_bf16"],
                           page_table=w["page_table"], page_size=w["page_size"],
                           tokens=tokens, n_threads=n_threads)


def oracle_setup(w: dict):
    import oracle
    pool = oracle.fill_pool(w)
    q8 = qs = None
    if w["name"].startswith("prefill_q8"):
        q8, qs = oracle.quantize_q8(w["q_bf16"])
    return pool, q8, qs


def cpu_baseline(w: dict, seconds: float) -> dict:
    """The oracle as it stands, on all host cores, over whole passes of the
    batch (writer of the step's new rows + attention for every token) until
    ``seconds`` have passed; for the prefill batch a 64-token slice per pass."""
    import oracle
    cores = len(os.sched_getaffinity(0))
    pool, q8, qs = oracle_setup(w)
    x_new, slots = step_rows(w)
    T = w["T"]
    tokens = np.arange(min(T, 64)) if w["name"].startswith("prefill_q8") else np.arange(T)
    done = 0
    t0 = time.perf_counter()
    while True:
        oracle.kv_write(w["layout"], x_new, slots, pool)
        oracle_pass(w, pool, tokens, cores, q8, qs)
        done += len(tokens)
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": round(done / dt, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{done // len(tokens)} passes x {len(tokens)} tokens of {w['name']} "
                      f"(writer of the step's rows + float64 attention), {dt:.1f} s"}


def run_reference(args, rank: int):
    if rank != 0:
        return None
    w = make_workload(args.workload, args.heads, args.layout)
    cores = len(os.sched_getaffinity(0))
    pool, q8, qs = oracle_setup(w)
    x_new, slots = step_rows(w)
    import oracle
    t0 = time.perf_counter()
    oracle_pass(w, pool, np.arange(min(cores, w["T"])), cores, q8, qs)
    per_tok = (time.perf_counter() - t0) / min(cores, w["T"])
    budget = 120.0
    n_tok = int(max(1, min(w["T"], budget / max(1, args.steps + args.warmup) / per_tok)))
    rng = np.random.default_rng(0)
    for _ in range(args.warmup):
        oracle.kv_write(w["layout"], x_new, slots, pool)
        oracle_pass(w, pool, np.sort(rng.choice(w["T"], n_tok, replace=False)), cores, q8, qs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.kv_write(w["layout"], x_new, slots, pool)
        oracle_pass(w, pool, np.sort(rng.choice(w["T"], n_tok, replace=False)), cores, q8, qs)
    dt = time.perf_counter() - t0
    value = n_tok * args.steps / dt
    sample = f"{n_tok} of {w['T']} tokens per step ({w['name']}), writer of the step's rows + float64 attention"
    return {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": args.workload, "T": w["T"], "H": w["H"], "K": w["K"], "layout": w["layout"]},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if args.impl == "reference":
        line = run_reference(args, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    import importlib
    importlib.import_module("sparse_mla_attention_page_gb300.build").build()
    if args.op in ("gather_dequant", "kv_write"):
        if rank == 0:
            print(json.dumps(run_gather(args) if args.op == "gather_dequant" else run_kv_write(args)), flush=True)
        return
    out = run_ours(args, rank, world, local_rank, dist)
    if out is not None:
        line, w = out
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
        else:
            line["cpu_baseline"] = None
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
