#!/usr/bin/env python3
"""Benchmark of the sparse FP8 MLA attention hot path on GB300.

One step = one pass of the hot path over one batch of the chosen workload:
the fused BF16 -> FP8 KV writer stores the batch's new latent rows, the
prefill batch quantises its queries to FP8, then the sparse attention call
(index translation, row gather, dequantisation, QK^T, softmax, PV, split-K
merge) produces O and LSE for every query token.

Default workload (the headline line): prefill_q8_raw512, the largest batch
(4096 query tokens, 32 heads, FP8 queries, top-k 2048 over a 16384-row raw
FP8 pool, page size 64).  L2 is flushed (a 2x-L2 buffer is written) before
every timed step and every timed call.  Timing: CUDA events on the launching
stream; the K timed steps give `value`; the attention call alone is timed in
5 runs of K calls (median of the runs' mean call time) for the roofline.
`per_config` carries every other workload measured the same way (decode
batches, writers, the writer sweep, the reader), each with its roofline.
Prints one JSON line (rank 0).

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
# the sources of the profiled kernel (ncu -k regex:sparse_attn_tc): its recorded
# counters stay valid while these hash the same
ATTN_SOURCES = ["sparse_mla_attention_page_gb300/csrc/sparse_attn_tc.cu",
                "sparse_mla_attention_page_gb300/csrc/tc_ptx.cuh",
                "sparse_mla_attention_page_gb300/csrc/dsa_common.cuh",
                "sparse_mla_attention_page_gb300/csrc/kernels.h"]
ATTN_KERNEL = "sparse_attn_tc_kernel + combine_kernel (the attention call)"
COMPUTE_DTYPE = "e4m3"         # tcgen05 kind::f8f6f4 MMAs (E4M3 operands, FP32 accumulation)
RUNS = 5                       # runs per roofline figure (median of the runs' mean call time)

ROW_BYTES = {"raw512": 512, "scaled528": 528, "rope656": 656}
WRITERS = {"raw512": lambda b: b.dsa_kv_write_raw, "scaled528": lambda b: b.dsa_kv_write_scaled,
           "rope656": lambda b: b.dsa_kv_write_rope656}

# per_config entries: (key, kind, workload, options)
PER_CONFIG = [
    ("tiny_decode_raw512", "attention", "tiny_decode_raw512", {}),
    ("decode_raw512", "attention", "decode_raw512", {}),
    ("decode_scaled528", "attention", "decode_scaled528", {}),
    ("prefill_q8_raw512", "attention", "prefill_q8_raw512", {}),
    ("kv_write_raw512", "kv_write", None, {"layout": "raw512"}),
    ("kv_write_scaled528", "kv_write", None, {"layout": "scaled528"}),
    ("writer_sweep_raw512_h8", "attention", "writer_sweep", {"heads": 8, "layout": "raw512"}),
    ("writer_sweep_raw512_h16", "attention", "writer_sweep", {"heads": 16, "layout": "raw512"}),
    ("writer_sweep_raw512_h32", "attention", "writer_sweep", {"heads": 32, "layout": "raw512"}),
    ("writer_sweep_scaled528_h8", "attention", "writer_sweep", {"heads": 8, "layout": "scaled528"}),
    ("writer_sweep_scaled528_h16", "attention", "writer_sweep", {"heads": 16, "layout": "scaled528"}),
    ("writer_sweep_scaled528_h32", "attention", "writer_sweep", {"heads": 32, "layout": "scaled528"}),
    ("decode_rope656", "attention", "decode_rope656", {}),
    ("prefill_q8_scaled528", "attention", "prefill_q8_scaled528", {}),
    ("kv_write_rope656", "kv_write", None, {"layout": "rope656"}),
    ("gather_dequant_decode_raw512", "gather_dequant", "decode_raw512", {}),
    ("gather_dequant_decode_scaled528", "gather_dequant", "decode_scaled528", {}),
    ("gather_dequant_tiny_decode_raw512", "gather_dequant", "tiny_decode_raw512", {}),
]


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=list(W.WORKLOADS), default="prefill_q8_raw512")
    p.add_argument("--cpu-seconds", type=float, default=8.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-per-config", action="store_true", help="time the headline workload only")
    p.add_argument("--only", default=None,
                   help="comma-separated per_config keys to time (default: all)")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--layout", choices=["raw512", "scaled528", "rope656"], default="raw512",
                   help="row layout of --workload writer_sweep (raw512, scaled528)")
    p.add_argument("--heads", type=int, default=16, help="head count of --workload writer_sweep")
    p.add_argument("--warm", action="store_true",
                   help="informational: no L2 flush between steps (inputs may stay in L2); "
                        "the default run flushes before every step")
    return p.parse_args(argv)


# ----------------------------------------------------------------- workloads

def make_workload(name: str, heads: int = 16, layout: str = "raw512") -> dict:
    if name == "writer_sweep":   # decode over freshly written rows: heads, layout
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


def is_prefill(w: dict) -> bool:
    return w["name"].startswith("prefill_q8")


def algorithmic_bytes(w: dict) -> int:
    """Bytes the attention call must move: each valid entry's row once, plus the
    query, q_scale, top-k list, O and LSE."""
    T, H, K = w["T"], w["H"], w["K"]
    R = ROW_BYTES[w["layout"]]
    valid = W.valid_entry_count(w["topk"])
    q8 = is_prefill(w)
    q_width = 576 if w["layout"] == "rope656" else 512
    q_bytes = T * H * q_width * (1 if q8 else 2) + (T * H * 4 if q8 else 0)
    return valid * R + q_bytes + T * K * 4 + T * H * 512 * 2 + T * H * 4


def attn_flops(w: dict) -> int:
    """QK^T over the key width (576 with RoPE) and PV over the 512 latent dims."""
    dk = 576 if w["layout"] == "rope656" else 512
    return 2 * w["H"] * (dk + 512) * W.valid_entry_count(w["topk"])


def gather_bytes(w: dict) -> int:
    """Bytes the reader must move: per valid entry its row and its BF16 output row
    (selected branch), or every pool row in and out once (full-pool branch), plus
    the top-k list read and the remapped list written."""
    T, K, R = w["T"], w["K"], ROW_BYTES[w["layout"]]
    width = 576 if w["layout"] == "rope656" else 512
    if T * K < w["pool_rows"]:
        rows = W.valid_entry_count(w["topk"])
    else:
        rows = w["pool_rows"]
    return rows * (R + 2 * width) + T * K * 8


def writer_bytes(n: int, layout: str) -> int:
    width = 576 if layout == "rope656" else 512
    return n * (width * 2 + ROW_BYTES[layout] + 8)     # BF16 row in, FP8 row out, slot


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


def recorded_profile(key: str) -> dict | None:
    """The committed ncu counters of one attention call (profiles/ncu_traffic.json),
    only while the kernel source is the one that was profiled."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not key or not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    e = rec.get(key)
    if not e or e.get("source_sha") != kernel_source_sha():
        return None
    return e


def recorded_traffic(key: str):
    """DRAM bytes per attention call from the committed ncu counters."""
    e = recorded_profile(key)
    return e.get("dram_bytes_per_call") if e else None


def torch_sms(dev) -> int:
    import torch
    return torch.cuda.get_device_properties(dev).multi_processor_count


SMEM_BYTES_PER_CLK = 128     # shared-memory banks of one SM: 32 x 4 bytes a clock


def smem_roofline(key: str, us: float, peaks: dict, sms: int) -> dict | None:
    """Shared-memory bank traffic of one attention call (ncu l1tex__data_bank_reads
    + _writes, 4 bytes each, recorded per kernel source) against 128 B a clock on
    every SM at the maximum SM clock."""
    e = recorded_profile(key)
    if not e or "smem_bank_bytes_per_call" not in e:
        return None
    mhz = float(peaks.get("sm_max_mhz", 2070.0))
    peak = SMEM_BYTES_PER_CLK * sms * mhz * 1e6 / 1e9
    b = e["smem_bank_bytes_per_call"]
    gbs = b / (us * 1e-6) / 1e9
    return {"achieved": round(gbs, 1), "peak": round(peak, 1), "unit": "GB/s", "frac": round(gbs / peak, 4),
            "bytes_per_call": b,
            "peak_source": f"{SMEM_BYTES_PER_CLK} B/clk x {sms} SMs x {mhz:.0f} MHz (maximum SM clock)"}


# -------------------------------------------------------------------- peaks

def measure_fp8_peak(dev) -> dict | None:
    """Dense FP8 (E4M3 x E4M3 -> BF16) throughput of one 8192^3 GEMM through
    torch._scaled_mm, best of 10 after warm-up (a burst figure, like the
    measured BF16 peak)."""
    import torch
    try:
        n = 8192
        a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()     # column-major operand
        one = torch.ones((), dtype=torch.float32, device=dev)

        def mm():
            return torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        for _ in range(3):
            mm()
        ts = []
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            mm()
            e1.record()
            torch.cuda.synchronize(dev)
            ts.append(e0.elapsed_time(e1) / 1e3)
        del a, b
        return {"tflops": round(2 * n ** 3 / min(ts) / 1e12, 1),
                "how": "torch._scaled_mm E4M3 x E4M3 -> BF16, 8192^3, best of 10 (burst)"}
    except Exception as e:  # noqa: BLE001 - report and fall back to the nominal ratio
        return {"tflops": None, "how": f"not measured ({type(e).__name__}: {e})"[:200]}


def tensor_peak(peaks: dict, fp8: dict | None) -> tuple[float, str]:
    if fp8 and fp8.get("tflops"):
        return float(fp8["tflops"]), "measured FP8 burst"
    bf16 = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    return 2.0 * bf16, "2 x BF16 burst (nominal FP8/BF16 ratio)"


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
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "20"]
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

class Timer:
    """CUDA-event timing of one call per step on the launching stream, with an
    L2 flush (a write of twice the L2 size) before every step."""

    def __init__(self, dev, warm: bool = False):
        import torch
        self.torch = torch
        self.dev = dev
        self.warm = warm
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.flush_buf = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)

    def flush(self):
        if not self.warm:
            self.flush_buf.zero_()

    def run(self, fn, steps: int) -> list:
        """Per-step milliseconds of `steps` flushed calls of fn."""
        torch = self.torch
        stream = torch.cuda.current_stream(self.dev)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for i in range(steps):
            self.flush()
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize(self.dev)
        return [e[0].elapsed_time(e[1]) for e in ev]

    def median_call_us(self, fn, steps: int, warmup: int, runs: int = RUNS) -> tuple[float, list]:
        """Median over `runs` runs of the mean flushed call time (microseconds)."""
        for _ in range(warmup):
            self.flush()
            fn()
        self.torch.cuda.synchronize(self.dev)
        means = [statistics.mean(self.run(fn, steps)) * 1e3 for _ in range(runs)]
        return statistics.median(means), [round(m, 3) for m in means]


class AttnCase:
    """Device state of one attention workload: the pool filled by the GPU writer,
    the step's new rows, queries, lists and outputs; `write()` is the step's
    writer (+ FP8 query quantiser for prefill), `attn()` the attention call."""

    def __init__(self, w: dict, dev, binding):
        import torch
        self.w, self.dev, self.b = w, dev, binding
        T, H, K = w["T"], w["H"], w["K"]
        self.layout = w["layout"]
        self.prefill = is_prefill(w)

        def to_dev(a, dtype=None):
            t = torch.from_numpy(np.ascontiguousarray(a))
            return (t.view(dtype) if dtype is not None else t).to(dev)

        self.to_dev = to_dev
        self.bf16 = lambda a: to_dev(a.view(np.int16), torch.bfloat16)
        self.writer = WRITERS[self.layout](binding)
        self.pool = torch.zeros(w["pool_rows"], ROW_BYTES[self.layout], dtype=torch.uint8, device=dev)
        kv_src = self.bf16(w["kv_src"])
        self.writer(kv_src, to_dev(w["kv_slots"]), self.pool)
        del kv_src
        self.x_new_h, self.slots_h = step_rows(w)
        self.x_new, self.slots = self.bf16(self.x_new_h), to_dev(self.slots_h)
        self.q = self.bf16(w["q_bf16"])
        self.topk = to_dev(w["topk"])
        self.pt = None if w["page_table"] is None else to_dev(w["page_table"])
        self.o = torch.empty(T, H, 512, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(T, H, dtype=torch.float32, device=dev)
        self.ws = binding.workspace_for(T, H, K, device=dev)
        self.q8 = torch.empty(T, H, 512, dtype=torch.uint8, device=dev) if self.prefill else None
        self.qs = torch.empty(T, H, dtype=torch.float32, device=dev) if self.prefill else None
        if self.prefill:
            binding.dsa_quantize_q8(self.q, self.q8, self.qs)

    def write(self):
        self.writer(self.x_new, self.slots, self.pool)
        if self.prefill:
            self.b.dsa_quantize_q8(self.q, self.q8, self.qs)

    def attn(self):
        w = self.w
        if self.prefill:
            self.b.dsa_sparse_attn_prefill_q8(self.q8, self.qs, self.pool, self.layout, self.topk, w["sm_scale"],
                                              self.o, self.lse, self.ws, page_table=self.pt,
                                              page_size=w["page_size"])
        else:
            self.b.dsa_sparse_attn_decode(self.q, self.pool, self.layout, self.topk, w["sm_scale"], self.o,
                                          self.lse, self.ws, page_table=self.pt, page_size=w["page_size"])

    def step(self):
        self.write()
        self.attn()

    def launches_per_step(self) -> int:
        # writer, [q8 quantiser], attention, [split-unit merge when a unit spans CTAs]
        return 1 + (1 if self.prefill else 0) + 1 + (1 if self.ws is not None else 0)


def attn_roofline(w: dict, us: float, peaks: dict, tpeak: float, tsrc: str, traffic, smem=None) -> dict:
    """Both rooflines of one attention call; `bound` names the binding one: HBM
    for the decode batches, the tensor pipe for the prefill batches (their pools
    sit in L2, so algorithmic HBM bytes there overstate what DRAM must move)."""
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    abytes = algorithmic_bytes(w)
    gbs = abytes / (us * 1e-6) / 1e9
    tfl = attn_flops(w) / (us * 1e-6) / 1e12
    bound = "tensor" if is_prefill(w) else "hbm"
    main = ({"achieved": round(tfl, 2), "peak": tpeak, "unit": "TFLOP/s", "frac": round(tfl / tpeak, 4)}
            if bound == "tensor" else
            {"achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4)})
    return {"bound": bound, **main, "traffic": traffic, "kernel": ATTN_KERNEL,
            "algorithmic_bytes_per_call": abytes, "algorithmic_flops_per_call": attn_flops(w),
            "attn_us_per_call": round(us, 3),
            "hbm": {"achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4),
                    "peak_source": "measured" if "hbm_gbs" in peaks else "fallback"},
            "tensor": {"achieved": round(tfl, 2), "peak": tpeak, "unit": "TFLOP/s",
                       "frac": round(tfl / tpeak, 4), "peak_source": tsrc},
            **({"smem": smem} if smem else {})}


def warm_call_us(fn, dev, calls: int = 10) -> float:
    """Per-call microseconds of `calls` back-to-back calls replayed from one CUDA
    graph (inputs left in L2 between calls; the host's launch cost is out of it)."""
    import torch
    stream = torch.cuda.Stream(dev)
    stream.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(stream):
        fn()                                   # anything lazily set up, outside the capture
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(calls):
            fn()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize(dev)
    times = []
    for _ in range(RUNS):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize(dev)
        times.append(a.elapsed_time(b) * 1e3 / calls)
    return statistics.median(times)


def per_config_attention(key, w, dev, binding, timer, args, peaks, tpeak, tsrc) -> dict:
    case = AttnCase(w, dev, binding)
    steps = max(5, min(args.steps, 20))
    us, runs = timer.median_call_us(case.attn, steps, args.warmup)
    warm = None
    if not is_prefill(w) and not timer.warm:
        # second column: back-to-back calls with no flush, the pool staying in L2
        # as far as it fits (informational; the cold figure is the roofline's)
        warm_us = warm_call_us(case.attn, dev)
        warm = {"attn_us_per_call": round(warm_us, 3),
                "hbm_frac": round(algorithmic_bytes(w) / (warm_us * 1e-6) / 1e9
                                  / float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS)), 4),
                "how": "10 calls captured in one CUDA graph, median of 5 replays (no host launch gaps)"}
    step_ms = timer.run(case.step, steps)
    sms = torch_sms(dev)
    roof = attn_roofline(w, us, peaks, tpeak, tsrc, recorded_traffic(key), smem_roofline(key, us, peaks, sms))
    return {"value": round(w["T"] * len(step_ms) / (sum(step_ms) / 1e3), 1), "unit": UNIT,
            "workload": w["name"], "T": w["T"], "H": w["H"], "K": w["K"], "layout": w["layout"],
            "pool_rows": w["pool_rows"], "valid_entries": W.valid_entry_count(w["topk"]),
            "attn_us_per_call": round(us, 3), "attn_us_runs": runs,
            "step_us": round(statistics.mean(step_ms) * 1e3, 3), "roofline": roof,
            **({"warm": warm} if warm else {})}


def per_config_kv_write(layout, dev, binding, timer, args, peaks) -> dict:
    """One fused BF16 -> FP8 KV writer on 16384 new rows (N(0,1) x U(0.1, 8)) into
    distinct random slots of a 262144-row pool."""
    import torch
    w = W.writer_rows()
    n = w["n_rows"]
    x = w["x_bf16"]
    if layout == "rope656":   # 576-wide input rows: 512 latent dims + 64 RoPE dims
        rope = W.f32_to_bf16_bits(W.rng_for(8).standard_normal((n, W.D_ROPE), dtype=np.float32))
        x = np.concatenate([x, rope], axis=1)
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(dev)
    slots = torch.from_numpy(w["slots"]).to(dev)
    pool = torch.zeros(w["pool_rows"], ROW_BYTES[layout], dtype=torch.uint8, device=dev)
    write = WRITERS[layout](binding)
    us, runs = timer.median_call_us(lambda: write(xd, slots, pool), max(5, min(args.steps, 20)), args.warmup)
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    abytes = writer_bytes(n, layout)
    gbs = abytes / (us * 1e-6) / 1e9
    return {"value": round(n / (us * 1e-6), 1), "unit": "rows/s", "op": "kv_write", "layout": layout,
            "n_rows": n, "pool_rows": w["pool_rows"], "us_per_call": round(us, 3), "us_runs": runs,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(gbs / hbm, 4), "algorithmic_bytes_per_call": abytes,
                         "kernel": "kv_write_*_kernel"}}


def per_config_gather(w, dev, binding, timer, args, peaks) -> dict:
    """The gather/dequantise reader over a workload's pool and lists."""
    import torch
    case = AttnCase(w, dev, binding)
    T, K = w["T"], w["K"]
    out = binding.gather_workspace_for(T, K, w["pool_rows"], w["layout"], device=dev)
    idx = torch.empty(T, K, dtype=torch.int32, device=dev)

    def call():
        binding.dsa_gather_dequant(case.pool, w["layout"], case.topk, out, idx, page_table=case.pt,
                                   page_size=w["page_size"])
    us, runs = timer.median_call_us(call, max(5, min(args.steps, 20)), args.warmup)
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    abytes = gather_bytes(w)
    gbs = abytes / (us * 1e-6) / 1e9
    return {"value": round(W.valid_entry_count(w["topk"]) / (us * 1e-6), 1), "unit": "entries/s",
            "op": "gather_dequant", "workload": w["name"], "T": T, "K": K, "layout": w["layout"],
            "pool_rows": w["pool_rows"], "branch": "selected" if T * K < w["pool_rows"] else "full pool",
            "workspace_bytes": binding.dsa_gather_dequant_workspace_bytes(T, K, w["pool_rows"], w["layout"]),
            "us_per_call": round(us, 3), "us_runs": runs,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(gbs / hbm, 4), "algorithmic_bytes_per_call": abytes,
                         "kernel": "gather_dequant_kernel"}}


def run_ours(args, rank: int, world: int, local_rank: int, dist):
    import torch

    from sparse_mla_attention_page_gb300 import binding

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = make_workload(args.workload, args.heads, args.layout)
    T, H, K = w["T"], w["H"], w["K"]
    layout = w["layout"]
    prefill = is_prefill(w)
    timer = Timer(dev, args.warm)
    stream = torch.cuda.current_stream(dev)
    case = AttnCase(w, dev, binding)

    for _ in range(args.warmup):
        timer.flush()
        case.step()
    torch.cuda.synchronize(dev)

    props = torch.cuda.get_device_properties(dev)
    gpu_id = None
    if all(hasattr(props, f) for f in ("pci_domain_id", "pci_bus_id", "pci_device_id")):
        gpu_id = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)
    # the K timed steps, events at the step boundaries only: the attention kernel is
    # a programmatic dependent launch and may start its set-up while the writer runs
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    step_ms = timer.run(case.step, args.steps)
    if dist is not None:
        dist.barrier()
    # the attention call alone, for the roofline: RUNS runs of K flushed calls
    attn_us, attn_runs = timer.median_call_us(case.attn, args.steps, 0)
    t_wall1 = time.time()
    time.sleep(0.2)
    sampler.stop()
    total_ms = max_over_ranks(float(sum(step_ms)), dist, dev)

    # end to end through the public API, host buffers in and out
    e2e_ms, n_e2e, in_n, out_n, e2e_flush = run_e2e(case, w, binding, dev, max(1, min(args.e2e_steps, args.steps)),
                                                    timer)
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)

    if rank != 0:
        return None
    peaks = measured_peaks()
    fp8 = measure_fp8_peak(dev)
    tpeak, tsrc = tensor_peak(peaks, fp8)
    pkey = args.workload if args.workload != "writer_sweep" else None
    roof = attn_roofline(w, attn_us, peaks, tpeak, tsrc, recorded_traffic(pkey),
                         smem_roofline(pkey, attn_us, peaks, torch_sms(dev)))
    roof["attn_us_runs"] = attn_runs
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
                          else f"flushed before every step ({timer.flush_buf.numel() >> 20} MiB write)"),
                   "timing": f"value: {args.steps} timed steps; roofline: median of {RUNS} runs of "
                             f"{args.steps} flushed calls",
                   "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "e2e": {"value": round(world * T * n_e2e / (e2e_ms / 1e3), 1), "unit": UNIT,
                "h2d_bytes_per_step": in_n, "d2h_bytes_per_step": out_n,
                "how": f"{n_e2e} steps through the C ABI from pinned host memory, pipelined over three "
                       "streams (inputs of step i+1 uploading and outputs of step i-1 downloading while "
                       "step i computes; two device buffer sets); "
                       + ("L2 flushed before each step's kernels (inside the timed region)" if e2e_flush else
                          f"no L2 flush: each step copies {(in_n + out_n) >> 20} MiB, more than L2")},
        "gpu_launches": case.launches_per_step() * args.steps,
        "clocks": sampler.summary(t_wall0, t_wall1),
        "fp8_peak": fp8,
    }
    del case
    torch.cuda.empty_cache()
    if world == 1 and not args.no_per_config:
        line["per_config"] = run_per_config(args, dev, binding, timer, peaks, tpeak, tsrc,
                                            headline=(args.workload, roof, value))
    return line, w


def run_e2e(case, w, binding, dev, n_steps: int, timer):
    """End to end through the public API: every step copies its inputs (queries,
    top-k lists, the new latent rows, their slots, the page table) from one
    pinned host buffer to the device, runs writer (+ quantiser) + attention on
    them, and copies O and LSE back to pinned host memory.  Steps are pipelined
    over three streams with two device buffer sets: the upload of step i+1 and
    the download of step i-1 overlap the kernels of step i.  Returns the summed
    milliseconds of n_steps steps (first upload to last download), the steps,
    the bytes copied per step each way, and whether L2 was flushed before each
    step (when a step copies less than L2 holds)."""
    import torch
    T, H = w["T"], w["H"]

    def packed(parts):
        """Byte offsets of 256-byte-aligned parts in one buffer, and its size."""
        offs, n = [], 0
        for a in parts:
            offs.append(n)
            n += (a.nbytes + 255) // 256 * 256
        return offs, n

    in_parts = [np.ascontiguousarray(w["q_bf16"]), np.ascontiguousarray(w["topk"]),
                np.ascontiguousarray(case.x_new_h), np.ascontiguousarray(case.slots_h)]
    if w["page_table"] is not None:
        in_parts.append(np.ascontiguousarray(w["page_table"]))
    in_offs, in_n = packed(in_parts)
    h_in = torch.empty(in_n, dtype=torch.uint8).pin_memory()
    for a, off in zip(in_parts, in_offs):
        h_in[off:off + a.nbytes].copy_(torch.from_numpy(a.view(np.uint8).reshape(-1)))
    (o_off, lse_off), out_n = packed([np.empty((T, H, 512), np.uint16), np.empty((T, H), np.float32)])

    def view(buf, off, a_shape, dtype):
        n = int(np.prod(a_shape)) * torch.empty(0, dtype=dtype).element_size()
        return buf[off:off + n].view(dtype).view(*a_shape)

    sets = []
    for _ in range(2):
        d_in = torch.empty(in_n, dtype=torch.uint8, device=dev)
        d_out = torch.empty(out_n, dtype=torch.uint8, device=dev)
        sets.append({
            "d_in": d_in, "d_out": d_out, "h_out": torch.empty(out_n, dtype=torch.uint8).pin_memory(),
            "q": view(d_in, in_offs[0], w["q_bf16"].shape, torch.bfloat16),
            "topk": view(d_in, in_offs[1], w["topk"].shape, torch.int32),
            "x": view(d_in, in_offs[2], case.x_new_h.shape, torch.bfloat16),
            "slots": view(d_in, in_offs[3], case.slots_h.shape, torch.int64),
            "pt": None if w["page_table"] is None else view(d_in, in_offs[4], w["page_table"].shape, torch.int32),
            "o": view(d_out, o_off, (T, H, 512), torch.bfloat16),
            "lse": view(d_out, lse_off, (T, H), torch.float32)})
    if case.prefill:
        q8 = torch.empty(T, H, 512, dtype=torch.uint8, device=dev)
        qs = torch.empty(T, H, dtype=torch.float32, device=dev)
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    flush_each = (in_n + out_n) < torch.cuda.get_device_properties(dev).L2_cache_size and not timer.warm

    def pipeline(n: int):
        ev = [{k: torch.cuda.Event() for k in ("in", "comp", "out")} for _ in range(n)]
        for i in range(n):
            b = sets[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev[i - 2]["comp"])          # the kernels of step i-2 read this set
                b["d_in"].copy_(h_in, non_blocking=True)
                ev[i]["in"].record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(ev[i]["in"])
                if i >= 2:
                    s_comp.wait_event(ev[i - 2]["out"])         # step i-2's outputs have left this set
                if flush_each:
                    timer.flush()
                case.writer(b["x"], b["slots"], case.pool)
                if case.prefill:
                    binding.dsa_quantize_q8(b["q"], q8, qs)
                    binding.dsa_sparse_attn_prefill_q8(q8, qs, case.pool, case.layout, b["topk"], w["sm_scale"],
                                                       b["o"], b["lse"], case.ws, page_table=b["pt"],
                                                       page_size=w["page_size"])
                else:
                    binding.dsa_sparse_attn_decode(b["q"], case.pool, case.layout, b["topk"], w["sm_scale"],
                                                   b["o"], b["lse"], case.ws, page_table=b["pt"],
                                                   page_size=w["page_size"])
                ev[i]["comp"].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev[i]["comp"])
                b["h_out"].copy_(b["d_out"], non_blocking=True)
                ev[i]["out"].record(s_out)
        return ev

    torch.cuda.synchronize(dev)
    pipeline(3)                                                  # warm-up
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    ev = pipeline(n_steps)
    for e in ev:                                                 # end after every step's download
        s_out.wait_event(e["out"])
    end.record(s_out)
    torch.cuda.synchronize(dev)
    ms = start.elapsed_time(end)
    del sets, h_in
    return ms, n_steps, in_n, out_n, flush_each


def run_per_config(args, dev, binding, timer, peaks, tpeak, tsrc, headline) -> dict:
    import torch
    only = None if args.only is None else set(args.only.split(","))
    out = {}
    for key, kind, wname, opt in PER_CONFIG:
        if only is not None and key not in only:
            continue
        if kind == "attention" and wname == headline[0] and not opt:
            out[key] = {"same_as": "headline line (roofline, value)"}
            continue
        t0 = time.time()
        try:
            if kind == "attention":
                w = make_workload(wname, opt.get("heads", 16), opt.get("layout", "raw512"))
                out[key] = per_config_attention(key, w, dev, binding, timer, args, peaks, tpeak, tsrc)
            elif kind == "kv_write":
                out[key] = per_config_kv_write(opt["layout"], dev, binding, timer, args, peaks)
            else:
                out[key] = per_config_gather(make_workload(wname), dev, binding, timer, args, peaks)
        except Exception as e:  # noqa: BLE001 - one failing config must not hide the others
            out[key] = {"error": f"{type(e).__name__}: {e}"[:300]}
        out[key]["wall_s"] = round(time.time() - t0, 1)
        torch.cuda.empty_cache()
    return out


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
    if is_prefill(w):
        q8, qs = oracle.quantize_q8(w["q_bf16"])
    return pool, q8, qs


def _oracle_rate(w, pool, q8, qs, n_threads: int, seconds: float, chunk: int):
    """Query-tokens/s of the oracle (writer of the step's rows + attention) over
    consecutive slices of `chunk` tokens until `seconds` have passed."""
    import oracle
    x_new, slots = step_rows(w)
    T = w["T"]
    done, start = 0, 0
    t0 = time.perf_counter()
    while True:
        tokens = (np.arange(chunk) + start) % T
        start = (start + chunk) % T
        oracle.kv_write(w["layout"], x_new, slots, pool)
        oracle_pass(w, pool, tokens, n_threads, q8, qs)
        done += chunk
        if time.perf_counter() - t0 >= seconds:
            break
    return done, time.perf_counter() - t0


def cpu_baseline(w: dict, seconds: float) -> dict:
    """The oracle as it stands on the host cores: all cores (the figure) and one
    thread, each over slices of the batch until its time has passed; each slice
    runs the writer of the step's new rows and the attention of its tokens."""
    cores = len(os.sched_getaffinity(0))
    pool, q8, qs = oracle_setup(w)
    T = w["T"]
    chunk_all = min(T, 64) if is_prefill(w) else T
    done, dt = _oracle_rate(w, pool, q8, qs, cores, seconds, chunk_all)
    chunk_one = min(T, 2 if is_prefill(w) else 16)
    done1, dt1 = _oracle_rate(w, pool, q8, qs, 1, seconds / 2, chunk_one)
    return {"value": round(done / dt, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{done} tokens of {w['name']} in slices of {chunk_all} (writer of the step's rows + "
                      f"float64 attention), {dt:.1f} s on {cores} threads",
            "single_thread": {"value": round(done1 / dt1, 3), "unit": UNIT, "cores": 1,
                              "sample": f"{done1} tokens in slices of {chunk_one}, {dt1:.1f} s on 1 thread"}}


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
