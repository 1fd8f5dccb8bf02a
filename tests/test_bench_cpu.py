"""CPU checks of bench.py: the byte and flop counts behind the roofline, its
defaults, the JSON line of the reference arm (the oracle, run on the host), and
the multi-rank path on two gloo ranks (max-over-ranks timing, rank 0 alone
printing)."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from sparse_mla_attention_page_gb300 import workloads as W  # noqa: E402


def test_algorithmic_bytes_decode():
    """Each valid entry's 512-byte row once, BF16 Q and O, int32 top-k, FP32 LSE."""
    w = W.tiny_decode_raw512()
    T, H, K = w["T"], w["H"], w["K"]
    valid = int((w["topk"] >= 0).sum())
    assert valid == T * (K - 16)                  # the tiny case masks a 16-entry tail
    expect = valid * 512 + T * H * 512 * 2 + T * K * 4 + T * H * 512 * 2 + T * H * 4
    assert bench.algorithmic_bytes(w) == expect
    assert bench.attn_flops(w) == 4 * H * 512 * valid


def test_algorithmic_bytes_prefill_and_rope():
    """Q8 prefill: one-byte queries plus an FP32 scale per (token, head); 656-byte rows:
    576-wide BF16 queries and keys, values over the 512 latent dims."""
    w = W.prefill_q8_raw512(T=8, context=256, pool_rows=512)
    T, H, K = w["T"], w["H"], w["K"]
    valid = int((w["topk"] >= 0).sum())
    assert valid == sum(min(K, 256 + t + 1) for t in range(T))
    expect = valid * 512 + T * H * 512 + T * H * 4 + T * K * 4 + T * H * 512 * 2 + T * H * 4
    assert bench.algorithmic_bytes(w) == expect
    r = W.decode_rope656(T=2, K=256, pool_rows=4096)
    v = int((r["topk"] >= 0).sum())
    assert bench.algorithmic_bytes(r) == (v * 656 + r["T"] * r["H"] * 576 * 2 + r["T"] * r["K"] * 4
                                          + r["T"] * r["H"] * 512 * 2 + r["T"] * r["H"] * 4)
    assert bench.attn_flops(r) == 2 * r["H"] * (576 + 512) * v


def test_defaults(monkeypatch):
    """The headline is the largest single-GPU batch (the Q8 prefill); at least
    3 warm-up steps; every per_config entry names a known workload or op."""
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse_args()
    assert (a.gpus, a.impl, a.workload) == (1, "ours", "prefill_q8_raw512")
    assert a.warmup >= 3 and a.steps >= 1 and not a.warm and not a.no_per_config
    keys = [k for k, _, _, _ in bench.PER_CONFIG]
    assert len(keys) == len(set(keys))
    for key, kind, wname, opt in bench.PER_CONFIG:
        assert kind in ("attention", "kv_write", "gather_dequant")
        assert wname is None or wname in W.WORKLOADS
        assert kind != "kv_write" or opt["layout"] in bench.ROW_BYTES
    for need in ("tiny_decode_raw512", "decode_raw512", "decode_scaled528", "kv_write_raw512",
                 "kv_write_scaled528", "writer_sweep_raw512_h32", "writer_sweep_scaled528_h8"):
        assert need in keys


def test_gather_and_writer_bytes():
    """The reader moves each valid entry's row and BF16 output row when entries
    are fewer than pool rows, else the whole pool once; plus the lists."""
    w = W.tiny_decode_raw512()
    v = int((w["topk"] >= 0).sum())
    assert bench.gather_bytes(w) == v * (512 + 1024) + w["T"] * w["K"] * 8
    w2 = W.decode_raw512(T=8, K=256, pool_rows=2048)
    assert w2["T"] * w2["K"] >= w2["pool_rows"]
    assert bench.gather_bytes(w2) == 2048 * (512 + 1024) + 8 * 256 * 8
    assert bench.writer_bytes(10, "scaled528") == 10 * (1024 + 528 + 8)
    assert bench.writer_bytes(10, "rope656") == 10 * (1152 + 656 + 8)


def test_tensor_peak_choice():
    assert bench.tensor_peak({"bf16_tflops": 1000.0}, {"tflops": 3500.0}) == (3500.0, "measured FP8 burst")
    assert bench.tensor_peak({"bf16_tflops": 1000.0}, {"tflops": None})[0] == 2000.0
    assert bench.tensor_peak({}, None)[0] == 2 * bench.FALLBACK_BF16_TFLOPS


def test_recorded_counters_follow_the_kernel_source(monkeypatch):
    """The DRAM and shared-memory figures of the ncu record are used only while
    the kernel source hashes to the profiled one; the bank roofline is bytes /
    time against 128 B a clock on every SM."""
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        rec = json.load(f)
    e = rec["prefill_q8_raw512"]
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: e["source_sha"])
    assert bench.recorded_traffic("prefill_q8_raw512") == e["dram_bytes_per_call"]
    r = bench.smem_roofline("prefill_q8_raw512", 1000.0, {"sm_max_mhz": 2000.0}, 100)
    assert r["peak"] == 128 * 100 * 2000e6 / 1e9
    assert abs(r["achieved"] - e["smem_bank_bytes_per_call"] / 1e-3 / 1e9) < 0.1
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-4
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: "0" * 16)
    assert bench.recorded_traffic("prefill_q8_raw512") is None
    assert bench.smem_roofline("prefill_q8_raw512", 1000.0, {}, 100) is None


def test_reference_arm_line():
    """The reference arm times the oracle on the host cores and prints one JSON line
    with the metric, the impl tag, a cpu_baseline and an e2e with no copies."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny_decode_raw512", "--steps", "1", "--warmup", "1"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and np.isfinite(d["value"])
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "tiny_decode_raw512" and d["higher_is_better"] is True


def _free_port() -> int:
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    v = bench.max_over_ranks(1.5 + rank, dist, "cpu")
    with open(os.path.join(out_dir, f"rank{rank}"), "w") as f:
        f.write(repr(v))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    """The timed region of a multi-rank run is the slowest rank's: every rank gets
    the maximum (two gloo ranks on the CPU)."""
    torch.multiprocessing.spawn(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    assert [float((tmp_path / f"rank{r}").read_text()) for r in range(2)] == [2.5, 2.5]
    assert bench.max_over_ranks(3.0, None, "cpu") == 3.0


def test_reference_arm_two_ranks():
    """Launched as the driver launches N > 1 (torchrun, one process per rank), the
    reference arm runs on rank 0 alone: one JSON line, every rank exits 0."""
    out = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                          "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
                          os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny_decode_raw512",
                          "--steps", "1", "--warmup", "1"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    assert json.loads(lines[0])["impl"] == "reference"
