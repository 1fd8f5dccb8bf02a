"""GPU writers and FP8 query quantiser against the oracle: bit-exact bytes."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import bf16_dev, dev
from sparse_mla_attention_page_gb300 import binding
from sparse_mla_attention_page_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _finite_bf16_patterns(include_inf: bool) -> np.ndarray:
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = W.bf16_bits_to_f32(bits)
    keep = ~np.isnan(f) if include_inf else np.isfinite(f)
    return bits[keep]


def _write_gpu(layout, x_bits, slots, pool_init):
    pool = dev(pool_init.copy())
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    fn = {"raw512": binding.dsa_kv_write_raw, "scaled528": binding.dsa_kv_write_scaled,
          "rope656": binding.dsa_kv_write_rope656}[layout]
    fn(bf16_dev(x_bits), dev(slots.astype(np.int64)), pool, err_flag=err)
    torch.cuda.synchronize()
    return pool.cpu().numpy(), int(err.item())


@pytest.mark.parametrize("layout", ["raw512", "scaled528"])
def test_every_bf16_input_bit_exact(layout):
    """Every BF16 bit pattern (NaN patterns have their own test; inf is
    excluded for the scaled layout, where it turns the group's scale into
    inf), shuffled into rows so that groups mix magnitudes."""
    bits = _finite_bf16_patterns(include_inf=(layout == "raw512"))
    rng = np.random.default_rng(100)
    bits = bits[rng.permutation(bits.size)]
    n = -(-bits.size // 512)
    x = np.zeros(n * 512, dtype=np.uint16)
    x[: bits.size] = bits
    x = x.reshape(n, 512)
    slots = rng.permutation(n + 7)[:n].astype(np.int64)
    init = np.full((n + 7, oracle.row_bytes(layout)), 0x5A, dtype=np.uint8)
    ref = init.copy()
    oracle.kv_write(layout, x, slots, ref)
    got, err = _write_gpu(layout, x, slots, init)
    assert err == 0
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} bytes differ, first at {bad[:3].tolist()}"


def _nan_bf16_patterns() -> np.ndarray:
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    return bits[np.isnan(W.bf16_bits_to_f32(bits))]


@pytest.mark.parametrize("layout", ["raw512", "scaled528", "rope656"])
def test_nan_inputs_bit_exact(layout):
    """Every BF16 NaN pattern (both signs, all payloads), scattered among
    finite values: the NaN encodes as 0x7F with the input's sign, and the
    group scales ignore it (they are taken over the finite values)."""
    nan = _nan_bf16_patterns()
    assert nan.size == 254
    rng = np.random.default_rng(101)
    width = 576 if layout == "rope656" else 512
    n = 32
    x = W.f32_to_bf16_bits((rng.standard_normal((n, width)) * rng.uniform(0.1, 8, (n, 1))).astype(np.float32))
    pos = rng.choice(n * 512, nan.size, replace=False)            # latent dims only
    flat = x[:, :512].reshape(-1).copy()
    flat[pos] = nan
    x[:, :512] = flat.reshape(n, 512)
    slots = rng.permutation(n + 5)[:n].astype(np.int64)
    init = np.full((n + 5, oracle.row_bytes(layout)), 0x3C, dtype=np.uint8)
    ref = init.copy()
    oracle.kv_write(layout, x, slots, ref)
    got, err = _write_gpu(layout, x, slots, init)
    assert err == 0
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} bytes differ, first at {bad[:3].tolist()}: got {got[tuple(bad[0])]:#x} want {ref[tuple(bad[0])]:#x}"


def test_quantizer_nan_inputs_bit_exact():
    """The FP8 query quantiser over vectors holding every BF16 NaN pattern."""
    nan = _nan_bf16_patterns()
    rng = np.random.default_rng(102)
    q = W.f32_to_bf16_bits(rng.standard_normal((8, 4, 512)).astype(np.float32))
    flat = q.reshape(-1).copy()
    flat[rng.choice(flat.size, nan.size, replace=False)] = nan
    q = flat.reshape(q.shape)
    q8r, qsr = oracle.quantize_q8(q)
    q8 = torch.empty(8, 4, 512, dtype=torch.uint8, device="cuda")
    qs = torch.empty(8, 4, dtype=torch.float32, device="cuda")
    binding.dsa_quantize_q8(bf16_dev(q), q8, qs)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(q8.cpu().numpy(), q8r)
    np.testing.assert_array_equal(qs.cpu().numpy().view(np.uint32), qsr.view(np.uint32))


@pytest.mark.parametrize("layout", ["raw512", "scaled528"])
def test_writer_workload_bit_exact(layout):
    """16384 rows N(0,1)*U(0.1,8) into distinct random slots of a 262144-row
    pool (page size 64, so writes cross page boundaries)."""
    w = W.writer_rows()
    init = np.full((w["pool_rows"], oracle.row_bytes(layout)), 0xA5, dtype=np.uint8)
    ref = init.copy()
    oracle.kv_write(layout, w["x_bf16"], w["slots"], ref)
    got, err = _write_gpu(layout, w["x_bf16"], w["slots"], init)
    assert err == 0
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("layout", ["raw512", "scaled528"])
def test_writer_slot_edge_cases(layout):
    rng = np.random.default_rng(101)
    x = W.f32_to_bf16_bits(rng.standard_normal((6, 512)).astype(np.float32))
    x[2, :128] = 0                                          # a zero group
    slots = np.array([3, -1, 63, 64, 200, 0], dtype=np.int64)  # -1 skipped, 200 out of range
    init = np.full((128, oracle.row_bytes(layout)), 0x33, dtype=np.uint8)
    ok = slots.copy()
    ok[4] = -1
    ref = init.copy()
    oracle.kv_write(layout, x, ok, ref)
    got, err = _write_gpu(layout, x, slots, init)
    assert err == binding.DSA_DEV_ERR_SLOT_RANGE
    assert np.array_equal(got, ref)


def test_rope656_writer_bit_exact():
    """656-byte rows: 8192 rows of the decode_rope656 source (latent N(0,1)*U(0.1,4),
    RoPE N(0,1)) plus rows of every finite BF16 pattern in both parts, into
    random slots; a skipped and an out-of-range slot."""
    w = W.decode_rope656(T=1, K=128, pool_rows=8192)
    rng = np.random.default_rng(102)
    bits = _finite_bf16_patterns(include_inf=False)
    bits = bits[rng.permutation(bits.size)]
    n_extra = -(-bits.size // 576)
    extra = np.zeros(n_extra * 576, dtype=np.uint16)
    extra[: bits.size] = bits
    x = np.concatenate([w["kv_src"], extra.reshape(n_extra, 576)])
    n = x.shape[0]
    slots = rng.permutation(n + 9)[:n].astype(np.int64)
    slots[5] = -1
    init = np.full((n + 9, 656), 0x3C, dtype=np.uint8)
    ok = slots.copy()
    slots[7] = n + 50                                        # beyond the pool: flagged, not written
    ok[7] = -1
    ref = init.copy()
    oracle.kv_write("rope656", x, ok, ref)
    got, err = _write_gpu("rope656", x, slots, init)
    assert err == binding.DSA_DEV_ERR_SLOT_RANGE
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} bytes differ, first at {bad[:3].tolist()}"


def test_writer_empty_is_noop():
    pool = torch.full((8, 512), 7, dtype=torch.uint8, device="cuda")
    binding.dsa_kv_write_raw(torch.empty(0, 512, dtype=torch.bfloat16, device="cuda"),
                             torch.empty(0, dtype=torch.int64, device="cuda"), pool)
    torch.cuda.synchronize()
    assert (pool == 7).all()


def test_quantize_q8_bit_exact():
    rng = np.random.default_rng(102)
    q = W.f32_to_bf16_bits((rng.standard_normal((64, 32, 512)) *
                            rng.uniform(1e-3, 100, (64, 32, 1))).astype(np.float32))
    q[5, 7] = 0
    q8_ref, sc_ref = oracle.quantize_q8(q)
    q8 = torch.empty(64, 32, 512, dtype=torch.uint8, device="cuda")
    sc = torch.empty(64, 32, dtype=torch.float32, device="cuda")
    binding.dsa_quantize_q8(bf16_dev(q), q8, sc)
    torch.cuda.synchronize()
    assert np.array_equal(q8.cpu().numpy(), q8_ref)
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), sc_ref.view(np.uint32))
