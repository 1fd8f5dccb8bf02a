"""Checks that tie the CPU oracle to something other than itself.

Each ``pin_*`` function raises AssertionError when the oracle (the library
currently loaded by ``oracle.lib()``) disagrees with an independent fact:
the OCP E4M3 table, PyTorch's own float8_e4m3fn conversion, hand-derived
worked examples, PyTorch's float64 scaled-dot-product attention and
logsumexp, closed forms and invariants of the attention definition.
The same functions run against deliberately broken copies of the oracle in
``test_oracle_mutants.py`` to show that each plausible mistake is caught.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle
from sparse_mla_attention_page_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _torch_decode(b: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def _torch_encode(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def _all_bf16_as_f32() -> np.ndarray:
    return W.bf16_bits_to_f32(np.arange(65536, dtype=np.uint32).astype(np.uint16))


# ------------------------------------------------------------------ FP8 codec

def pin_decode_spec():
    with open(os.path.join(GOLDEN, "e4m3_spec_values.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    for byte, val in rows:
        got = oracle.e4m3_decode(int(byte, 16))
        if val == "nan":
            assert math.isnan(got), byte
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val)), (byte, got, val)


def pin_decode_torch():
    b = np.arange(256, dtype=np.uint8)
    ours, ref = oracle.decode_table(), _torch_decode(b)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def pin_encode_exhaustive_bf16():
    """Every BF16 input: bisection == exhaustive search == PyTorch RNE (|x| <= 464),
    and saturation to +-448 above (PyTorch gives NaN there, it does not saturate)."""
    x = _all_bf16_as_f32()
    x = x[~np.isnan(x)]
    fast = oracle.e4m3_encode_array(x)
    brute = oracle.e4m3_encode_array(x, bruteforce=True)
    assert np.array_equal(fast, brute)
    small = np.abs(x) <= 464.0
    assert np.array_equal(fast[small], _torch_encode(x[small]))
    big = ~small
    assert np.array_equal(fast[big], np.where(np.signbit(x[big]), 0xFE, 0x7E).astype(np.uint8))


def pin_encode_ties_and_f32():
    """Exact midpoints between adjacent codes go to the even code; random FP32
    inputs over the whole range agree with PyTorch."""
    vals = oracle.decode_table()[:127]
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    assert np.array_equal(((vals[:-1] + vals[1:]) / 2), mids.astype(np.float64))  # exact in FP32
    got = oracle.e4m3_encode_array(mids)
    lo = np.arange(126)
    want = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8)
    assert np.array_equal(got, want)
    assert np.array_equal(oracle.e4m3_encode_array(-mids), want | 0x80)
    rng = np.random.default_rng(11)
    r = (rng.standard_normal(200000) * np.exp2(rng.uniform(-14, 9, 200000))).astype(np.float32)
    r = r[np.abs(r) <= 464.0]
    assert np.array_equal(oracle.e4m3_encode_array(r), _torch_encode(r))


def pin_encode_roundtrip():
    b = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    v = oracle.decode_table()[b].astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode_array(v), b)


# ------------------------------------------------------------------- writers

def pin_encode_nan():
    """NaN inputs: every FP32 NaN encoding (quiet and signalling payloads, both
    signs) and every BF16 NaN bit pattern encodes as PyTorch's float8_e4m3fn
    cast does: the FN NaN code 0x7F with the input's sign bit."""
    f32 = np.array([0x7FC00000, 0xFFC00000, 0x7F800001, 0xFF800001, 0x7FFFFFFF, 0xFFFFFFFF, 0x7FA00000],
                   dtype=np.uint32).view(np.float32)
    bf = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    bf = bf[((bf & 0x7F80) == 0x7F80) & ((bf & 0x7F) != 0)]
    x = np.concatenate([f32, W.bf16_bits_to_f32(bf)])
    assert np.isnan(x).all() and x.size == 7 + 2 * 127
    want = _torch_encode(x)
    for brute in (False, True):
        got = oracle.e4m3_encode_array(x, bruteforce=brute)
        np.testing.assert_array_equal(got, want)
    assert set(want.tolist()) == {0x7F, 0xFF}


def pin_nan_in_scaled_writer_and_quantiser():
    """NaN elements of a group-scaled row or of a query vector: the scale is
    taken over the other values (NumPy's nanmax / 448 in FP32) and the NaN
    encodes as 0x7F with its own sign, whatever sign a division would give."""
    rng = np.random.default_rng(17)
    xf = rng.standard_normal((4, 512)).astype(np.float32)
    nan_pos = [(0, 3, 0), (1, 200, 1), (2, 511, 0), (3, 0, 1), (3, 130, 1)]   # (row, dim, negative)
    x = W.f32_to_bf16_bits(xf)
    for r, d, neg in nan_pos:
        x[r, d] = 0xFFC0 if neg else 0x7FC0
    xv = W.bf16_bits_to_f32(x)
    pool = oracle.new_pool(4, "scaled528")
    oracle.kv_write("scaled528", x, np.arange(4), pool)
    sc = pool[:, 512:].copy().view("<f4")
    amax = np.nanmax(np.abs(xv.reshape(4, 4, 128)), axis=2)
    np.testing.assert_array_equal(sc, (amax / np.float32(448)).astype(np.float32))
    q8, qs = oracle.quantize_q8(x.reshape(4, 1, 512))
    np.testing.assert_array_equal(qs[:, 0], (np.nanmax(np.abs(xv), axis=1) / np.float32(448)).astype(np.float32))
    for r, d, neg in nan_pos:
        assert pool[r, d] == (0xFF if neg else 0x7F), (r, d, pool[r, d])
        assert q8[r, 0, d] == (0xFF if neg else 0x7F), (r, d, q8[r, 0, d])
    finite = ~np.isnan(xv)
    assert not np.isin(pool[:, :512][finite], [0x7F, 0xFF]).any()


def _bf16_row(values: np.ndarray) -> np.ndarray:
    bits = W.f32_to_bf16_bits(values.astype(np.float32))
    assert np.array_equal(W.bf16_bits_to_f32(bits), values.astype(np.float32)), "fixture not BF16-exact"
    return bits


def pin_scaled_worked_example():
    x = np.zeros(512, dtype=np.float32)
    want = np.zeros(528, dtype=np.uint8)
    scales = {}
    with open(os.path.join(GOLDEN, "scaled528_row_worked_example.txt")) as f:
        for ln in f:
            ln = ln.split("#")[0].split()
            if not ln:
                continue
            if ln[0] == "scale":
                scales[int(ln[1])] = int(ln[2], 16)
                continue
            g, i, v, byte = int(ln[0]), int(ln[1]), float(ln[2]), int(ln[3], 16)
            x[128 * g + i] = v
            want[128 * g + i] = byte
    for g, bits in scales.items():
        want[512 + 4 * g: 516 + 4 * g] = np.frombuffer(np.uint32(bits).tobytes(), dtype=np.uint8)
    pool = oracle.new_pool(3, "scaled528")
    pool[:] = 0xAB
    oracle.kv_write("scaled528", _bf16_row(x)[None, :], np.array([1]), pool)
    assert np.array_equal(pool[1], want), np.nonzero(pool[1] != want)
    assert (pool[0] == 0xAB).all() and (pool[2] == 0xAB).all()


def pin_raw_writer_torch():
    rng = np.random.default_rng(12)
    x = W.f32_to_bf16_bits((rng.standard_normal((40, 512)) * rng.uniform(0.01, 300, (40, 1))).astype(np.float32))
    slots = rng.choice(200, size=40, replace=False).astype(np.int64)
    slots[5] = -1
    pool = oracle.new_pool(200, "raw512")
    pool[:] = 0x11
    n = oracle.kv_write("raw512", x, slots, pool)
    assert n == 39
    xf = W.bf16_bits_to_f32(x)
    want = _torch_encode(np.clip(xf, -448, 448))
    for i, s in enumerate(slots):
        if s >= 0:
            assert np.array_equal(pool[s], want[i]), i
    untouched = np.setdiff1d(np.arange(200), slots[slots >= 0])
    assert (pool[untouched] == 0x11).all()


def pin_scaled_writer_invariants():
    rng = np.random.default_rng(13)
    n = 64
    xf = (rng.standard_normal((n, 512)) * rng.uniform(1e-3, 1e3, (n, 1))).astype(np.float32)
    xf[3, 128:256] = 0.0                                  # one zero group
    x = W.f32_to_bf16_bits(xf)
    xf = W.bf16_bits_to_f32(x)
    pool = oracle.new_pool(n, "scaled528")
    oracle.kv_write("scaled528", x, np.arange(n), pool)
    vals = _torch_decode(pool[:, :512]).reshape(n, 4, 128)
    sc = pool[:, 512:].copy().view("<f4").astype(np.float64)      # [n, 4]
    xg = xf.reshape(n, 4, 128).astype(np.float64)
    amax = np.abs(xg).max(axis=2)
    zero = amax == 0
    assert zero[3, 1] and zero.sum() == 1
    assert (sc[zero] == 0).all() and (pool[3, 128:256] == 0).all()
    nz = ~zero
    # the scale is amax/448 rounded to FP32 (within half an FP32 ulp)
    assert (np.abs(sc[nz] * 448 - amax[nz]) <= amax[nz] * 2.0 ** -23).all()
    # the group's largest element encodes to +-448
    arg = np.abs(xg).argmax(axis=2)
    top = np.take_along_axis(vals, arg[..., None], axis=2)[..., 0]
    sgn = np.sign(np.take_along_axis(xg, arg[..., None], axis=2)[..., 0])
    assert np.array_equal(top[nz], 448.0 * sgn[nz])
    # dequantisation error: half an E4M3 ulp of x/s (normal range) or 2^-10 s below
    deq = vals * sc[..., None]
    err = np.abs(deq - xg)
    r = np.abs(xg) / np.where(sc > 0, sc, 1)[..., None]
    bound = np.where(r >= 2.0 ** -6, np.abs(xg) * 2.0 ** -4, sc[..., None] * 2.0 ** -10) * (1 + 1e-6)
    assert (err[nz] <= bound[nz]).all()


# ----------------------------------------------------------------- attention

def _pool_rows_f64(pool: np.ndarray, layout: str, rows: np.ndarray) -> np.ndarray:
    r = pool[rows]
    v = _torch_decode(r[:, :512])
    if layout == "scaled528":
        sc = r[:, 512:].copy().view("<f4").astype(np.float64)
        v = v * np.repeat(sc, 128, axis=1)
    return v


def _phys(page_table, token_seq, t, idx, page_size=64):
    if page_table is None:
        return idx
    seq = 0 if token_seq is None else token_seq[t]
    return page_table[seq, idx // page_size] * page_size + idx % page_size


def _sdpa_reference(w: dict, pool: np.ndarray):
    """Float64 PyTorch scaled_dot_product_attention over each token's gathered rows."""
    T, H = w["T"], w["H"]
    q = torch.from_numpy(w["q_bf16"].astype(np.int16)).view(torch.bfloat16).to(torch.float64)
    O = np.zeros((T, H, 512))
    L = np.full((T, H), -np.inf)
    for t in range(T):
        idx = w["topk"][t]
        idx = idx[idx >= 0]
        if idx.size == 0:
            continue
        rows = np.array([_phys(w["page_table"], w.get("token_seq"), t, int(i)) for i in idx])
        k = torch.from_numpy(_pool_rows_f64(pool, w["layout"], rows))
        qt = q[t][None, :, None, :]                     # [1, H, 1, 512]
        kk = k[None, None].expand(1, H, -1, -1)
        o = torch.nn.functional.scaled_dot_product_attention(qt, kk, kk, scale=float(np.float32(w["sm_scale"])))
        O[t] = o[0, :, 0].numpy()
        logits = (q[t] @ k.T) * float(np.float32(w["sm_scale"]))
        L[t] = torch.logsumexp(logits, dim=-1).numpy()
    return O, L


def _oracle_run(w: dict, pool: np.ndarray, **kw):
    return oracle.sparse_attn(pool, w["layout"], w["topk"], w["sm_scale"], q_bf16=w["q_bf16"],
                              page_table=w["page_table"], page_size=w["page_size"],
                              token_seq=w.get("token_seq"), **kw)


def _tiny(layout: str, seed: int, T=5, H=4, K=256, pool_rows=1024, dup=False, seqs=1):
    rng = np.random.default_rng(seed)
    mult = rng.uniform(0.1, 4, (pool_rows, 1)) if layout == "scaled528" else 1.0
    kv = W.f32_to_bf16_bits((rng.standard_normal((pool_rows, 512)) * mult).astype(np.float32))
    pages = pool_rows // 64
    seq_pages = pages // seqs
    perm = rng.permutation(pages).astype(np.int32)
    page_table = perm[: seq_pages * seqs].reshape(seqs, seq_pages)
    token_seq = (np.arange(T) % seqs).astype(np.int32) if seqs > 1 else None
    span = seq_pages * 64
    if dup:
        topk = rng.integers(0, span, (T, K)).astype(np.int32)
    else:
        topk = np.stack([rng.choice(span, K, replace=False) for _ in range(T)]).astype(np.int32)
    topk[rng.random((T, K)) < 0.1] = -1
    q = W.f32_to_bf16_bits(rng.standard_normal((T, H, 512)).astype(np.float32))
    w = dict(layout=layout, T=T, H=H, K=K, q_bf16=q, kv_src=kv, kv_slots=np.arange(pool_rows),
             pool_rows=pool_rows, page_table=page_table, page_size=64, token_seq=token_seq,
             topk=topk, sm_scale=W.SM_SCALE)
    return w, oracle.fill_pool(w)


def pin_attn_sdpa():
    for layout, seed, dup, seqs in (("raw512", 21, False, 1), ("scaled528", 22, True, 2),
                                    ("raw512", 23, True, 3)):
        w, pool = _tiny(layout, seed, dup=dup, seqs=seqs)
        O, L, err = _oracle_run(w, pool, n_threads=2)
        Or, Lr = _sdpa_reference(w, pool)
        assert err == 0
        np.testing.assert_allclose(O, Or, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(L, Lr, rtol=1e-12, atol=1e-12)


def pin_attn_closed_forms():
    w, pool = _tiny("raw512", 31, T=4, H=3)
    topk = np.full_like(w["topk"], -1)
    topk[0, 17] = w["topk"][0, 0] if w["topk"][0, 0] >= 0 else 5      # one-hot
    # token 1: all masked (left as -1)
    topk[2, :40] = np.arange(40) * 3                                      # Q = 0 case below
    topk[3, :2] = [7, 7]                                                  # duplicate pair
    w2 = dict(w, topk=topk)
    q = w["q_bf16"].copy()
    q[2] = 0
    w2["q_bf16"] = q
    O, L, _ = _oracle_run(w2, pool)
    pt = w["page_table"]
    # one-hot: O = that row, LSE = its logit
    row = _phys(pt, None, 0, int(topk[0, 17]))
    k = _pool_rows_f64(pool, "raw512", np.array([row]))[0]
    qf = W.bf16_bits_to_f32(q[0]).astype(np.float64)
    np.testing.assert_allclose(O[0], np.broadcast_to(k, O[0].shape), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(L[0], float(np.float32(W.SM_SCALE)) * (qf @ k), rtol=1e-12, atol=1e-13)
    # all masked: O = 0, LSE = -inf
    assert (O[1] == 0).all() and np.isneginf(L[1]).all()
    # Q = 0: uniform weights, O = mean of the rows, LSE = ln(count)
    rows = np.array([_phys(pt, None, 2, int(i)) for i in topk[2, :40]])
    mean = _pool_rows_f64(pool, "raw512", rows).mean(axis=0)
    np.testing.assert_allclose(O[2], np.broadcast_to(mean, O[2].shape), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(L[2], math.log(40), rtol=1e-14)
    # a duplicated entry counts twice: LSE = logit + ln 2, O = the row
    row = _phys(pt, None, 3, 7)
    k = _pool_rows_f64(pool, "raw512", np.array([row]))[0]
    qf = W.bf16_bits_to_f32(q[3]).astype(np.float64)
    np.testing.assert_allclose(L[3], float(np.float32(W.SM_SCALE)) * (qf @ k) + math.log(2), rtol=1e-12)
    np.testing.assert_allclose(O[3], np.broadcast_to(k, O[3].shape), rtol=1e-12, atol=1e-14)


def pin_attn_invariances():
    w, pool = _tiny("scaled528", 41, dup=True)
    O, L, _ = _oracle_run(w, pool)
    rng = np.random.default_rng(42)
    # permuting each token's top-k list (the -1 slots too) changes nothing
    perm = np.stack([rng.permutation(w["K"]) for _ in range(w["T"])])
    O2, L2, _ = _oracle_run(dict(w, topk=np.take_along_axis(w["topk"], perm, axis=1)), pool)
    np.testing.assert_allclose(O2, O, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(L2, L, rtol=1e-13)
    # moving physical pages, with the page table updated to match, changes nothing
    pages = w["pool_rows"] // 64
    move = rng.permutation(pages)                       # old page p -> new page move[p]
    pool3 = np.empty_like(pool)
    pool3.reshape(pages, 64, -1)[move] = pool.reshape(pages, 64, -1)
    O3, L3, _ = _oracle_run(dict(w, page_table=move[w["page_table"]].astype(np.int32)), pool3)
    np.testing.assert_array_equal(O3, O)
    np.testing.assert_array_equal(L3, L)
    # a scaled row whose four scales are 1.0 reads like the raw row
    wr, praw = _tiny("raw512", 43)
    psc = np.zeros((praw.shape[0], 528), dtype=np.uint8)
    psc[:, :512] = praw
    psc[:, 512:] = np.frombuffer(np.array([1.0] * 4, dtype="<f4").tobytes(), dtype=np.uint8)
    Or, Lr, _ = _oracle_run(wr, praw)
    Os, Ls, _ = _oracle_run(dict(wr, layout="scaled528"), psc)
    np.testing.assert_array_equal(Os, Or)
    np.testing.assert_array_equal(Ls, Lr)


def pin_q8_matches_bf16_decode():
    """An FP8 query with power-of-two scales is exactly a BF16 query: the Q8
    path must give the BF16 path's answer for it."""
    w, pool = _tiny("raw512", 51, T=3, H=4)
    rng = np.random.default_rng(52)
    q8 = rng.integers(0, 256, (3, 4, 512)).astype(np.uint8)
    q8[(q8 & 0x7F) == 0x7F] = 0x3C                      # no NaN codes
    sc = np.exp2(rng.integers(-6, 3, (3, 4))).astype(np.float32)
    qf = _torch_decode(q8) * sc[..., None]
    qb = W.f32_to_bf16_bits(qf.astype(np.float32))
    assert np.array_equal(W.bf16_bits_to_f32(qb).astype(np.float64), qf)
    O8, L8, _ = oracle.sparse_attn(pool, "raw512", w["topk"], w["sm_scale"], q8=q8, q_scale=sc,
                                   page_table=w["page_table"])
    Ob, Lb, _ = oracle.sparse_attn(pool, "raw512", w["topk"], w["sm_scale"], q_bf16=qb,
                                   page_table=w["page_table"])
    np.testing.assert_array_equal(O8, Ob)
    np.testing.assert_array_equal(L8, Lb)


def pin_q8_quantiser():
    rng = np.random.default_rng(53)
    q = W.f32_to_bf16_bits((rng.standard_normal((6, 5, 512)) * rng.uniform(0.01, 50, (6, 5, 1))).astype(np.float32))
    q[2, 3] = 0
    q8, sc = oracle.quantize_q8(q)
    qf = W.bf16_bits_to_f32(q).astype(np.float64)
    amax = np.abs(qf).max(-1)
    assert sc[2, 3] == 0 and (q8[2, 3] == 0).all()
    nz = amax > 0
    assert (np.abs(sc[nz].astype(np.float64) * 448 - amax[nz]) <= amax[nz] * 2.0 ** -23).all()
    arg = np.abs(qf).argmax(-1)
    top = np.take_along_axis(_torch_decode(q8), arg[..., None], -1)[..., 0]
    assert np.array_equal(np.abs(top[nz]), np.full(nz.sum(), 448.0))
    deq = _torch_decode(q8) * sc[..., None]
    assert (np.abs(deq - qf) <= np.abs(qf) * 2.0 ** -4 + sc[..., None] * 2.0 ** -10 + 1e-30).all()


def pin_error_bits():
    w, pool = _tiny("raw512", 61, T=3, H=2, seqs=2)
    topk = w["topk"].copy()
    seq_pages = w["page_table"].shape[1]
    topk[0, 3] = seq_pages * 64 + 5           # beyond the page table's width
    O, L, err = _oracle_run(dict(w, topk=topk), pool)
    assert err == oracle.ERR_INDEX_RANGE
    ref = topk.copy()
    ref[0, 3] = -1
    O2, L2, err2 = _oracle_run(dict(w, topk=ref), pool)
    assert err2 == 0
    np.testing.assert_array_equal(O, O2)
    pt = w["page_table"].copy()
    first = int(topk[1][topk[1] >= 0][0])
    pt[1, first // 64] = w["pool_rows"] // 64 + 3          # page beyond the pool
    _, _, err3 = _oracle_run(dict(w, page_table=pt), pool)
    assert err3 == oracle.ERR_PAGE_RANGE
    # physical indices (no page table): index beyond the pool
    topk4 = np.array([[5, w["pool_rows"], -1, 9]], dtype=np.int32)
    _, _, err4 = oracle.sparse_attn(pool, "raw512", topk4, W.SM_SCALE, q_bf16=w["q_bf16"][:1])
    assert err4 == oracle.ERR_INDEX_RANGE


def pin_wrong_index_is_detected():
    """Negative control: one wrong row index moves O beyond the attention
    tolerance, so the parity comparison can see a gather mistake."""
    w, pool = _tiny("raw512", 71, T=2, H=8, K=128)
    topk = w["topk"].copy()
    topk[:, 1:] = -1                            # single valid entry: its row is O
    O, L, _ = _oracle_run(dict(w, topk=topk), pool)
    bad = topk.copy()
    bad[:, 0] = (bad[:, 0] + 1) % (w["page_table"].shape[1] * 64)
    Ob, Lb, _ = _oracle_run(dict(w, topk=bad), pool)
    diff = np.abs(Ob - O) - (1e-2 + 1e-2 * np.abs(O))
    assert (diff > 0).any()


def _torch_rows_bf16(pool: np.ndarray, layout: str, rows: np.ndarray) -> np.ndarray:
    """BF16 bits of physical rows dequantised by PyTorch: its own FP8 decode
    (raw rows, exact in BF16), or its FP32 product with the group scale cast
    to BF16; 656-byte rows append their stored RoPE bits."""
    rows = np.asarray(rows, dtype=np.int64)
    r = torch.from_numpy(np.ascontiguousarray(pool[rows, :512])).view(torch.float8_e4m3fn)
    if layout == "raw512":
        v = r.to(torch.bfloat16)
    else:
        sc = torch.from_numpy(np.ascontiguousarray(pool[rows, 512:528]).view("<f4").copy())
        v = (r.to(torch.float32) * sc.repeat_interleave(128, dim=1)).to(torch.bfloat16)
    out = v.view(torch.int16).numpy().view(np.uint16)
    if layout == "rope656":
        out = np.concatenate([out, np.ascontiguousarray(pool[rows, 528:656]).view("<u2")], axis=1)
    return out


def _tiny_rope(seed: int, T: int, K: int, pool_rows: int):
    w = W.decode_rope656(seed=seed, T=T, H=2, K=K, pool_rows=pool_rows)
    w["token_seq"] = None
    return w, oracle.fill_pool(w)


def pin_gather_selected_branch():
    """Fewer top-k entries than pool rows: the workspace has one row per entry
    (T*K rows), each the PyTorch dequantisation of the entry's physical row;
    the remapped index of an entry is its entry number, -1 where masked; an
    entry outside the page table is masked with the attention's error bit."""
    for layout, seed, seqs in (("raw512", 81, 1), ("scaled528", 82, 2)):
        w, pool = _tiny(layout, seed, T=4, K=128, seqs=seqs)
        topk = w["topk"].copy()
        T, K = topk.shape
        assert T * K < w["pool_rows"]
        out, idx, err = oracle.gather_dequant(pool, layout, topk, page_table=w["page_table"],
                                              page_size=64, token_seq=w["token_seq"])
        assert err == 0 and out.shape == (T * K, 512)
        want_idx = np.where(topk >= 0, np.arange(T * K, dtype=np.int32).reshape(T, K), -1)
        np.testing.assert_array_equal(idx, want_idx)
        e = np.nonzero(topk.reshape(-1) >= 0)[0]
        rows = np.array([_phys(w["page_table"], w["token_seq"], int(i) // K, int(topk.reshape(-1)[i]))
                         for i in e])
        np.testing.assert_array_equal(out[e], _torch_rows_bf16(pool, layout, rows))
        masked = np.nonzero(topk.reshape(-1) < 0)[0]
        assert masked.size and not out[masked].any()          # masked rows are not written
    bad = topk.copy()
    bad[0, 0] = w["page_table"].shape[1] * 64 + 1          # beyond the page table's width
    _, idx2, err2 = oracle.gather_dequant(pool, "scaled528", bad, page_table=w["page_table"],
                                          page_size=64, token_seq=w["token_seq"])
    assert err2 == oracle.ERR_INDEX_RANGE and idx2[0, 0] == -1


def pin_gather_full_pool_branch():
    """As many top-k entries as pool rows, or more: the workspace is the whole
    pool dequantised by PyTorch (pool_rows rows), and each entry's remapped
    index is its physical row (page table applied), -1 where masked.  The
    boundary T*K == pool_rows already takes this branch."""
    for layout, seed, T, K in (("raw512", 83, 4, 128), ("scaled528", 84, 6, 128)):
        w, pool = _tiny(layout, seed, T=T, K=K, pool_rows=512, seqs=2)
        topk = w["topk"]
        assert T * K >= w["pool_rows"]
        out, idx, err = oracle.gather_dequant(pool, layout, topk, page_table=w["page_table"],
                                              page_size=64, token_seq=w["token_seq"])
        assert err == 0 and out.shape == (w["pool_rows"], 512)
        np.testing.assert_array_equal(out, _torch_rows_bf16(pool, layout, np.arange(w["pool_rows"])))
        want = np.array([[_phys(w["page_table"], w["token_seq"], t, int(i)) if i >= 0 else -1
                          for i in topk[t]] for t in range(T)], dtype=np.int32)
        np.testing.assert_array_equal(idx, want)


def pin_gather_rows_bound():
    """The workspace row count is min(pool rows, selected entries): its BF16
    payload is bounded by min(physical_tokens, selected_entries) * 1024 bytes."""
    for pool_rows, n in ((1024, 512), (1024, 1023), (1024, 1024), (1024, 1025), (131072, 262144),
                         (16384, 8388608), (4096, 0)):
        assert oracle.gather_rows(pool_rows, n) == min(pool_rows, n), (pool_rows, n)


def pin_gather_rope656():
    """656-byte rows in both branches: 576-wide BF16 workspace rows, the
    latent dims dequantised as for 528-byte rows and the RoPE dims copied."""
    for T, K, pool_rows in ((2, 128, 1024), (4, 256, 1024)):
        w, pool = _tiny_rope(85 + T, T, K, pool_rows)
        topk = w["topk"]
        out, idx, err = oracle.gather_dequant(pool, "rope656", topk, page_table=w["page_table"], page_size=64)
        assert err == 0 and out.shape == (min(pool_rows, T * K), 576)
        for t in range(T):
            for j in range(K):
                if topk[t, j] < 0:
                    assert idx[t, j] == -1
                    continue
                row = _phys(w["page_table"], None, t, int(topk[t, j]))
                np.testing.assert_array_equal(out[idx[t, j]], _torch_rows_bf16(pool, "rope656", [row])[0])


def pin_rope656():
    """656-byte rows: the latent part is byte-identical to the group-scaled
    writer's row, the RoPE part is the input BF16 bits; attention over 576-wide
    keys with 512-wide values equals PyTorch's float64 scaled_dot_product_attention
    and logsumexp."""
    w = W.decode_rope656(seed=91, T=4, H=3, K=256, pool_rows=2048)
    pool = oracle.fill_pool(w)
    ref = oracle.new_pool(w["pool_rows"], "scaled528")
    oracle.kv_write("scaled528", np.ascontiguousarray(w["kv_src"][:, :512]), w["kv_slots"], ref)
    np.testing.assert_array_equal(pool[:, :528], ref)
    np.testing.assert_array_equal(pool[:, 528:].view("<u2"), w["kv_src"][:, 512:])
    O, L, err = oracle.sparse_attn(pool, "rope656", w["topk"], w["sm_scale"], q_bf16=w["q_bf16"],
                                   page_table=w["page_table"], page_size=64, n_threads=2)
    assert err == 0
    q = torch.from_numpy(w["q_bf16"].astype(np.int16)).view(torch.bfloat16).to(torch.float64)
    for t in range(w["T"]):
        idx = w["topk"][t]
        idx = idx[idx >= 0]
        rows = np.array([_phys(w["page_table"], None, t, int(i)) for i in idx])
        nope = torch.from_numpy(_pool_rows_f64(pool[:, :528], "scaled528", rows))
        rope = torch.from_numpy(np.ascontiguousarray(pool[rows, 528:]).view(np.int16)).view(torch.bfloat16)
        k = torch.cat([nope, rope.to(torch.float64)], dim=1)             # [n, 576]
        sc = float(np.float32(w["sm_scale"]))
        o = torch.nn.functional.scaled_dot_product_attention(q[t][:, None, :], k[None].expand(w["H"], -1, -1),
                                                             nope[None].expand(w["H"], -1, -1), scale=sc)
        np.testing.assert_allclose(O[t], o[:, 0].numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(L[t], torch.logsumexp((q[t] @ k.T) * sc, dim=-1).numpy(), rtol=1e-12, atol=1e-12)


ALL_PINS = [
    pin_decode_spec, pin_decode_torch, pin_encode_exhaustive_bf16, pin_encode_ties_and_f32,
    pin_encode_roundtrip, pin_scaled_worked_example, pin_raw_writer_torch,
    pin_scaled_writer_invariants, pin_attn_sdpa, pin_attn_closed_forms, pin_attn_invariances,
    pin_q8_matches_bf16_decode, pin_q8_quantiser, pin_error_bits, pin_wrong_index_is_detected,
    pin_gather_selected_branch, pin_gather_full_pool_branch,
    pin_gather_rows_bound, pin_gather_rope656, pin_rope656, pin_encode_nan,
    pin_nan_in_scaled_writer_and_quantiser,
]
