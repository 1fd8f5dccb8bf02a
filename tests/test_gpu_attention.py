"""Sparse attention through the C ABI against the CPU oracle.

Small cases are compared on every element; the full-size workloads (the
shapes the benchmark times) on every element where the oracle finishes in
seconds and on a fixed sample of tokens otherwise.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_attn_close, bf16_dev, dev, pool_dev, run_decode, run_prefill
from sparse_mla_attention_page_gb300 import binding
from sparse_mla_attention_page_gb300 import workloads as W

pytestmark = pytest.mark.gpu

_pools = {}


def pool_for(w, key):
    if key not in _pools:
        p = oracle.fill_pool(w)
        _pools[key] = (p, pool_dev(p))
    return _pools[key]


def oracle_decode(w, pool, tokens=None, topk=None, page_table=None):
    return oracle.sparse_attn(pool, w["layout"], w["topk"] if topk is None else topk, w["sm_scale"],
                              q_bf16=w["q_bf16"],
                              page_table=w["page_table"] if page_table is None else page_table,
                              page_size=w["page_size"], token_seq=w.get("token_seq"), tokens=tokens)


def sample_tokens(T, n, seed):
    if T <= n:
        return np.arange(T)
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, T - 1), n - 2, replace=False)
    return np.sort(np.concatenate([[0, T - 1], mid]))


# ----------------------------------------------------------------- workloads

def test_tiny_decode_raw512():
    w = W.tiny_decode_raw512()
    pool, pd = pool_for(w, "tiny")
    O, L, err = run_decode(w, pd)
    Or, Lr, erro = oracle_decode(w, pool)
    assert err == erro == 0
    assert_attn_close(O, L, Or, Lr, "tiny")


@pytest.mark.parametrize("T,K,pool_rows", [(16, 1024, 16384), (5, 384, 8192), (64, 2048, 131072)])
def test_decode_raw512(T, K, pool_rows):
    w = W.decode_raw512(T=T, K=K, pool_rows=pool_rows)
    pool, pd = pool_for(w, ("raw", T, K, pool_rows))
    O, L, err = run_decode(w, pd)
    Or, Lr, _ = oracle_decode(w, pool)
    assert err == 0
    assert_attn_close(O, L, Or, Lr, f"decode_raw512 T={T} K={K}")
    assert np.isneginf(L[1]).all() and (O[1] == 0).all()     # the all-masked token


@pytest.mark.parametrize("T,K,pool_rows,full", [(16, 512, 16384, True), (128, 2048, 131072, False)])
def test_decode_scaled528(T, K, pool_rows, full):
    w = W.decode_scaled528(T=T, K=K, pool_rows=pool_rows)
    pool, pd = pool_for(w, ("scaled", T, K, pool_rows))
    O, L, err = run_decode(w, pd)
    tok = None if full else sample_tokens(T, 24, 7)
    Or, Lr, _ = oracle_decode(w, pool, tokens=tok)
    assert err == 0
    if tok is not None:
        O, L = O[tok], L[tok]
    assert_attn_close(O, L, Or, Lr, f"decode_scaled528 T={T}")


@pytest.mark.parametrize("T,full", [(64, True), (4096, False)])
def test_prefill_q8_raw512(T, full):
    w = W.prefill_q8_raw512(T=T)
    pool, pd = pool_for(w, ("prefill", T))
    q8, qs = oracle.quantize_q8(w["q_bf16"])
    O, L, err = run_prefill(w, pd, q8, qs)
    tok = None if full else sample_tokens(T, 24, 8)
    Or, Lr, _ = oracle.sparse_attn(pool, "raw512", w["topk"], w["sm_scale"], q8=q8, q_scale=qs,
                                   page_table=w["page_table"], tokens=tok)
    assert err == 0
    if tok is not None:
        O, L = O[tok], L[tok]
    assert_attn_close(O, L, Or, Lr, f"prefill_q8 T={T}")


@pytest.mark.parametrize("H", [8, 16, 64])
def test_prefill_q8_head_counts(H):
    """FP8 queries with 8 and 16 heads (one head group) and 64 heads (two groups of 32,
    the one-P-buffer pipeline); a short context pads the first tokens' top-k with -1."""
    w = W.prefill_q8_raw512(T=24, H=H, context=1024, pool_rows=2048)
    pool, pd = pool_for(w, ("prefill_heads", H))
    q8, qs = oracle.quantize_q8(w["q_bf16"])
    O, L, err = run_prefill(w, pd, q8, qs)
    Or, Lr, _ = oracle.sparse_attn(pool, "raw512", w["topk"], w["sm_scale"], q8=q8, q_scale=qs,
                                   page_table=w["page_table"])
    assert err == 0
    assert_attn_close(O, L, Or, Lr, f"prefill_q8 H={H}")


@pytest.mark.parametrize("T,full", [(64, True), (4096, False)])
def test_prefill_q8_scaled528(T, full):
    """FP8 queries over group-scaled 528-byte rows (beyond the pages, which keep
    Q8 prefill to raw rows): the same definition, scales applied per group."""
    w = W.prefill_q8_scaled528(T=T)
    pool, pd = pool_for(w, ("prefill_scaled", T))
    q8, qs = oracle.quantize_q8(w["q_bf16"])
    O, L, err = run_prefill(w, pd, q8, qs)
    tok = None if full else sample_tokens(T, 24, 9)
    Or, Lr, _ = oracle.sparse_attn(pool, "scaled528", w["topk"], w["sm_scale"], q8=q8, q_scale=qs,
                                   page_table=w["page_table"], tokens=tok)
    assert err == 0
    if tok is not None:
        O, L = O[tok], L[tok]
    assert_attn_close(O, L, Or, Lr, f"prefill_q8_scaled528 T={T}")


@pytest.mark.parametrize("T,K,H,full", [(16, 512, 16, True), (8, 256, 8, True), (64, 2048, 16, False),
                                         (12, 384, 32, True), (5, 256, 64, True), (2, 256, 128, True),
                                         (64, 2048, 32, False)])
def test_decode_rope656(T, K, H, full):
    """656-byte rows: group-scaled latent plus 64 BF16 RoPE dims; 576-wide
    queries and keys (the RoPE scores by BF16 MMAs), 512-wide values; 32 and
    more heads run as head groups of 16."""
    w = W.decode_rope656(T=T, K=K, H=H, pool_rows=131072 if not full else 16384)
    pool, pd = pool_for(w, ("rope", T, K, H))
    O, L, err = run_decode(w, pd)
    tok = None if full else sample_tokens(T, 16, 10)
    Or, Lr, _ = oracle_decode(w, pool, tokens=tok)
    assert err == 0
    if tok is not None:
        O, L = O[tok], L[tok]
    assert_attn_close(O, L, Or, Lr, f"decode_rope656 T={T} H={H}")


@pytest.mark.parametrize("layout", ["raw512", "scaled528", "rope656", "q8_raw512"])
def test_peaked_softmax(layout):
    """Queries scaled up (x100) so each head's logits spread over far more than
    2^8 in log2 units and a handful of entries carry the softmax: O is then
    about the size of a KV row, so the tolerance sees errors in PV, and the
    running maximum is raised mid-segment (the O rescale path).  Besides the
    elementwise tolerance, the largest error must stay within 1 % of max |O|."""
    T, H, K = 8, 16, 1024
    if layout == "rope656":
        w = W.decode_rope656(seed=300, T=T, H=H, K=K, pool_rows=8192)
    elif layout == "scaled528":
        w = W.decode_scaled528(seed=301, T=T, H=H, K=K, pool_rows=8192)
    else:
        w = W.decode_raw512(seed=302, T=T, H=H, K=K, pool_rows=8192, special_tokens=False)
    q = W.bf16_bits_to_f32(w["q_bf16"]) * np.float32(100.0)
    w["q_bf16"] = W.f32_to_bf16_bits(q)
    pool, pd = pool_for(w, ("peaked", layout))
    if layout == "q8_raw512":
        q8, qs = oracle.quantize_q8(w["q_bf16"])
        O, L, err = run_prefill(w, pd, q8, qs)
        Or, Lr, _ = oracle.sparse_attn(pool, "raw512", w["topk"], w["sm_scale"], q8=q8, q_scale=qs,
                                       page_table=w["page_table"])
    else:
        O, L, err = run_decode(w, pd)
        Or, Lr, _ = oracle_decode(w, pool)
    assert err == 0
    st = assert_attn_close(O, L, Or, Lr, f"peaked {layout}")
    assert st["max_ref"] > 0.3, st                         # O is row-sized, not ~0.01
    assert st["rel_to_max"] <= 1e-2, st


@pytest.mark.parametrize("scale", [1.0, 4.0, 16.0])
@pytest.mark.parametrize("peaked", [False, True])
def test_prefill_q8_row_magnitudes(scale, peaked):
    """The error of O from the FP8 split of P grows with the rows' magnitudes
    (relative error of a P entry times max|V|): rows of N(0, scale^2) latents
    (entries up to about 70 at scale 16), with a flat and with a peaked softmax
    (queries scaled so the logits keep their spread), stay within the tolerance
    at 32 heads with FP8 queries."""
    T, H, K = 8, 32, 1024
    w = W.decode_raw512(seed=310, T=T, H=H, K=K, pool_rows=8192, special_tokens=False)
    w["kv_src"] = W.f32_to_bf16_bits(W.bf16_bits_to_f32(w["kv_src"]) * np.float32(2.0 * scale))
    if peaked:
        w["q_bf16"] = W.f32_to_bf16_bits(W.bf16_bits_to_f32(w["q_bf16"]) * np.float32(100.0 / scale))
    pool, pd = pool_for(w, ("magnitude", scale, peaked))
    q8, qs = oracle.quantize_q8(w["q_bf16"])
    O, L, err = run_prefill(w, pd, q8, qs)
    Or, Lr, _ = oracle.sparse_attn(pool, "raw512", w["topk"], w["sm_scale"], q8=q8, q_scale=qs,
                                   page_table=w["page_table"])
    assert err == 0
    assert_attn_close(O, L, Or, Lr, f"q8 rows x{scale} {'peaked' if peaked else 'flat'}")


def test_prefill_q8_short_context_padding():
    """Zero prior context: early tokens have fewer than K causal rows, so the
    list is padded with -1 (down to a single valid entry for the first token)."""
    w = W.prefill_q8_raw512(T=40, K=256, context=0, pool_rows=1024)
    pool, pd = pool_for(w, ("prefill_short",))
    q8, qs = oracle.quantize_q8(w["q_bf16"])
    assert (w["topk"][0] >= 0).sum() == 1
    O, L, _ = run_prefill(w, pd, q8, qs)
    Or, Lr, _ = oracle.sparse_attn(pool, "raw512", w["topk"], w["sm_scale"], q8=q8, q_scale=qs,
                                   page_table=w["page_table"])
    assert_attn_close(O, L, Or, Lr, "prefill short context")


@pytest.mark.parametrize("layout", ["raw512", "scaled528"])
@pytest.mark.parametrize("H", [8, 16, 32])
def test_writer_sweep_decode(layout, H):
    """Decode over rows the GPU writer just wrote (physical indices, no page
    table); one one-hot and one all-masked token."""
    w = W.writer_sweep(H=H, layout=layout)
    pool, _ = pool_for(w, ("sweep", layout))
    gpu_pool = torch.zeros(w["pool_rows"], oracle.row_bytes(layout), dtype=torch.uint8, device="cuda")
    fn = binding.dsa_kv_write_raw if layout == "raw512" else binding.dsa_kv_write_scaled
    fn(bf16_dev(w["kv_src"]), dev(w["kv_slots"]), gpu_pool)
    torch.cuda.synchronize()
    assert np.array_equal(gpu_pool.cpu().numpy(), pool)
    O, L, err = run_decode(w, gpu_pool)
    tok = sample_tokens(w["T"], 16, 9)
    Or, Lr, _ = oracle_decode(w, pool, tokens=tok)
    assert err == 0
    assert_attn_close(O[tok], L[tok], Or, Lr, f"sweep {layout} H={H}")
    k0 = int(w["topk"][0, 0])
    if layout == "raw512":
        row = oracle.decode_table()[pool[k0]]
    else:
        sc = pool[k0, 512:].copy().view("<f4").astype(np.float64)
        row = oracle.decode_table()[pool[k0, :512]] * np.repeat(sc, 128)
    np.testing.assert_allclose(O[0], np.broadcast_to(row, O[0].shape), rtol=1e-2, atol=1e-2)
    assert np.isneginf(L[1]).all() and (O[1] == 0).all()


# ---------------------------------------------------------------- edge cases

def _small(layout="raw512", T=6, H=16, K=256, pool_rows=2048, seed=200, **kw):
    if layout == "raw512":
        w = W.decode_raw512(seed=seed, T=T, H=H, K=K, pool_rows=pool_rows, special_tokens=False, **kw)
    else:
        w = W.decode_scaled528(seed=seed, T=T, H=H, K=K, pool_rows=pool_rows, **kw)
    return w


@pytest.mark.parametrize("H", [64, 128])
def test_many_heads(H):
    w = _small(H=H, T=3)
    pool, pd = pool_for(w, ("heads", H))
    O, L, _ = run_decode(w, pd)
    Or, Lr, _ = oracle_decode(w, pool)
    assert_attn_close(O, L, Or, Lr, f"H={H}")


def test_all_tokens_masked():
    w = _small(T=4)
    pool, pd = pool_for(w, ("masked",))
    topk = np.full_like(w["topk"], -1)
    O, L, _ = run_decode(w, pd, topk=topk)
    assert (O == 0).all() and np.isneginf(L).all()


@pytest.mark.parametrize("K", [128, 8192])
def test_topk_widths(K):
    w = _small(T=5, K=K, pool_rows=16384)
    pool, pd = pool_for(w, ("K", K))
    O, L, _ = run_decode(w, pd)
    Or, Lr, _ = oracle_decode(w, pool)
    assert_attn_close(O, L, Or, Lr, f"K={K}")


@pytest.mark.parametrize("mode", ["raw512", "scaled528", "q8", "rope656"])
def test_one_tile_segments(mode):
    """Many tokens with one-tile lists (K = 128): every tile is a segment of its
    own, so each CTA switches query buffers, resets the running state and runs
    the epilogue on every tile, and the tail CTAs' units split across CTAs."""
    T, H, K = 1000, 16, 128
    rng = np.random.default_rng(500)
    if mode == "rope656":
        w = W.decode_rope656(seed=501, T=T, H=H, K=K, pool_rows=8192)
    else:
        w = _small(layout="scaled528" if mode == "scaled528" else "raw512", T=T, H=H, K=K, pool_rows=8192,
                   seed=502)
    w["topk"] = np.stack([rng.choice(8192, K, replace=False) for _ in range(T)]).astype(np.int32)
    w["topk"][rng.random((T, K)) < 0.1] = -1
    pool, pd = pool_for(w, ("one-tile", mode))
    if mode == "q8":
        q8, qs = oracle.quantize_q8(w["q_bf16"])
        O, L, err = run_prefill(w, pd, q8, qs)
        Or, Lr, erro = oracle.sparse_attn(pool, "raw512", w["topk"], w["sm_scale"], q8=q8, q_scale=qs,
                                          page_table=w["page_table"], page_size=w["page_size"])
    else:
        O, L, err = run_decode(w, pd)
        Or, Lr, erro = oracle_decode(w, pool)
    assert err == erro == 0
    assert_attn_close(O, L, Or, Lr, f"one-tile segments {mode}")


@pytest.mark.parametrize("T,K,layout", [(1, 8192, "raw512"), (2, 16384, "raw512"), (1, 4096, "scaled528")])
def test_unit_spread_over_many_ctas(T, K, layout):
    """Few tokens with long top-k lists: each (token, head group) is split over
    dozens of CTAs, so the merge folds many partial results (several batches)."""
    w = _small(T=T, K=K, pool_rows=32768, layout=layout)
    pool, pd = pool_for(w, ("spread", T, K, layout))
    O, L, err = run_decode(w, pd)
    Or, Lr, _ = oracle_decode(w, pool)
    assert err == 0
    assert_attn_close(O, L, Or, Lr, f"T={T} K={K} {layout}")


def test_multi_sequence_page_tables():
    """Tokens of three sequences, each with its own page table row."""
    rng = np.random.default_rng(201)
    w = _small(T=9, K=256, pool_rows=4096)
    perm = rng.permutation(64).astype(np.int32)
    w["page_table"] = perm[:60].reshape(3, 20)
    w["token_seq"] = (np.arange(9) % 3).astype(np.int32)
    w["topk"] = np.stack([rng.choice(20 * 64, 256, replace=False) for _ in range(9)]).astype(np.int32)
    w["topk"][:, 200:] = -1
    pool, pd = pool_for(w, ("multi",))
    O, L, err = run_decode(w, pd)
    Or, Lr, erro = oracle_decode(w, pool)
    assert err == erro == 0
    assert_attn_close(O, L, Or, Lr, "multi-seq")


@pytest.mark.parametrize("page_size", [1, 16, 128, 256])
@pytest.mark.parametrize("mode", ["raw512", "scaled528", "q8"])
def test_page_sizes(page_size, mode):
    """Index translation row = page_table[seq][i / P] * P + i % P at page sizes
    other than the workloads' 64 (one row a page up to 256), over a shuffled
    page table; decode over both layouts and the FP8-query prefill."""
    rng = np.random.default_rng(400 + page_size)
    pool_rows = 4096
    w = _small(layout="scaled528" if mode == "scaled528" else "raw512", T=5, K=384, pool_rows=pool_rows,
               seed=401 + page_size)
    pages = pool_rows // page_size
    w["page_table"] = rng.permutation(pages).astype(np.int32).reshape(1, pages)
    w["page_size"] = page_size
    w["topk"] = np.stack([rng.choice(pool_rows, 384, replace=False) for _ in range(5)]).astype(np.int32)
    w["topk"][:, 300:] = -1
    pool, pd = pool_for(w, ("page_size", page_size, mode))
    if mode == "q8":
        q8, qs = oracle.quantize_q8(w["q_bf16"])
        O, L, err = run_prefill(w, pd, q8, qs)
        Or, Lr, erro = oracle.sparse_attn(pool, "raw512", w["topk"], w["sm_scale"], q8=q8, q_scale=qs,
                                          page_table=w["page_table"], page_size=page_size)
    else:
        O, L, err = run_decode(w, pd)
        Or, Lr, erro = oracle_decode(w, pool)
    assert err == erro == 0
    assert_attn_close(O, L, Or, Lr, f"page size {page_size} {mode}")


def test_duplicates_and_scattered_sentinels():
    w = _small("scaled528", T=6, K=384, pool_rows=2048, masked_frac=0.3)
    w["topk"][:, 10:50] = w["topk"][:, 50:90]                    # many duplicates
    pool, pd = pool_for(w, ("dups",))
    O, L, _ = run_decode(w, pd)
    Or, Lr, _ = oracle_decode(w, pool)
    assert_attn_close(O, L, Or, Lr, "duplicates")


def test_out_of_range_entries_masked_and_flagged():
    w = _small(T=4, K=256, pool_rows=4096)
    pool, pd = pool_for(w, ("oob",))
    topk = w["topk"].copy()
    width = w["page_table"].shape[1] * 64
    topk[0, 5] = width + 3                               # beyond the page table
    O, L, err = run_decode(w, pd, topk=topk)
    Or, Lr, erro = oracle_decode(w, pool, topk=topk)
    assert err == erro == binding.DSA_DEV_ERR_INDEX_RANGE
    assert_attn_close(O, L, Or, Lr, "index beyond page table")
    pt = w["page_table"].copy()
    pt[0, int(topk[1, 0]) // 64] = 10**6                   # page beyond the pool
    O, L, err = run_decode(w, pd, page_table=pt)
    Or, Lr, erro = oracle_decode(w, pool, page_table=pt)
    assert err == erro == binding.DSA_DEV_ERR_PAGE_RANGE
    assert_attn_close(O, L, Or, Lr, "bad page entry")


def test_physical_indices_out_of_range():
    w = W.writer_sweep(H=16, T=4, K=128, n_rows=512, pool_rows=1024)
    pool, pd = pool_for(w, ("phys_oob",))
    topk = w["topk"].copy()
    topk[2, 7] = w["pool_rows"] + 11
    O, L, err = run_decode(w, pd, topk=topk)
    Or, Lr, erro = oracle_decode(w, pool, topk=topk)
    assert err == erro == binding.DSA_DEV_ERR_INDEX_RANGE
    assert_attn_close(O, L, Or, Lr, "physical index beyond pool")


def test_repeatable_and_stream():
    w = _small(T=8, K=512, pool_rows=8192)
    pool, pd = pool_for(w, ("rep",))
    s = torch.cuda.Stream()
    O1, L1, _ = run_decode(w, pd)
    with torch.cuda.stream(s):
        O2, L2, _ = run_decode(w, pd, stream=s)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_cuda_graph_replay_with_changed_inputs():
    """Capture one decode call, then change indices, queries and the pool's
    scale words in place and replay: the result must follow the new inputs
    (no host read of device data, no allocation inside the call)."""
    w = _small("scaled528", T=8, K=256, pool_rows=4096)
    pool, _ = pool_for(w, ("graph",))
    pool_d = pool_dev(pool.copy())
    T, H, K = w["T"], w["H"], w["K"]
    q_d = bf16_dev(w["q_bf16"])
    topk_d = dev(w["topk"])
    pt_d = dev(w["page_table"])
    o = torch.empty(T, H, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(T, H, dtype=torch.float32, device="cuda")
    ws = binding.workspace_for(T, H, K)
    args = (q_d, pool_d, "scaled528", topk_d, w["sm_scale"], o, lse, ws)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        binding.dsa_sparse_attn_decode(*args, page_table=pt_d, page_size=64)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        binding.dsa_sparse_attn_decode(*args, page_table=pt_d, page_size=64)
    rng = np.random.default_rng(202)
    for rep in range(2):
        w2 = dict(w)
        w2["topk"] = np.stack([rng.choice(4096, K) for _ in range(T)]).astype(np.int32)
        w2["topk"][rng.random((T, K)) < 0.1] = -1
        w2["q_bf16"] = W.f32_to_bf16_bits(rng.standard_normal((T, H, 512)).astype(np.float32))
        pool2 = pool.copy()
        pool2[:, 512:] = np.frombuffer((pool[:, 512:].copy().view("<f4") * np.float32(1.5 + rep)).tobytes(),
                                       dtype=np.uint8).reshape(-1, 16)
        topk_d.copy_(dev(w2["topk"]))
        q_d.copy_(bf16_dev(w2["q_bf16"]))
        pool_d.copy_(pool_dev(pool2))
        g.replay()
        torch.cuda.synchronize()
        O = o.float().cpu().numpy().astype(np.float64)
        L = lse.cpu().numpy().astype(np.float64)
        Or, Lr, _ = oracle_decode(w2, pool2)
        assert_attn_close(O, L, Or, Lr, f"graph replay {rep}")


def test_t_zero_is_noop():
    w = _small(T=2)
    pool, pd = pool_for(w, ("t0",))
    o = torch.full((0, 16, 512), 1.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(0, 16, dtype=torch.float32, device="cuda")
    binding.dsa_sparse_attn_decode(torch.empty(0, 16, 512, dtype=torch.bfloat16, device="cuda"), pd,
                                   "raw512", torch.empty(0, 256, dtype=torch.int32, device="cuda"),
                                   0.1, o, lse)


def test_wrong_index_negative_control():
    """A deliberately wrong index on the host side makes the comparison fail:
    the parity check can see a single-row gather mistake."""
    w = _small(T=3, K=128)
    topk = w["topk"].copy()
    topk[:, 1:] = -1
    pool, pd = pool_for(w, ("neg",))
    O, L, _ = run_decode(w, pd, topk=topk)
    bad = topk.copy()
    bad[:, 0] = (bad[:, 0] + 1) % (w["page_table"].shape[1] * 64)
    Or, Lr, _ = oracle_decode(w, pool, topk=bad)
    with pytest.raises(AssertionError):
        assert_attn_close(O, L, Or, Lr, "negative control")
