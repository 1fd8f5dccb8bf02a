"""The gather/dequantise reader on the GPU against the oracle, in both of its
branches: fewer top-k entries than pool rows (a workspace row per entry) and
as many or more (the whole pool dequantised).  Workspace rows and remapped
indices bit-exact, error bits equal, rows the reader must not write left
untouched."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import dev, pool_dev
from sparse_mla_attention_page_gb300 import binding
from sparse_mla_attention_page_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SENTINEL = 0x7FBF          # a BF16 NaN pattern the reader never writes


def run_gather(pool_d, layout, topk, page_table=None, page_size=64, token_seq=None):
    T, K = topk.shape
    pool_rows = pool_d.shape[0]
    out = binding.gather_workspace_for(T, K, pool_rows, layout)
    assert out.numel() * 2 == binding.dsa_gather_dequant_workspace_bytes(T, K, pool_rows, layout)
    out.view(torch.int16).fill_(SENTINEL)
    idx = torch.full((T, K), 7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.dsa_gather_dequant(pool_d, layout, dev(topk.astype(np.int32)), out, idx,
                               page_table=None if page_table is None else dev(page_table.astype(np.int32)),
                               page_size=page_size,
                               token_seq=None if token_seq is None else dev(token_seq.astype(np.int32)),
                               err_flag=err)
    torch.cuda.synchronize()
    return out.view(torch.int16).cpu().numpy().view(np.uint16), idx.cpu().numpy(), int(err.item())


def check(pool, layout, topk, **kw):
    """Returns True when the full-pool branch ran."""
    out, idx, err = run_gather(pool_dev(pool), layout, topk, **kw)
    ro, ri, rerr = oracle.gather_dequant(pool, layout, topk, **kw)
    assert err == rerr
    assert out.shape == ro.shape
    np.testing.assert_array_equal(idx, ri)
    full = topk.size >= pool.shape[0]
    if full:
        np.testing.assert_array_equal(out, ro)                  # every pool row
    else:
        valid = ri.reshape(-1) >= 0
        np.testing.assert_array_equal(out[valid], ro[valid])
        assert (out[~valid] == SENTINEL).all()                 # masked entries' rows untouched
    return full


def _pool(layout, pool_rows, seed):
    rng = np.random.default_rng(seed)
    width = 576 if layout == "rope656" else 512
    w = dict(layout=layout, pool_rows=pool_rows, kv_slots=np.arange(pool_rows),
             kv_src=W.f32_to_bf16_bits((rng.standard_normal((pool_rows, width))
                                        * rng.uniform(0.1, 8, (pool_rows, 1))).astype(np.float32)))
    return oracle.fill_pool(w), rng


@pytest.mark.parametrize("layout", ["raw512", "scaled528", "rope656"])
@pytest.mark.parametrize("T,K", [(7, 200), (11, 200)])
def test_gather_small_paged(layout, T, K):
    """2048-row pool: 7 x 200 entries take the selected branch, 11 x 200 the
    full-pool branch; two sequences, 20 % -1, an all-masked token; K is not a
    multiple of 32 (a ragged chunk)."""
    pool_rows = 2048
    pool, rng = _pool(layout, pool_rows, {"raw512": 11, "scaled528": 12, "rope656": 14}[layout] + T)
    page_table = rng.permutation(pool_rows // 64).astype(np.int32).reshape(2, -1)
    token_seq = (np.arange(T) % 2).astype(np.int32)
    topk = rng.integers(0, page_table.shape[1] * 64, (T, K)).astype(np.int32)
    topk[rng.random((T, K)) < 0.2] = -1
    topk[3] = -1                                      # an all-masked token
    full = check(pool, layout, topk, page_table=page_table, page_size=64, token_seq=token_seq)
    assert full == (T * K >= pool_rows)


@pytest.mark.parametrize("page_size", [1, 16, 256])
@pytest.mark.parametrize("T,K", [(4, 128), (20, 128)])
def test_gather_page_sizes(page_size, T, K):
    """Index translation at page sizes other than 64 over two sequences, in the
    selected branch (4 x 128 entries over 2048 rows) and the full-pool branch
    (20 x 128)."""
    pool_rows = 2048
    pool, rng = _pool("scaled528", pool_rows, 16 + page_size)
    pages = pool_rows // page_size
    page_table = rng.permutation(pages).astype(np.int32).reshape(2, -1)
    token_seq = (np.arange(T) % 2).astype(np.int32)
    topk = rng.integers(0, page_table.shape[1] * page_size, (T, K)).astype(np.int32)
    topk[rng.random((T, K)) < 0.15] = -1
    full = check(pool, "scaled528", topk, page_table=page_table, page_size=page_size, token_seq=token_seq)
    assert full == (T * K >= pool_rows)


@pytest.mark.parametrize("delta", [-1, 0, 1])
def test_gather_branch_boundary(delta):
    """T*K = pool_rows - 1, pool_rows, pool_rows + 1 (physical indices): the
    full-pool branch starts at equality."""
    pool_rows = 1024
    pool, rng = _pool("scaled528", pool_rows, 15)
    T = 8
    K = (pool_rows + delta) // T if (pool_rows + delta) % T == 0 else None
    if K is None:
        T, K = 1, pool_rows + delta
    topk = rng.integers(0, pool_rows, (T, K)).astype(np.int32)
    topk[rng.random((T, K)) < 0.1] = -1
    assert check(pool, "scaled528", topk) == (T * K >= pool_rows)


def test_gather_errors_and_physical_indices():
    pool_rows = 1024
    pool, rng = _pool("raw512", pool_rows, 13)
    topk = rng.integers(0, pool_rows, (3, 64)).astype(np.int32)
    topk[0, 5] = pool_rows + 7                        # outside the pool: masked, index bit
    check(pool, "raw512", topk)
    out, idx, err = run_gather(pool_dev(pool), "raw512", topk)
    assert err == binding.DSA_DEV_ERR_INDEX_RANGE and idx[0, 5] == -1


@pytest.mark.parametrize("name", ["decode_raw512", "decode_scaled528", "tiny_decode_raw512"])
def test_gather_full_decode_batches(name):
    """The decode workloads' own lists: 64 x 2048 entries over 131072 rows and
    128 x 2048 over 131072 (full-pool branch), 4 x 128 over 4096 (selected)."""
    w = W.make(name)
    pool = oracle.fill_pool(w)
    full = check(pool, w["layout"], w["topk"], page_table=w["page_table"], page_size=w["page_size"])
    assert full == (name != "tiny_decode_raw512")
