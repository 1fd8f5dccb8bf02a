"""The gather/dequantise reader on the GPU against the oracle: BF16 rows and
remapped indices bit-exact, error bits equal, masked slots left untouched."""
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
    out = torch.full((T * K, 512), SENTINEL, dtype=torch.int16, device="cuda").view(torch.bfloat16)
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
    out, idx, err = run_gather(pool_dev(pool), layout, topk, **kw)
    ro, ri, rerr = oracle.gather_dequant(pool, layout, topk, **kw)
    assert err == rerr
    np.testing.assert_array_equal(idx, ri)
    valid = ri.reshape(-1) >= 0
    np.testing.assert_array_equal(out[valid], ro[valid])
    assert (out[~valid] == SENTINEL).all()          # masked slots are not written


@pytest.mark.parametrize("layout", ["raw512", "scaled528"])
def test_gather_small_paged(layout):
    rng = np.random.default_rng(11 if layout == "raw512" else 12)
    pool_rows, T, K = 2048, 7, 200                    # K not a multiple of 32 or 128: ragged tail
    w = dict(layout=layout, pool_rows=pool_rows, kv_slots=np.arange(pool_rows),
             kv_src=W.f32_to_bf16_bits((rng.standard_normal((pool_rows, 512))
                                        * rng.uniform(0.1, 8, (pool_rows, 1))).astype(np.float32)))
    pool = oracle.fill_pool(w)
    page_table = rng.permutation(pool_rows // 64).astype(np.int32).reshape(2, -1)
    token_seq = (np.arange(T) % 2).astype(np.int32)
    topk = rng.integers(0, page_table.shape[1] * 64, (T, K)).astype(np.int32)
    topk[rng.random((T, K)) < 0.2] = -1
    topk[3] = -1                                      # an all-masked token
    check(pool, layout, topk, page_table=page_table, page_size=64, token_seq=token_seq)


def test_gather_errors_and_physical_indices():
    rng = np.random.default_rng(13)
    pool_rows = 1024
    w = dict(layout="raw512", pool_rows=pool_rows, kv_slots=np.arange(pool_rows),
             kv_src=W.f32_to_bf16_bits(rng.standard_normal((pool_rows, 512)).astype(np.float32)))
    pool = oracle.fill_pool(w)
    topk = rng.integers(0, pool_rows, (3, 64)).astype(np.int32)
    topk[0, 5] = pool_rows + 7                        # outside the pool: masked, index bit
    check(pool, "raw512", topk)
    out, idx, err = run_gather(pool_dev(pool), "raw512", topk)
    assert err == binding.DSA_DEV_ERR_INDEX_RANGE and idx[0, 5] == -1


@pytest.mark.parametrize("name", ["decode_raw512", "decode_scaled528"])
def test_gather_full_decode_batches(name):
    w = W.make(name)
    pool = oracle.fill_pool(w)
    check(pool, w["layout"], w["topk"], page_table=w["page_table"], page_size=w["page_size"])
