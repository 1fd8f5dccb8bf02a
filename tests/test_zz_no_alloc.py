"""dsa_sparse_attn_decode_noalloc against dsa_sparse_attn_decode.

The no-allocation entry point serves callers that cannot obtain a device
workspace (an engine that gave all of HBM to its KV-cache pool, a plug-in
inside a host that owns the allocator, code that must not call cudaMalloc):
it runs the same decode with the library's own static device array as the
split-K workspace.  The kernels, the plan and the inputs are the same, so
its outputs must be bitwise identical to the workspace entry point's, on
two calls in a row with different inputs (neither a stale array nor the
first call's one-time set-up may change a result), for both row layouts;
one small split-K case is also checked against the oracle.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_attn_close, bf16_dev, dev, pool_dev
from sparse_mla_attention_page_gb300 import binding
from sparse_mla_attention_page_gb300 import build as build_mod
from sparse_mla_attention_page_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _same_bits(o_a, lse_a, o_b, lse_b):
    assert torch.equal(o_a.view(torch.int16), o_b.view(torch.int16)), "O differs bitwise"
    assert torch.equal(lse_a.view(torch.int32), lse_b.view(torch.int32)), "LSE differs bitwise"


def _both(w, pool, topk_d, q, pt):
    T, H, K = w["T"], w["H"], w["K"]
    o_ref = torch.empty(T, H, 512, dtype=torch.bfloat16, device="cuda")
    lse_ref = torch.empty(T, H, dtype=torch.float32, device="cuda")
    binding.dsa_sparse_attn_decode(q, pool, w["layout"], topk_d, w["sm_scale"], o_ref, lse_ref,
                                   binding.workspace_for(T, H, K), page_table=pt, page_size=64)
    o = torch.full((T, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.dsa_sparse_attn_decode_noalloc(q, pool, w["layout"], topk_d, w["sm_scale"], o, lse,
                                           page_table=pt, page_size=64, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return o, lse, o_ref, lse_ref


@pytest.mark.parametrize("layout", ["raw512", "scaled528"])
def test_noalloc_matches_workspace_entry_point_twice(layout):
    build_mod.build()
    T, K = 64, 2048
    H = 16 if layout == "raw512" else 32
    need = binding.dsa_sparse_attn_workspace_bytes(T, H, K)
    assert 0 < need <= (32 << 20), "the case must use split-K scratch and fit the static array"
    if layout == "raw512":
        w = W.decode_raw512(seed=77, T=T, H=H, K=K, pool_rows=16384)
    else:
        w = W.decode_scaled528(seed=79, T=T, H=H, K=K, pool_rows=16384)
    pool = pool_dev(oracle.fill_pool(w))
    pt = dev(w["page_table"])
    rng = np.random.default_rng(78)
    for call in range(2):
        topk = w["topk"].copy()
        if call == 1:                       # different inputs on the second call
            topk = np.stack([rng.permutation(r) for r in topk]).astype(np.int32)
            topk[5:9] = -1
        q = bf16_dev(W.f32_to_bf16_bits(rng.standard_normal((T, H, 512)).astype(np.float32)))
        o, lse, o_ref, lse_ref = _both(w, pool, dev(topk), q, pt)
        _same_bits(o, lse, o_ref, lse_ref)


def test_noalloc_split_units_against_oracle():
    """Two tokens with 4096 entries each: every unit is spread over dozens of
    CTAs, so the result passes through the static array's partials."""
    w = W.decode_raw512(seed=80, T=2, H=16, K=4096, pool_rows=16384, special_tokens=False)
    assert binding.dsa_sparse_attn_workspace_bytes(2, 16, 4096) > 0
    pool_np = oracle.fill_pool(w)
    pool = pool_dev(pool_np)
    o, lse, o_ref, lse_ref = _both(w, pool, dev(w["topk"]), bf16_dev(w["q_bf16"]), dev(w["page_table"]))
    _same_bits(o, lse, o_ref, lse_ref)
    Or, Lr, _ = oracle.sparse_attn(pool_np, "raw512", w["topk"], w["sm_scale"], q_bf16=w["q_bf16"],
                                   page_table=w["page_table"], page_size=64)
    assert_attn_close(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
                      Or, Lr, "noalloc split units")


def test_noalloc_array_covers_every_shape():
    """The split-K workspace holds two partial slots per SM, whatever T and K
    are, so on this GPU the static array serves every supported shape; a
    shape that did not fit would be refused with DSA_ERR_WORKSPACE before
    any launch."""
    build_mod.build()
    limit = 32 << 20
    for H in (8, 16, 32, 64, 128):
        for T in (1, 64, 4096, 1 << 20):
            for K in (128, 2048, 65536):
                assert binding.dsa_sparse_attn_workspace_bytes(T, H, K) <= limit, (T, H, K)
