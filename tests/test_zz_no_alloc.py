"""dsa_sparse_attn_decode_noalloc against dsa_sparse_attn_decode.

The no-allocation entry point serves callers that cannot obtain a device
workspace (an engine that gave all of HBM to its KV-cache pool, a plug-in
inside a host that owns the allocator, code that must not call cudaMalloc):
it runs the same decode with the library's own static device array as the
split-K workspace.  Two calls in a row, on different inputs, must each match
the workspace entry point within the attention tolerance, so neither a stale
workspace nor the first call's one-time set-up changes a result.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

from gpu_util import LSE_ATOL, O_ATOL, O_RTOL, bf16_dev, dev
from sparse_mla_attention_page_gb300 import binding
from sparse_mla_attention_page_gb300 import build as build_mod
from sparse_mla_attention_page_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _close(o_a, lse_a, o_b, lse_b):
    oa, ob = o_a.float().cpu().numpy(), o_b.float().cpu().numpy()
    assert (np.abs(oa - ob) <= O_ATOL + O_RTOL * np.abs(ob)).all()
    la, lb = lse_a.cpu().numpy(), lse_b.cpu().numpy()
    neg = np.isneginf(lb)
    assert np.array_equal(np.isneginf(la), neg)
    assert (np.abs(la[~neg] - lb[~neg]) <= LSE_ATOL).all()


def test_noalloc_matches_workspace_entry_point_twice():
    build_mod.build()
    T, H, K = 64, 16, 2048
    need = binding.dsa_sparse_attn_workspace_bytes(T, H, K)
    assert 0 < need <= (32 << 20), "the case must use split-K scratch and fit the static array"
    w = W.decode_raw512(seed=77, T=T, H=H, K=K, pool_rows=16384)
    pool = torch.zeros(w["pool_rows"], 512, dtype=torch.uint8, device="cuda")
    binding.dsa_kv_write_raw(bf16_dev(w["kv_src"]), dev(w["kv_slots"]), pool)
    pt = dev(w["page_table"])
    rng = np.random.default_rng(78)
    for call in range(2):
        topk = w["topk"].copy()
        if call == 1:                       # different inputs on the second call
            topk = np.stack([rng.permutation(r) for r in topk]).astype(np.int32)
            topk[5:9] = -1
        q = bf16_dev(W.f32_to_bf16_bits(rng.standard_normal((T, H, 512)).astype(np.float32)))
        topk_d = dev(topk)
        o_ref = torch.empty(T, H, 512, dtype=torch.bfloat16, device="cuda")
        lse_ref = torch.empty(T, H, dtype=torch.float32, device="cuda")
        ws = binding.workspace_for(T, H, K)
        binding.dsa_sparse_attn_decode(q, pool, "raw512", topk_d, w["sm_scale"], o_ref, lse_ref, ws,
                                       page_table=pt, page_size=64)
        o = torch.full((T, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        binding.dsa_sparse_attn_decode_noalloc(q, pool, "raw512", topk_d, w["sm_scale"], o, lse,
                                               page_table=pt, page_size=64, err_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        _close(o, lse, o_ref, lse_ref)


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
