"""Helpers for the GPU parity tests: move numpy inputs to the device, call the
library through its C-ABI binding, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

from sparse_mla_attention_page_gb300 import binding

# Attention tolerance: |O - O_ref| <= 1e-2 + 1e-2 |O_ref| per element (O in BF16),
# |LSE - LSE_ref| <= 1e-3 where finite, and -inf exactly where the oracle has -inf.
O_ATOL = 1e-2
O_RTOL = 1e-2
LSE_ATOL = 1e-3


def dev(a: np.ndarray, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    return dev(bits.astype(np.uint16).view(np.int16), torch.bfloat16)


def pool_dev(pool: np.ndarray) -> torch.Tensor:
    return dev(pool)


def run_decode(w: dict, pool_d: torch.Tensor, topk=None, q=None, err=None, page_table=None,
               stream=None):
    """Decode through the C ABI; returns O (float64 numpy), LSE (float64), err bits."""
    T, H = w["T"], w["H"]
    topk = w["topk"] if topk is None else topk
    q_d = bf16_dev(w["q_bf16"] if q is None else q)
    pt = w["page_table"] if page_table is None else page_table
    pt_d = None if pt is None else dev(pt.astype(np.int32))
    ts_d = None if w.get("token_seq") is None else dev(w["token_seq"].astype(np.int32))
    topk_d = dev(topk.astype(np.int32))
    o = torch.empty(T, H, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(T, H, dtype=torch.float32, device="cuda")
    ws = binding.workspace_for(T, H, topk.shape[1])
    err_d = torch.zeros(1, dtype=torch.int32, device="cuda") if err is None else err
    binding.dsa_sparse_attn_decode(q_d, pool_d, w["layout"], topk_d, w["sm_scale"], o, lse, ws,
                                   page_table=pt_d, page_size=w["page_size"], token_seq=ts_d,
                                   err_flag=err_d, stream=stream)
    torch.cuda.synchronize()
    return (o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
            int(err_d.item()))


def run_prefill(w: dict, pool_d: torch.Tensor, q8: np.ndarray, q_scale: np.ndarray):
    T, H = w["T"], w["H"]
    pt_d = None if w["page_table"] is None else dev(w["page_table"].astype(np.int32))
    o = torch.empty(T, H, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(T, H, dtype=torch.float32, device="cuda")
    ws = binding.workspace_for(T, H, w["topk"].shape[1])
    err_d = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.dsa_sparse_attn_prefill_q8(dev(q8), dev(q_scale.astype(np.float32)), pool_d, w["layout"],
                                       dev(w["topk"].astype(np.int32)), w["sm_scale"], o, lse, ws,
                                       page_table=pt_d, page_size=w["page_size"], err_flag=err_d)
    torch.cuda.synchronize()
    return (o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
            int(err_d.item()))


def attn_error_stats(O, L, Or, Lr) -> dict:
    """max |O - O_ref|, the same relative to max |O_ref| (how large the error is
    next to the output itself), and max |LSE - LSE_ref| where finite."""
    d = np.abs(O - Or)
    scale = float(np.abs(Or).max()) if Or.size else 0.0
    neg = np.isneginf(Lr)
    dl = np.abs(L[~neg] - Lr[~neg])
    return {"max_abs": float(d.max()) if d.size else 0.0,
            "rel_to_max": float(d.max() / scale) if d.size and scale > 0 else 0.0,
            "max_ref": scale, "lse_max_abs": float(dl.max()) if dl.size else 0.0}


def assert_attn_close(O, L, Or, Lr, what=""):
    """Elementwise tolerance check with a readable report of the worst offender
    and of the error relative to max |O_ref|; returns the error statistics."""
    assert O.shape == Or.shape and L.shape == Lr.shape
    st = attn_error_stats(O, L, Or, Lr) if np.isfinite(O).all() else {}
    excess = np.abs(O - Or) - (O_ATOL + O_RTOL * np.abs(Or))
    if (excess > 0).any() or not np.isfinite(O).all():
        i = np.unravel_index(np.nanargmax(np.where(np.isfinite(excess), excess, np.inf)), excess.shape)
        raise AssertionError(f"{what} O mismatch at {i}: got {O[i]} ref {Or[i]} "
                             f"({int((excess > 0).sum())} elements out of tolerance; {st})")
    neg = np.isneginf(Lr)
    assert np.array_equal(np.isneginf(L), neg), f"{what} LSE -inf pattern differs"
    d = np.abs(L[~neg] - Lr[~neg])
    if d.size and d.max() > LSE_ATOL:
        i = np.argmax(d)
        raise AssertionError(f"{what} LSE mismatch: max |diff| {d.max()} (got {L[~neg][i]} ref {Lr[~neg][i]}; {st})")
    return st
