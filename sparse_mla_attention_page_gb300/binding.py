"""Thin ctypes binding of the C ABI in include/dsa.h (argument marshalling only).

Every function here has the name of the C entry point it calls, takes torch
tensors that already live on the GPU, checks that they have the dtype and
shape the C function documents, passes their pointers and sizes, and turns a
non-zero status into ``DsaError``.  All computation happens in the CUDA
library; there is no fallback: if ``libdsa_gb300.so`` has not been built the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

DSA_KV_RAW512 = 0
DSA_KV_SCALED528 = 1
DSA_KV_ROPE656 = 2
LAYOUTS = {"raw512": DSA_KV_RAW512, "scaled528": DSA_KV_SCALED528, "rope656": DSA_KV_ROPE656}

DSA_DEV_ERR_INDEX_RANGE = 1
DSA_DEV_ERR_PAGE_RANGE = 2
DSA_DEV_ERR_TIMEOUT = 4
DSA_DEV_ERR_SLOT_RANGE = 8

_lock = threading.Lock()
_lib = None

# Every symbol include/dsa.h declares.
EXPORTS = (
    "dsa_status_string", "dsa_kv_row_bytes", "dsa_kv_write_raw", "dsa_kv_write_scaled", "dsa_kv_write_rope656",
    "dsa_quantize_q8", "dsa_sparse_attn_workspace_bytes", "dsa_sparse_attn_decode",
    "dsa_sparse_attn_prefill_q8", "dsa_gather_dequant_workspace_bytes", "dsa_gather_dequant",
    "dsa_sparse_attn_decode_noalloc", "dsa_set_wait_limit_ns",
)


class DsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def library_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: build the CUDA library first "
                                   "(sparse_mla_attention_page_gb300.build.build())")
            L = ctypes.CDLL(path)
            c = ctypes
            vp, i64, i32 = c.c_void_p, c.c_int64, c.c_int
            L.dsa_status_string.restype = c.c_char_p
            L.dsa_status_string.argtypes = [i32]
            L.dsa_set_wait_limit_ns.restype = c.c_uint64
            L.dsa_set_wait_limit_ns.argtypes = [c.c_uint64]
            L.dsa_kv_row_bytes.restype = c.c_size_t
            L.dsa_kv_row_bytes.argtypes = [i32]
            for f in (L.dsa_kv_write_raw, L.dsa_kv_write_scaled, L.dsa_kv_write_rope656):
                f.restype = i32
                f.argtypes = [vp, i64, vp, vp, i64, vp, vp]
            L.dsa_quantize_q8.restype = i32
            L.dsa_quantize_q8.argtypes = [vp, i64, vp, vp, vp]
            L.dsa_sparse_attn_workspace_bytes.restype = c.c_size_t
            L.dsa_sparse_attn_workspace_bytes.argtypes = [i32, i32, i32]
            L.dsa_sparse_attn_decode.restype = i32
            L.dsa_sparse_attn_decode.argtypes = [
                vp, i32, i32, i32, vp, i64, i32, i32, vp, i32, i32, i32, vp, vp, i32,
                c.c_float, vp, vp, vp, c.c_size_t, vp, vp]
            L.dsa_sparse_attn_prefill_q8.restype = i32
            L.dsa_sparse_attn_prefill_q8.argtypes = [
                vp, vp, i32, i32, i32, vp, i64, i32, i32, vp, i32, i32, i32, vp, vp, i32,
                c.c_float, vp, vp, vp, c.c_size_t, vp, vp]
            L.dsa_gather_dequant.restype = i32
            L.dsa_gather_dequant.argtypes = [vp, i64, i32, vp, i32, i32, i32, vp, vp, i32, i32, vp, c.c_size_t,
                                             vp, vp, vp]
            L.dsa_gather_dequant_workspace_bytes.restype = c.c_size_t
            L.dsa_gather_dequant_workspace_bytes.argtypes = [i32, i32, i64, i32]
            L.dsa_sparse_attn_decode_noalloc.restype = i32
            L.dsa_sparse_attn_decode_noalloc.argtypes = [
                vp, i32, i32, i32, vp, i64, i32, i32, vp, i32, i32, i32, vp, vp, i32,
                c.c_float, vp, vp, vp, vp]
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().dsa_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != 0:
        raise DsaError(status, where)


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, last: int | None = None):
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous CUDA {dtype} tensor")
    if last is not None and t.shape[-1] != last:
        raise ValueError(f"{name} must have last dimension {last}, got {tuple(t.shape)}")


def dsa_set_wait_limit_ns(ns: int) -> int:
    """Limit of the attention kernel's bounded waits for later calls; returns the old one."""
    return int(lib().dsa_set_wait_limit_ns(int(ns)))


def dsa_kv_row_bytes(layout) -> int:
    return int(lib().dsa_kv_row_bytes(LAYOUTS.get(layout, layout)))


def _write(fn_name, x_bf16, slots, pool, err_flag, stream, width=512):
    _need(x_bf16, "x_bf16", torch.bfloat16, width)
    _need(slots, "slots", torch.int64)
    _need(pool, "pool", torch.uint8)
    if err_flag is not None:
        _need(err_flag, "err_flag", torch.int32)
    n = x_bf16.numel() // width
    if slots.numel() != n:
        raise ValueError("slots must have one entry per row")
    rows = pool.shape[0]
    st = getattr(lib(), fn_name)(_ptr(x_bf16), n, _ptr(slots), _ptr(pool), rows, _ptr(err_flag), _stream(stream))
    _check(st, fn_name)


def dsa_kv_write_raw(x_bf16, slots, pool, err_flag=None, stream=None) -> None:
    """pool [rows, 512] uint8 <- e4m3(x) at rows ``slots`` (see include/dsa.h)."""
    if pool.dim() != 2 or pool.shape[1] != 512:
        raise ValueError("raw pool must be [rows, 512] uint8")
    _write("dsa_kv_write_raw", x_bf16, slots, pool, err_flag, stream)


def dsa_kv_write_scaled(x_bf16, slots, pool, err_flag=None, stream=None) -> None:
    """pool [rows, 528] uint8 <- group-scaled e4m3(x) at rows ``slots``."""
    if pool.dim() != 2 or pool.shape[1] != 528:
        raise ValueError("scaled pool must be [rows, 528] uint8")
    _write("dsa_kv_write_scaled", x_bf16, slots, pool, err_flag, stream)


def dsa_kv_write_rope656(x_bf16, slots, pool, err_flag=None, stream=None) -> None:
    """pool [rows, 656] uint8 <- group-scaled e4m3(x[:, :512]) and the BF16 RoPE
    dims x[:, 512:576] at rows ``slots``."""
    if pool.dim() != 2 or pool.shape[1] != 656:
        raise ValueError("RoPE pool must be [rows, 656] uint8")
    _write("dsa_kv_write_rope656", x_bf16, slots, pool, err_flag, stream, width=576)


def dsa_quantize_q8(q_bf16, q8, q_scale, stream=None) -> None:
    """q8 [..., 512] uint8 and q_scale [...] float32 from q_bf16 [..., 512]."""
    _need(q_bf16, "q_bf16", torch.bfloat16, 512)
    _need(q8, "q8", torch.uint8, 512)
    _need(q_scale, "q_scale", torch.float32)
    n = q_bf16.numel() // 512
    if q8.numel() != n * 512 or q_scale.numel() != n:
        raise ValueError("q8 / q_scale sizes do not match q_bf16")
    _check(lib().dsa_quantize_q8(_ptr(q_bf16), n, _ptr(q8), _ptr(q_scale), _stream(stream)),
           "dsa_quantize_q8")


def dsa_sparse_attn_workspace_bytes(T: int, H: int, K: int) -> int:
    return int(lib().dsa_sparse_attn_workspace_bytes(int(T), int(H), int(K)))


def workspace_for(T: int, H: int, K: int, device=None) -> torch.Tensor | None:
    """A device workspace of the size the attention entry points need (or None)."""
    n = dsa_sparse_attn_workspace_bytes(T, H, K)
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def _attn_common(q, pool, layout, topk, o, lse, page_table, token_seq, workspace, err_flag):
    T, H = q.shape[0], q.shape[1]
    _need(pool, "pool", torch.uint8)
    _need(topk, "topk", torch.int32)
    _need(o, "o", torch.bfloat16, 512)
    _need(lse, "lse", torch.float32)
    if topk.dim() != 2 or topk.shape[0] != T:
        raise ValueError("topk must be [T, K] int32")
    if tuple(o.shape) != (T, H, 512) or tuple(lse.shape) != (T, H):
        raise ValueError("o must be [T, H, 512] bf16 and lse [T, H] float32")
    lay = LAYOUTS.get(layout, layout)
    if page_table is not None:
        _need(page_table, "page_table", torch.int32)
        B, max_pages = page_table.shape
    else:
        B, max_pages = 1, 1
    if token_seq is not None:
        _need(token_seq, "token_seq", torch.int32)
    if err_flag is not None:
        _need(err_flag, "err_flag", torch.int32)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return T, H, lay, B, max_pages, ws_bytes


def dsa_gather_dequant_workspace_bytes(T: int, K: int, pool_rows: int, layout) -> int:
    return int(lib().dsa_gather_dequant_workspace_bytes(T, K, pool_rows, LAYOUTS.get(layout, layout)))


def gather_workspace_for(T: int, K: int, pool_rows: int, layout, device=None) -> torch.Tensor:
    """A BF16 workspace [min(pool_rows, T*K), 512 or 576] for dsa_gather_dequant."""
    lay = LAYOUTS.get(layout, layout)
    width = 576 if lay == DSA_KV_ROPE656 else 512
    rows = min(pool_rows, T * K)
    return torch.empty(rows, width, dtype=torch.bfloat16, device=device or "cuda")


def dsa_gather_dequant(pool, layout, topk, out, idx_out, page_table=None, page_size=64,
                       token_seq=None, err_flag=None, stream=None) -> None:
    """BF16 workspace out [min(pool_rows, T*K), 512 or 576] and remapped indices
    idx_out [T, K] for topk [T, K]."""
    lay = LAYOUTS.get(layout, layout)
    _need(pool, "pool", torch.uint8)
    _need(topk, "topk", torch.int32)
    _need(out, "out", torch.bfloat16, 576 if lay == DSA_KV_ROPE656 else 512)
    _need(idx_out, "idx_out", torch.int32)
    if topk.dim() != 2:
        raise ValueError("topk must be [T, K] int32")
    T, K = topk.shape
    if tuple(idx_out.shape) != (T, K):
        raise ValueError("idx_out must be [T, K] int32")
    if page_table is not None:
        _need(page_table, "page_table", torch.int32)
        B, max_pages = page_table.shape
    else:
        B, max_pages = 1, 1
    if token_seq is not None:
        _need(token_seq, "token_seq", torch.int32)
    if err_flag is not None:
        _need(err_flag, "err_flag", torch.int32)
    _check(lib().dsa_gather_dequant(_ptr(pool), pool.shape[0], lay, _ptr(page_table), B, max_pages,
                                    page_size, _ptr(token_seq), _ptr(topk), T, K, _ptr(out),
                                    out.numel() * out.element_size(), _ptr(idx_out), _ptr(err_flag),
                                    _stream(stream)),
           "dsa_gather_dequant")


def _kv_row_dim(pool, lay) -> int:
    """Key width held by one pool row (528- and 656-byte rows carry 16 bytes of
    scales; 656-byte rows add 64 BF16 RoPE dims)."""
    if lay == DSA_KV_ROPE656:
        return 512 + (pool.shape[1] - 528) // 2
    return pool.shape[1] - (16 if lay == DSA_KV_SCALED528 else 0)


def dsa_sparse_attn_decode(q_bf16, pool, layout, topk, sm_scale, o, lse, workspace=None,
                           page_table=None, page_size=64, token_seq=None, err_flag=None,
                           stream=None) -> None:
    """Sparse MLA decode with BF16 queries [T, H, 512] ([T, H, 576] over 656-byte
    rows; see include/dsa.h)."""
    _need(q_bf16, "q_bf16", torch.bfloat16, 576 if LAYOUTS.get(layout, layout) == DSA_KV_ROPE656 else 512)
    T, H, lay, B, max_pages, ws_bytes = _attn_common(q_bf16, pool, layout, topk, o, lse,
                                                     page_table, token_seq, workspace, err_flag)
    st = lib().dsa_sparse_attn_decode(
        _ptr(q_bf16), T, H, q_bf16.shape[-1], _ptr(pool), pool.shape[0], lay,
        _kv_row_dim(pool, lay),
        _ptr(page_table), B, max_pages, page_size, _ptr(token_seq), _ptr(topk), topk.shape[1],
        float(sm_scale), _ptr(o), _ptr(lse), _ptr(workspace), ws_bytes, _ptr(err_flag),
        _stream(stream))
    _check(st, "dsa_sparse_attn_decode")


def dsa_sparse_attn_prefill_q8(q8, q_scale, pool, layout, topk, sm_scale, o, lse, workspace=None,
                               page_table=None, page_size=64, token_seq=None, err_flag=None,
                               stream=None) -> None:
    """Sparse MLA prefill with E4M3 queries [T, H, 512] + FP32 scales [T, H]."""
    _need(q8, "q8", torch.uint8, 512)
    _need(q_scale, "q_scale", torch.float32)
    T, H, lay, B, max_pages, ws_bytes = _attn_common(q8, pool, layout, topk, o, lse,
                                                     page_table, token_seq, workspace, err_flag)
    st = lib().dsa_sparse_attn_prefill_q8(
        _ptr(q8), _ptr(q_scale), T, H, q8.shape[-1], _ptr(pool), pool.shape[0], lay,
        _kv_row_dim(pool, lay),
        _ptr(page_table), B, max_pages, page_size, _ptr(token_seq), _ptr(topk), topk.shape[1],
        float(sm_scale), _ptr(o), _ptr(lse), _ptr(workspace), ws_bytes, _ptr(err_flag),
        _stream(stream))
    _check(st, "dsa_sparse_attn_prefill_q8")


def dsa_sparse_attn_decode_noalloc(q_bf16, pool, layout, topk, sm_scale, o, lse, page_table=None,
                                   page_size=64, token_seq=None, err_flag=None, stream=None) -> None:
    """Decode using the library's own static workspace (no allocation by anyone);
    see include/dsa.h for its size limit and the sharing rules."""
    _need(q_bf16, "q_bf16", torch.bfloat16, 576 if LAYOUTS.get(layout, layout) == DSA_KV_ROPE656 else 512)
    T, H, lay, B, max_pages, _ = _attn_common(q_bf16, pool, layout, topk, o, lse,
                                              page_table, token_seq, None, err_flag)
    st = lib().dsa_sparse_attn_decode_noalloc(
        _ptr(q_bf16), T, H, q_bf16.shape[-1], _ptr(pool), pool.shape[0], lay, _kv_row_dim(pool, lay),
        _ptr(page_table), B, max_pages, page_size, _ptr(token_seq), _ptr(topk), topk.shape[1],
        float(sm_scale), _ptr(o), _ptr(lse), _ptr(err_flag), _stream(stream))
    _check(st, "dsa_sparse_attn_decode_noalloc")
