"""CPU oracle for the sparse FP8 MLA attention path (test infrastructure).

Only the tests, the smoke check and the benchmark's CPU-baseline leg (and its
reference arm) may import this package.  The CUDA library never does: the two
share no code.  The arithmetic lives in ``dsa_oracle.c`` (plain C, float64);
this module builds it with gcc and marshals numpy arrays to it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libdsa_oracle.so")
_lock = threading.Lock()
_lib = None

ERR_INDEX_RANGE = 1
ERR_PAGE_RANGE = 2


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call([
            "gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", _SRC, "-o", tmp, "-lm", "-lpthread"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load(path: str):
    """Open a compiled oracle library and declare its C signatures."""
    L = ctypes.CDLL(path)
    c = ctypes
    L.oracle_e4m3_decode.restype = c.c_double
    L.oracle_e4m3_decode.argtypes = [c.c_uint8]
    L.oracle_e4m3_encode.restype = c.c_uint8
    L.oracle_e4m3_encode.argtypes = [c.c_float]
    L.oracle_e4m3_encode_bruteforce.restype = c.c_uint8
    L.oracle_e4m3_encode_bruteforce.argtypes = [c.c_float]
    for fn in (L.oracle_kv_write_raw, L.oracle_kv_write_scaled, L.oracle_kv_write_rope656):
        fn.restype = c.c_int64
        fn.argtypes = [c.c_void_p, c.c_int64, c.c_void_p, c.c_void_p, c.c_int64]
    L.oracle_e4m3_encode_array.restype = None
    L.oracle_e4m3_encode_array.argtypes = [c.c_void_p, c.c_int64, c.c_void_p, c.c_int]
    L.oracle_e4m3_decode_array.restype = None
    L.oracle_e4m3_decode_array.argtypes = [c.c_void_p, c.c_int64, c.c_void_p]
    L.oracle_quantize_q8.restype = None
    L.oracle_quantize_q8.argtypes = [c.c_void_p, c.c_int64, c.c_int, c.c_void_p, c.c_void_p]
    L.oracle_sparse_attn.restype = c.c_int
    L.oracle_gather_rows.restype = c.c_int64
    L.oracle_gather_rows.argtypes = [c.c_int64, c.c_int64]
    L.oracle_gather_dequant.restype = c.c_int
    L.oracle_gather_dequant.argtypes = [c.c_void_p, c.c_int64, c.c_int, c.c_void_p, c.c_int, c.c_int, c.c_int,
                                        c.c_void_p, c.c_void_p, c.c_int, c.c_int, c.c_void_p, c.c_void_p]
    L.oracle_sparse_attn.argtypes = [
        c.c_int, c.c_void_p, c.c_void_p, c.c_int, c.c_int,
        c.c_void_p, c.c_int64, c.c_int,
        c.c_void_p, c.c_int, c.c_int, c.c_int,
        c.c_void_p, c.c_void_p, c.c_int, c.c_double,
        c.c_void_p, c.c_int, c.c_void_p, c.c_void_p, c.c_int]
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = load(_LIB_PATH)
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def e4m3_decode(b: int) -> float:
    return lib().oracle_e4m3_decode(int(b) & 0xFF)


def e4m3_encode(x: float) -> int:
    return lib().oracle_e4m3_encode(float(x))


def e4m3_encode_bruteforce(x: float) -> int:
    return lib().oracle_e4m3_encode_bruteforce(float(x))


def decode_table() -> np.ndarray:
    """float64 value of every byte 0..255 (NaN for 0x7F, 0xFF)."""
    return e4m3_decode_array(np.arange(256, dtype=np.uint8))


def e4m3_decode_array(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint8)
    out = np.empty(b.shape, dtype=np.float64)
    lib().oracle_e4m3_decode_array(_ptr(b), b.size, _ptr(out))
    return out


def e4m3_encode_array(x: np.ndarray, bruteforce: bool = False) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode_array(_ptr(x), x.size, _ptr(out), int(bruteforce))
    return out


LAYOUT_CODES = {"raw512": 0, "scaled528": 1, "rope656": 2}


def row_bytes(layout: str) -> int:
    return {"raw512": 512, "scaled528": 528, "rope656": 656}[layout]


def key_width(layout: str) -> int:
    """Query/key width: the 512 latent dims, plus 64 RoPE dims for 656-byte rows."""
    return 576 if layout == "rope656" else 512


def new_pool(pool_rows: int, layout: str) -> np.ndarray:
    return np.zeros((pool_rows, row_bytes(layout)), dtype=np.uint8)


def kv_write(layout: str, x_bf16: np.ndarray, slots: np.ndarray, pool: np.ndarray) -> int:
    """Write BF16 rows (uint16 bits [n, 512], or [n, 576] for 656-byte rows) into
    pool rows ``slots`` (in place)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    s = np.ascontiguousarray(slots, dtype=np.int64)
    assert pool.flags.c_contiguous and pool.dtype == np.uint8
    assert pool.shape[1] == row_bytes(layout) and x.shape[1] == key_width(layout) and x.shape[0] == s.shape[0]
    fn = {"raw512": lib().oracle_kv_write_raw, "scaled528": lib().oracle_kv_write_scaled,
          "rope656": lib().oracle_kv_write_rope656}[layout]
    n = fn(_ptr(x), x.shape[0], _ptr(s), _ptr(pool), pool.shape[0])
    if n < 0:
        raise ValueError("slot beyond the pool")
    return int(n)


def quantize_q8(q_bf16: np.ndarray):
    """Per-(token, head) E4M3 query with FP32 scale amax/448: returns (q8, scale)."""
    q = np.ascontiguousarray(q_bf16, dtype=np.uint16)
    d = q.shape[-1]
    n = q.size // d
    q8 = np.empty(q.shape, dtype=np.uint8)
    sc = np.empty(q.shape[:-1], dtype=np.float32)
    lib().oracle_quantize_q8(_ptr(q), n, d, _ptr(q8), _ptr(sc))
    return q8, sc


def sparse_attn(pool: np.ndarray, layout: str, topk: np.ndarray, sm_scale: float, *,
                q_bf16: np.ndarray | None = None, q8: np.ndarray | None = None,
                q_scale: np.ndarray | None = None, page_table: np.ndarray | None = None,
                page_size: int = 64, token_seq: np.ndarray | None = None,
                tokens=None, n_threads: int | None = None):
    """Reference O (float64 [n, H, 512]) and LSE (float64 [n, H]) and error bits.

    ``sm_scale`` is taken as the FP32 value the library receives.
    """
    topk = np.ascontiguousarray(topk, dtype=np.int32)
    T, K = topk.shape
    if q_bf16 is not None:
        q = np.ascontiguousarray(q_bf16, dtype=np.uint16)
        kind, qs = 0, None
    else:
        q = np.ascontiguousarray(q8, dtype=np.uint8)
        qs = np.ascontiguousarray(q_scale, dtype=np.float32)
        kind = 1
    assert q.shape[0] == T and q.shape[2] == (key_width(layout) if kind == 0 else 512)
    assert kind == 0 or layout != "rope656", "FP8 queries are defined over the 512 latent dims only"
    H = q.shape[1]
    pool = np.ascontiguousarray(pool, dtype=np.uint8)
    assert pool.shape[1] == row_bytes(layout)
    if page_table is not None:
        pt = np.ascontiguousarray(page_table, dtype=np.int32)
        B, max_pages = pt.shape
    else:
        pt, B, max_pages = None, 1, 0
    ts = None if token_seq is None else np.ascontiguousarray(token_seq, dtype=np.int32)
    if tokens is None:
        tok = None
        n = T
    else:
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        n = tok.shape[0]
    O = np.zeros((n, H, 512), dtype=np.float64)
    LSE = np.zeros((n, H), dtype=np.float64)
    if n_threads is None:
        n_threads = max(1, len(os.sched_getaffinity(0)))
    err = lib().oracle_sparse_attn(
        kind, _ptr(q), _ptr(qs), T, H,
        _ptr(pool), pool.shape[0], LAYOUT_CODES[layout],
        _ptr(pt), B, max_pages, page_size,
        _ptr(ts), _ptr(topk), K, float(np.float32(sm_scale)),
        _ptr(tok), n, _ptr(O), _ptr(LSE), int(n_threads))
    return O, LSE, int(err)


def gather_rows(pool_rows: int, n_selected: int) -> int:
    """Rows of the reader's BF16 workspace: min(pool_rows, selected entries)."""
    return int(lib().oracle_gather_rows(int(pool_rows), int(n_selected)))


def gather_dequant(pool: np.ndarray, layout: str, topk: np.ndarray, *,
                   page_table: np.ndarray | None = None, page_size: int = 64,
                   token_seq: np.ndarray | None = None):
    """The reader's BF16 workspace (uint16 [gather_rows(pool_rows, T*K), W],
    W = 512, or 576 for 656-byte rows; rows it leaves alone stay 0 here),
    remapped indices (int32 [T, K]) and error bits.  With T*K < pool_rows
    the workspace holds the selected rows and idx_out the entry numbers;
    otherwise it holds the whole pool and idx_out the physical rows."""
    topk = np.ascontiguousarray(topk, dtype=np.int32)
    T, K = topk.shape
    pool = np.ascontiguousarray(pool, dtype=np.uint8)
    assert pool.shape[1] == row_bytes(layout)
    if page_table is not None:
        pt = np.ascontiguousarray(page_table, dtype=np.int32)
        B, max_pages = pt.shape
    else:
        pt, B, max_pages = None, 1, 0
    ts = None if token_seq is None else np.ascontiguousarray(token_seq, dtype=np.int32)
    out = np.zeros((gather_rows(pool.shape[0], T * K), key_width(layout)), dtype=np.uint16)
    idx = np.zeros((T, K), dtype=np.int32)
    err = lib().oracle_gather_dequant(_ptr(pool), pool.shape[0], LAYOUT_CODES[layout],
                                      _ptr(pt), B, max_pages, page_size, _ptr(ts), _ptr(topk), T, K,
                                      _ptr(out), _ptr(idx))
    return out, idx, int(err)


def fill_pool(workload: dict) -> np.ndarray:
    """Pool bytes for a workload: its BF16 source rows through the oracle writer."""
    pool = new_pool(workload["pool_rows"], workload["layout"])
    kv_write(workload["layout"], workload["kv_src"], workload["kv_slots"], pool)
    return pool
