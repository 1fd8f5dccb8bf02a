"""Seeded synthetic inputs for the sparse FP8 MLA attention path.

This module only draws random numbers and lays them out: BF16 latent rows,
BF16 queries, page tables and top-k index lists.  It holds none of the
method's arithmetic (no FP8 cast, no scale, no attention): the KV pool bytes
are produced from `kv_src` by a writer (the oracle's in the tests, the CUDA
writer in the benchmark), and FP8 queries by a quantiser.  Both the CUDA path
and the CPU oracle are fed from here, so they see identical bytes.

Workloads (all 512-dim NoPE latent rows, page size 64, sm_scale = 1/sqrt(576)):

* ``tiny_decode_raw512``   4 tokens, 16 heads, 4096-row pool, top-k 128 with
  the last 16 entries -1.
* ``decode_raw512``        64 tokens, 16 heads, 131072-row pool of N(0, 0.5)
  rows, top-k 2048 distinct, valid count U[1536, 2048] (rest -1), one token
  all -1 and one token with a single valid entry.
* ``decode_scaled528``     128 tokens, 32 heads, 131072-row pool of
  N(0,1)*U(0.1,4) rows (one multiplier per row), top-k 2048 drawn with
  replacement (duplicates allowed), 5 % of entries -1 at random positions.
* ``decode_rope656``       64 tokens, 16 heads, 131072-row pool of 656-byte
  rows (group-scaled latent N(0,1)*U(0.1,4) per row plus a 64-dim BF16 RoPE
  part N(0,1)), 576-wide queries, top-k 2048 distinct, 5 % -1.
* ``prefill_q8_raw512``    4096 query tokens at positions 0..4095 after 8192
  context rows of one sequence, 32 heads, 16384-row pool; token at position
  p draws min(2048, 8193 + p) distinct causal indices from [0, 8192 + p],
  padded to a multiple of 128 with -1.
* ``prefill_q8_scaled528`` the same prefill batch over group-scaled 528-byte
  rows of N(0,1)*U(0.1,4) (one multiplier per row): FP8 queries over scaled
  rows, which the pages leave out.
* ``writer_sweep``         16384 new rows of N(0,1)*U(0.1,8) written to
  distinct random slots of a 262144-row pool; decode over the written slots
  (physical indices, no page table) at 8/16/32 heads, top-k 2048, with one
  one-hot and one all-masked token.

The sizes of every workload can be shrunk (``T``, ``H``, ``K``, ``pool_rows``
...) for tests that the CPU oracle must finish in seconds.
"""
from __future__ import annotations

import math

import numpy as np

D_LATENT = 512
D_ROPE = 64          # RoPE dims of a 656-byte row
PAGE_SIZE = 64
SM_SCALE = 1.0 / math.sqrt(576.0)

WORKLOADS = (
    "tiny_decode_raw512",
    "decode_raw512",
    "decode_scaled528",
    "decode_rope656",
    "prefill_q8_raw512",
    "prefill_q8_scaled528",
    "writer_sweep",
)


def rng_for(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 samples to the nearest BF16 (ties to even); returns uint16 bits.

    Only finite samples are produced here, so NaN handling is not needed.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = b + 0x7FFF + ((b >> 16) & 1)
    return (b >> 16).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _shuffled_page_table(rng, n_seq_pages: int, n_phys_pages: int) -> np.ndarray:
    """One sequence whose logical pages map to distinct random physical pages."""
    perm = rng.permutation(n_phys_pages)[:n_seq_pages].astype(np.int32)
    return perm.reshape(1, n_seq_pages)


def _distinct_indices(rng, n_tokens: int, k: int, upper: int) -> np.ndarray:
    """k distinct uniform indices in [0, upper) per token (upper >= k)."""
    out = np.empty((n_tokens, k), dtype=np.int32)
    for t in range(n_tokens):
        out[t] = rng.choice(upper, size=k, replace=False).astype(np.int32)
    return out


def tiny_decode_raw512(seed: int = 1, T: int = 4, H: int = 16, K: int = 128,
                       pool_rows: int = 4096, n_masked_tail: int = 16) -> dict:
    rng = rng_for(seed)
    q = f32_to_bf16_bits(rng.standard_normal((T, H, D_LATENT), dtype=np.float32))
    kv_src = f32_to_bf16_bits(rng.standard_normal((pool_rows, D_LATENT), dtype=np.float32))
    pages = pool_rows // PAGE_SIZE
    page_table = _shuffled_page_table(rng, pages, pages)
    topk = _distinct_indices(rng, T, K, pool_rows)
    if n_masked_tail:
        topk[:, K - n_masked_tail:] = -1
    return dict(name="tiny_decode_raw512", layout="raw512", T=T, H=H, K=K,
                q_bf16=q, kv_src=kv_src, kv_slots=np.arange(pool_rows, dtype=np.int64),
                pool_rows=pool_rows, page_table=page_table, page_size=PAGE_SIZE,
                token_seq=None, topk=topk, sm_scale=SM_SCALE)


def decode_raw512(seed: int = 2, T: int = 64, H: int = 16, K: int = 2048,
                  pool_rows: int = 131072, valid_lo: int | None = None,
                  special_tokens: bool = True) -> dict:
    rng = rng_for(seed)
    q = f32_to_bf16_bits(rng.standard_normal((T, H, D_LATENT), dtype=np.float32))
    kv_src = f32_to_bf16_bits(0.5 * rng.standard_normal((pool_rows, D_LATENT), dtype=np.float32))
    pages = pool_rows // PAGE_SIZE
    page_table = _shuffled_page_table(rng, pages, pages)
    topk = _distinct_indices(rng, T, K, pool_rows)
    lo = (3 * K) // 4 if valid_lo is None else valid_lo
    valid = rng.integers(lo, K + 1, size=T)
    for t in range(T):
        topk[t, valid[t]:] = -1
    if special_tokens and T >= 3:
        topk[1, :] = -1            # all-masked token
        topk[2, 1:] = -1           # a single valid entry
    return dict(name="decode_raw512", layout="raw512", T=T, H=H, K=K,
                q_bf16=q, kv_src=kv_src, kv_slots=np.arange(pool_rows, dtype=np.int64),
                pool_rows=pool_rows, page_table=page_table, page_size=PAGE_SIZE,
                token_seq=None, topk=topk, sm_scale=SM_SCALE)


def decode_scaled528(seed: int = 3, T: int = 128, H: int = 32, K: int = 2048,
                     pool_rows: int = 131072, masked_frac: float = 0.05) -> dict:
    rng = rng_for(seed)
    q = f32_to_bf16_bits(rng.standard_normal((T, H, D_LATENT), dtype=np.float32))
    mult = rng.uniform(0.1, 4.0, size=(pool_rows, 1)).astype(np.float32)
    kv_src = f32_to_bf16_bits(rng.standard_normal((pool_rows, D_LATENT), dtype=np.float32) * mult)
    pages = pool_rows // PAGE_SIZE
    page_table = _shuffled_page_table(rng, pages, pages)
    topk = rng.integers(0, pool_rows, size=(T, K)).astype(np.int32)   # duplicates allowed
    topk[rng.random((T, K)) < masked_frac] = -1
    return dict(name="decode_scaled528", layout="scaled528", T=T, H=H, K=K,
                q_bf16=q, kv_src=kv_src, kv_slots=np.arange(pool_rows, dtype=np.int64),
                pool_rows=pool_rows, page_table=page_table, page_size=PAGE_SIZE,
                token_seq=None, topk=topk, sm_scale=SM_SCALE)


def decode_rope656(seed: int = 7, T: int = 64, H: int = 16, K: int = 2048,
                   pool_rows: int = 131072, masked_frac: float = 0.05) -> dict:
    """Decode over 656-byte rows: the group-scaled latent (N(0,1) * U(0.1, 4) per
    row) plus a 64-dim BF16 RoPE part N(0,1); queries are 576 wide."""
    rng = rng_for(seed)
    q = f32_to_bf16_bits(rng.standard_normal((T, H, D_LATENT + D_ROPE), dtype=np.float32))
    mult = rng.uniform(0.1, 4.0, size=(pool_rows, 1)).astype(np.float32)
    nope = rng.standard_normal((pool_rows, D_LATENT), dtype=np.float32) * mult
    rope = rng.standard_normal((pool_rows, D_ROPE), dtype=np.float32)
    kv_src = f32_to_bf16_bits(np.concatenate([nope, rope], axis=1))
    pages = pool_rows // PAGE_SIZE
    page_table = _shuffled_page_table(rng, pages, pages)
    topk = _distinct_indices(rng, T, K, pool_rows)
    topk[rng.random((T, K)) < masked_frac] = -1
    return dict(name="decode_rope656", layout="rope656", T=T, H=H, K=K,
                q_bf16=q, kv_src=kv_src, kv_slots=np.arange(pool_rows, dtype=np.int64),
                pool_rows=pool_rows, page_table=page_table, page_size=PAGE_SIZE,
                token_seq=None, topk=topk, sm_scale=SM_SCALE)


def prefill_q8_raw512(seed: int = 4, T: int = 4096, H: int = 32, K: int = 2048,
                      context: int = 8192, pool_rows: int = 16384,
                  first_pos: int = 0) -> dict:
    """Query tokens sit at logical positions context+first_pos .. context+first_pos+T-1."""
    rng = rng_for(seed)
    q = f32_to_bf16_bits(rng.standard_normal((T, H, D_LATENT), dtype=np.float32))
    seq_len = context + first_pos + T
    seq_pages = -(-seq_len // PAGE_SIZE)
    phys_pages = pool_rows // PAGE_SIZE
    assert seq_pages <= phys_pages
    page_table = _shuffled_page_table(rng, seq_pages, phys_pages)
    kv_src = f32_to_bf16_bits(rng.standard_normal((pool_rows, D_LATENT), dtype=np.float32))
    topk = np.full((T, K), -1, dtype=np.int32)
    for t in range(T):
        upper = context + first_pos + t + 1          # causal: rows <= own position
        n = min(K, upper)
        topk[t, :n] = rng.choice(upper, size=n, replace=False).astype(np.int32)
    return dict(name="prefill_q8_raw512", layout="raw512", T=T, H=H, K=K,
                q_bf16=q, kv_src=kv_src, kv_slots=np.arange(pool_rows, dtype=np.int64),
                pool_rows=pool_rows, page_table=page_table, page_size=PAGE_SIZE,
                token_seq=None, topk=topk, sm_scale=SM_SCALE)


def prefill_q8_scaled528(seed: int = 6, T: int = 4096, H: int = 32, K: int = 2048,
                         context: int = 8192, pool_rows: int = 16384, first_pos: int = 0) -> dict:
    """The prefill batch over group-scaled 528-byte rows of N(0,1) * U(0.1, 4) per row."""
    w = prefill_q8_raw512(seed=seed, T=T, H=H, K=K, context=context, pool_rows=pool_rows,
                          first_pos=first_pos)
    rng = rng_for(seed + 1000)
    mult = rng.uniform(0.1, 4.0, size=(pool_rows, 1)).astype(np.float32)
    kv = rng.standard_normal((pool_rows, D_LATENT), dtype=np.float32) * mult
    w.update(name="prefill_q8_scaled528", layout="scaled528", kv_src=f32_to_bf16_bits(kv))
    return w


def writer_rows(seed: int = 5, n_rows: int = 16384, pool_rows: int = 262144,
                mult_hi: float = 8.0) -> dict:
    """New BF16 rows N(0,1)*U(0.1, mult_hi) and distinct random destination slots."""
    rng = rng_for(seed)
    mult = rng.uniform(0.1, mult_hi, size=(n_rows, 1)).astype(np.float32)
    x = f32_to_bf16_bits(rng.standard_normal((n_rows, D_LATENT), dtype=np.float32) * mult)
    slots = rng.choice(pool_rows, size=n_rows, replace=False).astype(np.int64)
    return dict(x_bf16=x, slots=slots, pool_rows=pool_rows, n_rows=n_rows)


def writer_sweep(seed: int = 5, H: int = 16, T: int = 64, K: int = 2048,
                 n_rows: int = 16384, pool_rows: int = 262144,
                 layout: str = "raw512") -> dict:
    """Decode over rows freshly written to random slots; physical indices (no page table)."""
    w = writer_rows(seed, n_rows, pool_rows)
    rng = rng_for(seed * 1000 + H)
    q = f32_to_bf16_bits(rng.standard_normal((T, H, D_LATENT), dtype=np.float32))
    topk = np.empty((T, K), dtype=np.int32)
    for t in range(T):
        topk[t] = w["slots"][rng.choice(n_rows, size=K, replace=False)].astype(np.int32)
    if T >= 2:
        topk[0, 1:] = -1            # one-hot token
        topk[1, :] = -1             # all-masked token
    return dict(name="writer_sweep", layout=layout, T=T, H=H, K=K,
                q_bf16=q, kv_src=w["x_bf16"], kv_slots=w["slots"],
                pool_rows=pool_rows, page_table=None, page_size=PAGE_SIZE,
                token_seq=None, topk=topk, sm_scale=SM_SCALE)


def make(name: str, **kw) -> dict:
    fn = {
        "tiny_decode_raw512": tiny_decode_raw512,
        "decode_raw512": decode_raw512,
        "decode_scaled528": decode_scaled528,
        "decode_rope656": decode_rope656,
        "prefill_q8_raw512": prefill_q8_raw512,
        "prefill_q8_scaled528": prefill_q8_scaled528,
        "writer_sweep": writer_sweep,
    }[name]
    return fn(**kw)


def valid_entry_count(topk: np.ndarray) -> int:
    return int((np.asarray(topk) >= 0).sum())
