/*
 * dsa.h - C ABI of a GB300 (sm_103a) library for DeepSeek-Sparse-Attention
 * style top-k sparse MLA attention over a paged FP8 (E4M3) KV cache of
 * 512-dim NoPE latent rows, and for the fused BF16 -> FP8 paged KV writer.
 *
 * Sources (web pages, cited by title and section):
 *   [P1] sglang pull request 44012 (CUDA TileLang raw FP8 KV path), sections
 *        "Motivation", "Modifications", "Speed Tests and Profiling".
 *   [P2] "[DSA] Support group-scaled FP8 NoPE KV reads for CUDA TileLang",
 *        sections "Motivation", "Modifications", "Accuracy Tests".
 *   [P3] "[DSA] Support flashmla_sparse_q8 prefill backend on CUDA",
 *        section "Modifications" and the review thread.
 *
 * Conventions for every entry point:
 *  - Pointers named *_dev are device pointers (cudaMalloc'd or equivalent);
 *    the caller owns all memory.  The library allocates nothing, keeps no
 *    state between calls, performs no host<->device copy and no
 *    synchronisation: each call only enqueues kernels on `stream`
 *    (a cudaStream_t passed as void*, NULL = the legacy default stream).
 *  - Arguments are validated on the host before anything is launched.  On a
 *    non-zero status nothing was launched and no output was touched.
 *    DSA_ERR_CUDA means a launch itself failed (cudaGetLastError).
 *  - Data-dependent faults (a top-k index outside the pool or the page table,
 *    a bad page-table entry, a bad destination slot) never trap: the entry
 *    is skipped and a bit is OR-ed into the caller's int32 *err_flag_dev
 *    (nullable; the library never clears it).
 *  - The FP8 format is OCP E4M3 "FN" (max 448, S.1111.111 = NaN) only;
 *    there is no format argument, so E4M3FNUZ cannot be requested [P1
 *    Modifications].  Saturating round-to-nearest-even everywhere.
 *  - Calls on different streams that write the same buffers race.
 *  - Only GPUs of compute capability 10.3 (GB300) are accepted.
 */
#ifndef DSA_GB300_H
#define DSA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

/* Physical KV row layouts [P1 Modifications; P2 Motivation]:
 *  DSA_KV_RAW512     512 unscaled E4M3 bytes per row.
 *  DSA_KV_SCALED528  512 E4M3 bytes, then four little-endian FP32 scales at
 *                    byte offsets 512 + 4g; scale g applies to dims
 *                    [128g, 128g + 128): value = e4m3(byte) * scale_g.
 *  DSA_KV_ROPE656    the 528-byte row, then the 64 RoPE dims of the key as
 *                    little-endian BF16 at byte offsets 528 + 2j: keys and
 *                    queries are 576 wide, values are the 512 latent dims
 *                    ["[DSA] Support group-scaled FP8 NoPE KV reads for CUDA
 *                    TileLang", Motivation: the 656-byte layout]. */
typedef enum { DSA_KV_RAW512 = 0, DSA_KV_SCALED528 = 1, DSA_KV_ROPE656 = 2 } dsa_kv_layout;

enum {
  DSA_OK = 0,
  DSA_ERR_NULL = 1,      /* a required pointer is NULL */
  DSA_ERR_SHAPE = 2,     /* a size is negative / zero where it must not be / overflows */
  DSA_ERR_LAYOUT = 3,    /* unknown layout, or a layout this entry point refuses */
  DSA_ERR_ROW_WIDTH = 4, /* query width or KV row width is not 512 [P1 Modifications] */
  DSA_ERR_TOPK_PAD = 5,  /* top-k width is not a positive multiple of 128 [P3 Modifications] */
  DSA_ERR_HEADS = 6,     /* head count not in {8, 16, 32, 64, 128} */
  DSA_ERR_WORKSPACE = 7, /* workspace missing or smaller than dsa_sparse_attn_workspace_bytes */
  DSA_ERR_DEVICE = 8,    /* no current CUDA device of compute capability 10.3 */
  DSA_ERR_CUDA = 9,      /* a kernel launch failed */
  DSA_ERR_ALIGN = 10     /* a pointer is not 16-byte aligned (workspace: 256-byte) */
};

/* Bits OR-ed into *err_flag_dev by the kernels. */
enum {
  DSA_DEV_ERR_INDEX_RANGE = 1, /* top-k index beyond the pool (no page table) or beyond
                                  the page table's width; the entry was masked */
  DSA_DEV_ERR_PAGE_RANGE = 2,  /* negative page-table entry, page beyond the pool, or a
                                  token's sequence id outside [0, B); entry masked */
  DSA_DEV_ERR_TIMEOUT = 4,     /* a bounded wait inside a kernel gave up; the outputs of
                                  that call are not valid */
  DSA_DEV_ERR_SLOT_RANGE = 8   /* writer slot >= pool_rows; the row was not written */
};

/* Human-readable name of a status code (static string). */
const char* dsa_status_string(int status);

/* Diagnostics: sets the limit, in nanoseconds, of every bounded wait inside
 * the attention kernel (default 1 s) for the attention calls made after it,
 * process-wide, and returns the previous limit.  A wait that runs out makes
 * the kernel give up: its other waits return at once, it waits (with a
 * separate 2 s bound) for its own copies and tensor-core operations in
 * flight, releases its tensor memory, returns, and ORs DSA_DEV_ERR_TIMEOUT
 * into err_flag_dev; that call's outputs are then not valid, and the CUDA
 * context stays usable.  A limit of 0 makes the first wait that is not
 * already complete give up, which lets a test exercise this path without
 * stalling the GPU.  Not meant to be changed while attention calls are being
 * issued from other threads. */
uint64_t dsa_set_wait_limit_ns(uint64_t ns);

/* Bytes of one physical KV row: 512, 528 or 656 ("exported buffer lengths",
 * [P1 Speed Tests and Profiling]); 0 for an unknown layout. */
size_t dsa_kv_row_bytes(int layout);

/* ------------------------------------------------------------- KV writers */

/* Stream ordering of the writers: each writer kernel releases its programmatic
 * dependents as it starts (griddepcontrol.launch_dependents).  A kernel that
 * the caller launches next on the same stream with programmatic stream
 * serialization may therefore begin while the writer still runs, and must
 * execute griddepcontrol.wait before it reads the pool (the attention entry
 * points below do).  Kernels launched without that attribute, copies and
 * events are ordered after the writer as usual. */

/* Fused cast + paged scatter of new latent rows into a raw512 pool
 * [P1 Motivation, Modifications: the fused cast/paged writer, selected by
 * raw versus scaled layout, NoPE rows with no RoPE tensor].
 *   x_bf16_dev  [n_rows, 512] BF16, row-major, 16-byte aligned.
 *   slots_dev   [n_rows] int64 physical destination rows; slot < 0 skips the
 *               row (padding); slot >= pool_rows sets DSA_DEV_ERR_SLOT_RANGE.
 *   pool_dev    [pool_rows, 512] bytes, 16-byte aligned.
 *   pool[slot][d] = e4m3_satrne((float)x[i][d]).  Duplicate slots within one
 *   call are a caller error (which row lands is unspecified).
 * n_rows == 0 is a no-op returning DSA_OK. */
int dsa_kv_write_raw(const void* x_bf16_dev, int64_t n_rows, const int64_t* slots_dev,
                     void* pool_dev, int64_t pool_rows, int32_t* err_flag_dev, void* stream);

/* Same for the group-scaled 528-byte layout [P2 Motivation: "512 FP8 values
 * and four FP32 scales per token"]: for each group g of 128 dims,
 * s_g = amax_g / 448 (FP32, IEEE division), byte = e4m3_satrne(x / s_g)
 * (FP32 IEEE division); amax_g == 0 stores s_g = 0 and zero bytes.
 *   pool_dev  [pool_rows, 528] bytes, 16-byte aligned. */
int dsa_kv_write_scaled(const void* x_bf16_dev, int64_t n_rows, const int64_t* slots_dev,
                        void* pool_dev, int64_t pool_rows, int32_t* err_flag_dev, void* stream);

/* Same for the 656-byte RoPE layout: x_bf16_dev is [n_rows, 576]; dims
 * [0, 512) are written as by dsa_kv_write_scaled, dims [512, 576) are stored
 * unchanged (BF16) at byte offsets 528 + 2j.
 *   x_bf16_dev  [n_rows, 576] BF16, 16-byte aligned.
 *   pool_dev    [pool_rows, 656] bytes, 16-byte aligned. */
int dsa_kv_write_rope656(const void* x_bf16_dev, int64_t n_rows, const int64_t* slots_dev,
                         void* pool_dev, int64_t pool_rows, int32_t* err_flag_dev, void* stream);

/* FP8 query quantiser (NoPE query preparation with a zero-dim RoPE part,
 * [P3 Modifications: zero-dimensional RoPE queries]): per vector of 512 dims
 * (one token and head), scale = amax / 448 (FP32), q8 = e4m3_satrne(q / scale);
 * amax == 0 gives scale 0 and zero bytes.
 *   q_bf16_dev   [n_vec, 512] BF16;  q8_dev [n_vec, 512] bytes;
 *   q_scale_dev  [n_vec] float.  All 16-byte aligned except q_scale (4). */
int dsa_quantize_q8(const void* q_bf16_dev, int64_t n_vec, void* q8_dev, float* q_scale_dev,
                    void* stream);

/* ------------------------------------------------------ sparse attention */

/* Workspace bytes the attention entry points need for (T, H, K) on the
 * current device, for any row layout: split-K partial results (two FP32
 * slots of [heads, 512] and [heads] per SM), needed only when a (token, head
 * group) is spread over several SMs.  May be 0.  Pass at least this many bytes, 256-byte aligned;
 * no initialisation is needed: each call writes every byte it reads. */
size_t dsa_sparse_attn_workspace_bytes(int T, int H, int K);

/* Sparse MLA decode with BF16 queries over a paged FP8 pool, either layout
 * [P1 Motivation: TileLang decode over raw FP8 KV; P2 Modifications: the
 * group-scaled reader; P3 Modifications: top-k padded to a multiple of 128
 * with -1 sentinels].
 *
 * For each token t and head h, over the valid entries j of topk[t]:
 *   row_j  = page_table[token_seq[t]][i / page_size] * page_size + i % page_size,
 *            i = topk[t][j]  (row_j = i when page_table is NULL);
 *   k_j    = dequantised 512-dim latent row (the same row is key and value);
 *   s_j    = sm_scale * <q[t][h], k_j>;
 *   LSE    = log(sum_j exp(s_j))            (natural log)
 *   O[t,h] = sum_j exp(s_j - LSE) * k_j     (BF16, round-to-nearest-even)
 * A negative index is masked.  A token with no valid entry gets O = 0 and
 * LSE = -inf.  Duplicate indices count once per slot.
 *
 *   q_bf16_dev      [T, H, 512] BF16, 16-byte aligned.
 *   D, kv_row_dim   must both be 512, or both 576 with DSA_KV_ROPE656 (else
 *                   DSA_ERR_ROW_WIDTH); over 656-byte rows the query is
 *                   [T, H, 576] (latent dims, then the 64 RoPE dims), the
 *                   scores use all 576 dims and O the 512 latent dims.
 *   pool_dev        [pool_rows, 512, 528 or 656] bytes, 16-byte aligned.
 *   page_table_dev  [B, max_pages] int32 physical page ids, or NULL.
 *   token_seq_dev   [T] int32 sequence id per token, or NULL (all sequence 0).
 *   topk_dev        [T, K] int32, K a positive multiple of 128.
 *   o_bf16_dev      [T, H, 512] BF16 out, 16-byte aligned.
 *   lse_dev         [T, H] float out.
 *   workspace_dev   ws_bytes >= dsa_sparse_attn_workspace_bytes(T, H, K).
 *   err_flag_dev    nullable int32 error bits.
 * H must be one of 8, 16, 32, 64, 128.
 * T == 0 is a no-op.
 * Launch: the attention kernel is launched with programmatic stream
 * serialization; it may start its set-up while the previous kernel on the
 * stream runs (if that kernel released its dependents early, as the writers
 * do) and executes griddepcontrol.wait before it reads or writes any global
 * memory, so the stream order of all inputs and outputs is kept.  The
 * split-unit merge that follows it is launched the same way. */
int dsa_sparse_attn_decode(const void* q_bf16_dev, int T, int H, int D,
                           const void* pool_dev, int64_t pool_rows, int layout, int kv_row_dim,
                           const int32_t* page_table_dev, int B, int max_pages, int page_size,
                           const int32_t* token_seq_dev, const int32_t* topk_dev, int K,
                           float sm_scale, void* o_bf16_dev, float* lse_dev,
                           void* workspace_dev, size_t ws_bytes, int32_t* err_flag_dev,
                           void* stream);

/* Sparse MLA prefill with FP8 queries ("Q8", [P3 Modifications]): the same
 * definition with q[t][h][d] = e4m3(q8[t][h][d]) * q_scale[t][h].  Both row
 * layouts are accepted.  The pages' Q8 prefill stops at raw rows and guards
 * against packed FP8 pools [P3 review thread: the packed-FP8 KPool guard;
 * "[DSA] Support group-scaled FP8 NoPE KV reads for CUDA TileLang",
 * Modifications: native FP8 attention over the scaled layout not included];
 * over 528-byte rows this library applies each group's scale exactly as the
 * BF16-query decode does.
 *   q8_dev       [T, H, 512] E4M3 bytes, 16-byte aligned.
 *   q_scale_dev  [T, H] float. */
int dsa_sparse_attn_prefill_q8(const void* q8_dev, const float* q_scale_dev, int T, int H, int D,
                               const void* pool_dev, int64_t pool_rows, int layout, int kv_row_dim,
                               const int32_t* page_table_dev, int B, int max_pages, int page_size,
                               const int32_t* token_seq_dev, const int32_t* topk_dev, int K,
                               float sm_scale, void* o_bf16_dev, float* lse_dev,
                               void* workspace_dev, size_t ws_bytes, int32_t* err_flag_dev,
                               void* stream);

/* ------------------------------------------- gather / dequantise reader */

/* Bytes of the BF16 workspace dsa_gather_dequant writes for T tokens with
 * top-k width K over a pool of pool_rows rows: min(pool_rows, T*K) rows of
 * 512 BF16 values (1024 bytes), or of 576 values (1152 bytes) for 656-byte
 * rows ["[DSA] Support group-scaled FP8 NoPE KV reads for CUDA TileLang",
 * Modifications: the BF16 payload workspace is bounded by
 * min(physical_tokens, selected_entries) * 1024 bytes].  The size follows
 * from the shapes alone, so sizing it needs no device data.  0 for a
 * negative size or an unknown layout. */
size_t dsa_gather_dequant_workspace_bytes(int T, int K, int64_t pool_rows, int layout);

/* Gather / dequantise reader: the rows a top-k list selects, dequantised to
 * BF16 in a workspace that BF16 consumers index with the remapped list
 * ["[DSA] Support group-scaled FP8 NoPE KV reads for CUDA TileLang",
 * Modifications: the full and paged readers, int64 physical addressing, the
 * selected-row workspace with remapped indices and kept masks; P3 review
 * thread: the paged gather with -1 padding].  Two branches, chosen by shape:
 *  - T*K < pool_rows (fewer selected entries than physical rows): workspace
 *    row e = t*K + j holds entry j of token t, idx_out[e] = e;
 *  - otherwise the whole pool is dequantised: workspace row r holds physical
 *    row r, idx_out[e] = the entry's physical row.
 * A masked entry (negative index, or one that fails to resolve, with the
 * attention's error bits in err_flag_dev) gets idx_out[e] = -1; in the first
 * branch its workspace row is left untouched.  In both branches
 * out[idx_out[e]] is entry e's row:
 *   out[.][d] = bf16_rn(fp32(e4m3(b_d) * s_g))   (raw rows: s = 1, exact),
 * followed, for 656-byte rows, by the row's 64 RoPE dims as stored.
 *   pool_dev        [pool_rows, 512, 528 or 656] bytes, 16-byte aligned.
 *   page_table_dev  [B, max_pages] int32, or NULL (indices are physical rows).
 *   token_seq_dev   [T] int32 or NULL.
 *   topk_dev        [T, K] int32, any K >= 1, T * K < 2^31.
 *   out_bf16_dev    out_bytes >= dsa_gather_dequant_workspace_bytes(T, K,
 *                   pool_rows, layout) (else DSA_ERR_WORKSPACE), 16-byte
 *                   aligned; row-major [rows, 512 or 576] BF16.
 *   idx_out_dev     [T, K] int32.
 * T == 0 is a no-op. */
int dsa_gather_dequant(const void* pool_dev, int64_t pool_rows, int layout,
                       const int32_t* page_table_dev, int B, int max_pages, int page_size,
                       const int32_t* token_seq_dev, const int32_t* topk_dev, int T, int K,
                       void* out_bf16_dev, size_t out_bytes, int32_t* idx_out_dev, int32_t* err_flag_dev,
                       void* stream);

/* ------------------------------------------- decode without allocation */

/* Largest split-K workspace dsa_sparse_attn_decode_noalloc can serve (32 MiB). */
#define DSA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/* dsa_sparse_attn_decode for callers that cannot allocate device memory.
 * The pages have no counterpart of this entry point; it exists for callers
 * that have no way to obtain the workspace buffer: an engine that gives all
 * of HBM to its KV-cache pool up front, a plug-in running inside a host that
 * owns the CUDA allocator, or code that must stay free of cudaMalloc.
 *
 * Arguments and results are those of dsa_sparse_attn_decode without the
 * workspace pair.  The workspace is a file-scope device array of
 * DSA_NOALLOC_SCRATCH_BYTES bytes inside this library: every GPU on which the
 * library is loaded holds that array until the process exits.  The call
 * itself allocates nothing (no cudaMalloc, no cudaFree, no allocating library
 * routine).
 *  - The first call on a device looks up the array's device address for that
 *    device (cudaGetSymbolAddress, with that device current); make that first
 *    call before any stream capture on the device.  The address is kept for
 *    the life of the process; after a cudaDeviceReset of that device it is
 *    stale, so a process that resets a device must not call this entry point
 *    on it again.
 *  - A (T, H, K) whose workspace (dsa_sparse_attn_workspace_bytes) exceeds
 *    DSA_NOALLOC_SCRATCH_BYTES is refused with DSA_ERR_WORKSPACE, nothing
 *    launched.
 *  - All calls share the one array, which keeps whatever the last call left
 *    in it; nothing in it needs clearing, because each call writes the
 *    partial results before it reads them.  Calls whose work overlaps on
 *    the GPU (other streams, other host threads) race on the array:
 *    serialise them. */
int dsa_sparse_attn_decode_noalloc(const void* q_bf16_dev, int T, int H, int D,
                                   const void* pool_dev, int64_t pool_rows, int layout, int kv_row_dim,
                                   const int32_t* page_table_dev, int B, int max_pages, int page_size,
                                   const int32_t* token_seq_dev, const int32_t* topk_dev, int K,
                                   float sm_scale, void* o_bf16_dev, float* lse_dev,
                                   int32_t* err_flag_dev, void* stream);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif

#ifdef __cplusplus
}
#endif

#endif /* DSA_GB300_H */
