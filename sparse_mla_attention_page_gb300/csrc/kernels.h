// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace dsa {

void launch_kv_write(int layout, const void* x, int64_t n_rows, const int64_t* slots, void* pool,
                     int64_t pool_rows, int32_t* err, int sms, cudaStream_t stream);

void launch_quantize_q8(const void* q, int64_t n_vec, void* q8, float* scale, int sms,
                        cudaStream_t stream);

// Everything one sparse-attention launch needs.
//
// Work is cut into units of (token, group of hg heads) and each unit's top-k
// list into tiles of 128 entries: n_tiles = T * hgs * tpt.  The persistent
// kernel runs `grid` CTAs; CTA c owns the contiguous global tiles
// [c * n_tiles / grid, (c + 1) * n_tiles / grid).  A unit whose tiles span more
// than one CTA leaves one partial result per CTA, merged by combine_kernel.
struct AttnArgs {
  const void* q;          // BF16 [T,H,512] or E4M3 [T,H,512]
  const float* q_scale;   // [T,H] for FP8 queries, else nullptr
  int T, H;
  int q_row;              // elements per query row: 512, or 576 over 656-byte rows
  const uint8_t* pool;
  int64_t pool_rows;
  bool scaled;            // 528-byte (or 656-byte) rows: group scales
  bool rope;              // 656-byte rows: 64 BF16 RoPE dims after the scales
  const int32_t* page_table;
  int B, max_pages, page_size;
  const int32_t* token_seq;
  const int32_t* topk;
  int K;
  float sm_scale;
  void* o;                // BF16 [T,H,512]
  float* lse;             // [T,H]
  int hg, hgs, tpt;       // heads per unit, units per token, tiles per unit
  int64_t n_tiles;
  int grid;
  float* ws_o;            // [grid][2][hg][512] normalised partial O (slot 0: the CTA's first unit)
  float* ws_lse;          // [grid][2][hg]
  int32_t* err;
  uint64_t wait_ns;       // limit of every bounded wait inside the kernel
};

// Launch plan shared by the workspace query and the launch.  Workspace (only
// when a unit spans two or more CTAs): split-K partials, two slots per CTA.
struct AttnPlan {
  int hg, hgs, tpt;
  int64_t n_tiles;
  int grid;
  bool split;
  size_t ws_o_offset, ws_lse_offset;
  size_t ws_bytes;
};
AttnPlan plan_attn(int T, int H, int K, int sms, bool rope);

// false when nothing was launched (a launch attribute could not be set, or the
// kernel was not built with the register count its register re-split needs).
bool launch_sparse_attn(const AttnArgs& a, bool q8, cudaStream_t stream);

// Gather / dequantise reader (see gather_dequant.cu).
struct GatherArgs {
  const uint8_t* pool;
  int64_t pool_rows;
  int layout;             // DSA_KV_RAW512, DSA_KV_SCALED528 or DSA_KV_ROPE656
  bool full_pool;         // T*K >= pool_rows: dequantise the whole pool
  const int32_t* page_table;
  int B, max_pages, page_size;
  const int32_t* token_seq;
  const int32_t* topk;    // [T, K]
  int T, K;
  void* out;              // BF16 [gather_rows(pool_rows, T*K), 512 or 576]
  int32_t* idx_out;       // [T, K]
  int32_t* err;
};
// Rows of the reader's workspace: min(pool_rows, selected entries).
int64_t gather_rows(int64_t pool_rows, int64_t n_selected);
void launch_gather_dequant(const GatherArgs& g, int sms, cudaStream_t stream);

// Merges the partial results of split units (after the attention kernel).
void launch_combine(const AttnArgs& a, cudaStream_t stream);

// DSA_OK and the SM count when the current device has compute capability
// 10.3, else DSA_ERR_DEVICE.
int current_device_sms(int* sms);

// Heads handled together by one CTA of the attention kernel: up to 32, up to
// 16 over 656-byte rows (whose RoPE operands take the shared memory of the
// larger groups).
int head_group(int H, bool rope);

// The persistent schedule: CTA c owns global tiles [tile_begin(c), tile_begin(c + 1)).
__host__ __device__ __forceinline__ int64_t tile_begin(int c, int64_t n_tiles, int grid) {
  return (int64_t)c * n_tiles / grid;
}
// The CTA that owns global tile x: the largest c with tile_begin(c) <= x.
__host__ __device__ __forceinline__ int cta_of_tile(int64_t x, int64_t n_tiles, int grid) {
  return (int)(((x + 1) * grid + n_tiles - 1) / n_tiles - 1);
}

}  // namespace dsa
