// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace dsa {

void launch_kv_write(bool scaled, const void* x, int64_t n_rows, const int64_t* slots, void* pool,
                     int64_t pool_rows, int32_t* err, int sms, cudaStream_t stream);

void launch_quantize_q8(const void* q, int64_t n_vec, void* q8, float* scale, int sms,
                        cudaStream_t stream);

// Everything one sparse-attention launch needs.
struct AttnArgs {
  const void* q;          // BF16 [T,H,512] or E4M3 [T,H,512]
  const float* q_scale;   // [T,H] for FP8 queries, else nullptr
  int T, H;
  const uint8_t* pool;
  int64_t pool_rows;
  bool scaled;            // 528-byte rows
  const int32_t* page_table;
  int B, max_pages, page_size;
  const int32_t* token_seq;
  const int32_t* topk;
  int K;
  float sm_scale;
  void* o;                // BF16 [T,H,512]
  float* lse;             // [T,H]
  float* ws_o;            // [n_splits,T,H,512] partial O (normalised), when n_splits > 1
  float* ws_lse;          // [n_splits,T,H]
  int n_splits, chunk;    // top-k entries [s*chunk, min(K,(s+1)*chunk)) go to split s
  int32_t* err;
};

// Split-K plan: how many top-k chunks per token, shared by the workspace
// query and the launch.
struct SplitPlan {
  int n_splits;
  int chunk;
  size_t ws_bytes;
  size_t ws_lse_offset;
};
SplitPlan plan_splits(int T, int H, int K, int sms);

void launch_sparse_attn(const AttnArgs& a, bool q8, cudaStream_t stream);
void launch_combine(const AttnArgs& a, cudaStream_t stream);

// Heads handled by one CTA of the attention kernel, and the most top-k
// entries one CTA can own (bounds the split plan).
int head_group(int H);
int max_chunk();

}  // namespace dsa
