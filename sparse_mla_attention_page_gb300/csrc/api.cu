// C ABI entry points (include/dsa.h): host-side validation, then launches.
// Every check runs before anything is enqueued; on a non-zero status nothing
// was launched.
#include <atomic>
#include <climits>
#include <cstdio>
#include <cstdlib>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/dsa.h"
#include "kernels.h"

namespace dsa {

// Current device must be compute capability 10.3; returns its SM count.
int current_device_sms(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return DSA_ERR_DEVICE;
  }
  int major = 0, minor = 0, count = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return DSA_ERR_DEVICE;
  }
  if (major != 10 || minor != 3) return DSA_ERR_DEVICE;
  *sms = count;
  return DSA_OK;
}

}  // namespace dsa

namespace {

using dsa::current_device_sms;

// Limit of the attention kernel's bounded waits (dsa_set_wait_limit_ns).
std::atomic<uint64_t> g_wait_ns{1000000000ull};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// A failed launch returns DSA_ERR_CUDA; with DSA_DEBUG set in the environment
// the CUDA error string is also printed to stderr.
int launch_status() {
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) return DSA_OK;
  if (std::getenv("DSA_DEBUG") != nullptr) std::fprintf(stderr, "dsa: launch failed: %s\n", cudaGetErrorString(e));
  return DSA_ERR_CUDA;
}

bool heads_ok(int H) { return H == 8 || H == 16 || H == 32 || H == 64 || H == 128; }

int validate_writer(const void* x, int64_t n_rows, const int64_t* slots, const void* pool,
                    int64_t pool_rows, int64_t row_bytes) {
  if (n_rows < 0 || pool_rows < 0) return DSA_ERR_SHAPE;
  if (n_rows == 0) return DSA_OK;
  if (x == nullptr || slots == nullptr || pool == nullptr) return DSA_ERR_NULL;
  if (pool_rows > INT64_MAX / row_bytes || n_rows > INT64_MAX / 1024) return DSA_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(pool, 16) || !aligned(slots, 8)) return DSA_ERR_ALIGN;
  return DSA_OK;
}

int write_rows(int layout, const void* x, int64_t n_rows, const int64_t* slots, void* pool,
               int64_t pool_rows, int32_t* err, void* stream) {
  int st = validate_writer(x, n_rows, slots, pool, pool_rows, (int64_t)dsa_kv_row_bytes(layout));
  if (st != DSA_OK || n_rows == 0) return st;
  int sms = 0;
  if ((st = current_device_sms(&sms)) != DSA_OK) return st;
  cudaGetLastError();  // a stale error from earlier work is not this call's
  dsa::launch_kv_write(layout, x, n_rows, slots, pool, pool_rows, err, sms,
                       static_cast<cudaStream_t>(stream));
  return launch_status();
}

int sparse_attn(bool q8, const void* q, const float* q_scale, int T, int H, int D, const void* pool,
                int64_t pool_rows, int layout, int kv_row_dim, const int32_t* page_table, int B,
                int max_pages, int page_size, const int32_t* token_seq, const int32_t* topk, int K,
                float sm_scale, void* o, float* lse, void* ws, size_t ws_bytes, int32_t* err,
                void* stream) {
  if (T < 0 || pool_rows < 0) return DSA_ERR_SHAPE;
  if (layout != DSA_KV_RAW512 && layout != DSA_KV_SCALED528 && layout != DSA_KV_ROPE656) return DSA_ERR_LAYOUT;
  const int width = layout == DSA_KV_ROPE656 ? 576 : 512;
  if (D != width || kv_row_dim != width) return DSA_ERR_ROW_WIDTH;
  if (q8 && layout == DSA_KV_ROPE656) return DSA_ERR_LAYOUT;
  if (K <= 0 || K % 128 != 0) return DSA_ERR_TOPK_PAD;
  if (!heads_ok(H)) return DSA_ERR_HEADS;
  if (T == 0) return DSA_OK;
  if (q == nullptr || pool == nullptr || topk == nullptr || o == nullptr || lse == nullptr ||
      (q8 && q_scale == nullptr))
    return DSA_ERR_NULL;
  if (pool_rows < 1 || pool_rows > INT32_MAX) return DSA_ERR_SHAPE;
  if (page_table != nullptr) {
    if (B < 1 || max_pages < 1 || page_size < 1) return DSA_ERR_SHAPE;
    if ((int64_t)max_pages * page_size > (int64_t)INT32_MAX + 1) return DSA_ERR_SHAPE;
  }
  if (!aligned(q, 16) || !aligned(pool, 16) || !aligned(o, 16) || !aligned(topk, 16) ||
      !aligned(lse, 4) || (q_scale && !aligned(q_scale, 4)))
    return DSA_ERR_ALIGN;
  int sms = 0;
  int st = current_device_sms(&sms);
  if (st != DSA_OK) return st;
  const dsa::AttnPlan plan = dsa::plan_attn(T, H, K, sms, layout == DSA_KV_ROPE656);
  if (plan.ws_bytes > 0) {
    if (ws == nullptr || ws_bytes < plan.ws_bytes) return DSA_ERR_WORKSPACE;
    if (!aligned(ws, 256)) return DSA_ERR_ALIGN;
  }
  dsa::AttnArgs a{};
  a.q = q;
  a.q_scale = q_scale;
  a.T = T;
  a.H = H;
  a.q_row = layout == DSA_KV_ROPE656 ? 576 : 512;
  a.pool = static_cast<const uint8_t*>(pool);
  a.pool_rows = pool_rows;
  a.scaled = layout == DSA_KV_SCALED528 || layout == DSA_KV_ROPE656;
  a.rope = layout == DSA_KV_ROPE656;
  a.page_table = page_table;
  a.B = B;
  a.max_pages = max_pages;
  a.page_size = page_table ? page_size : 1;
  a.token_seq = page_table ? token_seq : nullptr;
  a.topk = topk;
  a.K = K;
  a.sm_scale = sm_scale;
  a.o = o;
  a.lse = lse;
  a.hg = plan.hg;
  a.hgs = plan.hgs;
  a.tpt = plan.tpt;
  a.n_tiles = plan.n_tiles;
  a.grid = plan.grid;
  char* wsb = static_cast<char*>(ws);
  a.ws_o = plan.split ? reinterpret_cast<float*>(wsb + plan.ws_o_offset) : nullptr;
  a.ws_lse = plan.split ? reinterpret_cast<float*>(wsb + plan.ws_lse_offset) : nullptr;
  a.err = err;
  a.wait_ns = g_wait_ns.load();
  cudaGetLastError();
  const bool launched = dsa::launch_sparse_attn(a, q8, static_cast<cudaStream_t>(stream));
  const int st2 = launch_status();
  return st2 != DSA_OK ? st2 : launched ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* dsa_status_string(int status) {
  switch (status) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_NULL: return "DSA_ERR_NULL: a required pointer is NULL";
    case DSA_ERR_SHAPE: return "DSA_ERR_SHAPE: invalid size";
    case DSA_ERR_LAYOUT: return "DSA_ERR_LAYOUT: unsupported KV layout for this entry point";
    case DSA_ERR_ROW_WIDTH: return "DSA_ERR_ROW_WIDTH: query and KV row width must be 512";
    case DSA_ERR_TOPK_PAD: return "DSA_ERR_TOPK_PAD: top-k width must be a positive multiple of 128";
    case DSA_ERR_HEADS: return "DSA_ERR_HEADS: head count must be 8, 16, 32, 64 or 128";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE: workspace missing or too small";
    case DSA_ERR_DEVICE: return "DSA_ERR_DEVICE: current device is not a compute capability 10.3 GPU";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA: kernel launch failed";
    case DSA_ERR_ALIGN: return "DSA_ERR_ALIGN: pointer misaligned";
    default: return "unknown status";
  }
}

uint64_t dsa_set_wait_limit_ns(uint64_t ns) { return g_wait_ns.exchange(ns); }

size_t dsa_kv_row_bytes(int layout) {
  if (layout == DSA_KV_RAW512) return 512;
  if (layout == DSA_KV_SCALED528) return 528;
  if (layout == DSA_KV_ROPE656) return 656;
  return 0;
}

int dsa_kv_write_raw(const void* x_bf16_dev, int64_t n_rows, const int64_t* slots_dev,
                     void* pool_dev, int64_t pool_rows, int32_t* err_flag_dev, void* stream) {
  return write_rows(DSA_KV_RAW512, x_bf16_dev, n_rows, slots_dev, pool_dev, pool_rows, err_flag_dev, stream);
}

int dsa_kv_write_scaled(const void* x_bf16_dev, int64_t n_rows, const int64_t* slots_dev,
                        void* pool_dev, int64_t pool_rows, int32_t* err_flag_dev, void* stream) {
  return write_rows(DSA_KV_SCALED528, x_bf16_dev, n_rows, slots_dev, pool_dev, pool_rows, err_flag_dev, stream);
}

int dsa_kv_write_rope656(const void* x_bf16_dev, int64_t n_rows, const int64_t* slots_dev,
                         void* pool_dev, int64_t pool_rows, int32_t* err_flag_dev, void* stream) {
  return write_rows(DSA_KV_ROPE656, x_bf16_dev, n_rows, slots_dev, pool_dev, pool_rows, err_flag_dev, stream);
}

int dsa_quantize_q8(const void* q_bf16_dev, int64_t n_vec, void* q8_dev, float* q_scale_dev,
                    void* stream) {
  if (n_vec < 0) return DSA_ERR_SHAPE;
  if (n_vec == 0) return DSA_OK;
  if (q_bf16_dev == nullptr || q8_dev == nullptr || q_scale_dev == nullptr) return DSA_ERR_NULL;
  if (n_vec > INT64_MAX / 1024) return DSA_ERR_SHAPE;
  if (!aligned(q_bf16_dev, 16) || !aligned(q8_dev, 16) || !aligned(q_scale_dev, 4)) return DSA_ERR_ALIGN;
  int sms = 0;
  int st = current_device_sms(&sms);
  if (st != DSA_OK) return st;
  cudaGetLastError();
  dsa::launch_quantize_q8(q_bf16_dev, n_vec, q8_dev, q_scale_dev, sms, static_cast<cudaStream_t>(stream));
  return launch_status();
}

size_t dsa_gather_dequant_workspace_bytes(int T, int K, int64_t pool_rows, int layout) {
  if (T < 0 || K < 0 || pool_rows < 0 || dsa_kv_row_bytes(layout) == 0) return 0;
  const size_t width = layout == DSA_KV_ROPE656 ? 576 : 512;
  return (size_t)dsa::gather_rows(pool_rows, (int64_t)T * K) * width * 2;
}

int dsa_gather_dequant(const void* pool_dev, int64_t pool_rows, int layout,
                       const int32_t* page_table_dev, int B, int max_pages, int page_size,
                       const int32_t* token_seq_dev, const int32_t* topk_dev, int T, int K,
                       void* out_bf16_dev, size_t out_bytes, int32_t* idx_out_dev, int32_t* err_flag_dev,
                       void* stream) {
  if (T < 0 || K < 1 || pool_rows < 0) return DSA_ERR_SHAPE;
  if (layout != DSA_KV_RAW512 && layout != DSA_KV_SCALED528 && layout != DSA_KV_ROPE656) return DSA_ERR_LAYOUT;
  if (T == 0) return DSA_OK;
  if (pool_dev == nullptr || topk_dev == nullptr || out_bf16_dev == nullptr || idx_out_dev == nullptr)
    return DSA_ERR_NULL;
  if (pool_rows < 1 || pool_rows > INT32_MAX || (int64_t)T * K > INT32_MAX) return DSA_ERR_SHAPE;
  if (page_table_dev != nullptr) {
    if (B < 1 || max_pages < 1 || page_size < 1) return DSA_ERR_SHAPE;
    if ((int64_t)max_pages * page_size > (int64_t)INT32_MAX + 1) return DSA_ERR_SHAPE;
  }
  if (out_bytes < dsa_gather_dequant_workspace_bytes(T, K, pool_rows, layout)) return DSA_ERR_WORKSPACE;
  if (!aligned(pool_dev, 16) || !aligned(out_bf16_dev, 16) || !aligned(topk_dev, 4) ||
      !aligned(idx_out_dev, 4))
    return DSA_ERR_ALIGN;
  int sms = 0;
  int st = current_device_sms(&sms);
  if (st != DSA_OK) return st;
  dsa::GatherArgs g{};
  g.pool = static_cast<const uint8_t*>(pool_dev);
  g.pool_rows = pool_rows;
  g.layout = layout;
  g.full_pool = !((int64_t)T * K < pool_rows);
  g.page_table = page_table_dev;
  g.B = B;
  g.max_pages = max_pages;
  g.page_size = page_table_dev ? page_size : 1;
  g.token_seq = page_table_dev ? token_seq_dev : nullptr;
  g.topk = topk_dev;
  g.T = T;
  g.K = K;
  g.out = out_bf16_dev;
  g.idx_out = idx_out_dev;
  g.err = err_flag_dev;
  cudaGetLastError();
  dsa::launch_gather_dequant(g, sms, static_cast<cudaStream_t>(stream));
  return launch_status();
}

size_t dsa_sparse_attn_workspace_bytes(int T, int H, int K) {
  int sms = 0;
  if (current_device_sms(&sms) != DSA_OK) sms = 152;
  // enough for every layout: 656-byte rows use head groups of at most 16
  const size_t a = dsa::plan_attn(T, H, K, sms, false).ws_bytes;
  const size_t b = dsa::plan_attn(T, H, K, sms, true).ws_bytes;
  return a > b ? a : b;
}

int dsa_sparse_attn_decode(const void* q_bf16_dev, int T, int H, int D, const void* pool_dev,
                           int64_t pool_rows, int layout, int kv_row_dim,
                           const int32_t* page_table_dev, int B, int max_pages, int page_size,
                           const int32_t* token_seq_dev, const int32_t* topk_dev, int K,
                           float sm_scale, void* o_bf16_dev, float* lse_dev, void* workspace_dev,
                           size_t ws_bytes, int32_t* err_flag_dev, void* stream) {
  return sparse_attn(false, q_bf16_dev, nullptr, T, H, D, pool_dev, pool_rows, layout, kv_row_dim,
                     page_table_dev, B, max_pages, page_size, token_seq_dev, topk_dev, K, sm_scale,
                     o_bf16_dev, lse_dev, workspace_dev, ws_bytes, err_flag_dev, stream);
}

int dsa_sparse_attn_prefill_q8(const void* q8_dev, const float* q_scale_dev, int T, int H, int D,
                               const void* pool_dev, int64_t pool_rows, int layout, int kv_row_dim,
                               const int32_t* page_table_dev, int B, int max_pages, int page_size,
                               const int32_t* token_seq_dev, const int32_t* topk_dev, int K,
                               float sm_scale, void* o_bf16_dev, float* lse_dev,
                               void* workspace_dev, size_t ws_bytes, int32_t* err_flag_dev,
                               void* stream) {
  return sparse_attn(true, q8_dev, q_scale_dev, T, H, D, pool_dev, pool_rows, layout, kv_row_dim,
                     page_table_dev, B, max_pages, page_size, token_seq_dev, topk_dev, K, sm_scale,
                     o_bf16_dev, lse_dev, workspace_dev, ws_bytes, err_flag_dev, stream);
}

}  // extern "C"
