// Sparse MLA decode for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a device buffer for the split-K
// workspace: an engine that hands every byte of HBM to its KV-cache pool up
// front, a plug-in loaded into a host process that owns the CUDA allocator,
// or code running where a cudaMalloc would break an allocation-free
// guarantee.  dsa_sparse_attn_decode_noalloc serves them: it uses a
// file-scope device array as the workspace and otherwise runs exactly the
// work of dsa_sparse_attn_decode.
//
// The array's address is looked up once per device (cudaGetSymbolAddress,
// with that device current) on the first call made on that device; the host
// symbol itself is only a stand-in and is never handed to a kernel.  The
// address stays cached for the life of the process: a cudaDeviceReset, which
// unloads the module and may place the array elsewhere, invalidates it.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/dsa.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = DSA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device (set-up on first use).
int scratch_on_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return DSA_ERR_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDevices) return DSA_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return DSA_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return DSA_OK;
}

bool heads_supported(int H) { return H == 8 || H == 16 || H == 32 || H == 64 || H == 128; }

}  // namespace

extern "C" int dsa_sparse_attn_decode_noalloc(const void* q_bf16_dev, int T, int H, int D,
                                              const void* pool_dev, int64_t pool_rows, int layout,
                                              int kv_row_dim, const int32_t* page_table_dev, int B,
                                              int max_pages, int page_size,
                                              const int32_t* token_seq_dev, const int32_t* topk_dev,
                                              int K, float sm_scale, void* o_bf16_dev,
                                              float* lse_dev, int32_t* err_flag_dev, void* stream) {
  // the same first checks, in the same order, as dsa_sparse_attn_decode
  if (T < 0 || pool_rows < 0) return DSA_ERR_SHAPE;
  if (layout != DSA_KV_RAW512 && layout != DSA_KV_SCALED528 && layout != DSA_KV_ROPE656) return DSA_ERR_LAYOUT;
  const int width = layout == DSA_KV_ROPE656 ? 576 : 512;
  if (D != width || kv_row_dim != width) return DSA_ERR_ROW_WIDTH;
  if (K <= 0 || K % 128 != 0) return DSA_ERR_TOPK_PAD;
  if (!heads_supported(H)) return DSA_ERR_HEADS;
  if (T == 0) return DSA_OK;
  int sms = 0;
  if (dsa::current_device_sms(&sms) != DSA_OK) {
    // no usable device: the decode entry point's own checks give the status
    // (an argument error if there is one, else DSA_ERR_DEVICE); it launches
    // nothing on this path
    return dsa_sparse_attn_decode(q_bf16_dev, T, H, D, pool_dev, pool_rows, layout, kv_row_dim,
                                  page_table_dev, B, max_pages, page_size, token_seq_dev, topk_dev, K,
                                  sm_scale, o_bf16_dev, lse_dev, nullptr, 0, err_flag_dev, stream);
  }
  if (dsa_sparse_attn_workspace_bytes(T, H, K) > kScratchBytes) return DSA_ERR_WORKSPACE;
  void* ws = nullptr;
  const int st = scratch_on_current_device(&ws);
  if (st != DSA_OK) return st;
  return dsa_sparse_attn_decode(q_bf16_dev, T, H, D, pool_dev, pool_rows, layout, kv_row_dim,
                                page_table_dev, B, max_pages, page_size, token_seq_dev, topk_dev, K,
                                sm_scale, o_bf16_dev, lse_dev, ws, kScratchBytes, err_flag_dev, stream);
}
