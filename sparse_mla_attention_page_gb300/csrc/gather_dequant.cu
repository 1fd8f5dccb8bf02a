// Gather / dequantise reader: the rows a top-k list selects, dequantised to
// BF16 in a buffer padded to one slot per top-k entry, for consumers that
// attend in BF16 ("[DSA] Support group-scaled FP8 NoPE KV reads for CUDA
// TileLang", Modifications: the gather/cast reader; "[DSA] Support
// flashmla_sparse_q8 prefill backend on CUDA", review thread: the paged
// gather with -1 padding).  Slot e = t*K + j gets
//   out[e][d] = bf16_rn(fp32(e4m3(b_d) * s_g))   (raw rows: s = 1, exact)
// and idx_out[e] = e, or -1 when the entry is masked (out[e] untouched).
//
// Bandwidth-bound: each warp resolves 32 consecutive entries (one per lane)
// and then copies their rows four at a time, lane l converting bytes
// [16 l, 16 l + 16) of a row (16-byte loads, 32-byte stores, whole rows per
// warp instruction); grids are multiples of the SM count.
#include <cuda_bf16.h>

#include "dsa_common.cuh"
#include "kernels.h"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsInFlight = 4;

__global__ void __launch_bounds__(kThreads) gather_dequant_kernel(const GatherArgs g) {
  const int lane = threadIdx.x & 31;
  const int64_t n = (int64_t)g.T * g.K;
  const int64_t warp0 = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t n_warps = ((int64_t)gridDim.x * kThreads) >> 5;
  const int64_t R = g.scaled ? kScaledRow : kRawRow;
  for (int64_t base = warp0 * 32; base < n; base += n_warps * 32) {
    const int64_t e = base + lane;
    int64_t row = -1;
    if (e < n) {
      const int t = (int)(e / g.K);
      const int seq = g.token_seq ? __ldg(g.token_seq + t) : 0;
      row = resolve_row(__ldg(g.topk + e), g.page_table, g.B, g.max_pages, g.page_size, seq, g.pool_rows, g.err);
      g.idx_out[e] = row >= 0 ? (int32_t)e : -1;
    }
#pragma unroll 1
    for (int r0 = 0; r0 < 32; r0 += kRowsInFlight) {
      int64_t rr[kRowsInFlight];
      uint4 v[kRowsInFlight];
      float s[kRowsInFlight];
#pragma unroll
      for (int k = 0; k < kRowsInFlight; ++k) {
        rr[k] = __shfl_sync(0xffffffffu, row, r0 + k);
        v[k] = make_uint4(0, 0, 0, 0);
        s[k] = 1.f;
        if (rr[k] >= 0) {
          const uint8_t* src = g.pool + rr[k] * R;
          v[k] = __ldg(reinterpret_cast<const uint4*>(src) + lane);
          if (g.scaled) s[k] = __ldg(reinterpret_cast<const float*>(src + kD) + (lane * 16) / kGroup);
        }
      }
#pragma unroll
      for (int k = 0; k < kRowsInFlight; ++k) {
        if (rr[k] < 0) continue;
        const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float f[4];
          e4m3x4_to_f32(w[i], f);
          __nv_bfloat162 lo = __floats2bfloat162_rn(f[0] * s[k], f[1] * s[k]);
          __nv_bfloat162 hi = __floats2bfloat162_rn(f[2] * s[k], f[3] * s[k]);
          o[2 * i] = *reinterpret_cast<uint32_t*>(&lo);
          o[2 * i + 1] = *reinterpret_cast<uint32_t*>(&hi);
        }
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(g.out) + (base + r0 + k) * kD) + 2 * lane;
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
  }
}

}  // namespace

void launch_gather_dequant(const GatherArgs& g, int sms, cudaStream_t stream) {
  const int64_t n = (int64_t)g.T * g.K;
  const int64_t chunks = (n + 31) / 32;
  const int64_t want = (chunks + kThreads / 32 - 1) / (kThreads / 32);
  const int64_t cap = (int64_t)sms * 8;              // 8 blocks of 8 warps per SM
  const unsigned blocks = (unsigned)(want < cap ? want : cap);
  gather_dequant_kernel<<<blocks, kThreads, 0, stream>>>(g);
}

}  // namespace dsa
