// Gather / dequantise reader: the rows a top-k list selects, dequantised to
// BF16 in a workspace for consumers that attend in BF16 ("[DSA] Support
// group-scaled FP8 NoPE KV reads for CUDA TileLang", Modifications: the full
// and paged readers, the selected-row workspace with remapped indices and
// kept masks, bounded by min(physical rows, selected entries) rows; "[DSA]
// Support flashmla_sparse_q8 prefill backend on CUDA", review thread: the
// paged gather with -1 padding).
//
//   selected branch  (T*K < pool_rows): out[e] = dequant(row of entry e),
//                    idx_out[e] = e;
//   full-pool branch (T*K >= pool_rows): out[r] = dequant(physical row r)
//                    for every r, idx_out[e] = physical row of entry e;
//   masked entries:  idx_out[e] = -1 (selected branch: out[e] untouched).
// dequant(row)[d] = bf16_rn(fp32(e4m3(b_d) * s_g)) (raw rows: s = 1, exact);
// 656-byte rows append their 64 BF16 RoPE dims (576-wide output rows).
//
// Bandwidth-bound.  Work is cut into chunks of 32 rows or entries, one chunk
// per warp at a time: a warp resolves up to 32 (source row, destination row)
// pairs, one per lane, and then copies the rows four at a time, lane l
// converting bytes [16 l, 16 l + 16) of a row (16-byte loads, 32-byte stores,
// whole rows per warp instruction).  In the full-pool branch the chunks are
// the pool's rows (source = destination) followed by the top-k entries (index
// translation only).  Grids are multiples of the SM count.
#include <cuda_bf16.h>

#include "dsa_common.cuh"
#include "kernels.h"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsInFlight = 4;

template <int kLayout>
__global__ void __launch_bounds__(kThreads) gather_dequant_kernel(const GatherArgs g) {
  constexpr int64_t R = kLayout == DSA_KV_RAW512 ? kRawRow : kLayout == DSA_KV_SCALED528 ? kScaledRow : kRopeRow;
  constexpr int kW = kLayout == DSA_KV_ROPE656 ? kD + kRopeDims : kD;   // output row width (BF16)
  const int lane = threadIdx.x & 31;
  const int64_t n_sel = (int64_t)g.T * g.K;
  const int64_t row_chunks = g.full_pool ? (g.pool_rows + 31) / 32 : 0;
  const int64_t n_chunks = row_chunks + (n_sel + 31) / 32;
  const int64_t warp0 = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t n_warps = ((int64_t)gridDim.x * kThreads) >> 5;
  for (int64_t c = warp0; c < n_chunks; c += n_warps) {
    int64_t src = -1, dst = -1;
    if (c < row_chunks) {                    // full pool: every physical row, in place
      const int64_t r = c * 32 + lane;
      if (r < g.pool_rows) src = dst = r;
    } else {
      const int64_t e = (c - row_chunks) * 32 + lane;
      if (e < n_sel) {
        const int t = (int)(e / g.K);
        const int seq = g.token_seq ? __ldg(g.token_seq + t) : 0;
        const int64_t row =
            resolve_row(__ldg(g.topk + e), g.page_table, g.B, g.max_pages, g.page_size, seq, g.pool_rows, g.err);
        if (g.full_pool) {
          g.idx_out[e] = (int32_t)row;       // -1 where masked
        } else {
          g.idx_out[e] = row >= 0 ? (int32_t)e : -1;
          if (row >= 0) {
            src = row;
            dst = e;
          }
        }
      }
    }
    if (__ballot_sync(0xffffffffu, src >= 0) == 0) continue;
#pragma unroll 1
    for (int r0 = 0; r0 < 32; r0 += kRowsInFlight) {
      int64_t rs[kRowsInFlight], rd[kRowsInFlight];
      uint4 v[kRowsInFlight], rv[kRowsInFlight];
      float s[kRowsInFlight];
#pragma unroll
      for (int k = 0; k < kRowsInFlight; ++k) {
        rs[k] = __shfl_sync(0xffffffffu, src, r0 + k);
        rd[k] = __shfl_sync(0xffffffffu, dst, r0 + k);
        v[k] = make_uint4(0, 0, 0, 0);
        rv[k] = make_uint4(0, 0, 0, 0);
        s[k] = 1.f;
        if (rs[k] >= 0) {
          const uint8_t* p = g.pool + rs[k] * R;
          v[k] = __ldg(reinterpret_cast<const uint4*>(p) + lane);
          if (kLayout != DSA_KV_RAW512) s[k] = __ldg(reinterpret_cast<const float*>(p + kD) + (lane * 16) / kGroup);
          if (kLayout == DSA_KV_ROPE656 && lane < 8) rv[k] = __ldg(reinterpret_cast<const uint4*>(p + kScaledRow) + lane);
        }
      }
#pragma unroll
      for (int k = 0; k < kRowsInFlight; ++k) {
        if (rs[k] < 0) continue;
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
        uint16_t* out_row = static_cast<uint16_t*>(g.out) + rd[k] * kW;
        uint4* dst4 = reinterpret_cast<uint4*>(out_row) + 2 * lane;
        dst4[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst4[1] = make_uint4(o[4], o[5], o[6], o[7]);
        if (kLayout == DSA_KV_ROPE656 && lane < 8) reinterpret_cast<uint4*>(out_row + kD)[lane] = rv[k];
      }
    }
  }
}

}  // namespace

int64_t gather_rows(int64_t pool_rows, int64_t n_selected) {
  return n_selected < pool_rows ? n_selected : pool_rows;
}

void launch_gather_dequant(const GatherArgs& g, int sms, cudaStream_t stream) {
  const int64_t n_sel = (int64_t)g.T * g.K;
  const int64_t chunks = (g.full_pool ? (g.pool_rows + 31) / 32 : 0) + (n_sel + 31) / 32;
  const int64_t want = (chunks + kThreads / 32 - 1) / (kThreads / 32);
  const int64_t cap = (int64_t)sms * 8;              // 8 blocks of 8 warps per SM
  const unsigned blocks = (unsigned)(want < cap ? want : cap);
  if (g.layout == DSA_KV_ROPE656)
    gather_dequant_kernel<DSA_KV_ROPE656><<<blocks, kThreads, 0, stream>>>(g);
  else if (g.layout == DSA_KV_SCALED528)
    gather_dequant_kernel<DSA_KV_SCALED528><<<blocks, kThreads, 0, stream>>>(g);
  else
    gather_dequant_kernel<DSA_KV_RAW512><<<blocks, kThreads, 0, stream>>>(g);
}

}  // namespace dsa
