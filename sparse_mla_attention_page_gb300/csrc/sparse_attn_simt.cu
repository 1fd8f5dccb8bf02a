// Sparse MLA attention, first correct version on CUDA cores (FP32 FMA).
//
// Grid (split, token, head group of HG heads), 256 threads.  Each CTA walks its
// chunk of the token's top-k list in tiles of 32 entries: resolve rows through
// the page table, gather each row once (one warp per row, 16 bytes per lane,
// coalesced), score it against all HG queries, online softmax per head, then
// P*V from the row bytes kept in shared memory.  The row is both key and
// value (absorbed NoPE latent).  Partial results of a split go to the
// workspace and are merged by combine_kernel.
#include <atomic>
#include <cfloat>
#include <cuda_bf16.h>

#include "dsa_common.cuh"
#include "kernels.h"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 32;

template <int HG>
struct SimtSmem {
  float q[HG][kD];
  __align__(16) uint8_t kv[kTile][kD];
  float sc[kTile][4];
  int64_t row[kTile];
  float p[HG][kTile];
  float m[HG], l[HG], alpha[HG];
};

template <int HG, bool kScaled, bool kQ8>
__global__ void __launch_bounds__(kThreads) sparse_attn_simt_kernel(AttnArgs a) {
  constexpr int kHeadsPerThread = HG / 4;
  const int split = blockIdx.x, t = blockIdx.y, h0 = blockIdx.z * HG;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row_bytes = kScaled ? kScaledRow : kRawRow;

  extern __shared__ __align__(16) uint8_t smem_raw[];
  SimtSmem<HG>& sm = *reinterpret_cast<SimtSmem<HG>*>(smem_raw);
  auto& q_s = sm.q;
  auto& kv_s = sm.kv;
  auto& sc_s = sm.sc;
  auto& row_s = sm.row;
  auto& p_s = sm.p;
  auto& m_s = sm.m;
  auto& l_s = sm.l;
  auto& alpha_s = sm.alpha;

  for (int i = tid; i < HG * kD; i += kThreads) {
    const int h = i / kD, d = i % kD;
    const int64_t off = ((int64_t)t * a.H + h0 + h) * kD + d;
    float v;
    if (kQ8) {
      const uint8_t b = static_cast<const uint8_t*>(a.q)[off];
      float f[4];
      e4m3x4_to_f32(b, f);
      v = f[0] * a.q_scale[(int64_t)t * a.H + h0 + h];
    } else {
      v = bf16_bits_to_f32(static_cast<const uint16_t*>(a.q)[off]);
    }
    q_s[h][d] = v;
  }
  if (tid < HG) {
    m_s[tid] = -INFINITY;
    l_s[tid] = 0.f;
  }
  const int d8 = tid & 63, hq = tid >> 6;
  float acc[kHeadsPerThread][8];
#pragma unroll
  for (int i = 0; i < kHeadsPerThread; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;

  const int seq = a.token_seq ? __ldg(a.token_seq + t) : 0;
  const int k_begin = split * a.chunk;
  const int k_end = min(a.K, k_begin + a.chunk);
  __syncthreads();

  for (int kt = k_begin; kt < k_end; kt += kTile) {
    if (tid < kTile) {
      const int j = kt + tid;
      int64_t row = -1;
      if (j < k_end)
        row = resolve_row(__ldg(a.topk + (int64_t)t * a.K + j), a.page_table, a.B, a.max_pages,
                          a.page_size, seq, a.pool_rows, a.err);
      row_s[tid] = row;
    }
    __syncthreads();

    for (int jj = 0; jj < kTile / 8; ++jj) {
      const int j = warp * (kTile / 8) + jj;
      const int64_t row = row_s[j];
      if (row >= 0) {
        const uint8_t* rp = a.pool + row * row_bytes;
        const uint4 raw = *reinterpret_cast<const uint4*>(rp + lane * 16);
        *reinterpret_cast<uint4*>(&kv_s[j][lane * 16]) = raw;
        float kf[16];
        e4m3x4_to_f32(raw.x, kf);
        e4m3x4_to_f32(raw.y, kf + 4);
        e4m3x4_to_f32(raw.z, kf + 8);
        e4m3x4_to_f32(raw.w, kf + 12);
        if (kScaled) {
          const float sc = *reinterpret_cast<const float*>(rp + kD + 4 * (lane / 8));
#pragma unroll
          for (int i = 0; i < 16; ++i) kf[i] *= sc;
          if (lane < 4) sc_s[j][lane] = *reinterpret_cast<const float*>(rp + kD + 4 * lane);
        }
#pragma unroll 4
        for (int h = 0; h < HG; ++h) {
          float part = 0.f;
#pragma unroll
          for (int i = 0; i < 16; ++i) part = fmaf(q_s[h][lane * 16 + i], kf[i], part);
          part = warp_sum(part);
          if (lane == 0) p_s[h][j] = part * a.sm_scale;
        }
      } else {
        *reinterpret_cast<uint4*>(&kv_s[j][lane * 16]) = make_uint4(0, 0, 0, 0);
        if (kScaled && lane < 4) sc_s[j][lane] = 0.f;
        if (lane < HG) p_s[lane][j] = -INFINITY;
      }
    }
    __syncthreads();

    for (int h = warp; h < HG; h += kThreads / 32) {
      const float s = p_s[h][lane];
      const float mx = warp_max(s);
      const float m_old = m_s[h];
      const float m_new = fmaxf(m_old, mx);
      float alpha = 1.f, p = 0.f;
      if (m_new != -INFINITY) {
        alpha = expf(m_old - m_new);
        p = expf(s - m_new);
      }
      const float sum = warp_sum(p);
      p_s[h][lane] = p;
      if (lane == 0) {
        m_s[h] = m_new;
        l_s[h] = l_s[h] * alpha + sum;
        alpha_s[h] = alpha;
      }
    }
    __syncthreads();

#pragma unroll
    for (int i = 0; i < kHeadsPerThread; ++i) {
      const float al = alpha_s[hq + 4 * i];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[i][e] *= al;
    }
    for (int j = 0; j < kTile; ++j) {
      const uint2 raw = *reinterpret_cast<const uint2*>(&kv_s[j][d8 * 8]);
      float kf[8];
      e4m3x4_to_f32(raw.x, kf);
      e4m3x4_to_f32(raw.y, kf + 4);
      if (kScaled) {
        const float sc = sc_s[j][(d8 * 8) / kGroup];
#pragma unroll
        for (int e = 0; e < 8; ++e) kf[e] *= sc;
      }
#pragma unroll
      for (int i = 0; i < kHeadsPerThread; ++i) {
        const float p = p_s[hq + 4 * i][j];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(p, kf[e], acc[i][e]);
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < kHeadsPerThread; ++i) {
    const int h = hq + 4 * i;
    const float l = l_s[h];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse = l > 0.f ? m_s[h] + logf(l) : -INFINITY;
    const int64_t th = (int64_t)t * a.H + h0 + h;
    if (a.n_splits == 1) {
      __nv_bfloat16 ob[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) ob[e] = __float2bfloat16_rn(acc[i][e] * inv);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.o) + th * kD + d8 * 8) =
          *reinterpret_cast<const uint4*>(ob);
      if (d8 == 0) a.lse[th] = lse;
    } else {
      float* dst = a.ws_o + ((int64_t)split * a.T * a.H + th) * kD + d8 * 8;
      *reinterpret_cast<float4*>(dst) = make_float4(acc[i][0] * inv, acc[i][1] * inv, acc[i][2] * inv, acc[i][3] * inv);
      *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[i][4] * inv, acc[i][5] * inv, acc[i][6] * inv, acc[i][7] * inv);
      if (d8 == 0) a.ws_lse[(int64_t)split * a.T * a.H + th] = lse;
    }
  }
}

template <int HG, bool kScaled, bool kQ8>
void launch_one(const AttnArgs& a, cudaStream_t stream) {
  dim3 grid(a.n_splits, a.T, a.H / HG);
  const int smem = (int)sizeof(SimtSmem<HG>);
  static std::atomic<uint64_t> configured{0};   // one bit per device ordinal
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    cudaFuncSetAttribute(sparse_attn_simt_kernel<HG, kScaled, kQ8>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    configured.fetch_or(bit);
  }
  sparse_attn_simt_kernel<HG, kScaled, kQ8><<<grid, kThreads, smem, stream>>>(a);
}

}  // namespace

void launch_sparse_attn(const AttnArgs& a, bool q8, cudaStream_t stream) {
  if (a.H >= 16) {
    if (q8) launch_one<16, false, true>(a, stream);
    else if (a.scaled) launch_one<16, true, false>(a, stream);
    else launch_one<16, false, false>(a, stream);
  } else {
    if (q8) launch_one<8, false, true>(a, stream);
    else if (a.scaled) launch_one<8, true, false>(a, stream);
    else launch_one<8, false, false>(a, stream);
  }
  if (a.n_splits > 1) launch_combine(a, stream);
}

int head_group(int H) { return H >= 16 ? 16 : 8; }

int max_chunk() { return 1 << 30; }

}  // namespace dsa
