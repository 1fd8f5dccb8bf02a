// Merge of split units: a unit (token, head group) whose tiles the persistent
// attention grid spread over CTAs c0..c1 left one normalised partial per CTA
// (O_c, LSE_c).  Here LSE = logsumexp_c LSE_c and O = sum_c exp(LSE_c - LSE) O_c,
// folded part by part with a running maximum.
//
// One block per (CTA boundary, 256 of the unit's hg x 128 four-dim groups);
// the first boundary that falls inside a unit merges it.  The kernel is
// launched as a programmatic dependent of the attention kernel: its blocks
// take SMs as attention CTAs exit and wait for the whole attention grid
// (griddepcontrol.wait) before reading any partial.
#include <cuda_bf16.h>

#include "dsa_common.cuh"
#include "kernels.h"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 4;            // parts whose loads are issued together

__global__ void __launch_bounds__(kThreads) combine_kernel(const AttnArgs a) {
  // The block's unit and parts, worked out once by one thread (64-bit
  // divisions: issued by every thread they made the kernel instruction-bound).
  __shared__ int64_t s_th0;                // output row of the unit's first head
  __shared__ int s_c0, s_c1, s_slot0;      // s_c0 < 0: nothing to merge here
  if (threadIdx.x == 0) {
    const int k = blockIdx.x + 1;
    const int64_t bk = tile_begin(k, a.n_tiles, a.grid);
    const int64_t u0 = bk / a.tpt * a.tpt;
    int c0 = -1, c1 = -1, slot0 = 0;
    // a boundary inside a unit, and the first such boundary of that unit
    if (bk != u0 && !(k >= 2 && tile_begin(k - 1, a.n_tiles, a.grid) > u0)) {
      c0 = cta_of_tile(u0, a.n_tiles, a.grid);
      c1 = cta_of_tile(u0 + a.tpt - 1, a.n_tiles, a.grid);
      // slot 0 of a CTA holds the unit its range starts in, slot 1 its last
      // unit: the unit is the last one of CTA c0 unless its range starts at u0,
      // and the first one of every later CTA
      slot0 = 2 * c0 + (tile_begin(c0, a.n_tiles, a.grid) < u0 ? 1 : 0);
    }
    const int64_t u = u0 / a.tpt;
    const int t = (int)(u / a.hgs);
    s_th0 = (int64_t)t * a.H + (int)(u - (int64_t)t * a.hgs) * a.hg;
    s_c0 = c0;
    s_c1 = c1;
    s_slot0 = slot0;
  }
  __syncthreads();
  const int c0 = s_c0, c1 = s_c1;
  if (c0 < 0) return;
  const int item = blockIdx.y * kThreads + threadIdx.x;
  const int h = item / (kD / 4), d4 = item % (kD / 4);
  asm volatile("griddepcontrol.wait;" ::: "memory");               // every partial is written
  float m = -INFINITY, sum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int cb = c0; cb <= c1; cb += kBatch) {
    float ls[kBatch];
    float4 v[kBatch];
#pragma unroll
    for (int p = 0; p < kBatch; ++p) {
      const int c = cb + p;
      ls[p] = -INFINITY;
      v[p] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c <= c1) {
        const int64_t sb = (int64_t)(c == c0 ? s_slot0 : 2 * c) * a.hg + h;
        ls[p] = __ldcg(a.ws_lse + sb);
        v[p] = __ldcg(reinterpret_cast<const float4*>(a.ws_o + sb * kD) + d4);
      }
    }
#pragma unroll
    for (int p = 0; p < kBatch; ++p) {
      if (ls[p] == -INFINITY) continue;                            // a part with no valid entry
      const float mn = fmaxf(m, ls[p]);
      const float r = expf(m - mn), w = expf(ls[p] - mn);
      sum = sum * r + w;
      acc.x = fmaf(w, v[p].x, acc.x * r);
      acc.y = fmaf(w, v[p].y, acc.y * r);
      acc.z = fmaf(w, v[p].z, acc.z * r);
      acc.w = fmaf(w, v[p].w, acc.w * r);
      m = mn;
    }
  }
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  uint2 packed;
  packed.x = *reinterpret_cast<uint32_t*>(&lo);
  packed.y = *reinterpret_cast<uint32_t*>(&hi);
  const int64_t th = s_th0 + h;
  reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.o) + th * kD)[d4] = packed;
  if (d4 == 0) a.lse[th] = sum > 0.f ? m + logf(sum) : -INFINITY;
}

}  // namespace

void launch_combine(const AttnArgs& a, cudaStream_t stream) {
  if (a.grid < 2) return;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.grid - 1, a.hg * (kD / 4) / kThreads);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, combine_kernel, a);
}

}  // namespace dsa
