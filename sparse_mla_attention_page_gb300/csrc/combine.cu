// Split-K plan and merge of per-split partial results.
#include <cuda_bf16.h>

#include "dsa_common.cuh"
#include "kernels.h"

namespace dsa {
namespace {

// Merge split-K partials: LSE = logsumexp_s LSE_s, O = sum_s exp(LSE_s - LSE) O_s.
__global__ void __launch_bounds__(128) combine_kernel(AttnArgs a) {
  const int64_t th = blockIdx.x;
  const int64_t TH = (int64_t)a.T * a.H;
  float m = -INFINITY;
  for (int s = 0; s < a.n_splits; ++s) m = fmaxf(m, a.ws_lse[s * TH + th]);
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  float lse = -INFINITY;
  if (m != -INFINITY) {
    float sum = 0.f;
    for (int s = 0; s < a.n_splits; ++s) sum += expf(a.ws_lse[s * TH + th] - m);
    lse = m + logf(sum);
    for (int s = 0; s < a.n_splits; ++s) {
      const float ls = a.ws_lse[s * TH + th];
      if (ls == -INFINITY) continue;
      const float w = expf(ls - lse);
      const float4 v = reinterpret_cast<const float4*>(a.ws_o + (s * TH + th) * kD)[threadIdx.x];
      o.x = fmaf(w, v.x, o.x);
      o.y = fmaf(w, v.y, o.y);
      o.z = fmaf(w, v.z, o.z);
      o.w = fmaf(w, v.w, o.w);
    }
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(o.x, o.y), hi = __floats2bfloat162_rn(o.z, o.w);
  uint2 packed;
  packed.x = *reinterpret_cast<uint32_t*>(&lo);
  packed.y = *reinterpret_cast<uint32_t*>(&hi);
  reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.o) + th * kD)[threadIdx.x] = packed;
  if (threadIdx.x == 0) a.lse[th] = lse;
}

}  // namespace

// Each (token, head group) has K/128 tiles of top-k entries.  Choose the
// number of splits that minimises an estimated makespan: waves of CTAs over
// the SMs times (tiles per split + a fixed per-CTA start-up cost of about
// two tiles), subject to the per-CTA chunk limit of the attention kernel.
SplitPlan plan_splits(int T, int H, int K, int sms) {
  SplitPlan p{1, K, 0, 0};
  if (T <= 0 || H <= 0 || K <= 0 || sms <= 0) return p;
  const int64_t units = (int64_t)T * (H / head_group(H));
  const int tiles = (K + 127) / 128;
  const int min_splits = (K + max_chunk() - 1) / max_chunk();
  int64_t best_cost = -1;
  for (int n = min_splits < 1 ? 1 : min_splits; n <= tiles; ++n) {
    const int chunk_tiles = (tiles + n - 1) / n;
    const int n_eff = (tiles + chunk_tiles - 1) / chunk_tiles;
    const int64_t waves = (units * n_eff + sms - 1) / sms;
    const int64_t cost = waves * (chunk_tiles + 2);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      p.chunk = chunk_tiles * 128;
      p.n_splits = n_eff;
    }
  }
  if (p.n_splits > 1) {
    const size_t o_bytes = (size_t)p.n_splits * T * H * kD * sizeof(float);
    p.ws_lse_offset = (o_bytes + 255) / 256 * 256;
    p.ws_bytes = p.ws_lse_offset + (size_t)p.n_splits * T * H * sizeof(float);
  }
  return p;
}

void launch_combine(const AttnArgs& a, cudaStream_t stream) {
  combine_kernel<<<(unsigned)((int64_t)a.T * a.H), 128, 0, stream>>>(a);
}

}  // namespace dsa
