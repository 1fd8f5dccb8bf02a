// Launch plan and workspace layout of the persistent attention kernel.  Units
// (token, head group) whose tiles span two or more CTAs leave normalised
// partial results in the workspace; combine_kernel merges them.
#include "dsa_common.cuh"
#include "kernels.h"

namespace dsa {
// One persistent CTA per SM (fewer when there are fewer tiles than SMs).
AttnPlan plan_attn(int T, int H, int K, int sms, bool rope) {
  AttnPlan p{};
  if (T <= 0 || H <= 0 || K <= 0 || sms <= 0) return p;
  p.hg = head_group(H, rope);
  p.hgs = H / p.hg;
  p.tpt = (K + 127) / 128;
  p.n_tiles = (int64_t)T * p.hgs * p.tpt;
  p.grid = (int)(p.n_tiles < sms ? p.n_tiles : sms);
  for (int k = 1; k < p.grid && !p.split; ++k) p.split = tile_begin(k, p.n_tiles, p.grid) % p.tpt != 0;
  auto align = [](size_t x) { return (x + 255) / 256 * 256; };
  size_t end = 0;
  if (p.split) {
    p.ws_o_offset = 0;
    p.ws_lse_offset = align(p.ws_o_offset + (size_t)p.grid * 2 * p.hg * kD * sizeof(float));
    end = p.ws_lse_offset + (size_t)p.grid * 2 * p.hg * sizeof(float);
  }
  p.ws_bytes = end;
  return p;
}

}  // namespace dsa
