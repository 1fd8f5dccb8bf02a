// Device helpers shared by the library's kernels (sm_103a only).
#pragma once
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/dsa.h"

namespace dsa {

constexpr int kD = 512;          // latent width (kv_lora_rank, RoPE dim 0)
constexpr int kGroup = 128;      // dims per FP32 scale in the 528-byte row
constexpr int kRawRow = 512;
constexpr int kScaledRow = 528;
constexpr int kRopeRow = 656;    // 528-byte row + 64 BF16 RoPE dims
constexpr int kRopeDims = 64;

__device__ __forceinline__ void set_err(int32_t* flag, int bits) {
  if (flag != nullptr) atomicOr(flag, bits);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h16) {
  return __uint_as_float(h16 << 16);
}

// Two floats -> two E4M3 bytes with saturating round-to-nearest-even
// (cvt ... satfinite): result byte 0 <- lo, byte 1 <- hi.
__device__ __forceinline__ uint32_t e4m3x2_satrne(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Four floats -> 32-bit word of four E4M3 bytes (a in the low byte).
__device__ __forceinline__ uint32_t e4m3x4_satrne(float a, float b, float c, float d) {
  return e4m3x2_satrne(a, b) | (e4m3x2_satrne(c, d) << 16);
}

// Two E4M3 bytes (low 16 bits of v) -> two halves, exact (E4M3 is a subset of F16).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}

// Four E4M3 bytes of a 32-bit word -> four floats (exact).
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float out[4]) {
  uint32_t lo = e4m3x2_to_f16x2((uint16_t)(w & 0xFFFF));
  uint32_t hi = e4m3x2_to_f16x2((uint16_t)(w >> 16));
  __half2 l = *reinterpret_cast<__half2*>(&lo);
  __half2 h = *reinterpret_cast<__half2*>(&hi);
  float2 lf = __half22float2(l), hf = __half22float2(h);
  out[0] = lf.x; out[1] = lf.y; out[2] = hf.x; out[3] = hf.y;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Resolve top-k entry idx of token t to a physical row, or -1 when masked
// (negative index, or out of range: then an error bit is set).
__device__ __forceinline__ int64_t resolve_row(int32_t idx, const int32_t* __restrict__ page_table,
                                               int B, int max_pages, int page_size, int seq,
                                               int64_t pool_rows, int32_t* err) {
  if (idx < 0) return -1;
  if (page_table == nullptr) {
    if ((int64_t)idx >= pool_rows) { set_err(err, DSA_DEV_ERR_INDEX_RANGE); return -1; }
    return idx;
  }
  if (seq < 0 || seq >= B) { set_err(err, DSA_DEV_ERR_PAGE_RANGE); return -1; }
  int page = idx / page_size;
  int off = idx - page * page_size;
  if (page >= max_pages) { set_err(err, DSA_DEV_ERR_INDEX_RANGE); return -1; }
  int32_t phys = __ldg(page_table + (int64_t)seq * max_pages + page);
  if (phys < 0) { set_err(err, DSA_DEV_ERR_PAGE_RANGE); return -1; }
  int64_t row = (int64_t)phys * page_size + off;
  if (row >= pool_rows) { set_err(err, DSA_DEV_ERR_PAGE_RANGE); return -1; }
  return row;
}

}  // namespace dsa
