// Fused BF16 -> E4M3 cast + paged scatter of new latent rows (raw 512-byte and
// group-scaled 528-byte layouts) and the per-(token, head) FP8 query quantiser.
//
// One warp per 512-dim row: lane l owns dims [8l, 8l+8) and [256+8l, 256+8l+8),
// so every load instruction of the warp reads 512 contiguous bytes of the BF16
// row and every store writes 256 contiguous bytes of the FP8 row.  HBM-bound:
// 1 KiB read + 512 (528) bytes written per row.
#include "dsa_common.cuh"
#include "kernels.h"

namespace dsa {
namespace {

struct Row16 {
  float v[16];  // v[0..7]: dims 8l..8l+7, v[8..15]: dims 256+8l..256+8l+7
};

__device__ __forceinline__ void load_row16(const uint16_t* __restrict__ row, int lane, Row16& r) {
  const uint4 a = __ldcs(reinterpret_cast<const uint4*>(row) + lane);
  const uint4 b = __ldcs(reinterpret_cast<const uint4*>(row + 256) + lane);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    r.v[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
    r.v[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
  }
}

// Four floats -> four E4M3 bytes (saturating round-to-nearest-even); a NaN
// input gives the FN NaN code 0x7F with the input's sign bit (the cvt
// instruction alone returns 0x7F for NaN of either sign).
__device__ __forceinline__ uint32_t e4m3x4_keep_nan_sign(float a, float b, float c, float d) {
  uint32_t r = e4m3x4_satrne(a, b, c, d);
  const float v[4] = {a, b, c, d};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (v[i] != v[i]) r = (r & ~(0xFFu << (8 * i))) | ((0x7Fu | ((__float_as_uint(v[i]) >> 31) << 7)) << (8 * i));
  return r;
}

__device__ __forceinline__ void store_row16(uint8_t* __restrict__ row, int lane, const Row16& r) {
  uint2 lo, hi;
  lo.x = e4m3x4_keep_nan_sign(r.v[0], r.v[1], r.v[2], r.v[3]);
  lo.y = e4m3x4_keep_nan_sign(r.v[4], r.v[5], r.v[6], r.v[7]);
  hi.x = e4m3x4_keep_nan_sign(r.v[8], r.v[9], r.v[10], r.v[11]);
  hi.y = e4m3x4_keep_nan_sign(r.v[12], r.v[13], r.v[14], r.v[15]);
  reinterpret_cast<uint2*>(row)[lane] = lo;
  reinterpret_cast<uint2*>(row + 256)[lane] = hi;
}

// The KV writers let the next kernel in the stream, when it is launched as a
// programmatic dependent (the attention kernels are), start its set-up at
// once: it waits for this whole grid to complete before it reads anything.
// (The query quantiser does not: there the early start made a Q8 prefill step
// about 50 us slower, measured.)
__device__ __forceinline__ void allow_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__global__ void __launch_bounds__(256, 4) kv_write_raw_kernel(
    const uint16_t* __restrict__ x, int64_t n_rows, const int64_t* __restrict__ slots,
    uint8_t* __restrict__ pool, int64_t pool_rows, int32_t* err) {
  allow_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  auto put = [&](int64_t s, const Row16& r) {
    if (s < 0) return;
    if (s >= pool_rows) {
      if (lane == 0) set_err(err, DSA_DEV_ERR_SLOT_RANGE);
      return;
    }
    store_row16(pool + s * kRawRow, lane, r);
  };
  // two rows per warp and pass: both slots and both rows are loaded before
  // either is used, so a pass costs one load round trip
  for (int64_t i0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; i0 < n_rows; i0 += 2 * nwarps) {
    const int64_t i1 = i0 + nwarps;
    const bool two = i1 < n_rows;
    const int64_t s0 = __ldg(slots + i0);
    const int64_t s1 = two ? __ldg(slots + i1) : -1;
    Row16 r0, r1;
    load_row16(x + i0 * kD, lane, r0);
    if (two) load_row16(x + i1 * kD, lane, r1);
    put(s0, r0);
    if (two) put(s1, r1);
  }
}

// Group g of 128 dims is held by 16 lanes: groups 0 and 2 by lanes 0-15
// (first and second half of their registers), groups 1 and 3 by lanes 16-31.
// kRope: 656-byte rows, whose input rows are 576 wide; the 64 RoPE dims are
// stored as they are (BF16) after the scales, one 4-byte pair per lane.
template <bool kRope>
__global__ void __launch_bounds__(256, 4) kv_write_scaled_kernel(
    const uint16_t* __restrict__ x, int64_t n_rows, const int64_t* __restrict__ slots,
    uint8_t* __restrict__ pool, int64_t pool_rows, int32_t* err) {
  allow_dependents();
  constexpr int kIn = kRope ? kD + kRopeDims : kD;
  constexpr int kRowBytes = kRope ? kRopeRow : kScaledRow;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  auto put = [&](int64_t s, Row16& r, uint32_t rope_pair) {
    if (s < 0) return;
    if (s >= pool_rows) {
      if (lane == 0) set_err(err, DSA_DEV_ERR_SLOT_RANGE);
      return;
    }
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      a0 = fmaxf(a0, fabsf(r.v[k]));
      a1 = fmaxf(a1, fabsf(r.v[8 + k]));
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
      a0 = fmaxf(a0, __shfl_xor_sync(0xffffffffu, a0, o));
      a1 = fmaxf(a1, __shfl_xor_sync(0xffffffffu, a1, o));
    }
    const float s0 = a0 == 0.f ? 0.f : __fdiv_rn(a0, 448.0f);
    const float s1 = a1 == 0.f ? 0.f : __fdiv_rn(a1, 448.0f);
    // copysignf: the same quotient (s > 0), and a NaN keeps its input's sign
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      r.v[k] = s0 == 0.f ? 0.f : copysignf(__fdiv_rn(r.v[k], s0), r.v[k]);
      r.v[8 + k] = s1 == 0.f ? 0.f : copysignf(__fdiv_rn(r.v[8 + k], s1), r.v[8 + k]);
    }
    uint8_t* row = pool + s * kRowBytes;
    store_row16(row, lane, r);
    if (kRope) reinterpret_cast<uint32_t*>(row + kScaledRow)[lane] = rope_pair;
    const float g1 = __shfl_sync(0xffffffffu, s0, 16);
    const float g3 = __shfl_sync(0xffffffffu, s1, 16);
    if (lane == 0) {
      float4 sc = make_float4(s0, g1, s1, g3);
      *reinterpret_cast<float4*>(row + 512) = sc;
    }
  };
  // two rows per warp and pass, all loads issued before any is used
  for (int64_t i0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; i0 < n_rows; i0 += 2 * nwarps) {
    const int64_t i1 = i0 + nwarps;
    const bool two = i1 < n_rows;
    const int64_t s0 = __ldg(slots + i0);
    const int64_t s1 = two ? __ldg(slots + i1) : -1;
    Row16 r0, r1;
    load_row16(x + i0 * kIn, lane, r0);
    if (two) load_row16(x + i1 * kIn, lane, r1);
    uint32_t p0 = 0, p1 = 0;
    if (kRope) {
      p0 = __ldg(reinterpret_cast<const uint32_t*>(x + i0 * kIn + kD) + lane);
      if (two) p1 = __ldg(reinterpret_cast<const uint32_t*>(x + i1 * kIn + kD) + lane);
    }
    put(s0, r0, p0);
    if (two) put(s1, r1, p1);
  }
}

__global__ void __launch_bounds__(256, 4) quantize_q8_kernel(
    const uint16_t* __restrict__ q, int64_t n_vec, uint8_t* __restrict__ q8, float* __restrict__ scale) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  auto put = [&](int64_t i, Row16& r) {
    float a = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) a = fmaxf(a, fabsf(r.v[k]));
    a = warp_max(a);
    const float s = a == 0.f ? 0.f : __fdiv_rn(a, 448.0f);
#pragma unroll
    for (int k = 0; k < 16; ++k) r.v[k] = s == 0.f ? 0.f : copysignf(__fdiv_rn(r.v[k], s), r.v[k]);
    store_row16(q8 + i * kD, lane, r);
    if (lane == 0) scale[i] = s;
  };
  // two vectors per warp and pass, both loaded before either is used
  for (int64_t i0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; i0 < n_vec; i0 += 2 * nwarps) {
    const int64_t i1 = i0 + nwarps;
    const bool two = i1 < n_vec;
    Row16 r0, r1;
    load_row16(q + i0 * kD, lane, r0);
    if (two) load_row16(q + i1 * kD, lane, r1);
    put(i0, r0);
    if (two) put(i1, r1);
  }
}

// Two rows per warp and pass, eight warps per block; at most one wave of
// four blocks per SM (the kernels are built for four resident blocks).
int writer_grid(int64_t n_rows, int sms) {
  const int64_t rows_per_block = 16;
  int64_t blocks = (n_rows + rows_per_block - 1) / rows_per_block;
  const int64_t cap = (int64_t)sms * 4;
  if (blocks > cap) blocks = cap;
  return (int)(blocks < 1 ? 1 : blocks);
}

}  // namespace

void launch_kv_write(int layout, const void* x, int64_t n_rows, const int64_t* slots, void* pool,
                     int64_t pool_rows, int32_t* err, int sms, cudaStream_t stream) {
  const int grid = writer_grid(n_rows, sms);
  if (layout == DSA_KV_ROPE656)
    kv_write_scaled_kernel<true><<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(x), n_rows, slots,
                                                           static_cast<uint8_t*>(pool), pool_rows, err);
  else if (layout == DSA_KV_SCALED528)
    kv_write_scaled_kernel<false><<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(x), n_rows, slots,
                                                            static_cast<uint8_t*>(pool), pool_rows, err);
  else
    kv_write_raw_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(x), n_rows, slots,
                                                  static_cast<uint8_t*>(pool), pool_rows, err);
}

void launch_quantize_q8(const void* q, int64_t n_vec, void* q8, float* scale, int sms,
                        cudaStream_t stream) {
  quantize_q8_kernel<<<writer_grid(n_vec, sms), 256, 0, stream>>>(
      static_cast<const uint16_t*>(q), n_vec, static_cast<uint8_t*>(q8), scale);
}

}  // namespace dsa
