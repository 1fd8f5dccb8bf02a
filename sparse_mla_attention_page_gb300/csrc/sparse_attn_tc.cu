// Sparse MLA attention on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// One CTA = (split s, token t, group of HG <= 32 heads).  It owns top-k entries
// [s*chunk, (s+1)*chunk) of token t:
//
//   prologue   all warps: FP8 query operand in shared memory; the chunk's
//              indices are translated through the page table and compacted
//              (masked and out-of-range entries dropped, order kept), so that
//              tiles of 128 rows are dense except for the last one.
//   producer   4 warps: gather each tile's 128 latent rows (512 B, plus the
//              16-byte scale word for 528-byte rows) with 16-byte cp.async
//              straight into a 128-byte-swizzled K-major tile; a stage is
//              complete when every producer's copies have landed
//              (cp.async.mbarrier.arrive.noinc).  Two stages in flight.
//   MMA        1 thread: S^T = K Q^T   (M = 128 rows, N = query columns, K = 512)
//              and, one tile behind, O^T += V^T P^T (M = 128 latent dims x 4,
//              N = 2*HG, K = 128 rows), both kind::f8f6f4 with FP32
//              accumulators in tensor memory.  The same shared-memory tile is
//              the K-major A operand of the first and the MN-major A operand
//              of the second (V = K: one absorbed NoPE latent row).
//   softmax    4 warps, one thread per tile row (= TMEM lane): combines the
//              score columns, masks, reduces the tile max per head across the
//              128 rows, updates a lazy running max (rescaling O in TMEM only
//              when the max grows by more than 2^8), forms p = 2^(s - m),
//              accumulates the denominators and writes P as an FP8 operand.
//
// Exact FP8 operands for BF16 data: a BF16 query q is split per head into
// hi = e4m3(q * 2^a) and lo = e4m3((q * 2^a - hi) * 16) with a power-of-two
// 2^a; hi + lo/16 reproduces q * 2^a exactly (8 significant bits), so
// S = K.hi + K.lo/16 loses nothing but FP32 accumulation order.  P is split
// into three FP8 terms, p ~ hi + mid/16 + lo/256 (about 13 significant bits),
// because the output is a softmax-weighted sum of rows whose entries can be
// large while the sum cancels: two terms (8 bits) are not enough there.  For 528-byte rows the four
// group scales enter S per row (one accumulator per 128-dim group) and P per
// group (P_g = p * scale_g * 2^-e_g with a per-CTA power of two 2^e_g that
// bounds the chunk's scales), so the value rows never need dequantising.
#include <atomic>
#include <cuda_bf16.h>

#include "dsa_common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace dsa {
namespace {

using namespace tc;

constexpr int kRows = 128;          // top-k entries per tile = MMA M
constexpr int kStage = 65536;       // one tile: 128 rows x 512 FP8 bytes
constexpr int kMaxChunk = 2048;     // top-k entries one CTA can own
constexpr float kTau = 8.0f;        // lazy max threshold (log2 units)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kSoftmaxWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kProdWarp0 = 5;
constexpr int kProdWarps = 4;
constexpr int kThreads = 32 * (kSoftmaxWarps + 1 + kProdWarps);

template <int HG, bool kScaled, bool kQ8>
struct Cfg {
  static constexpr int G = kScaled ? 4 : 1;                    // score accumulators per tile
  static constexpr int NQ = kQ8 ? (HG < 16 ? 16 : HG) : 2 * HG;  // QK^T N (query operand rows)
  static constexpr int NP = (3 * HG + 15) / 16 * 16;          // PV N: P hi, mid, lo rows (+ zero pad)
  static constexpr int O_COLS = 4 * NP;
  static constexpr int GC = (G * NQ + O_COLS <= 512) ? G : G / 2;   // groups per QK^T chunk
  static constexpr int NQC = G / GC;                          // QK^T chunks per tile
  static constexpr int S_COLS = GC * NQ;
  static constexpr int NS = (2 * S_COLS + O_COLS <= 512) ? 2 : 1;
  static constexpr int O_COL0 = NS * S_COLS;
  static constexpr int USED = O_COL0 + O_COLS;
  static constexpr int TMEM_COLS =
      USED <= 32 ? 32 : USED <= 64 ? 64 : USED <= 128 ? 128 : USED <= 256 ? 256 : 512;
  static constexpr int NST = 2;                               // KV stages
  static constexpr int KV_OFF = 0;
  static constexpr int Q_OFF = KV_OFF + NST * kStage;
  static constexpr int P_OFF = Q_OFF + NQ * 512;
  static constexpr int SC_OFF = P_OFF + G * NP * 128;
  static constexpr int ROWS_OFF = SC_OFF + (kScaled ? NST * kRows * 16 : 0);
  static constexpr int MISC_OFF = ROWS_OFF + kMaxChunk * 4;
  static_assert(USED <= 512, "tensor memory budget");
  static_assert(Q_OFF % 1024 == 0 && P_OFF % 1024 == 0 && (NP * 128) % 1024 == 0, "operand alignment");
};

struct Misc {
  uint64_t kv_full[2];
  uint64_t kv_empty[2];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full;
  uint64_t o_done;
  uint64_t mma_final;
  uint32_t tmem_base;
  int abort;
  int n_valid;
  float red[2][4][32];
  float red2[4][32];
  float qsig[64];
  float gmax[kThreads / 32][4];
  float sc_pow[4], sc_inv[4];
  float linv[32], lse2[32];
};

template <int HG, bool kScaled, bool kQ8>
constexpr size_t smem_bytes() {
  return (size_t)Cfg<HG, kScaled, kQ8>::MISC_OFF + sizeof(Misc) + 1024;
}

// Byte offset of element (n, k) in a K-major operand of N rows whose K
// extent is split into 128-byte blocks (block-major), with the 128-byte
// swizzle: 16-byte chunk index XOR (row % 8).
template <int N>
__device__ __forceinline__ uint32_t kmajor_off(int n, int k) {
  return (k >> 7) * (N * 128) + (n >> 3) * 1024 + (n & 7) * 128 + ((((k >> 4) & 7) ^ (n & 7)) << 4) +
         (k & 15);
}

// Leaves in lane l the max (or sum) over the 32 lanes of v[l % N].
template <int N, bool kMax>
__device__ __forceinline__ float transpose_reduce(float (&v)[N], int lane) {
#pragma unroll
  for (int w = N / 2; w >= 1; w /= 2) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int k = 0; k < w; ++k) {
      const float send = upper ? v[k] : v[k + w];
      const float keep = upper ? v[k + w] : v[k];
      const float recv = __shfl_xor_sync(0xffffffffu, send, w);
      v[k] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
  float r = v[0];
#pragma unroll
  for (int off = N; off < 32; off *= 2) {
    const float o = __shfl_xor_sync(0xffffffffu, r, off);
    r = kMax ? fmaxf(r, o) : r + o;
  }
  return r;
}

__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t v16) {
  const uint32_t h = e4m3x2_to_f16x2((uint16_t)(v16 & 0xFFFFu));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

__device__ __forceinline__ void st_shared_u8(uint8_t* p, uint32_t v) {
  asm volatile("st.shared.u8 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

// ------------------------------------------------------------- prologue

// Query operand rows: decode -> [hi heads | lo heads] (exact split of BF16),
// Q8 -> the FP8 bytes (zero rows pad N to 16).  qsig[c] is the log2-domain
// multiplier of score column c (includes sm_scale and the power-of-two scale).
template <int HG, bool kScaled, bool kQ8>
__device__ void prepare_query(const AttnArgs& a, uint8_t* qop, Misc& ms, int t, int h0) {
  using C = Cfg<HG, kScaled, kQ8>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kWarps = kThreads / 32;
  const float base_sig = a.sm_scale * kLog2e;
  if (kQ8) {
    for (int n = warp; n < C::NQ; n += kWarps) {
      uint4 v = make_uint4(0, 0, 0, 0);
      float sig = 0.f;
      if (n < HG) {
        const int64_t th = (int64_t)t * a.H + h0 + n;
        v = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.q) + th * kD) + lane);
        sig = __ldg(a.q_scale + th) * base_sig;
      }
      *reinterpret_cast<uint4*>(qop + kmajor_off<C::NQ>(n, lane * 16)) = v;
      if (lane == 0) ms.qsig[n] = sig;
    }
    return;
  }
  for (int h = warp; h < HG; h += kWarps) {
    const int64_t th = (int64_t)t * a.H + h0 + h;
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) + th * kD + lane * 16);
    const uint4 u0 = __ldg(src), u1 = __ldg(src + 1);
    const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    float x[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
      x[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    amax = warp_max(amax);
    uint32_t hi[4] = {0, 0, 0, 0}, lo[4] = {0, 0, 0, 0};
    float sig = 0.f;
    if (amax > 0.f && amax <= 3.0e38f) {
      int e;
      const float f = frexpf(amax, &e);          // amax = f * 2^e, f in [0.5, 1)
      const int sh = (f <= 0.875f) ? 9 - e : 8 - e;   // largest sh with amax * 2^sh <= 448
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float y[4], r[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) y[k] = ldexpf(x[4 * i + k], sh);
        hi[i] = e4m3x4_satrne(y[0], y[1], y[2], y[3]);
        float yh[4];
        e4m3x4_to_f32(hi[i], yh);
#pragma unroll
        for (int k = 0; k < 4; ++k) r[k] = (y[k] - yh[k]) * 16.f;
        lo[i] = e4m3x4_satrne(r[0], r[1], r[2], r[3]);
      }
      sig = ldexpf(base_sig, -sh);
    }
    *reinterpret_cast<uint4*>(qop + kmajor_off<C::NQ>(h, lane * 16)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(qop + kmajor_off<C::NQ>(HG + h, lane * 16)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    if (lane == 0) {
      ms.qsig[h] = sig;
      ms.qsig[HG + h] = sig * 0.0625f;
    }
  }
}

// ------------------------------------------------------------------ roles

template <int HG, bool kScaled, bool kQ8>
__device__ void producer_role(const AttnArgs& a, uint8_t* sm, Misc& ms, int ntiles, int n_valid) {
  using C = Cfg<HG, kScaled, kQ8>;
  const int ptid = threadIdx.x - kProdWarp0 * 32;
  const int pw = ptid >> 5, lane = ptid & 31;
  const int32_t* rows = reinterpret_cast<const int32_t*>(sm + C::ROWS_OFF);
  constexpr int R = kScaled ? kScaledRow : kRawRow;
  volatile int* abort = &ms.abort;
  const uint32_t kv0 = smem_u32(sm + C::KV_OFF);
  for (int i = 0; i < ntiles; ++i) {
    const int stage = i % C::NST;
    if (i >= C::NST && !mbar_wait(smem_u32(&ms.kv_empty[stage]), ((i / C::NST) - 1) & 1, abort)) break;
    const uint32_t base = kv0 + stage * kStage;
#pragma unroll
    for (int rg = 0; rg < 4; ++rg) {
      const int r = 32 * pw + 8 * rg + (lane & 7);
      const int e = i * kRows + r;
      const int32_t row = rows[e < n_valid ? e : 0];
      const uint8_t* src = a.pool + (int64_t)row * R;
      const uint32_t dst_row = base + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
      for (int cg = 0; cg < 8; ++cg) {
        const int c = 4 * cg + (lane >> 3);   // 16-byte chunk 0..31 of the row
        cp_async_16(dst_row + (c >> 3) * 16384 + ((((c & 7) ^ (r & 7))) << 4), src + c * 16);
      }
    }
    if (kScaled) {
      const int e = i * kRows + ptid;
      const int32_t row = rows[e < n_valid ? e : 0];
      cp_async_16(smem_u32(sm + C::SC_OFF + stage * kRows * 16 + ptid * 16),
                  a.pool + (int64_t)row * kScaledRow + kD);
    }
    cp_async_arrive_noinc(smem_u32(&ms.kv_full[stage]));
  }
  cp_async_wait_all();
}

template <int HG, bool kScaled, bool kQ8>
__device__ void mma_role(uint8_t* sm, Misc& ms, uint32_t tmem, int ntiles) {
  using C = Cfg<HG, kScaled, kQ8>;
  if ((threadIdx.x & 31) != 0) return;
  volatile int* abort = &ms.abort;
  const uint32_t kv0 = smem_u32(sm + C::KV_OFF);
  const uint32_t q0 = smem_u32(sm + C::Q_OFF);
  const uint32_t p0 = smem_u32(sm + C::P_OFF);
  constexpr uint32_t kIdQK = idesc_e4m3(C::NQ, false);
  constexpr uint32_t kIdPV = idesc_e4m3(C::NP, true);
  for (int i = 0; i <= ntiles; ++i) {
    if (i < ntiles) {
      const int stage = i % C::NST;
      if (!mbar_wait(smem_u32(&ms.kv_full[stage]), (i / C::NST) & 1, abort)) break;
      fence_proxy_async_smem();   // rows landed through cp.async (generic proxy)
      const uint32_t a_base = kv0 + stage * kStage;
      bool stop = false;
#pragma unroll
      for (int qc = 0; qc < C::NQC; ++qc) {
        const int u = i * C::NQC + qc, sb = u % C::NS;
        if (u >= C::NS && !mbar_wait(smem_u32(&ms.s_free[sb]), ((u / C::NS) - 1) & 1, abort)) {
          stop = true;
          break;
        }
        tc_fence_after();
        const uint32_t d_base = tmem + sb * C::S_COLS;
        constexpr int kSteps = kScaled ? 4 * C::GC : 16;   // K = 32 per step
#pragma unroll
        for (int st = 0; st < kSteps; ++st) {
          const int ks = qc * kSteps + st;                  // global K step, 0..15
          const int kb = ks >> 2, kk = ks & 3;
          const uint64_t ad = sdesc_sw128(a_base + kb * 16384 + kk * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(q0 + kb * (C::NQ * 128) + kk * 32, 16, 1024);
          const uint32_t d = d_base + (kScaled ? (kb - qc * C::GC) * C::NQ : 0);
          const uint32_t acc = kScaled ? (kk > 0 ? 1u : 0u) : (ks > 0 ? 1u : 0u);
          mma_e4m3(d, ad, bd, kIdQK, acc);
        }
        mma_commit(smem_u32(&ms.s_full[sb]));
      }
      if (stop) break;
    }
    if (i >= 1) {
      const int j = i - 1, stage = j % C::NST;
      if (!mbar_wait(smem_u32(&ms.p_full), j & 1, abort)) break;
      fence_proxy_async_smem();
      tc_fence_after();
      const uint32_t a_base = kv0 + stage * kStage;
#pragma unroll
      for (int db = 0; db < 4; ++db) {
#pragma unroll
        for (int js = 0; js < 4; ++js) {
          const uint64_t ad = sdesc_sw128(a_base + db * 16384 + js * 4096, 1024, 1024);
          const uint64_t bd = sdesc_sw128(p0 + (kScaled ? db * (C::NP * 128) : 0) + js * 32, 16, 1024);
          mma_e4m3(tmem + C::O_COL0 + db * C::NP, ad, bd, kIdPV, (j > 0 || js > 0) ? 1u : 0u);
        }
      }
      mma_commit(smem_u32(&ms.kv_empty[stage]));
      mma_commit(smem_u32(&ms.o_done));
    }
  }
  // every MMA of this CTA completes before the tensor memory is released
  mma_commit(smem_u32(&ms.mma_final));
  volatile int no_abort = 0;
  mbar_wait(smem_u32(&ms.mma_final), 0, &no_abort, 2000000000ull);
}

template <int HG, bool kScaled, bool kQ8>
__device__ void softmax_role(const AttnArgs& a, uint8_t* sm, Misc& ms, uint32_t tmem, int ntiles, int n_valid,
                             int t, int h0, int split) {
  using C = Cfg<HG, kScaled, kQ8>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = threadIdx.x;                            // tile row = TMEM lane
  const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
  volatile int* abort = &ms.abort;
  uint8_t* pbuf = sm + C::P_OFF;
  float m_run[HG], l_part[HG];
  float m_lane = -INFINITY;                               // running max of head `lane`
#pragma unroll
  for (int h = 0; h < HG; ++h) {
    m_run[h] = -INFINITY;
    l_part[h] = 0.f;
  }
  bool ok = true;
  for (int i = 0; i < ntiles; ++i) {
    const int stage = i % C::NST;
    float sc4[4] = {1.f, 1.f, 1.f, 1.f};
    if (kScaled) {
      if (!(ok = mbar_wait(smem_u32(&ms.kv_full[stage]), (i / C::NST) & 1, abort))) break;
      const float4 v = *reinterpret_cast<const float4*>(sm + C::SC_OFF + stage * kRows * 16 + row * 16);
      sc4[0] = v.x; sc4[1] = v.y; sc4[2] = v.z; sc4[3] = v.w;
    }
    float s2[HG];
#pragma unroll
    for (int h = 0; h < HG; ++h) s2[h] = 0.f;
#pragma unroll
    for (int qc = 0; qc < C::NQC; ++qc) {
      const int u = i * C::NQC + qc, sb = u % C::NS;
      if (!(ok = mbar_wait(smem_u32(&ms.s_full[sb]), (u / C::NS) & 1, abort))) break;
      tc_fence_after();
#pragma unroll
      for (int gl = 0; gl < C::GC; ++gl) {
        const int g = qc * C::GC + gl;
        const uint32_t cbase = lane_base + sb * C::S_COLS + gl * C::NQ;
#pragma unroll
        for (int c0 = 0; c0 < HG; c0 += 8) {
          uint32_t hi[8], lo[8];
          tmem_ld8(cbase + c0, hi);
          if (!kQ8) tmem_ld8(cbase + HG + c0, lo);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            float v = __uint_as_float(hi[k]) * ms.qsig[c0 + k];
            if (!kQ8) v = fmaf(__uint_as_float(lo[k]), ms.qsig[HG + c0 + k], v);
            s2[c0 + k] = kScaled ? fmaf(sc4[g], v, s2[c0 + k]) : v;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&ms.s_free[sb]));
    }
    if (!ok) break;
    if (i * kRows + row >= n_valid) {
#pragma unroll
      for (int h = 0; h < HG; ++h) s2[h] = -INFINITY;
    }
    // tile max per head over the 128 rows
    float tmp[HG];
#pragma unroll
    for (int h = 0; h < HG; ++h) tmp[h] = s2[h];
    const float wmax = transpose_reduce<HG, true>(tmp, lane);
    if (lane < HG) ms.red[i & 1][warp][lane] = wmax;
    named_bar_sync(1, 128);
    float tile_max = -INFINITY;
    if (lane < HG)
      tile_max = fmaxf(fmaxf(ms.red[i & 1][0][lane], ms.red[i & 1][1][lane]),
                       fmaxf(ms.red[i & 1][2][lane], ms.red[i & 1][3][lane]));
    const bool need = lane < HG && tile_max > m_lane + kTau;
    const unsigned rmask = __ballot_sync(0xffffffffu, need);
    float alpha_lane = 1.f;
    if (need) {
      alpha_lane = exp2f(m_lane - tile_max);
      m_lane = tile_max;
    }
    float alpha[HG];
#pragma unroll
    for (int h = 0; h < HG; ++h) alpha[h] = 1.f;
    if (rmask) {
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        m_run[h] = __shfl_sync(0xffffffffu, m_lane, h);
        alpha[h] = __shfl_sync(0xffffffffu, alpha_lane, h);
        l_part[h] *= alpha[h];
      }
    }
    float p[HG];
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      p[h] = exp2f(s2[h] - m_run[h]);
      l_part[h] += p[h];
    }
    // the previous tile's PV has finished: P buffer free, O stable
    if (i > 0 && !(ok = mbar_wait(smem_u32(&ms.o_done), (i - 1) & 1, abort))) break;
    tc_fence_after();
    if (i > 0 && rmask) {
#pragma unroll
      for (int db = 0; db < 4; ++db) {
#pragma unroll
        for (int c0 = 0; c0 < C::NP; c0 += 8) {
          const uint32_t ca = lane_base + C::O_COL0 + db * C::NP + c0;
          uint32_t v[8];
          tmem_ld8(ca, v);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 8; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha[(c0 + k) % HG]);
          tmem_st8(ca, v);
        }
      }
      tmem_wait_st();
    }
#pragma unroll
    for (int g = 0; g < C::G; ++g) {
      const float mul = kScaled ? sc4[g] * ms.sc_inv[g] : 1.f;
      uint8_t* pg = pbuf + g * (C::NP * 128);
#pragma unroll
      for (int h = 0; h < HG; h += 2) {
        const float v0 = p[h] * mul, v1 = p[h + 1] * mul;
        const uint32_t hi2 = e4m3x2_satrne(v0, v1);
        const float2 hf = e4m3x2_to_f32x2(hi2);
        const float r0 = (v0 - hf.x) * 16.f, r1 = (v1 - hf.y) * 16.f;
        const uint32_t mid2 = e4m3x2_satrne(r0, r1);
        const float2 mf = e4m3x2_to_f32x2(mid2);
        const uint32_t lo2 = e4m3x2_satrne((r0 - mf.x) * 16.f, (r1 - mf.y) * 16.f);
        st_shared_u8(pg + kmajor_off<C::NP>(h, row), hi2 & 0xFFu);
        st_shared_u8(pg + kmajor_off<C::NP>(h + 1, row), (hi2 >> 8) & 0xFFu);
        st_shared_u8(pg + kmajor_off<C::NP>(HG + h, row), mid2 & 0xFFu);
        st_shared_u8(pg + kmajor_off<C::NP>(HG + h + 1, row), (mid2 >> 8) & 0xFFu);
        st_shared_u8(pg + kmajor_off<C::NP>(2 * HG + h, row), lo2 & 0xFFu);
        st_shared_u8(pg + kmajor_off<C::NP>(2 * HG + h + 1, row), (lo2 >> 8) & 0xFFu);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    mbar_arrive(smem_u32(&ms.p_full));
  }

  // ---- epilogue: denominators, O normalisation, stores
  float tmp[HG];
#pragma unroll
  for (int h = 0; h < HG; ++h) tmp[h] = l_part[h];
  const float wsum = transpose_reduce<HG, false>(tmp, lane);
  if (lane < HG) ms.red2[warp][lane] = wsum;
  named_bar_sync(1, 128);
  if (warp == 0 && lane < HG) {
    const float l = (ms.red2[0][lane] + ms.red2[1][lane]) + (ms.red2[2][lane] + ms.red2[3][lane]);
    ms.linv[lane] = l > 0.f ? 1.f / l : 0.f;
    ms.lse2[lane] = l > 0.f ? m_lane + log2f(l) : -INFINITY;
  }
  named_bar_sync(1, 128);
  const bool have_o = ok && ntiles > 0 &&
                      mbar_wait(smem_u32(&ms.o_done), (ntiles - 1) & 1, abort);
  tc_fence_after();
  const int64_t TH = (int64_t)a.T * a.H;
#pragma unroll
  for (int db = 0; db < 4; ++db) {
    const int d = db * kRows + row;
    const float pw = kScaled ? ms.sc_pow[db] : 1.f;
#pragma unroll
    for (int c0 = 0; c0 < HG; c0 += 8) {
      float o[8];
      if (have_o) {
        uint32_t hi[8], mid[8], lo[8];
        const uint32_t ob = lane_base + C::O_COL0 + db * C::NP + c0;
        tmem_ld8(ob, hi);
        tmem_ld8(ob + HG, mid);
        tmem_ld8(ob + 2 * HG, lo);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float acc = fmaf(__uint_as_float(lo[k]), 0.00390625f,
                                 fmaf(__uint_as_float(mid[k]), 0.0625f, __uint_as_float(hi[k])));
          o[k] = acc * pw * ms.linv[c0 + k];
        }
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) o[k] = 0.f;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int64_t th = (int64_t)t * a.H + h0 + c0 + k;
        if (a.n_splits == 1)
          static_cast<__nv_bfloat16*>(a.o)[th * kD + d] = __float2bfloat16_rn(o[k]);
        else
          a.ws_o[((int64_t)split * TH + th) * kD + d] = o[k];
      }
    }
  }
  if (warp == 0 && lane < HG) {
    const int64_t th = (int64_t)t * a.H + h0 + lane;
    const float lse = ms.lse2[lane] * kLn2;
    if (a.n_splits == 1) a.lse[th] = lse;
    else a.ws_lse[(int64_t)split * TH + th] = lse;
  }
}

template <int HG, bool kScaled, bool kQ8>
__global__ void __launch_bounds__(kThreads, 1) sparse_attn_tc_kernel(const AttnArgs a) {
  using C = Cfg<HG, kScaled, kQ8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Misc& ms = *reinterpret_cast<Misc*>(sm + C::MISC_OFF);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, t = blockIdx.y, h0 = blockIdx.z * HG;
  const int k_begin = split * a.chunk;
  const int n_chunk = min(a.K, k_begin + a.chunk) - k_begin;
  int32_t* rows = reinterpret_cast<int32_t*>(sm + C::ROWS_OFF);

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&ms.kv_full[s]), kProdWarps * 32);
      mbar_init(smem_u32(&ms.kv_empty[s]), 1);
      mbar_init(smem_u32(&ms.s_full[s]), 1);
      mbar_init(smem_u32(&ms.s_free[s]), kSoftmaxWarps * 32);
    }
    mbar_init(smem_u32(&ms.p_full), kSoftmaxWarps * 32);
    mbar_init(smem_u32(&ms.o_done), 1);
    mbar_init(smem_u32(&ms.mma_final), 1);
    ms.abort = 0;
    mbar_init_fence();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&ms.tmem_base), C::TMEM_COLS);
    tmem_relinquish();
  }
  prepare_query<HG, kScaled, kQ8>(a, sm + C::Q_OFF, ms, t, h0);

  // translate the chunk's indices to physical rows (-1: masked)
  const int seq = a.token_seq ? __ldg(a.token_seq + t) : 0;
  for (int e = tid; e < n_chunk; e += kThreads) {
    const int32_t idx = __ldg(a.topk + (int64_t)t * a.K + k_begin + e);
    rows[e] = (int32_t)resolve_row(idx, a.page_table, a.B, a.max_pages, a.page_size, seq, a.pool_rows, a.err);
  }
  __syncthreads();
  // stable in-place compaction of the valid rows
  if (warp == 0) {
    int base = 0;
    for (int e0 = 0; e0 < n_chunk; e0 += 32) {
      const int e = e0 + lane;
      const int32_t r = e < n_chunk ? rows[e] : -1;
      const unsigned m = __ballot_sync(0xffffffffu, r >= 0);
      if (r >= 0) rows[base + __popc(m & ((1u << lane) - 1u))] = r;
      base += __popc(m);
      __syncwarp();
    }
    if (lane == 0) ms.n_valid = base;
  }
  __syncthreads();
  const int n_valid = ms.n_valid;
  if (kScaled) {
    // a power of two bounding each group's scales over the chunk
    float gm[4] = {0.f, 0.f, 0.f, 0.f};
    for (int e = tid; e < n_valid; e += kThreads) {
      const float4 s = __ldg(reinterpret_cast<const float4*>(a.pool + (int64_t)rows[e] * kScaledRow + kD));
      gm[0] = fmaxf(gm[0], fabsf(s.x));
      gm[1] = fmaxf(gm[1], fabsf(s.y));
      gm[2] = fmaxf(gm[2], fabsf(s.z));
      gm[3] = fmaxf(gm[3], fabsf(s.w));
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) gm[g] = warp_max(gm[g]);
    if (lane == 0) {
#pragma unroll
      for (int g = 0; g < 4; ++g) ms.gmax[warp][g] = gm[g];
    }
    __syncthreads();
    if (tid < 4) {
      float mx = 0.f;
      for (int w = 0; w < kThreads / 32; ++w) mx = fmaxf(mx, ms.gmax[w][tid]);
      int ex = 0;
      if (mx > 0.f && mx <= 3.0e38f) {
        const float f = frexpf(mx, &ex);
        if (f == 0.5f) ex -= 1;                  // 2^ex >= mx, tight
      }
      ms.sc_pow[tid] = ldexpf(1.f, ex);
      ms.sc_inv[tid] = ldexpf(1.f, -ex);
    }
  }
  // P operand starts zeroed: its padding rows (N rounded up to 16) stay zero
  for (int i = tid; i < C::G * C::NP * 8; i += kThreads)
    reinterpret_cast<uint4*>(sm + C::P_OFF)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;
  const int ntiles = (n_valid + kRows - 1) / kRows;

  if (warp < kSoftmaxWarps)
    softmax_role<HG, kScaled, kQ8>(a, sm, ms, tmem, ntiles, n_valid, t, h0, split);
  else if (warp == kMmaWarp)
    mma_role<HG, kScaled, kQ8>(sm, ms, tmem, ntiles);
  else
    producer_role<HG, kScaled, kQ8>(a, sm, ms, ntiles, n_valid);

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (tid == 0 && ms.abort) set_err(a.err, DSA_DEV_ERR_TIMEOUT);
}

template <int HG, bool kScaled, bool kQ8>
void launch_tc(const AttnArgs& a, cudaStream_t stream) {
  constexpr size_t smem = smem_bytes<HG, kScaled, kQ8>();
  static_assert(smem <= 232448, "shared memory budget");
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    cudaFuncSetAttribute(sparse_attn_tc_kernel<HG, kScaled, kQ8>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    configured.fetch_or(bit);
  }
  dim3 grid(a.n_splits, a.T, a.H / HG);
  sparse_attn_tc_kernel<HG, kScaled, kQ8><<<grid, kThreads, smem, stream>>>(a);
}

template <int HG>
void launch_hg(const AttnArgs& a, bool q8, cudaStream_t stream) {
  if (q8) launch_tc<HG, false, true>(a, stream);
  else if (a.scaled) launch_tc<HG, true, false>(a, stream);
  else launch_tc<HG, false, false>(a, stream);
}

}  // namespace

int head_group(int H) { return H < 32 ? H : 32; }

void launch_sparse_attn(const AttnArgs& a, bool q8, cudaStream_t stream) {
  const int hg = head_group(a.H);
  if (hg == 8) launch_hg<8>(a, q8, stream);
  else if (hg == 16) launch_hg<16>(a, q8, stream);
  else launch_hg<32>(a, q8, stream);
  if (a.n_splits > 1) launch_combine(a, stream);
}

int max_chunk() { return kMaxChunk; }

}  // namespace dsa
