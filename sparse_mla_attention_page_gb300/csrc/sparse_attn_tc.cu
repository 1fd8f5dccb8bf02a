// Sparse MLA attention on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// Persistent kernel: one CTA per SM walks a contiguous range of 128-entry tiles
// of the global work list (unit = token x group of HG <= 32 heads; a unit's
// top-k list is tpt tiles).  Consecutive tiles of one unit form a segment;
// each segment ends with an epilogue that writes the unit's O and LSE (or a
// partial result when the unit spans CTAs).  Warp roles (24 warps):
//
//   index      1 warp: translates each tile's 128 top-k entries through the
//              page table into physical rows (top-k entries fetched three
//              tiles ahead, page-table reads one tile ahead, so no load
//              latency sits between tiles), publishes them in a ring of
//              kRing tiles for the producers; nothing ties it to the stages,
//              so it runs up to kRing tiles ahead of them.
//   producer   5 warps: publish a stage's valid-entry bits once the stage is
//              free, then gather each tile's rows with 16-byte cp.async into
//              the 128-byte-swizzled K-major tile, four rows x 128 bytes per
//              warp instruction (whole 128-byte lines), zero-filling masked
//              entries (source size 0: no memory read); 656-byte rows also
//              bring their 128-byte RoPE part into a tile of its own; a stage
//              is complete when every producer thread's copies have landed
//              (cp.async.mbarrier.arrive.noinc).  (Row gathers through the
//              tensor memory accelerator, tile::gather4, are issue-bound and
//              ran slower than cp.async here.)
//   QK^T       1 thread: S^T = K Q^T (M = 128 rows, N = query columns,
//              K = 512) per score chunk, kind::f8f6f4 with FP32 accumulators
//              in tensor memory; over 656-byte rows four kind::f16 MMAs per
//              tile add the BF16 RoPE scores K_rope Q_rope^T in extra columns.
//   PV         1 thread: O^T += V^T P^T (M = 128 latent dims x 4, N = P
//              columns, K = 128 rows).  The same shared-memory tile is the
//              K-major A operand of QK^T and the MN-major A operand of PV
//              (V = K: one absorbed NoPE latent row).  Two issuing threads
//              keep the tensor pipe fed while either one waits for its inputs.
//   softmax    16 warps, four per TMEM lane quarter, each thread one tile row
//              (= TMEM lane) and a quarter of the heads: combine the score
//              columns, mask, keep a lazy running max (one barrier with an
//              OR reduction asks whether any row exceeds its head's running
//              max by more than 2^8; only then are the per-head tile maxima
//              across the 128 rows formed and O in TMEM rescaled; 528-byte
//              rows, which also track the group-scale exponents, form them
//              every tile), form p = 2^(s - m), accumulate the denominators,
//              write P as an FP8 operand, build each segment's query operand
//              in shared memory (loads issued a tile ahead), and at the end of
//              a segment normalise O and store it (a unit whose tiles span
//              CTAs leaves a normalised partial O and LSE per CTA;
//              combine_kernel, launched right behind as a programmatic
//              dependent, merges them).
//
// FP8 operands for BF16 data: a BF16 query q is split per head into
// hi = e4m3(q * 2^a) and lo = e4m3((q * 2^a - hi) * 16) with a power-of-two
// 2^a placing the head's amax at the top of the E4M3 range; hi + lo/16
// reproduces q * 2^a exactly (8 significant bits) for every element within
// about 2^15 of the amax (smaller ones fall into the E4M3 subnormals and keep
// fewer bits, below 2^-15 of the largest term), so S = K.hi + K.lo/16 loses
// little beyond FP32 accumulation order.  P is split into three FP8 terms,
// p ~ hi + mid/16 + lo/256 (the FP16 value of p, 11 significant bits), because
// the output is a softmax-weighted sum of rows whose entries can be large
// while the sum cancels: two terms (8 bits, relative error up to 2^-8) broke
// the tolerance once rows held entries beyond about 20 (measured).  For
// 528-byte rows the four group scales enter S per row (one accumulator per
// 128-dim group) and P per group (P_g = p * scale_g * 2^-E_g, E_g a running
// power of two bounding the segment's scales), so value rows are never
// dequantised in shared memory.
#include <atomic>
#include <cstddef>
#include <cuda_bf16.h>

#include "dsa_common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace dsa {
namespace {

using namespace tc;

constexpr int kRows = 128;          // top-k entries per tile = MMA M
constexpr int kStage = 65536;       // one tile: 128 rows x 512 FP8 bytes
constexpr float kTau = 8.0f;        // lazy max threshold (log2 units)
constexpr float kNoMax = -1.0e30f;  // running max of a head with no valid entry yet (finite, so
                                    // 2^(s - m) needs no guard: masked s = -inf gives 0)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kSmxWarps = 16;       // softmax warps: warp w -> lane quarter w % 4, head quarter w / 4
constexpr int kSmxThreads = kSmxWarps * 32;
constexpr int kQkWarp = 16;         // issues QK^T
constexpr int kPvWarp = 17;         // issues PV
constexpr int kIdxWarp = 18;
constexpr int kProdWarp0 = 19;
constexpr int kProdWarps = 5;       // row gathers from L2/HBM scale with the warps issuing them
constexpr int kThreads = 32 * (kSmxWarps + 3 + kProdWarps);   // + QK, PV and index warps
constexpr int kQuads = kRows / 4;   // producer work unit: 4 rows (one warp instruction per 128-byte piece)
constexpr int kQuadsPerProd = (kQuads + kProdWarps - 1) / kProdWarps;
// registers per thread: the launch gives every thread 80 (768 threads, one CTA
// per SM, 24 warps of 10 x 256 registers); the four softmax warpgroups then take
// Cfg::SMX_REGS and the two others give back down to Cfg::OTHER_REGS, the two
// adding up to the launch's 61440 exactly
constexpr int kLaunchRegs = 80;
static_assert(kThreads == 768 && kSmxThreads == 512, "register split assumes 768 threads");
static_assert(kProdWarps >= 4, "scale words are fetched by four producer warps");
constexpr int kRing = 4;            // tiles of translated rows kept ahead of the producers
constexpr int kScStage = kRows * 16;   // scale words of one tile (528-byte rows)
constexpr int kSmemLimit = 232448;
constexpr int kMiscBytes = 6144;

struct Misc {
  uint64_t kv_full[3];
  uint64_t kv_empty[3];
  uint64_t meta_full[3];
  uint64_t idx_full[kRing];
  uint64_t idx_free[kRing];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t q_full[2];         // a segment's query operand is built (by the softmax warps)
  uint64_t p_full[2];         // P buffer b written (and O rescaled) by every softmax thread
  uint64_t pv_done[2];        // PV of the tiles that used P buffer b has completed
  uint64_t mma_final[2];      // drain of the QK^T and the PV issuer
  uint32_t tmem_base;
  int abort;
  uint8_t vflag[3][kRows];    // valid-entry flag of each row of each stage's tile
  __align__(16) int32_t ring[kRing][kRows];   // physical row of each entry (-1: masked)
  float red[2][4][4][8];      // [tile parity][head quarter][lane quarter][head] tile maxima
  float red_sc[2][4][4];      // [tile parity][lane quarter][group] maxima of the group scales
  float red2[4][4][8];        // [head quarter][lane quarter][head] denominators (epilogue)
  __align__(16) float qsig[2][64];   // log2-domain multiplier of each score column, per query buffer
  float linv[32], lse2[32];
};
static_assert(sizeof(Misc) <= kMiscBytes, "misc area");
static_assert(offsetof(Misc, ring) % 16 == 0 && offsetof(Misc, qsig) % 16 == 0, "vector access alignment");

template <int HG, bool kScaled, bool kQ8, bool kRope>
struct Cfg {
  static constexpr int HPT = HG / 4;                           // heads per softmax thread
  // P (and O) column order: with 8 heads a thread and unscaled rows, its
  // three terms are 24 adjacent columns (head quarter q: columns 24 q + 8 term
  // + head % 8), so a row of P goes out in one 16-byte and one 8-byte store;
  // otherwise column term * HG + head (measured: the interleaved order saved
  // 1.4 % on the FP8-query prefill and cost 0.6-1.8 % on 528-byte rows)
  static constexpr bool kPInter = HPT == 8 && !kScaled;
  static constexpr int G = kScaled ? 4 : 1;                    // score accumulators per tile
  // BF16 queries over 528-byte rows at 32 heads: the hi and lo halves of the
  // query are two K ranges of one N = HG operand (S = K.hi + K.lo in one
  // accumulator), not 2 HG columns, so that two groups' scores share a chunk
  static constexpr bool kHalvesK = kScaled && !kQ8 && !kRope && HG == 32;
  static constexpr int NQ = kQ8 ? (HG < 16 ? 16 : HG) : kHalvesK ? HG : 2 * HG;  // QK^T N (query operand rows)
  static constexpr int NP = (3 * HG + 15) / 16 * 16;          // PV N: P hi, mid, lo rows (+ zero pad)
  static constexpr int O_COLS = 4 * NP;
  // 656-byte rows: the RoPE part of the scores, S_rope = K_rope Q_rope^T (BF16
  // MMAs, N = NR query rows), accumulated in NR more columns of each score buffer
  static constexpr int NR = kRope ? (HG < 16 ? 16 : HG) : 0;
  // groups per QK^T chunk: the widest chunk for which two score buffers fit
  // beside O (so QK^T of the next chunk overlaps the read-out of this one),
  // else the widest that fits once
  static constexpr int GC = (2 * (G * NQ + NR) + O_COLS <= 512)       ? G
                            : (G >= 2 && 2 * (G / 2 * NQ + NR) + O_COLS <= 512) ? G / 2
                            : (G >= 4 && 2 * (G / 4 * NQ + NR) + O_COLS <= 512) ? G / 4
                            : (G * NQ + NR + O_COLS <= 512)             ? G
                                                                        : G / 2;
  static constexpr int NQC = G / GC;                          // QK^T chunks per tile
  static constexpr int S_COLS = GC * NQ + NR;
  static constexpr int NS = (2 * S_COLS + O_COLS <= 512) ? 2 : 1;
  static constexpr int O_COL0 = NS * S_COLS;
  static constexpr int USED = O_COL0 + O_COLS;
  static constexpr int TMEM_COLS =
      USED <= 32 ? 32 : USED <= 64 ? 64 : USED <= 128 ? 128 : USED <= 256 ? 256 : 512;
  static constexpr int Q_BYTES = NQ * 512 * (kHalvesK ? 2 : 1);
  static constexpr int P_BYTES = G * NP * 128;
  static constexpr int ROPE_STAGE = kRope ? kRows * 128 : 0;   // RoPE parts of a tile: 128 rows x 128 B
  static constexpr int QR_BYTES = NR * 128;                    // RoPE query operand
  static constexpr int STAGE = kStage + (kScaled ? kScStage : 0) + ROPE_STAGE;
  static constexpr int FIXED = kMiscBytes + 1024;             // + alignment slack
  // shared memory: three KV stages and two P buffers if they fit; else, with
  // one score group, three stages and one P buffer (the softmax forms P in
  // registers and waits for the previous PV only to store it); else two P
  // buffers; then a second query buffer
  static constexpr bool kFit3x2 = 3 * STAGE + Q_BYTES + 2 * P_BYTES + FIXED <= kSmemLimit;
  static constexpr bool kFit3x1 = G == 1 && 3 * STAGE + Q_BYTES + P_BYTES + FIXED <= kSmemLimit;
  static constexpr int NPB = kFit3x2 ? 2 : kFit3x1 ? 1 : (2 * STAGE + Q_BYTES + 2 * P_BYTES + FIXED <= kSmemLimit) ? 2 : 1;
  static constexpr int NST = (3 * STAGE + Q_BYTES + NPB * P_BYTES + FIXED <= kSmemLimit) ? 3 : 2;
  static constexpr int NQB =
      (NST * STAGE + 2 * (Q_BYTES + QR_BYTES) + NPB * P_BYTES + FIXED <= kSmemLimit) ? 2 : 1;
  static constexpr int KV_OFF = 0;
  static constexpr int Q_OFF = KV_OFF + NST * kStage;
  static constexpr int QR_OFF = Q_OFF + NQB * Q_BYTES;
  static constexpr int P_OFF = QR_OFF + NQB * QR_BYTES;
  static constexpr int ROPE_OFF = P_OFF + NPB * P_BYTES;
  static constexpr int SC_OFF = ROPE_OFF + NST * ROPE_STAGE;
  static constexpr int MISC_OFF = SC_OFF + (kScaled ? NST * kScStage : 0);
  static constexpr int SMEM = MISC_OFF + kMiscBytes + 1024;
  // softmax / other warpgroups' registers a thread (measured spill-free or least
  // spilling split per instantiation; the two add up to 256)
  static constexpr int SMX_REGS = HG <= 16 ? 88 : 96;
  static constexpr int OTHER_REGS = (kLaunchRegs * kThreads - SMX_REGS * kSmxThreads) / (kThreads - kSmxThreads);
  static_assert(HPT >= 2 && HPT <= 8, "heads per softmax thread");
  static_assert(USED <= 512, "tensor memory budget");
  static_assert(SMEM <= kSmemLimit, "shared memory budget");
  static_assert(Q_OFF % 1024 == 0 && P_OFF % 1024 == 0 && (NP * 128) % 1024 == 0, "operand alignment");
  static_assert(QR_OFF % 1024 == 0 && ROPE_OFF % 1024 == 0 && QR_BYTES % 1024 == 0, "RoPE operand alignment");
  static_assert(!kRope || (kScaled && !kQ8 && HG <= 16), "656-byte rows: BF16 queries, at most 16 heads");
};

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

// Three E4M3 terms of a pair of P values, p ~ hi + mid / 16 + lo / 256,
// formed in half precision: p is rounded to FP16 (11 significant bits) once;
// each residual (p - hi) * 16 is then exact in FP16, so the three terms (4
// significant bits each) represent the FP16 value exactly (bar saturation).
// About half the instructions of the same split in FP32.
__device__ __forceinline__ void split3_f16(float v0, float v1, uint32_t& hi2, uint32_t& mid2, uint32_t& lo2) {
  uint32_t p, t, r, r2;
  uint16_t h;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(p) : "f"(v1), "f"(v0));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(h) : "r"(p));
  hi2 = h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(t) : "h"(h));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(p), "r"(t));
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(r), "r"(0x4C004C00u));   // x 16
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(h) : "r"(r));
  mid2 = h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(t) : "h"(h));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r2) : "r"(r), "r"(t));
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r2) : "r"(r2), "r"(0x4C004C00u));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(h) : "r"(r2));
  lo2 = h;
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"((uint16_t)v) : "memory");
}
__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_shared_v2(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Byte offset of P column n (query column: head x term), tile row k in the
// PV B operand: MN-major without swizzle, core matrices of 8 rows x 16
// columns (128 bytes); the NP / 16 core matrices of one 8-row group are
// adjacent, so groups of 8 rows lie NP * 8 bytes apart.
template <int NP>
__device__ __forceinline__ uint32_t p_off(int n, int k) {
  return (n >> 4) * 128 + (k >> 3) * (NP * 8) + (k & 7) * 16 + (n & 15);
}

// 16-byte copy; bytes beyond src_bytes (0 or 16) are zero-filled and not read.
__device__ __forceinline__ void cp_async_16_zfill(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}

// Smallest power of two >= x (x > 0, finite), as an exponent.
__device__ __forceinline__ int ceil_log2(float x) {
  int e;
  const float f = frexpf(x, &e);     // x = f * 2^e, f in [0.5, 1)
  return f == 0.5f ? e - 1 : e;
}

// x * 2^e exactly for |e| up to 252 (two in-range power-of-two factors).
__device__ __forceinline__ float scale_pow2(float x, int e) {
  const int e1 = e / 2, e2 = e - e1;
  return __fmul_rn(__fmul_rn(x, __int_as_float((127 + e1) << 23)), __int_as_float((127 + e2) << 23));
}

// One arrival per warp on `bar`, after every lane's prior accesses (the
// caller fences them for the proxy they feed first): mbarriers fed by whole
// thread groups would otherwise take one serialised shared-memory atomic per
// thread.
__device__ __forceinline__ void warp_arrive(uint32_t bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Warp-uniform bounded wait (all lanes agree on the outcome).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort, uint64_t limit_ns) {
  const bool ok = mbar_wait(bar, parity, abort, limit_ns);
  return __all_sync(0xffffffffu, ok);
}

// Position of a CTA's tiles in the work list, advanced one tile at a time
// (no 64-bit division per tile): unit = t * hgs + hgi, tile within the unit.
struct TileCursor {
  int64_t unit;
  int tile, t, hgi;
  __device__ __forceinline__ TileCursor(const AttnArgs& a, int64_t g) {
    unit = g / a.tpt;
    tile = (int)(g - unit * a.tpt);
    t = (int)(unit / a.hgs);
    hgi = (int)(unit - (int64_t)t * a.hgs);
  }
  __device__ __forceinline__ void advance(const AttnArgs& a) {
    if (++tile == a.tpt) {
      tile = 0;
      ++unit;
      if (++hgi == a.hgs) {
        hgi = 0;
        ++t;
      }
    }
  }
  // first / last tile of a segment (the unit's tiles inside this CTA)
  __device__ __forceinline__ bool first(int it) const { return it == 0 || tile == 0; }
  __device__ __forceinline__ bool last(const AttnArgs& a, int it, int n_it) const {
    return it == n_it - 1 || tile == a.tpt - 1;
  }
};

// ------------------------------------------------------------ query operand

// The QK^T B operand of one unit (token t, heads h0 .. h0 + HG - 1), built by
// the softmax threads straight into a query buffer: K-major with the
// 128-byte swizzle, and the log2-domain multiplier of each score column.
// BF16 queries: rows [hi heads | lo heads], the exact two-term FP8 split
// hi = e4m3(q 2^sh), lo = e4m3((q 2^sh - hi) 16) with a power of two 2^sh per
// head; with kHalvesK the rows are the heads and lo = e4m3(q 2^sh - hi) sits
// at K offset 512 of the same row (exact while the residual is an E4M3
// normal, for elements within about 2^10 of the head's amax; smaller ones
// keep fewer bits, below 2^-18 of the amax).  FP8 queries: the bytes as they
// are, multiplier q_scale (rows past HG stay zero).  Thread -> head tid / TPH,
// dims [DPT (tid % TPH), + DPT).
template <int HG, bool kQ8, bool kRope, bool kHalvesK>
struct QueryBuild {
  static constexpr int kThr = kSmxThreads < 32 * HG ? kSmxThreads : 32 * HG;   // threads that build
  static constexpr int TPH = kThr / HG;                   // threads per head (one warp at most)
  static constexpr int DPT = kD / TPH;                    // dims per thread
  static constexpr int NV = kQ8 ? DPT / 16 : DPT / 8;     // 16-byte loads per thread
  static constexpr int NR = kRope ? (HG < 16 ? 16 : HG) : 0;   // RoPE operand rows (zero past HG)
  uint4 v[NV];
  uint4 rv;                                               // RoPE: 8 dims of head tid / 8
  float qs;                                               // FP8 queries: q_scale of the head

  __device__ __forceinline__ void load(const AttnArgs& a, int t, int h0) {
    const int head = threadIdx.x / TPH, part = threadIdx.x % TPH;
    if (threadIdx.x < kThr) {        // whole warps
      const int64_t th = (int64_t)t * a.H + h0 + head;
      const uint4* src = kQ8 ? reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.q) + th * kD + part * DPT)
                             : reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) + th * a.q_row + part * DPT);
#pragma unroll
      for (int i = 0; i < NV; ++i) v[i] = __ldg(src + i);
      qs = kQ8 ? __ldg(a.q_scale + th) : 0.f;
    }
    if constexpr (kRope) {
      const int rh = threadIdx.x >> 3, rc = threadIdx.x & 7;   // head, 16-byte chunk of its 64 dims
      rv = make_uint4(0, 0, 0, 0);
      if (rh < HG) {
        const uint16_t* qr = static_cast<const uint16_t*>(a.q) + ((int64_t)t * a.H + h0 + rh) * a.q_row + kD;
        rv = __ldg(reinterpret_cast<const uint4*>(qr) + rc);
      }
    }
  }

  // Writes the operand into qbuf (NQ rows), the multipliers into qsig and,
  // for 656-byte rows, the BF16 RoPE operand (NR rows x 64 dims) into rbuf.
  template <int NQ>
  __device__ __forceinline__ void store(const AttnArgs& a, uint8_t* qbuf, float* qsig, uint8_t* rbuf) const {
    const int head = threadIdx.x / TPH, part = threadIdx.x % TPH;
    const float base_sig = a.sm_scale * kLog2e;
    if constexpr (kRope) {
      const int rh = threadIdx.x >> 3, rc = threadIdx.x & 7;
      if (rh < NR)
        *reinterpret_cast<uint4*>(rbuf + (rh >> 3) * 1024 + (rh & 7) * 128 + ((rc ^ (rh & 7)) << 4)) = rv;
    }
    if (threadIdx.x >= kThr) return;   // whole warps
    if constexpr (kQ8) {
#pragma unroll
      for (int i = 0; i < NV; ++i) *reinterpret_cast<uint4*>(qbuf + kmajor_off<NQ>(head, part * DPT + 16 * i)) = v[i];
      if (part == 0) qsig[head] = qs * base_sig;
    } else {
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_f32(w[j] & 0xFFFFu)), fabsf(bf16_bits_to_f32(w[j] >> 16))));
      }
#pragma unroll
      for (int off = TPH / 2; off >= 1; off /= 2) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      int sh = 0;
      float sig = 0.f;
      const bool live = amax > 0.f && amax <= 3.0e38f;
      if (live) {
        int e;
        const float f = frexpf(amax, &e);                // amax = f * 2^e, f in [0.5, 1)
        sh = (f <= 0.875f) ? 9 - e : 8 - e;              // largest sh with amax * 2^sh <= 448
        sig = scale_pow2(base_sig, -sh);
      }
#pragma unroll
      for (int c = 0; c < NV / 2; ++c) {                  // 16 dims per chunk
        uint32_t hi[4] = {0, 0, 0, 0}, lo[4] = {0, 0, 0, 0};
        if (live) {
          const uint32_t w[8] = {v[2 * c].x, v[2 * c].y, v[2 * c].z, v[2 * c].w,
                                 v[2 * c + 1].x, v[2 * c + 1].y, v[2 * c + 1].z, v[2 * c + 1].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float y[4], r[4], yh[4];
            y[0] = scale_pow2(bf16_bits_to_f32(w[2 * i] & 0xFFFFu), sh);
            y[1] = scale_pow2(bf16_bits_to_f32(w[2 * i] >> 16), sh);
            y[2] = scale_pow2(bf16_bits_to_f32(w[2 * i + 1] & 0xFFFFu), sh);
            y[3] = scale_pow2(bf16_bits_to_f32(w[2 * i + 1] >> 16), sh);
            hi[i] = e4m3x4_satrne(y[0], y[1], y[2], y[3]);
            e4m3x4_to_f32(hi[i], yh);
#pragma unroll
            for (int j = 0; j < 4; ++j) r[j] = kHalvesK ? y[j] - yh[j] : (y[j] - yh[j]) * 16.f;
            lo[i] = e4m3x4_satrne(r[0], r[1], r[2], r[3]);
          }
        }
        const int k0 = part * DPT + 16 * c;
        *reinterpret_cast<uint4*>(qbuf + kmajor_off<NQ>(head, k0)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        if constexpr (kHalvesK)   // lo = q 2^sh - hi at K offset 512 of the same row
          *reinterpret_cast<uint4*>(qbuf + kmajor_off<NQ>(head, kD + k0)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        else
          *reinterpret_cast<uint4*>(qbuf + kmajor_off<NQ>(HG + head, k0)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      if (part == 0) {
        qsig[head] = sig;
        if constexpr (!kHalvesK) qsig[HG + head] = sig * 0.0625f;
      }
    }
  }
};

// ------------------------------------------------------------------ roles

// Index warp of the FP8-query kernels: per tile, the physical rows of the 128
// top-k entries (lane l owns entries 4l .. 4l + 3) into the ring, starting
// after the CTA's set-up.  The BF16-query kernels use IndexWarp below, which
// starts its loads before the set-up; the two loops translate alike.  Both
// forms are kept because the early-start form, measured in the FP8-query
// kernels (a few hundred tiles a CTA, where the start is negligible), raised
// their instruction-cache misses several-fold and cost 3.5 %, while in the
// decode kernels (about seven tiles a CTA) it saves about 1 us a call.
template <int HG, bool kScaled, bool kQ8, bool kRope>
__device__ void index_role(const AttnArgs& a, uint8_t* sm, Misc& ms, int64_t b0, int n_it) {
  using C = Cfg<HG, kScaled, kQ8, kRope>;
  constexpr int kAhead = 3;
  const int lane = threadIdx.x & 31;
  volatile int* abort = &ms.abort;
  int4 win[kAhead];           // top-k entries of tiles it + 1 .. it + kAhead (after the shift)
  int wseq[kAhead];
  TileCursor ahead(a, b0);    // the next tile whose entries are loaded
  auto load_entries = [&](int it2, int4& dst, int& sq) {
    if (it2 < n_it) {
      // K is a multiple of 128 and the top-k rows are 16-byte aligned
      dst = __ldg(reinterpret_cast<const int4*>(a.topk + (int64_t)ahead.t * a.K + ahead.tile * kRows) + lane);
      sq = a.token_seq ? __ldg(a.token_seq + ahead.t) : 0;
      ahead.advance(a);
    } else {
      dst = make_int4(-1, -1, -1, -1);
      sq = 0;
    }
  };
  // Translation in two halves so that the page-table loads of tile it + 1 are
  // in flight while tile it is handed over: issue() checks an entry and
  // starts its page-table load, finish() completes the physical row.  The
  // checks and error bits are those of resolve_row().  off: -1 masked or
  // rejected, -2 row already final (no page table), else the in-page offset.
  auto issue = [&](const int4& e4, int sq, int32_t (&v)[4], int32_t (&off)[4]) {
    const int32_t idx[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int32_t e = idx[k];
      v[k] = -1;
      off[k] = -1;
      if (e < 0) continue;
      if (a.page_table == nullptr) {
        if ((int64_t)e >= a.pool_rows) set_err(a.err, DSA_DEV_ERR_INDEX_RANGE);
        else { v[k] = e; off[k] = -2; }
        continue;
      }
      if (sq < 0 || sq >= a.B) { set_err(a.err, DSA_DEV_ERR_PAGE_RANGE); continue; }
      const int page = e / a.page_size;
      if (page >= a.max_pages) { set_err(a.err, DSA_DEV_ERR_INDEX_RANGE); continue; }
      off[k] = e - page * a.page_size;
      v[k] = __ldg(a.page_table + (int64_t)sq * a.max_pages + page);
    }
  };
  auto finish = [&](const int32_t (&v)[4], const int32_t (&off)[4], int32_t (&rows)[4]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      rows[k] = -1;
      if (off[k] == -2) { rows[k] = v[k]; continue; }
      if (off[k] < 0) continue;
      if (v[k] < 0) { set_err(a.err, DSA_DEV_ERR_PAGE_RANGE); continue; }
      const int64_t row = (int64_t)v[k] * a.page_size + off[k];
      if (row >= a.pool_rows) { set_err(a.err, DSA_DEV_ERR_PAGE_RANGE); continue; }
      rows[k] = (int32_t)row;
    }
  };
  int4 cur_e;
  int cur_sq;
  load_entries(0, cur_e, cur_sq);
#pragma unroll
  for (int d = 0; d < kAhead; ++d) load_entries(1 + d, win[d], wseq[d]);
  int32_t pv[4], poff[4];
  issue(cur_e, cur_sq, pv, poff);
  for (int it = 0; it < n_it; ++it) {
    int32_t rows[4];
    finish(pv, poff, rows);
    // publish the rows first: the producers wait for them, nothing here waits
    // for the loads of later tiles still in flight
    const int slot = it % kRing;
    if (it >= kRing && !warp_wait(smem_u32(&ms.idx_free[slot]), ((it / kRing) - 1) & 1, abort, a.wait_ns)) break;
    *reinterpret_cast<int4*>(&ms.ring[slot][4 * lane]) = make_int4(rows[0], rows[1], rows[2], rows[3]);
    warp_arrive(smem_u32(&ms.idx_full[slot]));
    // entries of tile it + 1 + kAhead; page-table reads of tile it + 1
    const int4 nxt = win[0];
    const int nxt_sq = wseq[0];
#pragma unroll
    for (int d = 0; d + 1 < kAhead; ++d) {
      win[d] = win[d + 1];
      wseq[d] = wseq[d + 1];
    }
    load_entries(it + 1 + kAhead, win[kAhead - 1], wseq[kAhead - 1]);
    issue(nxt, nxt_sq, pv, poff);
  }
}

// Index warp of the BF16-query kernels: per tile, the physical rows of the
// 128 top-k entries (lane l owns entries 4l .. 4l + 3) into the ring.
// prologue() runs before the CTA's set-up barrier: it waits for the previous
// grid (this warp alone) and starts the loads of the first tiles' entries and
// their page-table rows, so that the set-up of the other warps hides their
// latency; run() is the loop.
template <int HG, bool kScaled, bool kQ8, bool kRope>
struct IndexWarp {
  static constexpr int kAhead = 3;
  const int n_it;
  const int lane;
  int4 cur_e;                 // top-k entries of tile 0
  int cur_sq;
  int4 win[kAhead];           // top-k entries of tiles it + 1 .. it + kAhead (after the shift)
  int wseq[kAhead];
  TileCursor ahead;           // the next tile whose entries are loaded
  int32_t pv[4], poff[4];     // page-table rows in flight and in-page offsets

  // The arguments are passed to every method rather than kept in the object:
  // read straight from the kernel's parameter space they cost no loads.
  __device__ __forceinline__ IndexWarp(const AttnArgs& a, int64_t b0, int n_it_)
      : n_it(n_it_), lane(threadIdx.x & 31), ahead(a, b0) {}

  __device__ __forceinline__ void load_entries(const AttnArgs& a, int it2, int4& dst, int& sq) {
    if (it2 < n_it) {
      // K is a multiple of 128 and the top-k rows are 16-byte aligned
      dst = __ldg(reinterpret_cast<const int4*>(a.topk + (int64_t)ahead.t * a.K + ahead.tile * kRows) + lane);
      sq = a.token_seq ? __ldg(a.token_seq + ahead.t) : 0;
      ahead.advance(a);
    } else {
      dst = make_int4(-1, -1, -1, -1);
      sq = 0;
    }
  }
  // Translation in two halves so that the page-table loads of tile it + 1 are
  // in flight while tile it is handed over: issue() checks an entry and
  // starts its page-table load, finish() completes the physical row.  The
  // checks and error bits are those of resolve_row().  off: -1 masked or
  // rejected, -2 row already final (no page table), else the in-page offset.
  __device__ __forceinline__ void issue(const AttnArgs& a, const int4& e4, int sq) {
    const int32_t idx[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int32_t e = idx[k];
      pv[k] = -1;
      poff[k] = -1;
      if (e < 0) continue;
      if (a.page_table == nullptr) {
        if ((int64_t)e >= a.pool_rows) set_err(a.err, DSA_DEV_ERR_INDEX_RANGE);
        else { pv[k] = e; poff[k] = -2; }
        continue;
      }
      if (sq < 0 || sq >= a.B) { set_err(a.err, DSA_DEV_ERR_PAGE_RANGE); continue; }
      const int page = e / a.page_size;
      if (page >= a.max_pages) { set_err(a.err, DSA_DEV_ERR_INDEX_RANGE); continue; }
      poff[k] = e - page * a.page_size;
      pv[k] = __ldg(a.page_table + (int64_t)sq * a.max_pages + page);
    }
  }
  __device__ __forceinline__ void finish(const AttnArgs& a, int32_t (&rows)[4]) const {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      rows[k] = -1;
      if (poff[k] == -2) { rows[k] = pv[k]; continue; }
      if (poff[k] < 0) continue;
      if (pv[k] < 0) { set_err(a.err, DSA_DEV_ERR_PAGE_RANGE); continue; }
      const int64_t row = (int64_t)pv[k] * a.page_size + poff[k];
      if (row >= a.pool_rows) { set_err(a.err, DSA_DEV_ERR_PAGE_RANGE); continue; }
      rows[k] = (int32_t)row;
    }
  }

  __device__ __forceinline__ void prologue(const AttnArgs& a) {
    grid_dependency_wait();   // the lists and the page table are the previous grid's to write
    load_entries(a, 0, cur_e, cur_sq);
#pragma unroll
    for (int d = 0; d < kAhead; ++d) load_entries(a, 1 + d, win[d], wseq[d]);
    issue(a, cur_e, cur_sq);
  }

  __device__ __forceinline__ void run(const AttnArgs& a, Misc& ms) {
    volatile int* abort = &ms.abort;
    for (int it = 0; it < n_it; ++it) {
      int32_t rows[4];
      finish(a, rows);
      // publish the rows first: the producers wait for them, nothing here waits
      // for the loads of later tiles still in flight
      const int slot = it % kRing;
      if (it >= kRing && !warp_wait(smem_u32(&ms.idx_free[slot]), ((it / kRing) - 1) & 1, abort, a.wait_ns)) break;
      *reinterpret_cast<int4*>(&ms.ring[slot][4 * lane]) = make_int4(rows[0], rows[1], rows[2], rows[3]);
      warp_arrive(smem_u32(&ms.idx_full[slot]));
      // entries of tile it + 1 + kAhead; page-table reads of tile it + 1
      const int4 nxt = win[0];
      const int nxt_sq = wseq[0];
#pragma unroll
      for (int d = 0; d + 1 < kAhead; ++d) {
        win[d] = win[d + 1];
        wseq[d] = wseq[d + 1];
      }
      load_entries(a, it + 1 + kAhead, win[kAhead - 1], wseq[kAhead - 1]);
      issue(a, nxt, nxt_sq);
    }
  }
};

// Producers: copy the rows of each tile into its stage.  Producer warp pw
// owns the row quads q = pw, pw + kProdWarps, ...; one warp instruction moves
// 128-byte piece kb of the four rows of a quad (lane: row 4q + lane / 8,
// 16-byte chunk lane % 8).  Scale words of 528-byte rows: warps 0-3, one row
// per lane.
template <int HG, bool kScaled, bool kQ8, bool kRope>
__device__ void producer_role(const AttnArgs& a, uint8_t* sm, Misc& ms, int n_it) {
  using C = Cfg<HG, kScaled, kQ8, kRope>;
  constexpr int R = kRope ? kRopeRow : kScaled ? kScaledRow : kRawRow;
  const int ptid = threadIdx.x - kProdWarp0 * 32;
  const int pw = ptid >> 5, lane = ptid & 31;
  const int rq = lane >> 3, ch = lane & 7;
  volatile int* abort = &ms.abort;
  const uint32_t kv0 = smem_u32(sm + C::KV_OFF);
  for (int it = 0; it < n_it; ++it) {
    const int stage = it % C::NST, slot = it % kRing;
    if (it >= C::NST && !warp_wait(smem_u32(&ms.kv_empty[stage]), ((it / C::NST) - 1) & 1, abort, a.wait_ns)) break;
    if (!warp_wait(smem_u32(&ms.idx_full[slot]), (it / kRing) & 1, abort, a.wait_ns)) break;
    int32_t rows[kQuadsPerProd];
#pragma unroll
    for (int i = 0; i < kQuadsPerProd; ++i) {
      const int q = pw + i * kProdWarps;
      rows[i] = q < kQuads ? ms.ring[slot][4 * q + rq] : -1;
    }
    const int32_t sc_row = (kScaled && pw < 4) ? ms.ring[slot][32 * pw + lane] : -1;
    warp_arrive(smem_u32(&ms.idx_free[slot]));
    // valid flags of the stage (its previous tile's softmax is done: PV of
    // that tile released the stage)
#pragma unroll
    for (int i = 0; i < kQuadsPerProd; ++i) {
      const int q = pw + i * kProdWarps;
      if (q < kQuads && ch == 0) ms.vflag[stage][4 * q + rq] = rows[i] >= 0 ? 1 : 0;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&ms.meta_full[stage]));
    const uint32_t base = kv0 + stage * kStage;
    const uint32_t rope_base = smem_u32(sm + C::ROPE_OFF) + stage * C::ROPE_STAGE;
#pragma unroll
    for (int i = 0; i < kQuadsPerProd; ++i) {
      const int q = pw + i * kProdWarps;
      if (q >= kQuads) break;
      const int r = 4 * q + rq;
      const int32_t row = rows[i];
      const uint8_t* src = a.pool + (int64_t)(row >= 0 ? row : 0) * R + ch * 16;
      const uint32_t n = row >= 0 ? 16u : 0u;
      const uint32_t dst = base + (r >> 3) * 1024 + (r & 7) * 128 + ((ch ^ (r & 7)) << 4);
#pragma unroll
      for (int kb = 0; kb < 4; ++kb) cp_async_16_zfill(dst + kb * 16384, src + kb * 128, n);
      if (kRope)   // the row's 64 BF16 RoPE dims: one 128-byte swizzled row of the RoPE tile
        cp_async_16_zfill(rope_base + (r >> 3) * 1024 + (r & 7) * 128 + ((ch ^ (r & 7)) << 4),
                          src + kScaledRow, n);
    }
    if (kScaled && pw < 4) {
      const int r = 32 * pw + lane;
      cp_async_16_zfill(smem_u32(sm + C::SC_OFF + stage * kScStage + r * 16),
                        a.pool + (int64_t)(sc_row >= 0 ? sc_row : 0) * R + kD, sc_row >= 0 ? 16u : 0u);
    }
    cp_async_arrive_noinc(smem_u32(&ms.kv_full[stage]));
  }
  cp_async_wait_all();
}

// A shared-memory descriptor moved `bytes` further (the start address field
// holds address / 16 and never overflows inside the 227 KB window).
__device__ __forceinline__ uint64_t desc_add(uint64_t desc, uint32_t bytes) { return desc + (uint64_t)(bytes >> 4); }

// PV of one tile: O^T += V^T P^T over the four 128-dim blocks of the tile,
// K = 32 rows per MMA.  Descriptors are the stage's and the P buffer's base
// descriptors plus compile-time offsets, so each MMA costs a few instructions
// to issue.
template <class C, bool kFirst>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint64_t ad0, uint64_t bd0, uint32_t idesc) {
#pragma unroll
  for (int db = 0; db < 4; ++db) {
#pragma unroll
    for (int js = 0; js < 4; ++js) {
      // V^T: rows 32 js .. of dims block db (MN-major, 128-byte swizzle);
      // P: rows 32 js .. = four groups of 8 rows (MN-major, no swizzle)
      const uint64_t ad = desc_add(ad0, db * 16384 + js * 4096);
      const uint64_t bd = desc_add(bd0, (C::G > 1 ? db * (C::NP * 128) : 0) + js * 4 * (C::NP * 8));
      mma_e4m3(o_tmem + db * C::NP, ad, bd, idesc, (!kFirst || js > 0) ? 1u : 0u);
    }
  }
}

// Waits (bounded) for every tcgen05 operation this thread issued, so that the
// tensor memory can be released.
__device__ __forceinline__ void drain_mma(uint32_t bar) {
  mma_commit(bar);
  volatile int no_abort = 0;
  mbar_wait(bar, 0, &no_abort, 2000000000ull);
}

// QK^T issuer (one thread): per tile chunk, once its stage, query operand and
// score buffer are in place, S^T = K_tile Q^T into the score buffer.
template <int HG, bool kScaled, bool kQ8, bool kRope>
__device__ void qk_role(const AttnArgs& a, uint8_t* sm, Misc& ms, uint32_t tmem, int64_t b0, int n_it) {
  using C = Cfg<HG, kScaled, kQ8, kRope>;
  if ((threadIdx.x & 31) != 0) return;
  volatile int* abort = &ms.abort;
  const uint32_t kv0 = smem_u32(sm + C::KV_OFF);
  const uint32_t q0 = smem_u32(sm + C::Q_OFF);
  constexpr uint32_t kIdQK = idesc_e4m3(C::NQ, false);
  constexpr uint32_t kIdRope = idesc_bf16(C::NR > 0 ? C::NR : 16);
  const uint32_t rope0 = smem_u32(sm + C::ROPE_OFF);
  const uint32_t qr0 = smem_u32(sm + C::QR_OFF);
  int seg = -1;
  bool ok = true;
  TileCursor cur(a, b0);
  for (int it = 0; it < n_it && ok; ++it, cur.advance(a)) {
    const int stage = it % C::NST;
    if (cur.first(it)) {
      ++seg;
      ok = mbar_wait(smem_u32(&ms.q_full[seg % C::NQB]), (seg / C::NQB) & 1, abort, a.wait_ns);
    }
    ok = ok && mbar_wait(smem_u32(&ms.kv_full[stage]), (it / C::NST) & 1, abort, a.wait_ns);
    fence_proxy_async_smem();   // rows landed through cp.async (generic proxy)
#pragma unroll 1
    for (int qc = 0; qc < C::NQC && ok; ++qc) {
      const int u = it * C::NQC + qc, sb = u % C::NS;
      if (u >= C::NS) ok = mbar_wait(smem_u32(&ms.s_free[sb]), ((u / C::NS) - 1) & 1, abort, a.wait_ns);
      if (!ok) break;
      tc_fence_after();
      const uint64_t ad0 = sdesc_sw128(kv0 + stage * kStage + qc * (C::GC * 16384), 16, 1024);
      const uint64_t bd0 = sdesc_sw128(q0 + (seg % C::NQB) * C::Q_BYTES + qc * (C::GC * C::NQ * 128), 16, 1024);
      const uint32_t d_base = tmem + sb * C::S_COLS;
      constexpr int kSteps = kScaled ? 4 * C::GC : 16;   // K = 32 per step
#pragma unroll
      for (int st = 0; st < kSteps; ++st) {
        const int kb = st >> 2, kk = st & 3;              // 128-dim block within the chunk, K step in it
        const uint64_t ad = desc_add(ad0, kb * 16384 + kk * 32);
        const uint64_t bd = desc_add(bd0, kb * (C::NQ * 128) + kk * 32);
        // 528-byte rows: one accumulator per group (scaled by its rows' scales later)
        mma_e4m3(d_base + (kScaled ? kb * C::NQ : 0), ad, bd, kIdQK, (kScaled ? kk > 0 : st > 0) ? 1u : 0u);
        // the query's lo half: K offset 512 of the same rows, same accumulator
        if constexpr (C::kHalvesK)
          mma_e4m3(d_base + kb * C::NQ, ad, desc_add(bd, 4 * (C::NQ * 128)), kIdQK, 1u);
      }
      if (kRope && qc == 0) {
        // S_rope = K_rope Q_rope^T: 64 BF16 dims, K = 16 per MMA
        const uint32_t ra = rope0 + stage * C::ROPE_STAGE;
        const uint32_t rb = qr0 + (seg % C::NQB) * C::QR_BYTES;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(d_base + C::GC * C::NQ, sdesc_sw128(ra + kk * 32, 16, 1024), sdesc_sw128(rb + kk * 32, 16, 1024),
                   kIdRope, kk > 0 ? 1u : 0u);
      }
      mma_commit(smem_u32(&ms.s_full[sb]));
    }
  }
  drain_mma(smem_u32(&ms.mma_final[0]));
}

// PV issuer (one thread): per tile, once every softmax thread has written its
// P rows; its commits release the P buffer and the stage.
template <int HG, bool kScaled, bool kQ8, bool kRope>
__device__ void pv_role(const AttnArgs& a, uint8_t* sm, Misc& ms, uint32_t tmem, int64_t b0, int n_it) {
  using C = Cfg<HG, kScaled, kQ8, kRope>;
  if ((threadIdx.x & 31) != 0) return;
  volatile int* abort = &ms.abort;
  const uint32_t kv0 = smem_u32(sm + C::KV_OFF);
  const uint32_t p0 = smem_u32(sm + C::P_OFF);
  constexpr uint32_t kIdPV = idesc_e4m3(C::NP, true, true);
  TileCursor cur(a, b0);
  for (int it = 0; it < n_it; ++it, cur.advance(a)) {
    const int pb = it % C::NPB, stage = it % C::NST;
    if (!mbar_wait(smem_u32(&ms.p_full[pb]), (it / C::NPB) & 1, abort, a.wait_ns)) break;
    fence_proxy_async_smem();   // P and the stage were written through the generic proxy
    tc_fence_after();
    const uint64_t ad0 = sdesc_sw128(kv0 + stage * kStage, 1024, 1024);
    const uint64_t bd0 = sdesc_mn_none(p0 + pb * C::P_BYTES, C::NP * 8, 128);
    if (cur.first(it)) issue_pv<C, true>(tmem + C::O_COL0, ad0, bd0, kIdPV);
    else issue_pv<C, false>(tmem + C::O_COL0, ad0, bd0, kIdPV);
    mma_commit(smem_u32(&ms.kv_empty[stage]));
    mma_commit(smem_u32(&ms.pv_done[pb]));
  }
  drain_mma(smem_u32(&ms.mma_final[1]));
}

// Loads columns [c, c + HPT) of a 32-lane TMEM slice, HPT in {4, 8, 16}.
template <int HPT>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&v)[HPT]) {
  if constexpr (HPT == 2) {
    tmem_ld2(taddr, v);
  } else if constexpr (HPT == 4) {
    tmem_ld4(taddr, v);
  } else {
#pragma unroll
    for (int c = 0; c < HPT; c += 8) {
      uint32_t t8[8];
      tmem_ld8(taddr + c, t8);
#pragma unroll
      for (int k = 0; k < 8; ++k) v[c + k] = t8[k];
    }
  }
}

template <int HPT>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&v)[HPT]) {
  if constexpr (HPT == 2) {
    tmem_st2(taddr, v);
  } else if constexpr (HPT == 4) {
    tmem_st4(taddr, v);
  } else {
#pragma unroll
    for (int c = 0; c < HPT; c += 8) {
      uint32_t t8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) t8[k] = v[c + k];
      tmem_st8(taddr + c, t8);
    }
  }
}

template <int HG, bool kScaled, bool kQ8, bool kRope>
__device__ void softmax_role(const AttnArgs& a, uint8_t* sm, Misc& ms, uint32_t tmem, int64_t b0, int n_it,
                             int cta) {
  using C = Cfg<HG, kScaled, kQ8, kRope>;
  constexpr int HPT = C::HPT;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3, hq = warp >> 2;         // TMEM lane quarter, head quarter
  const int row = 32 * quarter + lane;                    // tile row = TMEM lane
  const int hbase = hq * HPT;                             // first head of this thread
  // P / O column of this thread's first head in term t (0 hi, 1 mid, 2 lo)
  auto tcol = [&](int t) { return C::kPInter ? hq * 24 + t * 8 : t * HG + hbase; };
  const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16);
  volatile int* abort = &ms.abort;
  float m_run[HPT], l_part[HPT];
  float m_thr[HPT];                // m_run + kTau: a score above it makes the running max grow
  float m_lane = kNoMax;           // running max of head hbase + (lane % HPT), log2 units
  int e_grp[4] = {-1000, -1000, -1000, -1000};   // running scale exponents (528-byte rows)
  int seg = -1;
  bool ok = true;                  // false once a wait gave up: keep going through every barrier
  TileCursor cur(a, b0);
  QueryBuild<HG, kQ8, kRope, C::kHalvesK> qnext;   // the next segment's query, loaded ahead of its build
  qnext.load(a, cur.t, cur.hgi * a.hg);
  qnext.template store<C::NQ>(a, sm + C::Q_OFF, ms.qsig[0], sm + C::QR_OFF);
  fence_proxy_async_smem();
  warp_arrive(smem_u32(&ms.q_full[0]));
  for (int it = 0; it < n_it; ++it, cur.advance(a)) {
    const bool first = cur.first(it), last = cur.last(a, it, n_it);
    const int stage = it % C::NST, pb = it % C::NPB;
    const bool build_next = last && it + 1 < n_it;      // the next tile starts a new segment
    if (first) {
      ++seg;
      const int qb = seg % C::NQB;
      ok &= mbar_wait(smem_u32(&ms.q_full[qb]), (seg / C::NQB) & 1, abort, a.wait_ns);
      m_lane = kNoMax;
#pragma unroll
      for (int h = 0; h < HPT; ++h) {
        m_run[h] = kNoMax;
        m_thr[h] = kNoMax + kTau;
        l_part[h] = 0.f;
      }
#pragma unroll
      for (int g = 0; g < 4; ++g) e_grp[g] = -1000;
    }
    const int qb = seg % C::NQB;
    ok &= mbar_wait(smem_u32(&ms.meta_full[stage]), (it / C::NST) & 1, abort, a.wait_ns);
    const bool valid = ms.vflag[stage][row] != 0;
    float sc4[4] = {1.f, 1.f, 1.f, 1.f};
    if (kScaled) {
      ok &= mbar_wait(smem_u32(&ms.kv_full[stage]), (it / C::NST) & 1, abort, a.wait_ns);
      const float4 v = *reinterpret_cast<const float4*>(sm + C::SC_OFF + stage * kScStage + row * 16);
      sc4[0] = v.x; sc4[1] = v.y; sc4[2] = v.z; sc4[3] = v.w;
    }
    float s2[HPT];
#pragma unroll
    for (int h = 0; h < HPT; ++h) s2[h] = 0.f;
#pragma unroll
    for (int qc = 0; qc < C::NQC; ++qc) {
      const int u = it * C::NQC + qc, sb = u % C::NS;
      ok &= mbar_wait(smem_u32(&ms.s_full[sb]), (u / C::NS) & 1, abort, a.wait_ns);
      tc_fence_after();
#pragma unroll
      for (int gl = 0; gl < C::GC; ++gl) {
        const int g = qc * C::GC + gl;
        const uint32_t cbase = lane_base + sb * C::S_COLS + gl * C::NQ;
        uint32_t hi[HPT], lo[HPT];
        tmem_ld_cols<HPT>(cbase + hbase, hi);
        if (!kQ8 && !C::kHalvesK) tmem_ld_cols<HPT>(cbase + HG + hbase, lo);
        tmem_wait_ld();
        float qs_hi[HPT], qs_lo[HPT];   // score column multipliers (16-byte aligned runs)
#pragma unroll
        for (int k = 0; k < HPT; k += 4) {
          const float4 m4 = *reinterpret_cast<const float4*>(&ms.qsig[qb][hbase + k]);
          qs_hi[k] = m4.x; qs_hi[k + 1] = m4.y; qs_hi[k + 2] = m4.z; qs_hi[k + 3] = m4.w;
          if (!kQ8 && !C::kHalvesK) {
            const float4 l4 = *reinterpret_cast<const float4*>(&ms.qsig[qb][HG + hbase + k]);
            qs_lo[k] = l4.x; qs_lo[k + 1] = l4.y; qs_lo[k + 2] = l4.z; qs_lo[k + 3] = l4.w;
          }
        }
#pragma unroll
        for (int k = 0; k < HPT; ++k) {
          float v = __uint_as_float(hi[k]) * qs_hi[k];
          if (!kQ8 && !C::kHalvesK) v = fmaf(__uint_as_float(lo[k]), qs_lo[k], v);
          s2[k] = kScaled ? fmaf(sc4[g], v, s2[k]) : v;
        }
      }
      if (kRope && qc == 0) {
        uint32_t rv[HPT];
        tmem_ld_cols<HPT>(lane_base + sb * C::S_COLS + C::GC * C::NQ + hbase, rv);
        tmem_wait_ld();
        const float rsig = a.sm_scale * kLog2e;
#pragma unroll
        for (int k = 0; k < HPT; ++k) s2[k] = fmaf(__uint_as_float(rv[k]), rsig, s2[k]);
      }
      tc_fence_before();
      warp_arrive(smem_u32(&ms.s_free[sb]));
    }
    // the next segment's query: its loads fly while this tile's P is formed
    if (build_next) {
      const int nt = cur.hgi + 1 == a.hgs ? cur.t + 1 : cur.t;
      const int nh0 = cur.hgi + 1 == a.hgs ? 0 : (cur.hgi + 1) * a.hg;
      qnext.load(a, nt, nh0);
    }
    if (!valid) {
#pragma unroll
      for (int h = 0; h < HPT; ++h) s2[h] = -INFINITY;
    }
    // Does a head's running maximum have to grow?  Each thread tests its own
    // row and one barrier ORs the answers; only then are the tile maxima
    // formed (each segment's first tile and the rare tiles whose maximum
    // exceeds the running one by more than 2^kTau).  528-byte rows also track
    // the group-scale exponents; testing those per row cost more than the
    // exchange it saves (measured), so their tiles always form the maxima.
    bool grow = false;
#pragma unroll
    for (int h = 0; h < HPT; ++h) grow |= s2[h] > m_thr[h];
    float tmp[HPT];
    unsigned rmask = 0;
    float alpha_lane = 1.f;
    float beta[4] = {1.f, 1.f, 1.f, 1.f};
    bool bchange = false;
    if (kScaled || named_bar_red_or(1, kSmxThreads, grow)) {
      // tile maxima over the 128 rows: per head, and per scale group
#pragma unroll
      for (int h = 0; h < HPT; ++h) tmp[h] = s2[h];
      const float wmax = transpose_reduce<HPT, true>(tmp, lane);
      if (lane < HPT) ms.red[it & 1][hq][quarter][lane] = wmax;
      if (kScaled && hq == 0) {
        float sct[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) sct[g] = valid ? fabsf(sc4[g]) : 0.f;
        const float wsc = transpose_reduce<4, true>(sct, lane);
        if (lane < 4) ms.red_sc[it & 1][quarter][lane] = wsc;
      }
      named_bar_sync(1, kSmxThreads);
      const int hl = lane % HPT;
      const float tile_max = fmaxf(fmaxf(ms.red[it & 1][hq][0][hl], ms.red[it & 1][hq][1][hl]),
                                   fmaxf(ms.red[it & 1][hq][2][hl], ms.red[it & 1][hq][3][hl]));
      const bool need = tile_max > m_lane + kTau;
      rmask = __ballot_sync(0xffffffffu, need);
      if (need) {
        alpha_lane = ex2_approx(m_lane - tile_max);
        m_lane = tile_max;
      }
      if (rmask) {
#pragma unroll
        for (int h = 0; h < HPT; ++h) {
          m_run[h] = __shfl_sync(0xffffffffu, m_lane, h);
          m_thr[h] = m_run[h] + kTau;
          l_part[h] *= __shfl_sync(0xffffffffu, alpha_lane, h);
        }
      }
      if (kScaled) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const float mx = fmaxf(fmaxf(ms.red_sc[it & 1][0][g], ms.red_sc[it & 1][1][g]),
                                 fmaxf(ms.red_sc[it & 1][2][g], ms.red_sc[it & 1][3][g]));
          if (mx > 0.f && mx <= 3.0e38f) {
            const int e = ceil_log2(mx);
            if (e > e_grp[g]) {
              beta[g] = e_grp[g] == -1000 ? 0.f : scale_pow2(1.f, e_grp[g] - e);
              e_grp[g] = e;
              bchange = true;
            }
          }
        }
      }
    }
    // O holds this segment's earlier tiles: rescale it after their PV has finished
    if (!first && (rmask || bchange)) {
      float alpha[HPT];
#pragma unroll
      for (int h = 0; h < HPT; ++h) alpha[h] = __shfl_sync(0xffffffffu, alpha_lane, h);
      ok &= mbar_wait(smem_u32(&ms.pv_done[(it - 1) % C::NPB]), ((it - 1) / C::NPB) & 1, abort, a.wait_ns);
      tc_fence_after();
#pragma unroll
      for (int db = 0; db < 4; ++db) {
#pragma unroll
        for (int term = 0; term < 3; ++term) {
          const uint32_t ca = lane_base + C::O_COL0 + db * C::NP + tcol(term);
          uint32_t v[HPT];
          tmem_ld_cols<HPT>(ca, v);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < HPT; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha[k] * beta[db]);
          tmem_st_cols<HPT>(ca, v);
        }
      }
      tmem_wait_st();
    }
    // this P buffer was last read by PV(it - NPB); with a single buffer the
    // wait comes after P is formed in registers, just before it is stored
    constexpr bool kLateWait = C::NPB == 1 && C::G == 1;
    if (!kLateWait && it >= C::NPB) ok &= mbar_wait(smem_u32(&ms.pv_done[pb]), ((it / C::NPB) - 1) & 1, abort, a.wait_ns);
    const uint32_t pbuf = smem_u32(sm + C::P_OFF + pb * C::P_BYTES);
    // p = 2^(s - m) (0 while the head has seen no valid entry), denominators, P operand
#pragma unroll
    for (int h = 0; h < HPT; ++h) {
      s2[h] = ex2_approx(s2[h] - m_run[h]);
      l_part[h] += s2[h];
    }
    // three E4M3 terms of a pair of P values: v ~ hi + mid / 16 + lo / 256
    auto split = [](float v0, float v1, uint32_t& hi2, uint32_t& mid2, uint32_t& lo2) {
      split3_f16(v0, v1, hi2, mid2, lo2);
    };
    // this row's P bytes: one term's HPT bytes are consecutive in the MN-major
    // operand; with the interleaved order all three terms' 24 bytes are, and
    // they go out as 16 + 8 bytes (even head quarter) or 8 + 16 (odd)
    auto store_p = [&](uint32_t pg, const uint32_t (&hi2)[HPT / 2], const uint32_t (&mid2)[HPT / 2],
                       const uint32_t (&lo2)[HPT / 2]) {
      if constexpr (C::kPInter) {
        const int n0 = hq * 24;
        const uint32_t w0 = hi2[0] | (hi2[1] << 16), w1 = hi2[2] | (hi2[3] << 16);
        const uint32_t w2 = mid2[0] | (mid2[1] << 16), w3 = mid2[2] | (mid2[3] << 16);
        const uint32_t w4 = lo2[0] | (lo2[1] << 16), w5 = lo2[2] | (lo2[3] << 16);
        if ((hq & 1) == 0) {
          st_shared_v4(pg + p_off<C::NP>(n0, row), w0, w1, w2, w3);
          st_shared_v2(pg + p_off<C::NP>(n0 + 16, row), w4, w5);
        } else {
          st_shared_v2(pg + p_off<C::NP>(n0, row), w0, w1);
          st_shared_v4(pg + p_off<C::NP>(n0 + 8, row), w2, w3, w4, w5);
        }
      } else {
        auto store_term = [&](int term, const uint32_t (&t2)[HPT / 2]) {
          const uint32_t addr = pg + p_off<C::NP>(tcol(term), row);
          if constexpr (HPT == 8)
            st_shared_v2(addr, t2[0] | (t2[1] << 16), t2[2] | (t2[3] << 16));
          else if constexpr (HPT == 4)
            st_shared_u32(addr, t2[0] | (t2[1] << 16));
          else
            st_shared_u16(addr, t2[0]);
        };
        store_term(0, hi2);
        store_term(1, mid2);
        store_term(2, lo2);
      }
    };
    if constexpr (kLateWait) {
      uint32_t hi2[HPT / 2], mid2[HPT / 2], lo2[HPT / 2];
#pragma unroll
      for (int h = 0; h < HPT; h += 2) split(s2[h], s2[h + 1], hi2[h / 2], mid2[h / 2], lo2[h / 2]);
      if (it >= 1) ok &= mbar_wait(smem_u32(&ms.pv_done[0]), (it - 1) & 1, abort, a.wait_ns);
      store_p(pbuf, hi2, mid2, lo2);
    } else {
#pragma unroll
      for (int g = 0; g < C::G; ++g) {
        const float mul = kScaled ? (e_grp[g] == -1000 ? 0.f : scale_pow2(sc4[g], -e_grp[g])) : 1.f;
        const uint32_t pg = pbuf + g * (C::NP * 128);
        uint32_t hi2[HPT / 2], mid2[HPT / 2], lo2[HPT / 2];
#pragma unroll
        for (int h = 0; h < HPT; h += 2) split(s2[h] * mul, s2[h + 1] * mul, hi2[h / 2], mid2[h / 2], lo2[h / 2]);
        store_p(pg, hi2, mid2, lo2);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    warp_arrive(smem_u32(&ms.p_full[pb]));
    // every thread passed this tile's barrier after its last read of the scores'
    // multipliers, and QK^T of this tile (the last reader of the operand) is done
    if (build_next) {
      const int nqb = (seg + 1) % C::NQB;
      qnext.template store<C::NQ>(a, sm + C::Q_OFF + nqb * C::Q_BYTES, ms.qsig[nqb], sm + C::QR_OFF + nqb * C::QR_BYTES);
      fence_proxy_async_smem();
      warp_arrive(smem_u32(&ms.q_full[nqb]));
    }

    if (!last) continue;
    // ---- end of a segment: denominators, O normalisation, stores
#pragma unroll
    for (int h = 0; h < HPT; ++h) tmp[h] = l_part[h];
    const float wsum = transpose_reduce<HPT, false>(tmp, lane);
    if (lane < HPT) ms.red2[hq][quarter][lane] = wsum;
    named_bar_sync(1, kSmxThreads);
    if (quarter == 0 && lane < HPT) {
      const float l = (ms.red2[hq][0][lane] + ms.red2[hq][1][lane]) + (ms.red2[hq][2][lane] + ms.red2[hq][3][lane]);
      ms.linv[hbase + lane] = l > 0.f ? 1.f / l : 0.f;
      ms.lse2[hbase + lane] = l > 0.f ? m_lane + log2f(l) : -INFINITY;
    }
    named_bar_sync(1, kSmxThreads);
    ok &= mbar_wait(smem_u32(&ms.pv_done[pb]), (it / C::NPB) & 1, abort, a.wait_ns);
    tc_fence_after();
    const int64_t u0 = cur.unit * a.tpt;
    const int h0 = cur.hgi * a.hg;
    const bool whole = cta_of_tile(u0, a.n_tiles, a.grid) == cta_of_tile(u0 + a.tpt - 1, a.n_tiles, a.grid);
    const int64_t slot = (int64_t)cta * 2 + (b0 >= u0 ? 0 : 1);
    constexpr int kCh = HPT < 8 ? HPT : 8;               // columns per TMEM load
#pragma unroll
    for (int db = 0; db < 4; ++db) {
      const int d = db * kRows + row;
      const float pw2 = kScaled && e_grp[db] != -1000 ? scale_pow2(1.f, e_grp[db]) : 1.f;
#pragma unroll
      for (int c0 = 0; c0 < HPT; c0 += kCh) {
        uint32_t hi[kCh], mid[kCh], lo[kCh];
        const uint32_t ob = lane_base + C::O_COL0 + db * C::NP + c0;
        tmem_ld_cols<kCh>(ob + tcol(0), hi);
        tmem_ld_cols<kCh>(ob + tcol(1), mid);
        tmem_ld_cols<kCh>(ob + tcol(2), lo);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < kCh; ++k) {
          const int h = hbase + c0 + k;
          const float li = ms.linv[h];
          const float acc = fmaf(__uint_as_float(lo[k]), 0.00390625f,
                                 fmaf(__uint_as_float(mid[k]), 0.0625f, __uint_as_float(hi[k])));
          const float o = li == 0.f ? 0.f : acc * pw2 * li;
          if (whole)
            static_cast<__nv_bfloat16*>(a.o)[((int64_t)cur.t * a.H + h0 + h) * kD + d] = __float2bfloat16_rn(o);
          else
            a.ws_o[(slot * a.hg + h) * kD + d] = o;
        }
      }
    }
    if (quarter == 0 && lane < HPT) {
      const int h = hbase + lane;
      const float lse = ms.lse2[h] * kLn2;
      if (whole) a.lse[(int64_t)cur.t * a.H + h0 + h] = lse;
      else a.ws_lse[slot * a.hg + h] = lse;
    }
  }
  (void)ok;
}

// Register re-split after the launch (Cfg::SMX_REGS): executed by whole warpgroups.
template <int kRegs>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
}
template <int kRegs>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
}

template <int HG, bool kScaled, bool kQ8, bool kRope>
__global__ void __launch_bounds__(kThreads, 1) sparse_attn_tc_kernel(const __grid_constant__ AttnArgs a) {
  using C = Cfg<HG, kScaled, kQ8, kRope>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Misc& ms = *reinterpret_cast<Misc*>(sm + C::MISC_OFF);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int cta = blockIdx.x;
  const int64_t b0 = tile_begin(cta, a.n_tiles, a.grid);
  const int n_it = (int)(tile_begin(cta + 1, a.n_tiles, a.grid) - b0);

  IndexWarp<HG, kScaled, kQ8, kRope> idx(a, b0, n_it);
  if constexpr (!kQ8) { if (warp == kIdxWarp) idx.prologue(a); }
  if (tid == 0) {
    for (int s = 0; s < 3; ++s) {
      mbar_init(smem_u32(&ms.kv_full[s]), kProdWarps * 32);
      mbar_init(smem_u32(&ms.kv_empty[s]), 1);
      mbar_init(smem_u32(&ms.meta_full[s]), kProdWarps);
    }
    for (int s = 0; s < kRing; ++s) {
      mbar_init(smem_u32(&ms.idx_full[s]), 1);            // the index warp (one arrival a warp)
      mbar_init(smem_u32(&ms.idx_free[s]), kProdWarps);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&ms.s_full[s]), 1);
      mbar_init(smem_u32(&ms.s_free[s]), kSmxWarps);
      mbar_init(smem_u32(&ms.q_full[s]), kSmxWarps);
      mbar_init(smem_u32(&ms.p_full[s]), kSmxWarps);
      mbar_init(smem_u32(&ms.pv_done[s]), 1);
    }
    mbar_init(smem_u32(&ms.mma_final[0]), 1);
    mbar_init(smem_u32(&ms.mma_final[1]), 1);
    ms.abort = 0;
    mbar_init_fence();
  }
  if (warp == kQkWarp) {
    tmem_alloc(smem_u32(&ms.tmem_base), C::TMEM_COLS);
    tmem_relinquish();
  }
  // the query and P operands start zeroed: their padding rows (N rounded up
  // to 16) stay zero
  for (int i = tid; i < (C::NQB * (C::Q_BYTES + C::QR_BYTES) + C::NPB * C::P_BYTES) / 16; i += kThreads)
    reinterpret_cast<uint4*>(sm + C::Q_OFF)[i] = make_uint4(0, 0, 0, 0);
  for (int i = tid; i < 2 * 64; i += kThreads) (&ms.qsig[0][0])[i] = 0.f;
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;
  // launched as a programmatic dependent: everything above overlapped the
  // previous kernel in the stream, whose results are visible from here on
  grid_dependency_wait();
  // the split-unit merge may be scheduled now: its blocks take SMs as CTAs
  // of this grid exit and wait for the whole grid before reading partials
  grid_launch_dependents();

  // 24 warps: the four softmax warpgroups (warps 0-15) grow to SMX_REGS
  // registers a thread, the two others (MMA issuers, index, producers) shrink
  // to OTHER_REGS
  static_assert(C::SMX_REGS % 8 == 0 && C::OTHER_REGS % 8 == 0 && C::SMX_REGS > kLaunchRegs &&
                C::OTHER_REGS < kLaunchRegs && C::OTHER_REGS >= 24 &&
                C::SMX_REGS * kSmxThreads + C::OTHER_REGS * (kThreads - kSmxThreads) == kLaunchRegs * kThreads,
                "setmaxnreg values");
  if (warp < kSmxWarps) regs_inc<C::SMX_REGS>();
  else regs_dec<C::OTHER_REGS>();
  if (warp < kSmxWarps)
    softmax_role<HG, kScaled, kQ8, kRope>(a, sm, ms, tmem, b0, n_it, cta);
  else if (warp == kQkWarp)
    qk_role<HG, kScaled, kQ8, kRope>(a, sm, ms, tmem, b0, n_it);
  else if (warp == kPvWarp)
    pv_role<HG, kScaled, kQ8, kRope>(a, sm, ms, tmem, b0, n_it);
  else if (warp == kIdxWarp) {
    if constexpr (kQ8) index_role<HG, kScaled, kQ8, kRope>(a, sm, ms, b0, n_it);
    else idx.run(a, ms);
  }
  else
    producer_role<HG, kScaled, kQ8, kRope>(a, sm, ms, n_it);

  tc_fence_before();
  __syncthreads();
  if (warp == kQkWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (tid == 0 && ms.abort) set_err(a.err, DSA_DEV_ERR_TIMEOUT);
}

template <int HG, bool kScaled, bool kQ8, bool kRope>
bool launch_tc(const AttnArgs& a, cudaStream_t stream) {
  using C = Cfg<HG, kScaled, kQ8, kRope>;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    if (cudaFuncSetAttribute(sparse_attn_tc_kernel<HG, kScaled, kQ8, kRope>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
      return false;   // the launch is skipped; the caller sees the attribute error
    // the in-kernel register re-split adds up only if every thread starts with
    // exactly kLaunchRegs registers; otherwise a warpgroup could wait forever
    // for registers, so refuse to launch
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, sparse_attn_tc_kernel<HG, kScaled, kQ8, kRope>) != cudaSuccess ||
        fa.numRegs != kLaunchRegs)
      return false;
    configured.fetch_or(bit);
  }
  // programmatic dependent launch: the set-up (barriers, tensor memory,
  // zeroed operands) may overlap the tail of the previous kernel
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sparse_attn_tc_kernel<HG, kScaled, kQ8, kRope>, a) == cudaSuccess;
}

template <int HG>
bool launch_hg(const AttnArgs& a, bool q8, cudaStream_t stream) {
  bool ok = false;
  if (a.rope) {
    if constexpr (HG <= 16) ok = launch_tc<HG, true, false, true>(a, stream);   // head_group caps HG at 16
  } else if (q8 && a.scaled) {
    ok = launch_tc<HG, true, true, false>(a, stream);
  } else if (q8) {
    ok = launch_tc<HG, false, true, false>(a, stream);
  } else if (a.scaled) {
    ok = launch_tc<HG, true, false, false>(a, stream);
  } else {
    ok = launch_tc<HG, false, false, false>(a, stream);
  }
  if (ok && a.ws_o != nullptr) launch_combine(a, stream);
  return ok;
}

}  // namespace

int head_group(int H, bool rope) {
  const int cap = rope ? 16 : 32;
  return H < cap ? H : cap;
}

bool launch_sparse_attn(const AttnArgs& a, bool q8, cudaStream_t stream) {
  if (a.hg == 8) return launch_hg<8>(a, q8, stream);
  if (a.hg == 16) return launch_hg<16>(a, q8, stream);
  return launch_hg<32>(a, q8, stream);
}

}  // namespace dsa
