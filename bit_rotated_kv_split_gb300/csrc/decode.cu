// Decode attention over BF16 sink | INT2 history | BF16 recent window.
//
// myzaker.com OSCAR article, part "从离线校准到在线推理的 pipeline": the INT2
// kernel unpacks, dequantises with scale/zero point and accumulates in float;
// a BF16 kernel handles sink and recent; an online-softmax merge joins them.
// gist.science "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV
// Cache Quantization", Technical summary 2.2 B: the inverse rotation is fused
// into the attention kernel with no extra memory traffic.  Here it is applied
// as q~ = q . R_K once per query head and one o . R_V^T per head after the
// history partials are merged, instead of rotating every token.
//
// One launch (programmatic dependent launch: it waits for the previous
// kernel's writes first and lets the next kernel become resident early).
// CTA (split, kv, b) of W warps (16 for GQA 4, 12 for GQA 8; one CTA per SM)
// owns a contiguous range of INT2 pages of one (request, KV head) and a
// share of its BF16 sink/recent tokens:
//   1. R_K is requested first (TMA bulk copy); lane 0 of each warp starts
//      1-D TMA bulk copies of the warp's first pages (one 1152-byte page
//      block per stage, a ring of 6 (GQA 4) or 8 (GQA 8) stages per warp,
//      mbarrier completion, bounded waits);
//   2. all warps but the last two compute q~ = q . R_K for the GQA group
//      (fp32) and build the 32 lanes' tensor-core B fragments once in shared
//      memory, while the last two scan the CTA's BF16 tokens;
//   3. every warp streams its INT2 pages through its ring, 4 (GQA 4) or 3
//      (GQA 8) per online-softmax step, keeping its own state; after a step
//      its lanes start the copies of the freed stages together;
//   4. one warp per head weighs the CTA's warp states against their common
//      maximum; the history part is rotated back with R_V (four 2-D TMA
//      copies with the 128-byte swizzle, issued after step 2) and joined
//      with the BF16 part into one partial (m, l, o) per query head;
//   5. the last CTA of the (request, KV head) to finish (acquire-release
//      ticket, no waiting) merges all partials (one warp per head) and
//      writes the normalised output, then resets the ticket.
//
// INT2 arithmetic on the tensor cores (mma.sync m16n8k16, fp32 accumulate):
//   QK: A = codes of 16 tokens x 128 channels, B = q~ with column 2i + e the
//       hi (e = 0) or lo (e = 1) fp16 part of head 4 nt + i, so
//       q~ . k^ = s (q~ . c) + z sum(q~).  A lane's accumulator then holds
//       both parts of one head (column group tig) for its two tokens.
//   PV: A = codes^T (128 channels x 16 tokens), B = p s_V in the same column
//       order (the lane's own values, transposed by movmatrix), so
//       o~ = sum p (s_V c + z_V) = (p s_V) . c + sum(p z_V).
//   A 2-bit code c at bit offset 2k of a 16-bit half is taken as the fp16
//   subnormal c * 4^k * 2^-24 by a single AND (no conversion); the 4^k and
//   2^-24 factors are folded into the B operand (QK) or the output (PV).
//   The contraction order of channels is free, so B is permuted to match.
//
// Codec variants (template arguments; page block sizes and ring depths above
// are those of one quantisation group per vector):
//   - NGK / NGV > 1 quantisation groups: the page format stores codes so that
//     K-step j reads K group j / (8 / NGK) and 16-row tile mt reads V group
//     mt / (8 / NGV); QK folds each group's sum with its scale as soon as its
//     K-steps are done, PV takes one p s_V operand per V group, and the
//     zero-point terms are summed per group.
//   - codebook levels: a level l[c] = l_0 + d1 c + a2 (2 b1) + b (b0 b1) of
//     the code's bits, so QK and PV run over the three bit planes c, 2 b1 and
//     b0 b1 (single ANDs at the same operand positions) with the level
//     coefficients on the QK sums and on the PV operands.
#include <cfloat>
#include <type_traits>

#include <cudaTypedefs.h>

#include "kernels.h"
#include "ptx.cuh"

// Tunables (compile-time): warps per CTA for GQA 4 / GQA 8, ring stages per
// warp, and the number of independent accumulator chains of the QK MMA.
#ifndef OSCAR_WARPS_G4
#define OSCAR_WARPS_G4 16
#endif
#ifndef OSCAR_WARPS_G8
#define OSCAR_WARPS_G8 12
#endif
#ifndef OSCAR_STAGES_G4
#define OSCAR_STAGES_G4 6
#endif
#ifndef OSCAR_STAGES_G8
#define OSCAR_STAGES_G8 8
#endif
#ifndef OSCAR_QK_CHAINS_G4
#define OSCAR_QK_CHAINS_G4 2
#endif
#ifndef OSCAR_QK_CHAINS_G8
#define OSCAR_QK_CHAINS_G8 1
#endif
// 1: every page copy is waited for right after it is issued, so no copy
// ever overlaps the computation (a verification build: its results must be
// bit-identical to the default build's, which overlaps them)
#ifndef OSCAR_SERIAL_COPIES
#define OSCAR_SERIAL_COPIES 0
#endif
// INT2 pages a warp processes per step (one online-softmax update per step)
// for GQA 4 / GQA 8
#ifndef OSCAR_GROUP_G4
#define OSCAR_GROUP_G4 3
#endif
#ifndef OSCAR_GROUP_G8
#define OSCAR_GROUP_G8 3
#endif
// splits per (request, KV head): 0 = the planner's model; n > 0 forces n
// (tuning builds)
#ifndef OSCAR_PLAN_SPLITS
#define OSCAR_PLAN_SPLITS 0
#endif

namespace oscar {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr uint32_t kFull = 0xffffffffu;
constexpr int kMaxSplits = 128;               // bounds the last CTA's merge scratch
constexpr int kBf16Warps = 2;                 // warps that scan the BF16 sink/recent tokens
constexpr uint32_t kPrologueBarrier = 1;      // named barrier of the q~ prologue

// NGK / NGV: quantisation groups per token-head of K / V (1, 2 or 4); they
// fix the page block size and, through it, how many ring stages fit.
template <int G, int NGK = 1, int NGV = 1, bool LV = false>
struct Geo {
  static constexpr int NT = (2 * G + 7) / 8;          // column tiles holding hi | lo parts
  static constexpr int HS = G >= 8 ? G / 4 : 2;       // BF16 head slots per lane
  static constexpr int NH = G / 4;                    // INT2 heads per lane (head 4 nt + tig)
  static constexpr int NTQ = (G + 7) / 8;             // BF16 QK column tiles
  static constexpr int W = G <= 4 ? OSCAR_WARPS_G4 : OSCAR_WARPS_G8;  // warps per CTA
  static constexpr int T = W * 32;
  // the last kBf16Warps warps scan the BF16 tokens while the others build q~
  static constexpr int PT = (W - kBf16Warps) * 32;
  // pages per step (GQA 8 with several quantisation groups or codebook
  // levels: 2, which keeps the extra state within the register budget)
  // (larger blocks leave room for fewer stages: two pages per step where
  // three would not give the ring two parts)
  static constexpr int kGroup = G <= 4 ? (NGK * NGV >= 16 ? 2 : OSCAR_GROUP_G4)
                                       : (NGK * NGV > 1 || LV ? 2 : OSCAR_GROUP_G8);
  static constexpr int kQkChains = G <= 4 ? OSCAR_QK_CHAINS_G4 : OSCAR_QK_CHAINS_G8;   // QK accumulators
  static constexpr int kBlock = block_bytes(NGK, NGV);   // one (page, KV head) block
  // union: R_K (64 KB, prologue) then R_V (epilogue), followed by the q~
  // scratch (prologue) that the CTA merge reuses
  static constexpr size_t kRotBytes = size_t(kHeadDim) * kHeadDim * 4;
  static constexpr size_t kQScratch = (6 * G * kHeadDim + 16 * G + 32 * NH * 16) * 4;
  static constexpr size_t kUnion = kRotBytes + kQScratch;   // R_K then R_V | q~ scratch
  static constexpr size_t kBf16State = size_t(kBf16Warps) * G * kPartStride * 4;
  // ring stages per warp: the tuned count, fewer when larger blocks (more
  // quantisation groups) would not fit the 227 KB with everything else
  // the ring is kParts parts of kGroup stages: a step consumes one part
  // while the others' copies are in flight
  static constexpr int kStagesTuned = G <= 4 ? OSCAR_STAGES_G4 : OSCAR_STAGES_G8;
  static constexpr int kStagesFit =
      int((227 * 1024 - (1024 + kUnion + kBf16State + 16 + 1024)) / (size_t(W) * kBlock));
  static constexpr int kStagesMax = kStagesTuned < kStagesFit ? kStagesTuned : kStagesFit;
  static constexpr int kParts = kStagesMax / kGroup;
  static constexpr int kStages = kParts * kGroup;
  static_assert(kGroup >= 1 && kParts >= 2, "a step leaves a part of the ring in flight");
  static constexpr size_t kStageBytes = size_t(W) * kStages * kBlock;
  // ring barriers + the R_K, R_V and prologue-done barriers, padded so the
  // region after it stays 128-byte aligned (TMA destinations need at least 16)
  static constexpr size_t kBarBytes = ((size_t(W) * kStages + 3) * 8 + 127) / 128 * 128;
  static_assert(kBarBytes <= 1024, "barrier region within its budget");
  // (+1 KB: the union starts at the next 1024-byte boundary, which the
  // swizzled R_V boxes need)
  static constexpr size_t kSmem = kStageBytes + kBarBytes + 1024 + kUnion + kBf16State + 16;
  static_assert(kStageBytes % 128 == 0 && kBarBytes % 128 == 0, "TMA destinations must stay aligned");
  static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
  // each warp's ring slice holds its INT2 state once its pages are done
  static_assert(G * kPartStride * 4 <= kStages * kBlock, "warp state in the ring slice");
  // CTA merge scratch (after R_V in the union): merged outputs and weights
  static_assert((2 * G * kHeadDim + 32 * G) * 4 <= kQScratch, "CTA merge scratch");
  // ring region once the warp states are consumed: rotation quarters, then
  // the last CTA's split weights
  static_assert(4 * G * kHeadDim * 4 <= kStageBytes && G * kMaxSplits * 4 <= kStageBytes, "merge scratch");
};

// head owned by head slot hs of a lane with column group tig
template <int G>
__device__ __forceinline__ int slot_head(int tig, int hs) {
  if (G <= 4) return (2 * tig + hs) & (G - 1);
  return 8 * (hs >> 1) + 2 * tig + (hs & 1);
}

// head slot of accumulator component c of column tile nt
template <int G>
__device__ __forceinline__ int acc_slot(int nt, int c) {
  if constexpr (G <= 4) {
    return c & 1;
  } else {
    return 2 * (nt % (Geo<G>::NT / 2)) + (c & 1);
  }
}

// (code j, code j+8) of the 16-code word w as an fp16x2 of subnormals
// c * 4^pos(j) * 2^-24, pos(j) = j (j < 5) or j - 3; wsh = w >> 6.
__device__ __forceinline__ uint32_t code_pair(uint32_t w, uint32_t wsh, int j) {
  return j < 5 ? (w & (0x00030003u << (2 * j))) : (wsh & (0x00030003u << (2 * (j - 3))));
}

__device__ __forceinline__ int code_pos(int j) { return j < 5 ? j : j - 3; }

__device__ __forceinline__ float split_lo(float x) {
  return x - __half2float(__float2half_rn(x));
}

// x as an fp16 (hi, lo) pair in one register, hi in the low half: hi = x
// with its 13 low significand bits cleared (11 significant bits, exact in
// fp16 within its normal range), lo = fp16(x - hi) (the difference is
// exact), so hi + lo keeps about 22 bits of x.
__device__ __forceinline__ uint32_t split_hi_lo(float x) {
  const float hi = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(x - hi), "f"(hi));
  return r;
}

// 2^x by the ex2.approx instruction (relative error about 2^-22; results
// below 2^-126 flush to zero, far below what the fp32 sums resolve)
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void flag(int32_t* st, int bit) {
  if (st) atomicOr(st, bit);
}

// ------------------------------------------------------------------ warp state and pages

template <int G>
struct WarpState {
  static constexpr int NT = Geo<G>::NT, HS = Geo<G>::HS;
  float acc[NT][8][4];
  float m[HS], l[HS], z[HS];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[nt][mt][c] = 0.f;
#pragma unroll
    for (int hs = 0; hs < HS; ++hs) {
      m[hs] = -INFINITY;
      l[hs] = 0.f;
      z[hs] = 0.f;
    }
  }
  // online-softmax update of the running max from this page's scores; lanes
  // rescale their state only when a head's max grew past the lazy threshold
  __device__ __forceinline__ void update_max(const float (&sc)[HS][2]) {
    bool need = false;
#pragma unroll
    for (int hs = 0; hs < HS; ++hs) need |= fmaxf(sc[hs][0], sc[hs][1]) > m[hs] + kRescaleLog2;
    if (!__any_sync(kFull, need)) return;
#pragma unroll
    for (int hs = 0; hs < HS; ++hs) {
      float pm = fmaxf(sc[hs][0], sc[hs][1]);
      pm = fmaxf(pm, __shfl_xor_sync(kFull, pm, 4));
      pm = fmaxf(pm, __shfl_xor_sync(kFull, pm, 8));
      pm = fmaxf(pm, __shfl_xor_sync(kFull, pm, 16));
      if (pm > m[hs]) {
        const float f = exp2f(m[hs] - pm);
        m[hs] = pm;
        l[hs] *= f;
        z[hs] *= f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int c = 0; c < 4; ++c)
              if (acc_slot<G>(nt, c) == hs) acc[nt][mt][c] *= f;
      }
    }
  }
  // B fragments of the PV MMA from the probabilities pp[hs][t] (t = 0: token
  // gid, 1: token gid + 8), hi parts in columns [0, G), lo parts in [G, 2G)
  template <bool kHalf>
  __device__ __forceinline__ void pv_operand(const float (&pp)[HS][2], int tig,
                                             uint32_t (&pb)[NT][2]) const {
    auto pack = [](float a, float b) { return kHalf ? pack_half2(a, b) : pack_bf162(a, b); };
    auto lo_of = [](float x) {
      return kHalf ? split_lo(x) : x - __bfloat162float(__float2bfloat16_rn(x));
    };
    if (G <= 4) {
      const bool lo = tig >= G / 2;
      const float a = lo ? lo_of(pp[0][0]) : pp[0][0], b2 = lo ? lo_of(pp[1][0]) : pp[1][0];
      const float c = lo ? lo_of(pp[0][1]) : pp[0][1], d = lo ? lo_of(pp[1][1]) : pp[1][1];
      pb[0][0] = movmatrix_trans(pack(a, b2));
      pb[0][1] = movmatrix_trans(pack(c, d));
    } else {
#pragma unroll
      for (int nt = 0; nt < NT / 2; ++nt) {
        const int h0 = 2 * nt, h1 = 2 * nt + 1;
        pb[nt][0] = movmatrix_trans(pack(pp[h0][0], pp[h1][0]));
        pb[nt][1] = movmatrix_trans(pack(pp[h0][1], pp[h1][1]));
        pb[nt + NT / 2][0] = movmatrix_trans(pack(lo_of(pp[h0][0]), lo_of(pp[h1][0])));
        pb[nt + NT / 2][1] = movmatrix_trans(pack(lo_of(pp[h0][1]), lo_of(pp[h1][1])));
      }
    }
  }
};

// INT2 state of a lane: heads 4 nt + tig (nt < G / 4), its tokens gid and
// gid + 8 of each page; acc[nt][mt] holds output channels 16 gid + mt
// (c < 2) and 16 gid + 8 + mt (c >= 2), columns hi (c even) and lo (c odd).
// z[nt][q]: the zero-point term sum p z_V of V group q.
template <int G, int NGV>
struct HistState {
  static constexpr int NH = Geo<G>::NH;
  float acc[NH][8][4];
  float m[NH], l[NH], z[NH][NGV];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int nt = 0; nt < NH; ++nt) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) acc[nt][mt][0] = acc[nt][mt][1] = acc[nt][mt][2] = acc[nt][mt][3] = 0.f;
      m[nt] = -INFINITY;
      l[nt] = 0.f;
#pragma unroll
      for (int q = 0; q < NGV; ++q) z[nt][q] = 0.f;
    }
  }
};

// QK of one INT2 page (one K group): d[nt] = 2^-24 sigma (q~ . c) of (token
// gid | gid + 8) x (head 4 nt + tig hi, lo), K-steps spread over kQkChains
// accumulators.
template <int G>
__device__ __forceinline__ void int2_qk(const uint8_t* __restrict__ pg, int gid, int tig,
                                        const uint32_t (&qb)[Geo<G>::NH][8][2], float (&d)[Geo<G>::NH][4]) {
  constexpr int NH = Geo<G>::NH, kQkChains = Geo<G>::kQkChains;
  const uint2 kw0 = *reinterpret_cast<const uint2*>(pg + 32 * gid + 8 * tig);
  const uint2 kw1 = *reinterpret_cast<const uint2*>(pg + 32 * (gid + 8) + 8 * tig);
  float dc[kQkChains][NH][4];
#pragma unroll
  for (int ch = 0; ch < kQkChains; ++ch)
#pragma unroll
    for (int nt = 0; nt < NH; ++nt) dc[ch][nt][0] = dc[ch][nt][1] = dc[ch][nt][2] = dc[ch][nt][3] = 0.f;
  const uint32_t w00 = kw0.x, w01 = kw0.y, w10 = kw1.x, w11 = kw1.y;
  const uint32_t s00 = w00 >> 6, s01 = w01 >> 6, s10 = w10 >> 6, s11 = w11 >> 6;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t a0 = code_pair(w00, s00, j), a1 = code_pair(w10, s10, j);
    const uint32_t a2 = code_pair(w01, s01, j), a3 = code_pair(w11, s11, j);
#pragma unroll
    for (int nt = 0; nt < NH; ++nt) mma_f16(dc[j % kQkChains][nt], a0, a1, a2, a3, qb[nt][j][0], qb[nt][j][1]);
  }
#pragma unroll
  for (int nt = 0; nt < NH; ++nt)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float v = dc[0][nt][c];
#pragma unroll
      for (int ch = 1; ch < kQkChains; ++ch) v += dc[ch][nt][c];
      d[nt][c] = v;
    }
}

// QK of one INT2 page with NGK > 1 K groups, each group folded into the
// score sums as soon as its K-steps are done (one live accumulator set):
// a[nt][t] = sum_q s_q 2^-24 sigma (q~ . c)_q of token gid (t = 0) or
// gid + 8 (t = 1).  The page format puts group q in K-steps q J .. q J + J - 1
// (J = 8 / NGK); ksz0 / ksz1: the tokens' (scale, zero) pairs.
template <int G, int NGK>
__device__ __forceinline__ void int2_qk_groups(const uint8_t* __restrict__ pg, int gid, int tig,
                                               const uint32_t (&qb)[Geo<G>::NH][8][2], const uint32_t (&ksz0)[NGK],
                                               const uint32_t (&ksz1)[NGK], float (&a)[Geo<G>::NH][2]) {
  constexpr int NH = Geo<G>::NH, J = 8 / NGK;
  const uint2 kw0 = *reinterpret_cast<const uint2*>(pg + 32 * gid + 8 * tig);
  const uint2 kw1 = *reinterpret_cast<const uint2*>(pg + 32 * (gid + 8) + 8 * tig);
  const uint32_t w00 = kw0.x, w01 = kw0.y, w10 = kw1.x, w11 = kw1.y;
  const uint32_t s00 = w00 >> 6, s01 = w01 >> 6, s10 = w10 >> 6, s11 = w11 >> 6;
#pragma unroll
  for (int nt = 0; nt < NH; ++nt) a[nt][0] = a[nt][1] = 0.f;
#pragma unroll
  for (int q = 0; q < NGK; ++q) {
    float dq[NH][4];
#pragma unroll
    for (int nt = 0; nt < NH; ++nt) dq[nt][0] = dq[nt][1] = dq[nt][2] = dq[nt][3] = 0.f;
#pragma unroll
    for (int jj = 0; jj < J; ++jj) {
      const int j = q * J + jj;
      const uint32_t a0 = code_pair(w00, s00, j), a1 = code_pair(w10, s10, j);
      const uint32_t a2 = code_pair(w01, s01, j), a3 = code_pair(w11, s11, j);
#pragma unroll
      for (int nt = 0; nt < NH; ++nt) mma_f16(dq[nt], a0, a1, a2, a3, qb[nt][j][0], qb[nt][j][1]);
    }
    const float2 kz0 = half2_to_float2(ksz0[q]), kz1 = half2_to_float2(ksz1[q]);
#pragma unroll
    for (int nt = 0; nt < NH; ++nt) {
      a[nt][0] = fmaf(kz0.x, dq[nt][0] + dq[nt][1], a[nt][0]);
      a[nt][1] = fmaf(kz1.x, dq[nt][2] + dq[nt][3], a[nt][1]);
    }
  }
}

// The (scale, zero) fp16 pairs of token slot t of a page block: NGK K pairs
// then NGV V pairs at kPairs + 4 (NGK + NGV) t.  load_pairs reads both sets
// (one 8-byte load with one group each); load_group_pairs reads N pairs
// from pair index `first` on.  The vector width of the loads is the largest
// that every token slot's address allows: A words apart, with A the largest
// power of two (at most 4) dividing both NGK + NGV and `first`.
constexpr int pair_align(int n, int first) {
  return (n % 4 == 0 && first % 4 == 0) ? 4 : (n % 2 == 0 && first % 2 == 0) ? 2 : 1;
}

template <int N, int A>
__device__ __forceinline__ void load_words(const uint8_t* a, uint32_t (&w)[N]) {
  constexpr int V = A < N ? A : (N % 4 == 0 ? 4 : N % 2 == 0 ? 2 : 1);
  static_assert(N % V == 0, "vector width divides the word count");
#pragma unroll
  for (int i = 0; i < N / V; ++i) {
    if constexpr (V == 4) {
      const uint4 v = reinterpret_cast<const uint4*>(a)[i];
      w[4 * i] = v.x;
      w[4 * i + 1] = v.y;
      w[4 * i + 2] = v.z;
      w[4 * i + 3] = v.w;
    } else if constexpr (V == 2) {
      const uint2 v = reinterpret_cast<const uint2*>(a)[i];
      w[2 * i] = v.x;
      w[2 * i + 1] = v.y;
    } else {
      w[i] = reinterpret_cast<const uint32_t*>(a)[i];
    }
  }
}

template <int NGK, int NGV>
__device__ __forceinline__ void load_pairs(const uint8_t* pg, int t, uint32_t (&ksz)[NGK], uint32_t (&vsz)[NGV]) {
  constexpr int N = NGK + NGV;
  uint32_t w[N];
  load_words<N, pair_align(N, 0)>(pg + kPairs + 4 * N * t, w);
#pragma unroll
  for (int q = 0; q < NGK; ++q) ksz[q] = w[q];
#pragma unroll
  for (int q = 0; q < NGV; ++q) vsz[q] = w[NGK + q];
}

template <int NGK, int NGV, int kFirst, int N>
__device__ __forceinline__ void load_group_pairs(const uint8_t* pg, int t, uint32_t (&sz)[N]) {
  load_words<N, pair_align(NGK + NGV, kFirst)>(pg + kPairs + 4 * (NGK + NGV) * t + 4 * kFirst, sz);
}

// Scores (log2 units) of the lane's two tokens of one page from its QK
// accumulators and the tokens' K (scale, zero); -inf where not valid.
// kMasked = false: every token of the page is valid (no selects).
// Scores (log2 units) of the lane's two tokens of one page from its QK
// accumulators and the tokens' K (scale, zero); -inf where not valid.
// kMasked = false: every token of the page is valid (no selects).
template <int G, bool kMasked>
__device__ __forceinline__ void int2_scores(const float (&d)[Geo<G>::NH][4], uint32_t ksz0, uint32_t ksz1,
                                            bool ok0, bool ok1, const float (&uns)[Geo<G>::NH],
                                            const float (&qz)[Geo<G>::NH][1], float (&sc)[Geo<G>::NH][2]) {
  const float2 kz0 = half2_to_float2(ksz0), kz1 = half2_to_float2(ksz1);
#pragma unroll
  for (int nt = 0; nt < Geo<G>::NH; ++nt) {
    const float s0 = fmaf(kz0.x * (d[nt][0] + d[nt][1]), uns[nt], kz0.y * qz[nt][0]);
    const float s1 = fmaf(kz1.x * (d[nt][2] + d[nt][3]), uns[nt], kz1.y * qz[nt][0]);
    sc[nt][0] = (!kMasked || ok0) ? s0 : -INFINITY;
    sc[nt][1] = (!kMasked || ok1) ? s1 : -INFINITY;
  }
}

// With NGK > 1 groups: score = unscale sum_q s_q (q~ . c)_q + sum_q z_q qz_q,
// from the folded sums of int2_qk_groups.
template <int G, int NGK, bool kMasked>
__device__ __forceinline__ void int2_scores_groups(const float (&a)[Geo<G>::NH][2], const uint32_t (&ksz0)[NGK],
                                                   const uint32_t (&ksz1)[NGK], bool ok0, bool ok1,
                                                   const float (&uns)[Geo<G>::NH],
                                                   const float (&qz)[Geo<G>::NH][NGK], float (&sc)[Geo<G>::NH][2]) {
#pragma unroll
  for (int nt = 0; nt < Geo<G>::NH; ++nt) {
    float z0 = 0.f, z1 = 0.f;
#pragma unroll
    for (int q = 0; q < NGK; ++q) {
      z0 = fmaf(half2_to_float2(ksz0[q]).y, qz[nt][q], z0);
      z1 = fmaf(half2_to_float2(ksz1[q]).y, qz[nt][q], z1);
    }
    const float s0 = fmaf(a[nt][0], uns[nt], z0), s1 = fmaf(a[nt][1], uns[nt], z1);
    sc[nt][0] = (!kMasked || ok0) ? s0 : -INFINITY;
    sc[nt][1] = (!kMasked || ok1) ? s1 : -INFINITY;
  }
}

// Lazy online-softmax maximum over a step's scores: raised only when a score
// exceeds it by 2^kRescaleLog2; the 8 lanes of a column group share a head.
// The INT2 state keeps its maximum lowered by pv_log2 (st.m = max - pv_log2),
// so that p = 2^(s - st.m) carries the PV operand scale 2^pv_log2 with it;
// `lift` = kRescaleLog2 + pv_log2.
template <int G, int NGV, int P>
__device__ __forceinline__ void int2_update_max(const float (&sc)[P][Geo<G>::NH][2], HistState<G, NGV>& st,
                                                float pv_log2, float lift) {
  constexpr int NH = Geo<G>::NH;
  bool need = false;
#pragma unroll
  for (int pg = 0; pg < P; ++pg)
#pragma unroll
    for (int nt = 0; nt < NH; ++nt) need |= fmaxf(sc[pg][nt][0], sc[pg][nt][1]) > st.m[nt] + lift;
  if (!__any_sync(kFull, need)) return;
#pragma unroll
  for (int nt = 0; nt < NH; ++nt) {
    float pm = fmaxf(sc[0][nt][0], sc[0][nt][1]);
#pragma unroll
    for (int pg = 1; pg < P; ++pg) pm = fmaxf(pm, fmaxf(sc[pg][nt][0], sc[pg][nt][1]));
    pm = fmaxf(pm, __shfl_xor_sync(kFull, pm, 4));
    pm = fmaxf(pm, __shfl_xor_sync(kFull, pm, 8));
    pm = fmaxf(pm, __shfl_xor_sync(kFull, pm, 16));
    pm -= pv_log2;
    if (pm > st.m[nt]) {
      const float f = exp2f(st.m[nt] - pm);
      st.m[nt] = pm;
      st.l[nt] *= f;
#pragma unroll
      for (int q = 0; q < NGV; ++q) st.z[nt][q] *= f;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        st.acc[nt][mt][0] *= f;
        st.acc[nt][mt][1] *= f;
        st.acc[nt][mt][2] *= f;
        st.acc[nt][mt][3] *= f;
      }
    }
  }
}

// Probabilities of one page -> PV B fragments: the lane packs (hi, lo) of
// p s_V for token gid (row gid, columns 2 tig, 2 tig + 1) and token gid + 8,
// with p = 2^(s - st.m) already carrying the operand scale 2^pv_log2;
// movmatrix transposes them into the B layout (rows = tokens).  With NGV
// groups there is one operand per V group q (its own s_V), and the
// zero-point term accumulates per group.
// (kMasked = false: every token valid, so stale ring bytes never reach a
// product and no select is needed.)
template <int G, int NGV, bool kMasked>
__device__ __forceinline__ void int2_probs(const float (&sc)[Geo<G>::NH][2], const uint32_t (&vsz0)[NGV],
                                           const uint32_t (&vsz1)[NGV], bool ok0, bool ok1,
                                           HistState<G, NGV>& st, uint32_t (&pb)[NGV][Geo<G>::NH][2]) {
  float2 vz0[NGV], vz1[NGV];
#pragma unroll
  for (int q = 0; q < NGV; ++q) {
    vz0[q] = half2_to_float2(vsz0[q]);
    vz1[q] = half2_to_float2(vsz1[q]);
  }
#pragma unroll
  for (int nt = 0; nt < Geo<G>::NH; ++nt) {
    float p0 = fast_exp2(sc[nt][0] - st.m[nt]);
    float p1 = fast_exp2(sc[nt][1] - st.m[nt]);
    if constexpr (kMasked) {
      p0 = ok0 ? p0 : 0.f;
      p1 = ok1 ? p1 : 0.f;
    }
    st.l[nt] += p0 + p1;
#pragma unroll
    for (int q = 0; q < NGV; ++q) {
      float q0, q1;
      if constexpr (kMasked) {
        st.z[nt][q] += (ok0 ? p0 * vz0[q].y : 0.f) + (ok1 ? p1 * vz1[q].y : 0.f);
        q0 = ok0 ? p0 * vz0[q].x : 0.f;
        q1 = ok1 ? p1 * vz1[q].x : 0.f;
      } else {
        st.z[nt][q] = fmaf(p0, vz0[q].y, fmaf(p1, vz1[q].y, st.z[nt][q]));
        q0 = p0 * vz0[q].x;
        q1 = p1 * vz1[q].x;
      }
      pb[q][nt][0] = movmatrix_trans(split_hi_lo(q0));
      pb[q][nt][1] = movmatrix_trans(split_hi_lo(q1));
    }
  }
}

// PV of one INT2 page: acc[nt][mt] += codes^T . P, code positions 16 gid + mt
// (+8); 16-row tile mt holds V group mt / (8 / NGV) (the page format's code
// order) and takes that group's operand.  The V rows interleave slot pairs
// by 16-bit halves, so the words at 64 a + 8 gid hold halves 2 gid and
// 2 gid + 1 (code positions 16 gid .. 16 gid + 15) of tokens 2a and 2a + 1:
// the lane's A operand rows, one 8-byte load per token pair.
template <int G, int NGV>
__device__ __forceinline__ void int2_pv(const uint8_t* __restrict__ pg, int gid, int tig,
                                        const uint32_t (&pb)[NGV][Geo<G>::NH][2], HistState<G, NGV>& st) {
  const uint8_t* pv = pg + kVCodes;
  const uint2 w0 = *reinterpret_cast<const uint2*>(pv + 64 * tig + 8 * gid);
  const uint2 w8 = *reinterpret_cast<const uint2*>(pv + 64 * (tig + 4) + 8 * gid);
  const uint32_t x0l = w0.x, x0h = w0.y, x8l = w8.x, x8h = w8.y;
  const uint32_t y0l = x0l >> 6, y0h = x0h >> 6, y8l = x8l >> 6, y8h = x8h >> 6;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const uint32_t a0 = code_pair(x0l, y0l, mt), a1 = code_pair(x0h, y0h, mt);
    const uint32_t a2 = code_pair(x8l, y8l, mt), a3 = code_pair(x8h, y8h, mt);
    const int q = mt / (8 / NGV);
#pragma unroll
    for (int nt = 0; nt < Geo<G>::NH; ++nt) mma_f16(st.acc[nt][mt], a0, a1, a2, a3, pb[q][nt][0], pb[q][nt][1]);
  }
}

// INT2 warp state -> ws[h * kPartStride + (0, 1, 4 + channel)] in the
// rotated basis: o~ = (hi + lo) 2^24 4^-pos(mt) + zeta_q, where code position
// c = 16 gid + mt (+8) holds the page format's V channel.  Every term of the
// state carries the factor 2^pv_log2 and its maximum is lowered by pv_log2,
// so (m, l, o~) is a softmax state like any other.
template <int G, int NGV>
__device__ __forceinline__ void store_hist_state(HistState<G, NGV>& st, float* ws, int gid, int tig,
                                                 float pv_unscale) {
  constexpr int NH = Geo<G>::NH;
#pragma unroll
  for (int nt = 0; nt < NH; ++nt) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      st.l[nt] += __shfl_xor_sync(kFull, st.l[nt], o);
#pragma unroll
      for (int q = 0; q < NGV; ++q) st.z[nt][q] += __shfl_xor_sync(kFull, st.z[nt][q], o);
    }
    const int h = 4 * nt + tig;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const float f = pv_unscale * __int_as_float((127 - 2 * code_pos(mt)) << 23);
      const float zq = st.z[nt][mt / (8 / NGV)];
      const int c0 = storage_channel_v(NGV, 16 * gid + mt), c8 = storage_channel_v(NGV, 16 * gid + 8 + mt);
      ws[h * kPartStride + 4 + c0] = fmaf(st.acc[nt][mt][0] + st.acc[nt][mt][1], f, zq);
      ws[h * kPartStride + 4 + c8] = fmaf(st.acc[nt][mt][2] + st.acc[nt][mt][3], f, zq);
    }
    if (gid == 0) {
      ws[h * kPartStride + 0] = st.m[nt];
      ws[h * kPartStride + 1] = st.l[nt];
    }
  }
}

// ---------------------------------------------------------------- codebook levels
// A code c = b0 + 2 b1 with level l[c] = l_0 + d1 c + a2 (2 b1) + b (b0 b1):
// the three bit planes c, 2 b1 and b0 b1 are taken by single ANDs at the
// positions code_pair uses (so they meet the same B fragments), with b0 b1
// read from t = w & (w >> 1).

__device__ __forceinline__ uint32_t plane_pair(uint32_t w, uint32_t wsh, int j, uint32_t m) {
  return j < 5 ? (w & (m << (2 * j))) : (wsh & (m << (2 * (j - 3))));
}

// QK of one page with levels: e[nt][t] = sum over planes k = (c, 2 b1, b0 b1)
// of coef[1 + k] 2^-24 sigma (q~ . plane_k) of token gid (t = 0) or gid + 8,
// the planes taken one after another and folded (one live accumulator set).
template <int G>
__device__ __forceinline__ void int2_qk_levels(const uint8_t* __restrict__ pg, int gid, int tig,
                                               const uint32_t (&qb)[Geo<G>::NH][8][2], const float* coef,
                                               float (&e)[Geo<G>::NH][2]) {
  constexpr int NH = Geo<G>::NH;
  const uint2 kw0 = *reinterpret_cast<const uint2*>(pg + 32 * gid + 8 * tig);
  const uint2 kw1 = *reinterpret_cast<const uint2*>(pg + 32 * (gid + 8) + 8 * tig);
  const uint32_t w[4] = {kw0.x, kw1.x, kw0.y, kw1.y};   // a0, a1, a2, a3 sources
#pragma unroll
  for (int nt = 0; nt < NH; ++nt) e[nt][0] = e[nt][1] = 0.f;
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    uint32_t src[4], sh[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      src[r] = k == 2 ? (w[r] & (w[r] >> 1)) : w[r];
      sh[r] = src[r] >> 6;
    }
    const uint32_t m = k == 0 ? 0x00030003u : k == 1 ? 0x00020002u : 0x00010001u;
    float d[NH][4];
#pragma unroll
    for (int nt = 0; nt < NH; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t a0 = plane_pair(src[0], sh[0], j, m), a1 = plane_pair(src[1], sh[1], j, m);
      const uint32_t a2 = plane_pair(src[2], sh[2], j, m), a3 = plane_pair(src[3], sh[3], j, m);
#pragma unroll
      for (int nt = 0; nt < NH; ++nt) mma_f16(d[nt], a0, a1, a2, a3, qb[nt][j][0], qb[nt][j][1]);
    }
#pragma unroll
    for (int nt = 0; nt < NH; ++nt) {
      e[nt][0] = fmaf(coef[1 + k], d[nt][0] + d[nt][1], e[nt][0]);
      e[nt][1] = fmaf(coef[1 + k], d[nt][2] + d[nt][3], e[nt][1]);
    }
  }
}

// Scores with levels: q~ . k^ = s (d1 S_c + a2 S_2b1 + b S_b0b1) + (z + s l_0) sum q~.
template <int G, bool kMasked>
__device__ __forceinline__ void int2_scores_levels(const float (&e)[Geo<G>::NH][2], uint32_t ksz0, uint32_t ksz1,
                                                   bool ok0, bool ok1, const float (&uns)[Geo<G>::NH],
                                                   const float (&qz)[Geo<G>::NH][1], const float* coef,
                                                   float (&sc)[Geo<G>::NH][2]) {
  const float2 kz0 = half2_to_float2(ksz0), kz1 = half2_to_float2(ksz1);
  const float z0 = fmaf(kz0.x, coef[0], kz0.y), z1 = fmaf(kz1.x, coef[0], kz1.y);
#pragma unroll
  for (int nt = 0; nt < Geo<G>::NH; ++nt) {
    const float s0 = fmaf(kz0.x * e[nt][0], uns[nt], z0 * qz[nt][0]);
    const float s1 = fmaf(kz1.x * e[nt][1], uns[nt], z1 * qz[nt][0]);
    sc[nt][0] = (!kMasked || ok0) ? s0 : -INFINITY;
    sc[nt][1] = (!kMasked || ok1) ? s1 : -INFINITY;
  }
}

// Probabilities with levels: z[nt][0] += sum p z_V, z[nt][1] += sum p s_V (the
// l_0 part), and one PV operand per plane k: p s_V coef[1 + k] (p carries
// the operand scale 2^pv_log2).
template <int G, bool kMasked>
__device__ __forceinline__ void int2_probs_levels(const float (&sc)[Geo<G>::NH][2], uint32_t vsz0, uint32_t vsz1,
                                                  bool ok0, bool ok1, const float* coef,
                                                  HistState<G, 2>& st, uint32_t (&pb)[3][Geo<G>::NH][2]) {
  const float2 vz0 = half2_to_float2(vsz0), vz1 = half2_to_float2(vsz1);
#pragma unroll
  for (int nt = 0; nt < Geo<G>::NH; ++nt) {
    float p0 = fast_exp2(sc[nt][0] - st.m[nt]);
    float p1 = fast_exp2(sc[nt][1] - st.m[nt]);
    float q0, q1;
    if constexpr (kMasked) {
      // a masked token's (scale, zero) may be stale ring bytes: selects, not
      // products with p = 0
      p0 = ok0 ? p0 : 0.f;
      p1 = ok1 ? p1 : 0.f;
      st.l[nt] += p0 + p1;
      st.z[nt][0] += (ok0 ? p0 * vz0.y : 0.f) + (ok1 ? p1 * vz1.y : 0.f);
      st.z[nt][1] += (ok0 ? p0 * vz0.x : 0.f) + (ok1 ? p1 * vz1.x : 0.f);
      q0 = ok0 ? p0 * vz0.x : 0.f;
      q1 = ok1 ? p1 * vz1.x : 0.f;
    } else {
      st.l[nt] += p0 + p1;
      st.z[nt][0] = fmaf(p0, vz0.y, fmaf(p1, vz1.y, st.z[nt][0]));
      st.z[nt][1] = fmaf(p0, vz0.x, fmaf(p1, vz1.x, st.z[nt][1]));
      q0 = p0 * vz0.x;
      q1 = p1 * vz1.x;
    }
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      pb[k][nt][0] = movmatrix_trans(split_hi_lo(q0 * coef[1 + k]));
      pb[k][nt][1] = movmatrix_trans(split_hi_lo(q1 * coef[1 + k]));
    }
  }
}

// PV with levels: acc += sum over planes of plane^T . pb[plane].
template <int G>
__device__ __forceinline__ void int2_pv_levels(const uint8_t* __restrict__ pg, int gid, int tig,
                                               const uint32_t (&pb)[3][Geo<G>::NH][2], HistState<G, 2>& st) {
  const uint8_t* pv = pg + kVCodes;
  const uint2 w0 = *reinterpret_cast<const uint2*>(pv + 64 * tig + 8 * gid);
  const uint2 w8 = *reinterpret_cast<const uint2*>(pv + 64 * (tig + 4) + 8 * gid);
  const uint32_t x[4] = {w0.x, w0.y, w8.x, w8.y};
  uint32_t xs[4], t[4], ts[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    xs[r] = x[r] >> 6;
    t[r] = x[r] & (x[r] >> 1);
    ts[r] = t[r] >> 6;
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    uint32_t a[3][4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      a[0][r] = plane_pair(x[r], xs[r], mt, 0x00030003u);
      a[1][r] = plane_pair(x[r], xs[r], mt, 0x00020002u);
      a[2][r] = plane_pair(t[r], ts[r], mt, 0x00010001u);
    }
#pragma unroll
    for (int k = 0; k < 3; ++k)
#pragma unroll
      for (int nt = 0; nt < Geo<G>::NH; ++nt)
        mma_f16(st.acc[nt][mt], a[k][0], a[k][1], a[k][2], a[k][3], pb[k][nt][0], pb[k][nt][1]);
  }
}

// INT2 warp state with levels -> ws: o~ = (hi + lo) 2^24 4^-pos(mt)
// + sum p z_V + l_0 sum p s_V (every term carries 2^pv_log2, as above).
template <int G>
__device__ __forceinline__ void store_hist_state_levels(HistState<G, 2>& st, float* ws, int gid, int tig,
                                                        float pv_unscale, float l0) {
  constexpr int NH = Geo<G>::NH;
#pragma unroll
  for (int nt = 0; nt < NH; ++nt) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      st.l[nt] += __shfl_xor_sync(kFull, st.l[nt], o);
      st.z[nt][0] += __shfl_xor_sync(kFull, st.z[nt][0], o);
      st.z[nt][1] += __shfl_xor_sync(kFull, st.z[nt][1], o);
    }
    const int h = 4 * nt + tig;
    const float zt = fmaf(l0, st.z[nt][1], st.z[nt][0]);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const float f = pv_unscale * __int_as_float((127 - 2 * code_pos(mt)) << 23);
      ws[h * kPartStride + 4 + 16 * gid + mt] = fmaf(st.acc[nt][mt][0] + st.acc[nt][mt][1], f, zt);
      ws[h * kPartStride + 4 + 16 * gid + 8 + mt] = fmaf(st.acc[nt][mt][2] + st.acc[nt][mt][3], f, zt);
    }
    if (gid == 0) {
      ws[h * kPartStride + 0] = st.m[nt];
      ws[h * kPartStride + 1] = st.l[nt];
    }
  }
}

// ------------------------------------------------------------------ BF16 page

template <int G>
__device__ __forceinline__ void bf16_page(const uint16_t* const (&krow)[2],
                                          const uint16_t* const (&vrow)[4], const bool (&kok)[2],
                                          const bool (&vok)[4], int gid, int tig,
                                          const uint32_t (&qf)[Geo<G>::NTQ][8][2],
                                          WarpState<G>& st) {
  constexpr int NT = Geo<G>::NT, HS = Geo<G>::HS, NTQ = Geo<G>::NTQ;
  const float scale = kLog2e * rsqrtf(float(kHeadDim));
  float d[NTQ][4];
#pragma unroll
  for (int nt = 0; nt < NTQ; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint4 k0[2], k1[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      k0[u] = __ldg(reinterpret_cast<const uint4*>(krow[0] + 32 * tig + 16 * half + 8 * u));
      k1[u] = __ldg(reinterpret_cast<const uint4*>(krow[1] + 32 * tig + 16 * half + 8 * u));
    }
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int j = 4 * half + jj;
      const uint4& a = k0[jj >> 1];
      const uint4& b = k1[jj >> 1];
      const uint32_t a0 = (jj & 1) ? a.z : a.x, a2 = (jj & 1) ? a.w : a.y;
      const uint32_t a1 = (jj & 1) ? b.z : b.x, a3 = (jj & 1) ? b.w : b.y;
#pragma unroll
      for (int nt = 0; nt < NTQ; ++nt) mma_bf16(d[nt], a0, a1, a2, a3, qf[nt][j][0], qf[nt][j][1]);
    }
  }
  float sc[HS][2];
  if (G <= 4) {
#pragma unroll
    for (int c = 0; c < 4; ++c) sc[c & 1][c >> 1] = d[0][c] * scale;
  } else {
#pragma unroll
    for (int nt = 0; nt < NTQ; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) sc[2 * nt + (c & 1)][c >> 1] = d[nt][c] * scale;
  }
#pragma unroll
  for (int hs = 0; hs < HS; ++hs) {
    if (!kok[0]) sc[hs][0] = -INFINITY;
    if (!kok[1]) sc[hs][1] = -INFINITY;
  }
  st.update_max(sc);
  float pp[HS][2];
#pragma unroll
  for (int hs = 0; hs < HS; ++hs) {
    pp[hs][0] = kok[0] ? exp2f(sc[hs][0] - st.m[hs]) : 0.f;
    pp[hs][1] = kok[1] ? exp2f(sc[hs][1] - st.m[hs]) : 0.f;
    st.l[hs] += pp[hs][0] + pp[hs][1];
  }
  uint32_t pb[NT][2];
  st.template pv_operand<false>(pp, tig, pb);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint4 v[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      v[t] = vok[t] ? __ldg(reinterpret_cast<const uint4*>(vrow[t] + 16 * gid + 8 * half))
                    : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int mm = 0; mm < 4; ++mm) {
      const int mt = 4 * half + mm;
      const uint32_t wa = mm == 0 ? v[0].x : mm == 1 ? v[0].y : mm == 2 ? v[0].z : v[0].w;
      const uint32_t wb = mm == 0 ? v[1].x : mm == 1 ? v[1].y : mm == 2 ? v[1].z : v[1].w;
      const uint32_t wc = mm == 0 ? v[2].x : mm == 1 ? v[2].y : mm == 2 ? v[2].z : v[2].w;
      const uint32_t wd = mm == 0 ? v[3].x : mm == 1 ? v[3].y : mm == 2 ? v[3].z : v[3].w;
      const uint32_t a0 = prmt(wa, wb, 0x5410), a1 = prmt(wa, wb, 0x7632);
      const uint32_t a2 = prmt(wc, wd, 0x5410), a3 = prmt(wc, wd, 0x7632);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_bf16(st.acc[nt][mt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
    }
  }
}

// ------------------------------------------------------------------ warp -> smem state

// kInt2: channel of (mt, c) is 16gid + mt (+8 for c >= 2), value scaled by
// 2^24 4^-pos(mt) plus the zero-point term; BF16: 16gid + 2mt (+1).
template <int G, bool kInt2>
__device__ __forceinline__ void store_warp_state(WarpState<G>& st, float* ws, int gid, int tig,
                                                 float pv_unscale) {
  constexpr int NT = Geo<G>::NT, HS = Geo<G>::HS;
#pragma unroll
  for (int hs = 0; hs < HS; ++hs) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      st.l[hs] += __shfl_xor_sync(kFull, st.l[hs], o);
      st.z[hs] += __shfl_xor_sync(kFull, st.z[hs], o);
    }
  }
  if (G <= 4) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        st.acc[0][mt][c] += __shfl_xor_sync(kFull, st.acc[0][mt][c], G / 2);
  } else {
#pragma unroll
    for (int nt = 0; nt < NT / 2; ++nt)
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int c = 0; c < 4; ++c) st.acc[nt][mt][c] += st.acc[nt + NT / 2][mt][c];
  }
  if (G <= 4 && tig >= G / 2) return;
  constexpr int NHI = G <= 4 ? 1 : NT / 2;
#pragma unroll
  for (int nt = 0; nt < NHI; ++nt) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const float f = kInt2 ? pv_unscale * ldexpf(1.f, -2 * code_pos(mt)) : 1.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int hs = acc_slot<G>(nt, c);
        const int h = slot_head<G>(tig, hs);
        const int ch = kInt2 ? 16 * gid + mt + (c >= 2 ? 8 : 0) : 16 * gid + 2 * mt + (c >= 2 ? 1 : 0);
        ws[h * kPartStride + 4 + ch] = kInt2 ? fmaf(st.acc[nt][mt][c], f, st.z[hs]) : st.acc[nt][mt][c];
      }
    }
  }
  if (gid == 0) {
#pragma unroll
    for (int hs = 0; hs < HS; ++hs) {
      const int h = slot_head<G>(tig, hs);
      ws[h * kPartStride + 0] = st.m[hs];
      ws[h * kPartStride + 1] = st.l[hs];
    }
  }
}

// ------------------------------------------------------------------ q~ and its fragments

// Shared-memory scratch of the prologue, in floats: qs[G][128] | part[4][G][128]
// | qt[G][128] | aux[G][8] | red[2][G][4] | frag[32][NH*16] (u32).
template <int G>
struct QScratch {
  static constexpr int kQs = 0, kPart = G * kHeadDim, kQt = 5 * G * kHeadDim, kAux = 6 * G * kHeadDim;
  static constexpr int kRed = kAux + 8 * G, kFrag = kRed + 8 * G;
  static constexpr int kFloats = kFrag + 32 * Geo<G>::NH * 16;
  static_assert(kFrag % 4 == 0, "fragment rows are read as uint4");
};

// q~ = q . R_K for the G query heads of (b, hkv) in fp32 (fixed summation
// order) from R_K and q already in shared memory (`rks` by a TMA issued at
// kernel start, qs filled at kernel start).  Per head a power-of-two scale sigma puts max|q~ sigma| in
// [2^13, 2^14) so the fp16 hi part is normal and the lo part precise.  The
// 32 lanes' B fragments of the QK MMA are built once per CTA: column
// gid of column tile nt is the hi (gid even) or lo (gid odd) part of head
// 4 nt + gid / 2; register r = 0 holds channels (32tig + j, 32tig + j + 8),
// r = 1 (32tig + 16 + j, 32tig + 24 + j), each scaled by sigma 4^-pos(j);
// these are code positions, holding the page format's K channels for NGK
// groups.  aux[h] = (sigma, unscale, qz[0 .. NGK-1]), qz[q] the scaled sum
// of q~ over K group q.
template <int G, int NGK>
__device__ void rotate_query(const DecodeParams& p, int b, int hkv, const float* rks, uint64_t* rbar,
                             float* scratch) {
  constexpr int T = Geo<G>::PT, NH = Geo<G>::NH;
  using S = QScratch<G>;
  static_assert(S::kFloats * 4 <= Geo<G>::kQScratch, "prologue scratch");
  float* qs = scratch + S::kQs;
  float* part = scratch + S::kPart;
  float* qt = scratch + S::kQt;
  float* aux = scratch + S::kAux;
  float* red = scratch + S::kRed;
  uint32_t* frag = reinterpret_cast<uint32_t*>(scratch + S::kFrag);
  const int tid = threadIdx.x;
  named_barrier(kPrologueBarrier, T);   // qs was filled at kernel start
  if (!mbar_wait_bounded(rbar, 0, kWaitLimitNs) && tid == 0) flag(p.dev_status, 0x4);
  for (int task = tid; task < 4 * kHeadDim; task += T) {
    const int ig = task / kHeadDim, j = task % kHeadDim;
    float acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = 0.f;
#pragma unroll 2
    for (int i4 = 0; i4 < 8; ++i4) {
      const int i0 = 32 * ig + 4 * i4;
      const float r0 = rks[(i0 + 0) * kHeadDim + j], r1 = rks[(i0 + 1) * kHeadDim + j];
      const float r2 = rks[(i0 + 2) * kHeadDim + j], r3 = rks[(i0 + 3) * kHeadDim + j];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float4 qv = *reinterpret_cast<const float4*>(qs + h * kHeadDim + i0);
        acc[h] = fmaf(qv.w, r3, fmaf(qv.z, r2, fmaf(qv.y, r1, fmaf(qv.x, r0, acc[h]))));
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) part[(ig * G + h) * kHeadDim + j] = acc[h];
  }
  named_barrier(kPrologueBarrier, T);
  for (int idx = tid; idx < G * kHeadDim; idx += T) {
    const float v = ((part[idx] + part[G * kHeadDim + idx]) + part[2 * G * kHeadDim + idx]) +
                    part[3 * G * kHeadDim + idx];
    qt[idx] = v;
    float mx = fabsf(v), sm = v;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
      sm += __shfl_xor_sync(kFull, sm, o);
    }
    if ((idx & 31) == 0) {
      red[(idx >> 7) * 4 + ((idx >> 5) & 3)] = mx;
      red[4 * G + (idx >> 7) * 4 + ((idx >> 5) & 3)] = sm;
    }
  }
  named_barrier(kPrologueBarrier, T);
  // sigma = 2^e of head h, max|q~ sigma| in [2^13, 2^14): e from the exponent
  // field of the head's maximum (the frexp exponent is that field - 126)
  auto sigma_exp = [&](int h) {
    const float mx = fmaxf(fmaxf(red[h * 4], red[h * 4 + 1]), fmaxf(red[h * 4 + 2], red[h * 4 + 3]));
    const int e = mx > 0.f ? 14 - (((__float_as_int(mx) >> 23) & 255) - 126) : 0;
    return max(-100, min(100, e));
  };
  if (tid < G) {
    // sums of q~ over 32-channel chunks; K group q spans chunks
    // [q 4 / NGK, (q + 1) 4 / NGK)
    const float* rs = red + 4 * G + tid * 4;
    const int e = sigma_exp(tid);
    const float scale = kLog2e * rsqrtf(float(kHeadDim));
    aux[tid * 8 + 0] = __int_as_float((127 + e) << 23);
    aux[tid * 8 + 1] = __int_as_float((151 - e) << 23) * scale;   // 2^24 / sigma * log2(e) / sqrt(d)
    if constexpr (NGK == 1) {
      aux[tid * 8 + 2] = (((rs[0] + rs[1]) + rs[2]) + rs[3]) * scale;
    } else if constexpr (NGK == 2) {
      aux[tid * 8 + 2] = (rs[0] + rs[1]) * scale;
      aux[tid * 8 + 3] = (rs[2] + rs[3]) * scale;
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) aux[tid * 8 + 2 + q] = rs[q] * scale;
    }
  }
  for (int idx = tid; idx < 32 * NH * 16; idx += T) {
    const int ln = idx / (NH * 16), rem = idx % (NH * 16);
    const int nt = rem / 16, j = (rem / 2) % 8, rr = rem % 2;
    const int gid = ln >> 2, tig = ln & 3;
    const int h = 4 * nt + gid / 2;
    const float f = __int_as_float((127 + sigma_exp(h) - 2 * code_pos(j)) << 23);   // sigma 4^-pos(j)
    const int c0 = 32 * tig + 16 * rr + j;   // code position; +8: the pair's second
    float v0 = qt[h * kHeadDim + storage_channel_k(NGK, c0)] * f;
    float v1 = qt[h * kHeadDim + storage_channel_k(NGK, c0 + 8)] * f;
    if (gid & 1) {
      v0 = split_lo(v0);
      v1 = split_lo(v1);
    }
    frag[idx] = pack_half2(v0, v1);
  }
  named_barrier(kPrologueBarrier, T);
}

// ------------------------------------------------------------------ split kernel

// kLevels: codebook levels (one quantisation group per vector only).
template <int G, int NGK, int NGV, bool kLevels>
__global__ void __launch_bounds__(Geo<G>::T, 1) split_kernel(const __grid_constant__ DecodeParams p) {
  using Gm = Geo<G, NGK, NGV, kLevels>;
  static_assert(!kLevels || (NGK == 1 && NGV == 1), "codebook levels with one group per vector");
  constexpr int NZ = kLevels ? 2 : NGV;   // zero-point sums per head
  constexpr int NTQ = Geo<G>::NTQ, W = Geo<G>::W, T = Geo<G>::T;
  constexpr int kStages = Gm::kStages;
  constexpr int kParts = Gm::kParts;
  constexpr int kBlock = Gm::kBlock;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stage = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Gm::kStageBytes);
  uint64_t* rbar = bars + W * kStages;       // R_K; rbar + 1: R_V
  uint8_t* uni = smem + Gm::kStageBytes + Gm::kBarBytes;
  uni += (1024u - (smem_addr(uni) & 1023u)) & 1023u;
  float* rks = reinterpret_cast<float*>(uni);                         // prologue only
  float* qscratch = reinterpret_cast<float*>(uni + Geo<G>::kRotBytes);
  float* st_bf16x = reinterpret_cast<float*>(uni + Geo<G>::kUnion);   // [kBf16Warps][G][kPartStride]
  int* s_last = reinterpret_cast<int*>(uni + Geo<G>::kUnion + Geo<G>::kBf16State);
  uint64_t* pro_done = bars + W * kStages + 2;   // q~ fragments ready (after R_K, R_V)
  constexpr int PT = Geo<G>::PT;

  // grid (KV head, request, split): CTAs start split-major, so the first
  // splits of every request (full when its history reaches past them) go
  // first and the shorter or empty later splits fill the last waves
  const int split = blockIdx.z, hkv = blockIdx.x, b = blockIdx.y;
  const int pair = b * p.n_kv + hkv;
  const int n_splits = p.n_splits;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool bf16_warp = warp >= W - kBf16Warps;
  const int gid = lane >> 2, tig = lane & 3;
  const int pbeg = split * p.pages_per_split;
  // L2 prefetch of what the first phases read (R_K, this split's page-table
  // entries, the query rows, the lengths): hints that read nothing, so they
  // may precede the wait for the previous kernel
  if (pbeg < p.max_pages) {
    const char* rk = reinterpret_cast<const char*>(p.r_k + int64_t(hkv) * kHeadDim * kHeadDim);
    for (int i = tid; i < kHeadDim * kHeadDim * 4 / 128; i += T)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(rk + 128 * i));
    if (warp == W - 1) {
      const int32_t* row = p.page_table + int64_t(b) * p.max_pages + pbeg;
      const int n = min(p.pages_per_split, p.max_pages - pbeg);
      for (int i = 32 * lane; i < n; i += 32 * 32) asm volatile("prefetch.global.L2 [%0];" ::"l"(row + i));
      if (lane < 2 * G)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p.q + (int64_t(b) * p.n_kv * G + int64_t(hkv) * G) * kHeadDim + 64 * lane));
      if (lane == 0) {
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p.hist_len + b));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p.sink_len + b));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p.recent_len + b));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p.recent_start + b));
      }
    }
  }
  if (bf16_warp) {
    // the K and V rows of this warp's BF16 virtual pages (lane: token
    // lane % 16, K or V, both 128-byte lines of the row); the ring start
    // is read ahead of the wait only to place these hints, so a stale
    // value costs nothing but useless lines
    const int bw = warp - (W - kBf16Warps);
    const int n_vp = p.sink_cap / kPage + p.recent_cap / kPage;
    int start = 0;
    if (p.recent_cap > 0) {
      start = *reinterpret_cast<const volatile int32_t*>(p.recent_start + b) % p.recent_cap;
      start += start < 0 ? p.recent_cap : 0;
    }
    const int64_t hstride = int64_t(p.n_kv) * kHeadDim;
    for (int vp = split + bw * n_splits; vp < n_vp; vp += kBf16Warps * n_splits) {
      const int u = vp * kPage + (lane & 15);
      const bool kv = lane >= 16;
      const uint16_t* a;
      if (u < p.sink_cap) {
        a = (kv ? p.sink_v : p.sink_k) + (int64_t(b) * p.sink_cap + u) * hstride;
      } else {
        const int slot = (start + u - p.sink_cap) % p.recent_cap;
        a = (kv ? p.recent_v : p.recent_k) + (int64_t(b) * p.recent_cap + slot) * hstride;
      }
      a += int64_t(hkv) * kHeadDim;
      asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
      asm volatile("prefetch.global.L2 [%0];" ::"l"(a + 64));
    }
  }
  pdl_wait();                 // the previous kernel's writes are visible
  pdl_launch_dependents();

  // ---------------- R_K -> shared memory first: nothing it depends on
  if (tid == 0) {
    mbar_init(rbar, 1);
    mbar_init(rbar + 1, 1);   // R_V
    mbar_init(pro_done, 1);
    fence_mbar_init();
  }
  if (tid == 0 && pbeg < p.max_pages) {
    mbar_arrive_expect_tx(rbar, uint32_t(Geo<G>::kRotBytes));
    const float* rk = p.r_k + int64_t(hkv) * kHeadDim * kHeadDim;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      bulk_copy_g2s(rks + c * (kHeadDim * kHeadDim / 4), rk + c * (kHeadDim * kHeadDim / 4),
                    uint32_t(Geo<G>::kRotBytes / 4), rbar);
  }

  uint16_t qv[(G * kHeadDim + PT - 1) / PT];
  {
    const uint16_t* qg = p.q + (int64_t(b) * p.n_kv * G + int64_t(hkv) * G) * kHeadDim;
#pragma unroll
    for (int i0 = 0; i0 < (G * kHeadDim + PT - 1) / PT; ++i0) {
      const int i = tid + i0 * PT;
      // (q may sit in pinned host memory: cache-volatile loads)
      qv[i0] = (pbeg < p.max_pages && !bf16_warp && i < G * kHeadDim)
                   ? uint16_t(__ldcv(reinterpret_cast<const unsigned short*>(qg + i)))
                   : uint16_t(0);
    }
  }

  // ---------------- INT2 pages of this CTA: warp w first copies pages
  // pbeg + kStages w + s (s < kStages) into its ring, requested before the
  // history length is known (pages past it are read but never used; ids
  // outside the pool are never copied).  The ring is kParts parts of kGroup
  // consecutive pages; once a step has consumed a part, the part takes the
  // warp's next kGroup pages.
  const int32_t* ptab = p.page_table + int64_t(b) * p.max_pages;
  const int spec_end = min(pbeg + p.pages_per_split, p.max_pages);
  int hist = p.hist_len[b];
  uint8_t* ring = stage + size_t(warp) * kStages * kBlock;
  uint64_t* bar = bars + warp * kStages;
  const uint8_t* pool = p.pages + int64_t(hkv) * kBlock;
  const int64_t page_stride = int64_t(p.n_kv) * kBlock;
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(bar + s, 1);
    fence_mbar_init();
  }
  __syncwarp();
  // lane s < kStages copies the warp's s-th first page into stage s
  uint32_t copied_bits, issued_bits;
  {
    const int j = pbeg + kStages * warp + lane;
    const bool in = lane < kStages && j < spec_end;
    const int pid = in ? __ldg(ptab + j) : -1;
    const bool ok = in && pid >= 0 && pid < p.n_pages;
    if (in) {
      if (!ok) {
        // no copy: complete the stage's phase without bytes so the ring stays in step
        mbar_arrive(bar + lane);
      } else {
        mbar_arrive_expect_tx(bar + lane, kBlock);
        bulk_copy_g2s(ring + lane * kBlock, pool + int64_t(pid) * page_stride, kBlock, bar + lane);
      }
    }
    copied_bits = __ballot_sync(kFull, ok);
    issued_bits = __ballot_sync(kFull, in);
    if (OSCAR_SERIAL_COPIES) {
      if (in) mbar_wait_bounded(bar + lane, 0, kDrainWaitNs);
      __syncwarp();
    }
  }

  __syncthreads();   // the R_K / R_V / prologue barriers are initialised

  // ---------------- the query rows -> shared memory (used by the prologue;
  // requested before the page copies, stored after them)
  if (pbeg < p.max_pages && !bf16_warp) {
#pragma unroll
    for (int i0 = 0; i0 < (G * kHeadDim + PT - 1) / PT; ++i0) {
      const int i = tid + i0 * PT;
      if (i < G * kHeadDim) qscratch[QScratch<G>::kQs + i] = __uint_as_float(uint32_t(qv[i0]) << 16);
    }
  }

  if (hist < 0 || hist > p.max_pages * kPage) {
    if (tid == 0) flag(p.dev_status, 0x2);
    hist = max(0, min(hist, p.max_pages * kPage));
  }
  const int n_pg = (hist + kPage - 1) / kPage;
  if (n_pg > n_splits * p.pages_per_split && split == 0 && tid == 0)
    flag(p.dev_status, 0x2);  // longer than the host bound max_hist: tail not read
  const int pend = min(pbeg + p.pages_per_split, n_pg);

  // ---------------- q~ and the lane's QK fragments (prologue warps); the
  // BF16 warps scan the sink/recent tokens meanwhile and read the fragments
  // once the prologue is done
  constexpr int NH = Geo<G>::NH;
  uint32_t qb[NH][8][2];
  float unscale[NH], qz[NH][NGK];
  const bool any_pages = pend > pbeg;
  float* rvs = rks;
  uint64_t* vbar = rbar + 1;
  auto load_fragments = [&]() {
    using S = QScratch<G>;
    const uint4* fr = reinterpret_cast<const uint4*>(qscratch + S::kFrag) + lane * NH * 4;
#pragma unroll
    for (int i = 0; i < NH * 4; ++i) {
      const uint4 v = fr[i];
      const int e = 4 * i;
      qb[e / 16][(e % 16) / 2][0] = v.x;
      qb[e / 16][(e % 16) / 2][1] = v.y;
      qb[(e + 2) / 16][((e + 2) % 16) / 2][0] = v.z;
      qb[(e + 2) / 16][((e + 2) % 16) / 2][1] = v.w;
    }
#pragma unroll
    for (int nt = 0; nt < NH; ++nt) {
      const int h = 4 * nt + tig;
      unscale[nt] = qscratch[S::kAux + h * 8 + 1];
#pragma unroll
      for (int q = 0; q < NGK; ++q) qz[nt][q] = qscratch[S::kAux + h * 8 + 2 + q];
    }
  };
  if (!bf16_warp) {
    if (any_pages) {
      rotate_query<G, NGK>(p, b, hkv, rks, rbar, qscratch);
      load_fragments();
    } else if (tid == 0 && pbeg < p.max_pages) {
      // R_K was requested: let it land before this region is reused
      if (!mbar_wait_bounded(rbar, 0, kWaitLimitNs)) flag(p.dev_status, 0x4);
    }
    named_barrier(kPrologueBarrier, PT);   // prologue reads of R_K are done
    // R_V -> shared memory (replacing R_K) for this CTA's output rotation:
    // box qq = columns 32 qq .. 32 qq + 31 of all 128 rows, 16-byte chunks
    // of row c swizzled to chunk ^ (c & 7)
    if (tid == 0) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(vbar, uint32_t(Geo<G>::kRotBytes));
#pragma unroll
      for (int qq = 0; qq < 4; ++qq)
        tma_load_2d(rvs + qq * (kHeadDim * kHeadDim / 4), &p.tm_rv, 32 * qq, hkv * kHeadDim, vbar);
      mbar_arrive(pro_done);
    }
  } else {
    // ---------------- BF16 sink / recent tokens owned by this CTA: virtual
    // pages split, split + n_splits, ...; the j-th goes to BF16 warp j % 2
    int sink_len = p.sink_len[b], rec_len = p.recent_len[b];
    const int rec_start = p.recent_start[b];
    const int bw = warp - (W - kBf16Warps);
    if (sink_len < 0 || sink_len > p.sink_cap || rec_len < 0 || rec_len > p.recent_cap ||
        rec_start < 0 || rec_start >= max(p.recent_cap, 1)) {
      if (bw == 0 && lane == 0) flag(p.dev_status, 0x2);
      sink_len = max(0, min(sink_len, p.sink_cap));
      rec_len = max(0, min(rec_len, p.recent_cap));
    }
    const int start = min(max(rec_start, 0), max(p.recent_cap - 1, 0));
    const int n_vp = p.sink_cap / kPage + p.recent_cap / kPage;
    const int64_t hstride = int64_t(p.n_kv) * kHeadDim;
    WarpState<G> st;
    st.init();
    const int mine = split + bw * n_splits;
    if (mine < n_vp) {
      uint32_t qf[NTQ][8][2];
#pragma unroll
      for (int nt = 0; nt < NTQ; ++nt) {
        const int h = (8 * nt + gid) % G;
        const uint16_t* qrow = p.q + (int64_t(b) * p.n_kv * G + hkv * G + h) * kHeadDim + 32 * tig;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 v = __ldcv(reinterpret_cast<const uint4*>(qrow + 8 * u));
          qf[nt][2 * u][0] = v.x;
          qf[nt][2 * u][1] = v.y;
          qf[nt][2 * u + 1][0] = v.z;
          qf[nt][2 * u + 1][1] = v.w;
        }
      }
      auto row_of = [&](int u, bool kv, bool& ok) -> const uint16_t* {
        if (u < p.sink_cap) {
          ok = u < sink_len;
          const uint16_t* base = kv ? p.sink_v : p.sink_k;
          return base + (int64_t(b) * p.sink_cap + u) * hstride + int64_t(hkv) * kHeadDim;
        }
        const int i = u - p.sink_cap;
        ok = i < rec_len;
        const int slot = (start + i) % p.recent_cap;
        const uint16_t* base = kv ? p.recent_v : p.recent_k;
        return base + (int64_t(b) * p.recent_cap + slot) * hstride + int64_t(hkv) * kHeadDim;
      };
      for (int vp = mine; vp < n_vp; vp += kBf16Warps * n_splits) {
        const int u0 = vp * kPage;
        bool kok[2], vok[4];
        const uint16_t* krow[2] = {row_of(u0 + gid, false, kok[0]), row_of(u0 + gid + 8, false, kok[1])};
        const uint16_t* vrow[4] = {row_of(u0 + 2 * tig, true, vok[0]), row_of(u0 + 2 * tig + 1, true, vok[1]),
                                   row_of(u0 + 2 * tig + 8, true, vok[2]),
                                   row_of(u0 + 2 * tig + 9, true, vok[3])};
        bf16_page<G>(krow, vrow, kok, vok, gid, tig, qf, st);
      }
    }
    store_warp_state<G, false>(st, st_bf16x + bw * G * kPartStride, gid, tig, 1.f);
    if (any_pages) {
      if (!mbar_wait_bounded(pro_done, 0, kWaitLimitNs)) {
        if (lane == 0) flag(p.dev_status, 0x4);
      } else {
        load_fragments();
      }
    }
  }
  // each warp's INT2 state goes into its own ring slice once its pages are done
  float* my_state = reinterpret_cast<float*>(ring);

  constexpr int kGroup = Gm::kGroup;
  // K and V pairs of a token in one load, kept from QK to PV (one group
  // each, GQA 4); the other variants load the V pairs again for PV, which
  // keeps their register budget
  constexpr bool kJointPairs = NGK == 1 && NGV == 1 && G <= 4;
  // ---------------- INT2 pages, one ring part (kGroup pages) per step: QK
  // of the step's pages, one maximum update, then their probabilities and
  // PV.  The loop body is unrolled over the kParts parts, so every stage
  // index is a compile-time constant.  A warp's pages only grow in
  // consumption order, so the first part past the history ends them.  A page with an invalid id is computed on stale ring data
  // with every token masked.
  {
    HistState<G, NZ> st;
    st.init();
    const float lift = float(kRescaleLog2) + p.pv_log2;   // rescale test against st.m (see int2_update_max)
    const int n_full = hist / kPage;                     // pages below it hold kPage valid tokens
    constexpr uint32_t kPartBits = (1u << kGroup) - 1u;
    // first page of each part and its copied pages (bit u: page base + u)
    int base[kParts];
    uint32_t good[kParts];
#pragma unroll
    for (int h = 0; h < kParts; ++h) {
      base[h] = pbeg + kStages * warp + kGroup * h;
      good[h] = (copied_bits >> (kGroup * h)) & kPartBits;
    }
    // stages whose arrival is not yet consumed, and each stage's parity
    uint32_t pending = issued_bits & ((1u << kStages) - 1u);
    uint32_t parity = 0u;
    bool timed_out = false, done = false;
    // the next refill, one step ahead: its first page and lane u's page id
    // refill n of warp w takes pages pbeg + kStages W + (n W + w) kGroup
    // onwards: a fixed schedule (the order of every sum is fixed, so results
    // are bit-reproducible), in step with the initial fill
    int n_refill = 0;
    auto grab = [&]() { return pbeg + kStages * W + (n_refill++ * W + warp) * kGroup; };
    int g_next = grab();
    int pid_next = lane < kGroup && g_next + lane < pend ? __ldg(ptab + g_next + lane) : -1;
    // the scan's time budget (page_wait_ns from its start): a warp past it
    // gives up its remaining pages as if a copy had stalled
    const uint64_t t_scan = global_timer_ns();
    while (!done) {
#pragma unroll
      for (int h = 0; h < kParts; ++h) {
        if (done) break;
        const int j0 = base[h];
        if (j0 >= pend) {
          done = true;
          break;
        }
        if (h == 0 && global_timer_ns() - t_scan > p.page_wait_ns) {   // once per ring cycle
          timed_out = true;
          done = true;
          break;
        }
        const int nv = min(kGroup, pend - j0);   // this part's pages within the history
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
          const int s = kGroup * h + u;
          if (u == 0 || u < nv) {
            if (!mbar_wait_bounded(bar + s, (parity >> s) & 1u, p.page_wait_ns)) {
              timed_out = true;
            } else {
              pending &= ~(1u << s);
              parity ^= 1u << s;
            }
          }
        }
        if (timed_out) {
          done = true;
          break;
        }
        const uint8_t* pg[kGroup];
#pragma unroll
        for (int u = 0; u < kGroup; ++u) pg[u] = ring + (kGroup * h + u) * kBlock;
        const bool all_full = nv == kGroup && good[h] == kPartBits && j0 + kGroup <= n_full;
        // token validity of the lane's two tokens per page (masked steps only)
        bool ok[kGroup][2];
        if (!all_full) {
#pragma unroll
          for (int u = 0; u < kGroup; ++u) {
            const bool copied = (good[h] >> u) & 1u;
            if (u < nv && !copied && lane == 0) flag(p.dev_status, 0x1);
            const int ntok = u < nv && copied ? hist - kPage * (j0 + u) : 0;
            ok[u][0] = gid < ntok;
            ok[u][1] = gid + 8 < ntok;
          }
        }
        // QK of the step's pages, one maximum update, probabilities and PV;
        // steps whose tokens are all valid (every step but the history's last)
        // take the select-free variant; in the other, pages past the history
        // are skipped (warp-uniform branches)
        auto step = [&](auto masked) {
          constexpr bool kMasked = decltype(masked)::value;
          float sc[kGroup][NH][2];
          uint32_t vsz0[kGroup][NGV], vsz1[kGroup][NGV];   // the pages' V (scale, zero) pairs
#pragma unroll
          for (int u = 0; u < kGroup; ++u) {
            if (kMasked && u > 0 && u >= nv) {
#pragma unroll
              for (int nt = 0; nt < NH; ++nt) sc[u][nt][0] = sc[u][nt][1] = -INFINITY;
              continue;
            }
            uint32_t ksz0[NGK], ksz1[NGK];
            if constexpr (kJointPairs) {
              load_pairs<NGK, NGV>(pg[u], gid, ksz0, vsz0[u]);
              load_pairs<NGK, NGV>(pg[u], gid + 8, ksz1, vsz1[u]);
            } else {
              load_group_pairs<NGK, NGV, 0>(pg[u], gid, ksz0);
              load_group_pairs<NGK, NGV, 0>(pg[u], gid + 8, ksz1);
            }
            if constexpr (kLevels) {
              float e[NH][2];
              int2_qk_levels<G>(pg[u], gid, tig, qb, p.coef_k, e);
              int2_scores_levels<G, kMasked>(e, ksz0[0], ksz1[0], ok[u][0], ok[u][1], unscale, qz, p.coef_k, sc[u]);
            } else if constexpr (NGK == 1) {
              float d[NH][4];
              int2_qk<G>(pg[u], gid, tig, qb, d);
              int2_scores<G, kMasked>(d, ksz0[0], ksz1[0], ok[u][0], ok[u][1], unscale, qz, sc[u]);
            } else {
              float a[NH][2];
              int2_qk_groups<G, NGK>(pg[u], gid, tig, qb, ksz0, ksz1, a);
              int2_scores_groups<G, NGK, kMasked>(a, ksz0, ksz1, ok[u][0], ok[u][1], unscale, qz, sc[u]);
            }
          }
          int2_update_max<G, NZ, kGroup>(sc, st, p.pv_log2, lift);
#pragma unroll
          for (int u = 0; u < kGroup; ++u) {
            if (kMasked && u > 0 && u >= nv) continue;
            if constexpr (!kJointPairs) {
              load_group_pairs<NGK, NGV, NGK>(pg[u], gid, vsz0[u]);
              load_group_pairs<NGK, NGV, NGK>(pg[u], gid + 8, vsz1[u]);
            }
            if constexpr (kLevels) {
              uint32_t pb[3][NH][2];
              int2_probs_levels<G, kMasked>(sc[u], vsz0[u][0], vsz1[u][0], ok[u][0], ok[u][1], p.coef_v, st, pb);
              int2_pv_levels<G>(pg[u], gid, tig, pb, st);
            } else {
              uint32_t pb[NGV][NH][2];
              int2_probs<G, NGV, kMasked>(sc[u], vsz0[u], vsz1[u], ok[u][0], ok[u][1], st, pb);
              int2_pv<G, NGV>(pg[u], gid, tig, pb, st);
            }
          }
        };
        if (all_full) {
          step(std::false_type{});
        } else {
          step(std::true_type{});
        }
        __syncwarp();
        // the part takes the pages g_next .. g_next + kGroup - 1 (ids loaded
        // one step ahead): lane u < kGroup starts the copy into its stage
        {
          const bool want = lane < kGroup && g_next + lane < pend;
          const bool good_id = want && pid_next >= 0 && pid_next < p.n_pages;
          if (want) {
            const int s = kGroup * h + lane;
            if (!good_id) {
              mbar_arrive(bar + s);   // no copy: complete the phase without bytes
            } else {
              mbar_arrive_expect_tx(bar + s, kBlock);
              bulk_copy_g2s(ring + s * kBlock, pool + int64_t(pid_next) * page_stride, kBlock, bar + s);
            }
            if (OSCAR_SERIAL_COPIES) mbar_wait_bounded(bar + s, (parity >> s) & 1u, kDrainWaitNs);
          }
          if (OSCAR_SERIAL_COPIES) __syncwarp();
          pending |= (__ballot_sync(kFull, want) & kPartBits) << (kGroup * h);
          good[h] = __ballot_sync(kFull, good_id) & kPartBits;
          base[h] = g_next;
          g_next = grab();
          pid_next = lane < kGroup && g_next + lane < pend ? __ldg(ptab + g_next + lane) : -1;
        }
      }
    }
    if (timed_out && lane == 0) flag(p.dev_status, 0x4);
    // copies still in flight (after a timeout, or requested speculatively
    // past the history) land before the CTA's shared memory goes away; each
    // wait is bounded
    for (int s = 0; s < kStages; ++s)
      if ((pending >> s) & 1u) mbar_wait_bounded(bar + s, (parity >> s) & 1u, kDrainWaitNs);
    __syncwarp();
    if constexpr (kLevels) {
      store_hist_state_levels<G>(st, my_state, gid, tig, p.pv_unscale, p.coef_v[0]);
    } else {
      store_hist_state<G, NGV>(st, my_state, gid, tig, p.pv_unscale);
    }
  }

  __syncthreads();

  // ---------------- CTA merge of the warps -> one partial per head: the
  // history part is rotated back with R_V and joined with the BF16 part, so
  // the CTA writes one (m, l, o) per head in the original basis.
  // Warp h weighs head h's W history states (ring slices) and kBf16Warps
  // BF16 states against their common maximum; lane i holds state i.
  float* os = qscratch;                       // [G][128] merged history output (rotated basis)
  float* ob = os + G * kHeadDim;              // [G][128] merged BF16 output
  float* wts = ob + G * kHeadDim;             // [G][32] state weights
  const int slice = kStages * kBlock / 4;   // floats between two warps' states
  const float* states = reinterpret_cast<const float*>(stage);
  float* part = p.partials + (int64_t(pair) * n_splits + split) * G * kPartStride;
  static_assert(W + kBf16Warps <= 32, "one lane per warp state");
  static_assert(G <= W, "one warp per head");
  if (warp < G) {
    const int h = warp;
    float m = -INFINITY, l = 0.f;
    if (lane < W) {
      m = states[lane * slice + h * kPartStride];
      l = states[lane * slice + h * kPartStride + 1];
    } else if (lane < W + kBf16Warps) {
      m = st_bf16x[(lane - W) * G * kPartStride + h * kPartStride];
      l = st_bf16x[(lane - W) * G * kPartStride + h * kPartStride + 1];
    }
    float mx = l > 0.f ? m : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    const float f = l > 0.f ? fast_exp2(m - mx) : 0.f;
    float lsum = l * f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(kFull, lsum, o);
    wts[h * 32 + lane] = f;
    if (lane == 0) {
      part[h * kPartStride + 0] = mx;
      part[h * kPartStride + 1] = lsum;
    }
  }
  __syncthreads();
  for (int idx = tid; idx < G * kHeadDim; idx += T) {
    const int h = idx / kHeadDim, c = idx % kHeadDim;
    const float* wh = wts + h * 32;
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) o = fmaf(wh[w], states[w * slice + h * kPartStride + 4 + c], o);
    float o2 = 0.f;
#pragma unroll
    for (int w = 0; w < kBf16Warps; ++w)
      o2 = fmaf(wh[W + w], st_bf16x[w * G * kPartStride + h * kPartStride + 4 + c], o2);
    os[idx] = o;
    ob[idx] = o2;
  }
  __syncthreads();
  if (!mbar_wait_bounded(vbar, 0, kWaitLimitNs) && tid == 0) flag(p.dev_status, 0x4);
  // history partial back in the original basis, o[c] = sum_j o~[j] R_V[c][j]:
  // thread (row c, quarter qq of j), a warp holding 32 consecutive rows of
  // one quarter; the swizzled boxes put chunk k4 of 8 consecutive rows in 8
  // bank groups while every lane reads the same o~ chunk (a broadcast); the
  // quarters are summed through shared memory (the ring, whose warp states
  // are consumed)
  float* red4 = reinterpret_cast<float*>(stage);   // [4][G][128]
  for (int task = tid; task < 4 * kHeadDim; task += T) {
    const int c = task & (kHeadDim - 1), qq = task >> 7;
    const float4* rrow = reinterpret_cast<const float4*>(rvs + qq * (kHeadDim * kHeadDim / 4)) + 8 * c;
    float4 r[8];
#pragma unroll
    for (int k4 = 0; k4 < 8; ++k4) r[k4] = rrow[k4 ^ (c & 7)];
    float d[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float4* o = reinterpret_cast<const float4*>(os + h * kHeadDim + 32 * qq);
      float acc = 0.f;
#pragma unroll
      for (int k4 = 0; k4 < 8; ++k4) {
        const float4 ov = o[k4];
        acc = fmaf(ov.x, r[k4].x, fmaf(ov.y, r[k4].y, fmaf(ov.z, r[k4].z, fmaf(ov.w, r[k4].w, acc))));
      }
      d[h] = acc;
    }
#pragma unroll
    for (int h = 0; h < G; ++h) red4[(qq * G + h) * kHeadDim + c] = d[h];
  }
  __syncthreads();
  for (int idx = tid; idx < G * kHeadDim; idx += T) {
    const int h = idx / kHeadDim, c = idx % kHeadDim;
    const float d = (red4[(0 * G + h) * kHeadDim + c] + red4[(1 * G + h) * kHeadDim + c]) +
                    (red4[(2 * G + h) * kHeadDim + c] + red4[(3 * G + h) * kHeadDim + c]);
    part[h * kPartStride + 4 + c] = d + ob[idx];
  }

  // ---------------- ticket: the last CTA of this (request, KV head) merges.
  // The barrier orders the CTA's partial writes before thread 0's
  // acquire-release add, which publishes them; in the last CTA the same add
  // acquires the other CTAs' partials, and the barrier after it extends
  // that to the merging warps.
  __syncthreads();
  if (tid == 0) {
    const unsigned t = atom_add_acq_rel_gpu(p.counters + pair, 1u);
    *s_last = (t == unsigned(n_splits - 1)) ? 1 : 0;
  }
  __syncthreads();
  if (!*s_last || warp >= G) return;

  // Merge of the n_splits partials: warp h merges head h on its own (lane =
  // channel quad).  The first kPre partial outputs and the (m, l) pairs are
  // requested back to back, so that all of them share one latency.
  {
    const int h = warp, NP = n_splits;
    const float* pp = p.partials + int64_t(pair) * n_splits * G * kPartStride;
    // the outputs first: the weights wait on the (m, l) loads issued last,
    // by which time every load of the batch is in flight
    constexpr int kPre = 24;
    float4 pre[kPre];
#pragma unroll
    for (int j = 0; j < kPre; ++j) {
      pre[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      ld_cg_if(pre[j], pp + int64_t(j * G + h) * kPartStride + 4 + 4 * lane, j < NP);
    }
    // (m, l) of partials lane, lane + 32, ... (NP <= kMaxSplits = 4 x 32)
    float2 ml[kMaxSplits / 32];
#pragma unroll
    for (int u = 0; u < kMaxSplits / 32; ++u) {
      const int i = lane + 32 * u;
      ml[u] = make_float2(-INFINITY, 0.f);
      ld_cg_if(ml[u], pp + int64_t(i * G + h) * kPartStride, i < NP);
    }
    auto o_of = [&](int i) {
      return __ldcg(reinterpret_cast<const float4*>(pp + int64_t(i * G + h) * kPartStride + 4) + lane);
    };
    float mx = -INFINITY;
#pragma unroll
    for (int u = 0; u < kMaxSplits / 32; ++u)
      if (ml[u].y > 0.f) mx = fmaxf(mx, ml[u].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    float lsum = 0.f;
    float* wh = reinterpret_cast<float*>(stage) + h * kMaxSplits;   // [G][kMaxSplits] weights
#pragma unroll
    for (int u = 0; u < kMaxSplits / 32; ++u) {
      const float f = ml[u].y > 0.f ? exp2f(ml[u].x - mx) : 0.f;
      wh[lane + 32 * u] = f;
      lsum = fmaf(ml[u].y, f, lsum);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(kFull, lsum, o);
    __syncwarp();
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kPre; ++j) {
      const float f = wh[j];   // 0 past NP
      a.x = fmaf(f, pre[j].x, a.x);
      a.y = fmaf(f, pre[j].y, a.y);
      a.z = fmaf(f, pre[j].z, a.z);
      a.w = fmaf(f, pre[j].w, a.w);
    }
    for (int i = kPre; i < NP; ++i) {
      const float4 v = o_of(i);
      const float f = wh[i];
      a.x = fmaf(f, v.x, a.x);
      a.y = fmaf(f, v.y, a.y);
      a.z = fmaf(f, v.z, a.z);
      a.w = fmaf(f, v.w, a.w);
    }
    const float s = lsum > 0.f ? 1.f / lsum : 0.f;
    const float4 res = make_float4(a.x * s, a.y * s, a.z * s, a.w * s);
    const int64_t oi = ((int64_t(b) * p.n_kv + hkv) * G + h) * kHeadDim;
    reinterpret_cast<float4*>(p.out + oi)[lane] = res;
    if (p.out_host) reinterpret_cast<float4*>(p.out_host + oi)[lane] = res;   // over the CPU-GPU link
    if (h == 0 && lane == 0) p.counters[pair] = 0u;   // ready for the next call
  }
}

// (every group variant also holds one CTA per SM: the planning uses the
// one-group kernel)
template <int G>
int occupancy() {
  int occ = 0;
  cudaFuncSetAttribute(split_kernel<G, 1, 1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       int(Geo<G>::kSmem));
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, split_kernel<G, 1, 1, false>, Geo<G>::T,
                                                    Geo<G>::kSmem) !=
      cudaSuccess)
    return 0;
  return occ;
}

template <int G, int NGK, int NGV, bool kLevels = false>
cudaError_t launch_g(const DecodeParams& p, cudaStream_t stream) {
  constexpr size_t smem = Geo<G, NGK, NGV, kLevels>::kSmem;
  cudaError_t e = set_smem_limit<split_kernel<G, NGK, NGV, kLevels>>(int(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(split_kernel<G, NGK, NGV, kLevels>, dim3(p.n_kv, p.batch, p.n_splits), dim3(Geo<G>::T),
                    smem, stream, p);
}

template <int G, int NGK>
cudaError_t launch_gk(const DecodeParams& p, cudaStream_t stream) {
  if (p.ng_v == 1) return launch_g<G, NGK, 1>(p, stream);
  if (p.ng_v == 2) return launch_g<G, NGK, 2>(p, stream);
  if (p.ng_v == 4) return launch_g<G, NGK, 4>(p, stream);
  return cudaErrorInvalidValue;
}

template <int G>
cudaError_t launch_gq(const DecodeParams& p, cudaStream_t stream) {
  if (p.codebook) return p.ng_k == 1 && p.ng_v == 1 ? launch_g<G, 1, 1, true>(p, stream) : cudaErrorInvalidValue;
  if (p.ng_k == 1) return launch_gk<G, 1>(p, stream);
  if (p.ng_k == 2) return launch_gk<G, 2>(p, stream);
  if (p.ng_k == 4) return launch_gk<G, 4>(p, stream);
  return cudaErrorInvalidValue;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

bool encode_rv_map(DecodeParams* p) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const cuuint64_t dims[2] = {cuuint64_t(kHeadDim), cuuint64_t(p->n_kv) * kHeadDim};
  const cuuint64_t strides[1] = {cuuint64_t(kHeadDim) * 4};
  const cuuint32_t box[2] = {32, cuuint32_t(kHeadDim)};
  const cuuint32_t estr[2] = {1, 1};
  return encode(&p->tm_rv, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(p->r_v), dims, strides, box,
                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int plan_decode(int batch, int n_kv, int group, int sink_cap, int recent_cap, int max_hist,
                DecodePlan* plan, cudaError_t* err) {
  (void)sink_cap;
  (void)recent_cap;
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return 0;
  static int sm_cache[64] = {0};
  int sms = dev < 64 ? sm_cache[dev] : 0;
  if (sms == 0) {
    *err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (*err != cudaSuccess) return 0;
    if (dev < 64) sm_cache[dev] = sms;
  }
  static int occ_cache[64][2] = {{0}};
  const int gi = group == 4 ? 0 : 1;
  int occ = dev < 64 ? occ_cache[dev][gi] : 0;
  if (occ == 0) {
    occ = group == 4 ? occupancy<4>() : occupancy<8>();
    if (occ <= 0) {
      *err = cudaGetLastError();
      if (*err == cudaSuccess) *err = cudaErrorInvalidConfiguration;
      return 0;
    }
    if (dev < 64) occ_cache[dev][gi] = occ;
  }
  const int warps = group == 4 ? Geo<4>::W : Geo<8>::W;
  const int64_t slots = int64_t(sms) * occ;
  const int64_t pairs = int64_t(batch) * n_kv;
  const int pages_max = (max_hist + kPage - 1) / kPage;
  // splits per (request, KV head): the count that minimises a simple model
  // of the launch time, waves x (pages per warp x time per page + fixed
  // per-CTA time), with the measured ~1 us per page per warp (GQA 4; ~1.5 us
  // for GQA 8) and ~10 us of fixed prologue + merge latency per CTA
  const double t_page = group == 4 ? 0.95 : 1.5, t_fixed = 10.0;
  int n_splits = 1;
  double best = 1e300;
  for (int n = 1; n <= kMaxSplits; ++n) {
    const int64_t pps_n = (pages_max + n - 1) / n;
    if (n > 1 && (pages_max + pps_n - 1) / pps_n < n) break;   // no finer split exists
    const int64_t waves = (pairs * n + slots - 1) / slots;
    const double cost = double(waves) * (double((pps_n + warps - 1) / warps) * t_page + t_fixed);
    if (cost < best * 0.999) {
      best = cost;
      n_splits = n;
    }
  }
  if (OSCAR_PLAN_SPLITS > 0) n_splits = min(OSCAR_PLAN_SPLITS, kMaxSplits);
  int pps = max(1, (pages_max + n_splits - 1) / n_splits);
  n_splits = max(1, (pages_max + pps - 1) / pps);
  plan->n_splits = n_splits;
  plan->pages_per_split = pps;
  size_t off = 0;
  plan->off_counters = off;
  off = align256(off + size_t(pairs) * 4);
  plan->off_partials = off;
  off = align256(off + size_t(pairs) * n_splits * group * kPartStride * 4);
  plan->total_bytes = off;
  *err = cudaSuccess;
  return occ;
}

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
  if (p.group == 4) return launch_gq<4>(p, stream);
  if (p.group == 8) return launch_gq<8>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace oscar
