// Decode attention over BF16 sink | INT2 history | BF16 recent window.
//
// myzaker.com OSCAR article, part "从离线校准到在线推理的 pipeline": the INT2
// kernel unpacks, dequantises with scale/zero point and accumulates in float;
// a BF16 kernel handles sink and recent; an online-softmax merge joins them.
// gist.science "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV
// Cache Quantization", Technical summary 2.2 B: the inverse rotation is fused
// into the attention kernel with no extra memory traffic.  Here it is applied
// as q~ = q . R_K once per query head and one o . R_V^T per head and split,
// instead of rotating every token.
//
// One launch; CTA (split, KV head, request) of 16 warps, one CTA per SM, owns
// a contiguous range of INT2 pages of one (request, KV head) and a share of
// its BF16 sink/recent tokens.  The INT2 pages are processed in tiles of 8
// pages (128 tokens) by a warp-specialised tcgen05 pipeline:
//   warp 12     producer: 1-D TMA bulk copies of the tile's 8 page blocks into
//               a ring of tile slots (mbarrier transaction counts);
//   warps 8-11  K path, thread = token: unpack the token's 128 K codes into
//               fp16 in tensor memory (A of QK); then lane 0 of warp 8 + j
//               issues the QK MMAs of K-steps 2j, 2j+1 into accumulator j:
//               D[token][col] = codes[token][k] . B_qk[k][col];
//   warps 0-3   softmax, thread = token: sum the 4 accumulators, scores,
//               online softmax with a running maximum per warp and head,
//               p s_V (hi | lo fp16) into shared memory (B of PV);
//   warps 4-7   V path, thread = channel: unpack the channel's codes of the
//               tile's 128 tokens into fp16 in tensor memory (A of PV); lane 0
//               of warp 4 + j issues the PV MMAs of K-steps 2j, 2j+1 (the
//               tokens of softmax warp j) into output accumulator j:
//               O_j[channel][col] += codes^T[channel][token] . P[token][col];
//   warps 14-15 the BF16 sink/recent tokens (mma.sync, bf16), concurrently;
//   warp 13     owns the tensor-memory allocation.
// MMAs are M = 128, N = 16, K = 16, fp16 in, fp32 accumulate in tensor
// memory, completion signalled by tcgen05.commit.  They are issued from 8
// threads because one thread issues only about one MMA per 50 cycles.  The
// columns of B are the GQA heads' hi parts then lo parts (fp16 hi + lo split
// of an fp32 value), so each MMA carries about fp32 precision.  A 2-bit code
// c at bit offset 2k of a 16-bit half is read as the fp16 subnormal
// c * 4^k * 2^-24 by one AND; the 4^k factors go into B and 2^-24 into the
// output scale.  A softmax warp raises its maximum lazily (only when a score
// exceeds it by 2^8); its output accumulator is then rescaled in place by
// the V warps before the next PV MMAs.  The 4 accumulators are merged at the
// end with their warps' maxima.
//
// Epilogue: the CTA rotates its history partial back with R_V (staged by TMA
// during the scan) and writes it and its BF16 partial; the last CTA of the
// (request, KV head) to finish (atomic ticket, no waiting) merges all
// partials and writes the normalised output, then resets the ticket.
// Every wait is an mbarrier wait bounded at 1 s; a timeout sets a device
// status bit and an abort flag that ends every role's loop.
#include <cfloat>

#include "kernels.h"
#include "ptx.cuh"

// ring depth in tiles of 8 pages
#ifndef OSCAR_TILE_SLOTS
#define OSCAR_TILE_SLOTS 6
#endif

namespace oscar {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr uint32_t kFull = 0xffffffffu;
constexpr int kMaxSplits = 128;               // bounds the last CTA's merge scratch

constexpr int kTilePages = 8;
constexpr int kTileTokens = kTilePages * kPage;           // 128
constexpr int kTileBytes = kTilePages * kBlockBytes;      // 9216
constexpr int kSlots = OSCAR_TILE_SLOTS;
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
// warp roles
constexpr int kVWarp0 = 4, kKWarp0 = 8, kProducerWarp = 12, kTmemWarp = 13, kBf16Warp = 14;
constexpr int kN = 16;                                      // MMA N: hi | lo columns
constexpr uint32_t kIdesc = idesc_f16_f32(128, kN);
constexpr int kBBytes = kN * kTileTokens * 2;               // one B operand tile (K = 128)
// operand buffering: A_K and D_qk double, A_V triple, P quadruple, so the V
// warps and the softmax can run ahead of the PV MMAs
constexpr int kAvBufs = 3, kBpBufs = 4;
// tensor-memory columns: A_K[2] | A_V[3] | D_qk[2][4 accumulators] | O[4 accumulators]
constexpr uint32_t kColAK = 0, kColAV = 128, kColQK = kColAV + 64 * kAvBufs, kColPV = kColQK + 128,
                   kTmemCols = 512;
static_assert(kColPV + 4 * kN <= kTmemCols, "tensor memory columns");

template <int G>
struct Geo {
  static constexpr int NT = (2 * G + 7) / 8;          // BF16 PV column tiles (hi | lo)
  static constexpr int HS = G >= 8 ? G / 4 : 2;       // BF16 head slots per lane
  static constexpr int NTQ = (G + 7) / 8;             // BF16 QK column tiles
  static constexpr size_t kStageBytes = size_t(kSlots) * kTileBytes;
  static constexpr size_t kRotBytes = size_t(kHeadDim) * kHeadDim * 4;
  // q~ scratch: qs[G][128] | part[4][G][128] | qt[G][128] | aux[G][4] | red[2][G][4]
  static constexpr size_t kQFloats = 6 * G * kHeadDim + 12 * G;
  static constexpr size_t kUnion = kRotBytes + kQFloats * 4;        // R_K then R_V | scratch
  static constexpr size_t kBf16State = size_t(2) * G * kPartStride * 4;
  // full, empty | ak qk_done qk_free | av | bp | pv | rs bqk rk rv fin
  static constexpr int kBars = 2 * kSlots + 3 * 2 + kAvBufs + 2 * kBpBufs + 5;
  static constexpr size_t kBarBytes = (kBars * 8 + 127) / 128 * 128;
  static constexpr size_t kMiscBytes = 2048;
  static constexpr size_t oStage = 0;
  static constexpr size_t oBqk = oStage + kStageBytes;
  static constexpr size_t oBp = oBqk + kBBytes;
  static constexpr size_t oUni = oBp + kBpBufs * kBBytes;
  static constexpr size_t oBf16 = oUni + kUnion;
  static constexpr size_t oBars = (oBf16 + kBf16State + 127) / 128 * 128;
  static constexpr size_t oMisc = oBars + kBarBytes;
  static constexpr size_t kSmem = oMisc + kMiscBytes;
  static_assert(kStageBytes % 128 == 0 && oBqk % 128 == 0 && oUni % 128 == 0, "TMA / UMMA operands aligned");
  static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
  // CTA merge scratch after R_V in the union; last-CTA scratch in the ring
  static_assert((G * kHeadDim + 8 * G) * 4 <= kQFloats * 4, "CTA merge scratch");
  static_assert((2 * G + 2 * G * kMaxSplits + 2 * G * kHeadDim) * 4 <= kStageBytes, "merge scratch");
};

// head owned by head slot hs of a lane with column group tig (BF16 mma.sync)
template <int G>
__device__ __forceinline__ int slot_head(int tig, int hs) {
  if (G <= 4) return (2 * tig + hs) & (G - 1);
  return 8 * (hs >> 1) + 2 * tig + (hs & 1);
}

// head slot of accumulator component c of column tile nt (BF16 mma.sync)
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

__device__ __forceinline__ void flag(int32_t* st, int bit) {
  if (st) atomicOr(st, bit);
}

// Byte offset of element (row n, k) in a K-major, unswizzled B tile of
// N = 16 rows x K = 128: 8x16-byte core matrices, 128 bytes between K halves
// (LBO), 256 bytes between 8-row groups (SBO), 512 bytes per 16-wide k-step.
__device__ __forceinline__ int b_offset(int n, int k) {
  return (k >> 4) * 512 + (n >> 3) * 256 + ((k >> 3) & 1) * 128 + (n & 7) * 16 + (k & 7) * 2;
}

// The first 2G columns (G = 4: 8, G = 8: 16) of one accumulator, this lane.
template <int G>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[2 * G]) {
  if constexpr (G == 4) {
    tmem_ld8(taddr, r);
  } else {
    tmem_ld16(taddr, r);
  }
}
template <int G>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[2 * G]) {
  if constexpr (G == 4) {
    tmem_st8(taddr, r);
  } else {
    tmem_st16(taddr, r);
  }
}

// Unpacks 8 code words (16 codes each) into 64 fp16x2 TMEM columns of this
// lane: column 8i + j = (code j, code j + 8) of word i, scaled 4^pos(j) 2^-24.
__device__ __forceinline__ void codes_to_tmem(uint32_t taddr, const uint32_t (&wv)[8]) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t rr[32];
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) {
      const uint32_t w = wv[4 * half + ii], wsh = w >> 6;
#pragma unroll
      for (int j = 0; j < 8; ++j) rr[8 * ii + j] = code_pair(w, wsh, j);
    }
    tmem_st32(taddr + 32u * half, rr);
  }
}

// Bounded mbarrier wait that also ends early once another role aborted.
struct Waiter {
  volatile int* abort_flag;
  int32_t* dev_status;
  __device__ __forceinline__ bool wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait_sleep(bar, parity, 1000000u)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
      if (*abort_flag) return false;
      if (mbar_try_wait_sleep(bar, parity, 1000000u)) return true;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        flag(dev_status, 0x4);
        return false;
      }
    }
  }
};

// ------------------------------------------------------------------ BF16 path (mma.sync)

template <int G>
struct WarpState {
  static constexpr int NT = Geo<G>::NT, HS = Geo<G>::HS;
  float acc[NT][8][4];
  float m[HS], l[HS];
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
  __device__ __forceinline__ void pv_operand(const float (&pp)[HS][2], int tig,
                                             uint32_t (&pb)[NT][2]) const {
    auto pack = [](float a, float b) { return pack_bf162(a, b); };
    auto lo_of = [](float x) { return x - __bfloat162float(__float2bfloat16_rn(x)); };
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
  st.pv_operand(pp, tig, pb);
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

// A BF16 warp's (m, l, o) per head -> ws[h * kPartStride + (0, 1, 4 + channel)];
// the accumulator of (mt, c) holds channel 16 gid + 2 mt (+1 for c >= 2).
template <int G>
__device__ __forceinline__ void store_warp_state(WarpState<G>& st, float* ws, int gid, int tig) {
  constexpr int NT = Geo<G>::NT, HS = Geo<G>::HS;
#pragma unroll
  for (int hs = 0; hs < HS; ++hs) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) st.l[hs] += __shfl_xor_sync(kFull, st.l[hs], o);
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
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int h = slot_head<G>(tig, acc_slot<G>(nt, c));
        ws[h * kPartStride + 4 + 16 * gid + 2 * mt + (c >= 2 ? 1 : 0)] = st.acc[nt][mt][c];
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
// ------------------------------------------------------------------ q~ and the QK operand

// Shared-memory scratch of the prologue, in floats: qs[G][128] | part[4][G][128]
// | qt[G][128] | aux[G][4] | red[2][G][4].
template <int G>
struct QScratch {
  static constexpr int kQs = 0, kPart = G * kHeadDim, kQt = 5 * G * kHeadDim, kAux = 6 * G * kHeadDim;
  static constexpr int kRed = kAux + 4 * G;
  static constexpr int kFloats = kRed + 8 * G;
  static_assert(kFloats <= int(Geo<G>::kQFloats), "scratch fits");
};

constexpr int kPrologueThreads = 256;   // warps 0-7
constexpr uint32_t kPrologueBarrier = 1;

// q~ = q . R_K for the G query heads of (b, hkv) in fp32 (fixed summation
// order), by warps 0-7, from R_K (TMA, barrier `rbar`) and q already in
// shared memory.  Per head a power-of-two scale sigma puts max|q~ sigma| in
// [2^13, 2^14) so the fp16 hi part is normal and the lo part precise.  The
// QK B operand is written once: row n is head n (hi part) for n < G, head
// n - G (lo part) for n < 2G, zero otherwise; K index k = 2 col + e holds
// channel 16 (col / 8) + col % 8 + 8 e scaled by sigma 4^-pos(col % 8).
// aux[h] = (sigma, 2^24 / sigma * log2(e) / sqrt(d), sum(q~) log2(e) / sqrt(d)).
template <int G>
__device__ void rotate_query(const float* rks, uint64_t* rbar, float* scratch, uint8_t* bqk,
                             uint64_t* bqk_ready, int32_t* dev_status) {
  constexpr int T = kPrologueThreads;
  using S = QScratch<G>;
  const float* qs = scratch + S::kQs;
  float* part = scratch + S::kPart;
  float* qt = scratch + S::kQt;
  float* aux = scratch + S::kAux;
  float* red = scratch + S::kRed;
  const int tid = threadIdx.x;
  if (!mbar_wait_bounded(rbar, 0, kWaitLimitNs) && tid == 0) flag(dev_status, 0x4);
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
  if (tid < G) {
    const float mx = fmaxf(fmaxf(red[tid * 4], red[tid * 4 + 1]), fmaxf(red[tid * 4 + 2], red[tid * 4 + 3]));
    const float sm = ((red[4 * G + tid * 4] + red[4 * G + tid * 4 + 1]) + red[4 * G + tid * 4 + 2]) +
                     red[4 * G + tid * 4 + 3];
    int e = 0;
    if (mx > 0.f) {
      frexpf(mx, &e);              // mx in [2^(e-1), 2^e)
      e = max(-100, min(100, 14 - e));
    }
    const float scale = kLog2e * rsqrtf(float(kHeadDim));
    aux[tid * 4 + 0] = ldexpf(1.f, e);
    aux[tid * 4 + 1] = ldexpf(1.f, 24 - e) * scale;
    aux[tid * 4 + 2] = sm * scale;
  }
  named_barrier(kPrologueBarrier, T);
  for (int idx = tid; idx < kN * 64; idx += T) {
    const int n = idx / 64, col = idx % 64;
    const int w = col / 8, j = col % 8;
    uint32_t v = 0u;
    if (n < 2 * G) {
      const int h = n < G ? n : n - G;
      const float f = aux[h * 4] * __int_as_float((127 - 2 * code_pos(j)) << 23);   // sigma 4^-pos(j)
      float v0 = qt[h * kHeadDim + 16 * w + j] * f, v1 = qt[h * kHeadDim + 16 * w + 8 + j] * f;
      if (n >= G) {
        v0 = split_lo(v0);
        v1 = split_lo(v1);
      }
      v = pack_half2(v0, v1);
    }
    *reinterpret_cast<uint32_t*>(bqk + b_offset(n, 2 * col)) = v;
  }
  fence_proxy_async_smem();
  mbar_arrive(bqk_ready);   // the QK issuers wait for this
  named_barrier(kPrologueBarrier, T);
}

// ------------------------------------------------------------------ split kernel

template <int G>
__global__ void __launch_bounds__(kThreads, 1) split_kernel(DecodeParams p) {
  constexpr int T = kThreads;
  using Gm = Geo<G>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stage = smem + Gm::oStage;
  uint8_t* bqk = smem + Gm::oBqk;
  uint8_t* bp = smem + Gm::oBp;
  float* rks = reinterpret_cast<float*>(smem + Gm::oUni);          // R_K, then R_V
  float* qscratch = reinterpret_cast<float*>(smem + Gm::oUni + Gm::kRotBytes);
  float* st_bf16 = reinterpret_cast<float*>(smem + Gm::oBf16);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Gm::oBars);
  uint64_t* full = bars;
  uint64_t* empty = full + kSlots;
  uint64_t* ak_full = empty + kSlots;
  uint64_t* qk_done = ak_full + 2;
  uint64_t* qk_free = qk_done + 2;
  uint64_t* av_full = qk_free + 2;                // [kAvBufs]
  uint64_t* bp_full = av_full + kAvBufs;          // [kBpBufs]
  uint64_t* pv_done = bp_full + kBpBufs;          // [kBpBufs], PV of tile u -> u % kBpBufs
  uint64_t* rsbar = pv_done + kBpBufs;
  uint64_t* bqk_ready = rsbar + 1;
  uint64_t* rbar = bqk_ready + 1;
  uint64_t* vbar = rbar + 1;
  uint64_t* fin = vbar + 1;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Gm::oMisc);
  uint32_t* tmem_slot = misc;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  int* s_last = reinterpret_cast<int*>(misc + 2);
  constexpr int kMaskWords = (kSlots + 3) / 4 * 4;
  uint32_t* tile_mask = misc + 4;                                    // [kSlots]
  int* rs_flag = reinterpret_cast<int*>(misc + 4 + kMaskWords);      // [kBpBufs][4], 16-byte aligned
  float* rs_f = reinterpret_cast<float*>(rs_flag + 4 * kBpBufs);     // [kBpBufs][4][G] rescale factors
  float* st_m = rs_f + 4 * kBpBufs * G;                              // [4][G] softmax warps' maxima
  float* st_l = st_m + 4 * G;                                        // [4][G] sums of p
  float* st_z = st_l + 4 * G;                                        // [4][G] sums of p z_V
  static_assert(4 + kMaskWords + 4 * kBpBufs + (4 * kBpBufs + 12) * G <= int(Gm::kMiscBytes / 4), "misc fits");

  const int split = blockIdx.x, hkv = blockIdx.y, b = blockIdx.z;
  const int pair = b * p.n_kv + hkv;
  const int n_splits = p.n_splits;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const int pbeg = split * p.pages_per_split;

  // ---------------- barriers, R_K, tensor memory
  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 384);                 // softmax, V and K warps
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(ak_full + i, 128);
      mbar_init(qk_done + i, 4);                 // one commit per QK issuer
      mbar_init(qk_free + i, 128);
    }
    for (int i = 0; i < kAvBufs; ++i) mbar_init(av_full + i, 128);
    for (int i = 0; i < kBpBufs; ++i) {
      mbar_init(bp_full + i, 128);
      mbar_init(pv_done + i, 4);                 // one commit per PV issuer
    }
    mbar_init(rsbar, 128);
    mbar_init(bqk_ready, kPrologueThreads);
    mbar_init(rbar, 1);
    mbar_init(vbar, 1);
    mbar_init(fin, 8);                           // every MMA issuer, once
    *abort_flag = 0;
    fence_mbar_init();
    if (pbeg < p.max_pages) {
      mbar_arrive_expect_tx(rbar, uint32_t(Gm::kRotBytes));
      const float* rk = p.r_k + int64_t(hkv) * kHeadDim * kHeadDim;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        bulk_copy_g2s(rks + c * (kHeadDim * kHeadDim / 4), rk + c * (kHeadDim * kHeadDim / 4),
                      uint32_t(Gm::kRotBytes / 4), rbar);
    }
  }
  if (warp == kTmemWarp) tmem_alloc(tmem_slot, kTmemCols);
  if (warp < 8 && pbeg < p.max_pages) {
    const uint16_t* qg = p.q + (int64_t(b) * p.n_kv * G + int64_t(hkv) * G) * kHeadDim;
    for (int i = tid; i < G * kHeadDim; i += kPrologueThreads)
      qscratch[QScratch<G>::kQs + i] = __uint_as_float(uint32_t(qg[i]) << 16);
    // P operand buffers: rows >= 2G stay zero
    for (int i = tid; i < kBpBufs * kBBytes / 16; i += kPrologueThreads)
      reinterpret_cast<uint4*>(bp)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }

  // ---------------- history range of this CTA
  const int32_t* ptab = p.page_table + int64_t(b) * p.max_pages;
  int hist = p.hist_len[b];
  if (hist < 0 || hist > p.max_pages * kPage) {
    if (tid == 0) flag(p.dev_status, 0x2);
    hist = max(0, min(hist, p.max_pages * kPage));
  }
  const int n_pg = (hist + kPage - 1) / kPage;
  if (n_pg > n_splits * p.pages_per_split && split == 0 && tid == 0)
    flag(p.dev_status, 0x2);  // longer than the host bound max_hist: tail not read
  const int pend = min(pbeg + p.pages_per_split, n_pg);
  const int n_tiles = pend > pbeg ? (pend - pbeg + kTilePages - 1) / kTilePages : 0;
  const uint8_t* pool = p.pages + int64_t(hkv) * kBlockBytes;
  const int64_t page_stride = int64_t(p.n_kv) * kBlockBytes;

  tc_fence_before();
  __syncthreads();   // barriers initialised, TMEM address published
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  Waiter wt{abort_flag, p.dev_status};
  bool pv_final = false;   // V warps: the last PV products have landed

  if (warp < 8) {
    // ================= prologue: q~ and the QK operand (warps 0-7)
    float uns[G], qzh[G];
    if (n_tiles > 0) {
      rotate_query<G>(rks, rbar, qscratch, bqk, bqk_ready, p.dev_status);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        uns[h] = qscratch[QScratch<G>::kAux + h * 4 + 1];
        qzh[h] = qscratch[QScratch<G>::kAux + h * 4 + 2];
      }
    } else if (tid == 0 && pbeg < p.max_pages) {
      // R_K was requested: let it land before the CTA moves on
      if (!mbar_wait_bounded(rbar, 0, kWaitLimitNs)) flag(p.dev_status, 0x4);
    }
    // R_V -> shared memory (replacing R_K) for the output rotation
    if (tid == 0 && n_tiles > 0) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(vbar, uint32_t(Gm::kRotBytes));
      const float* rv = p.r_v + int64_t(hkv) * kHeadDim * kHeadDim;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        bulk_copy_g2s(rks + c * (kHeadDim * kHeadDim / 4), rv + c * (kHeadDim * kHeadDim / 4),
                      uint32_t(Gm::kRotBytes / 4), vbar);
    }

    if (warp < 4) {
      // ================= softmax: thread r = token r of a tile
      const int r = tid;
      const uint32_t lane_addr = tmem + (uint32_t(warp * 32) << 16);
      const int pg_in_tile = r >> 4, slot = r & 15;
      const float pos_scale = __int_as_float((127 - 2 * code_pos(slot & 7)) << 23);   // 4^-pos
      const int kslot = 2 * (8 * pg_in_tile + (slot & 7)) + (slot >> 3);
      float m[G], l[G], z[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
        z[h] = 0.f;
      }
      for (int t = 0; t < n_tiles; ++t) {
        const int s = t % kSlots;
        if (!wt.wait(full + s, (t / kSlots) & 1)) break;
        const uint8_t* pg = stage + s * kTileBytes + pg_in_tile * kBlockBytes;
        const uint32_t ksz = *reinterpret_cast<const uint32_t*>(pg + 512 + 4 * slot);
        const uint32_t vsz = *reinterpret_cast<const uint32_t*>(pg + kHalfBytes + 512 + 4 * slot);
        const uint32_t mask = tile_mask[s];
        mbar_arrive(empty + s);
        if (!wt.wait(qk_done + (t & 1), (t >> 1) & 1)) break;
        tc_fence_after();
        float dq[2 * G];
        {
          uint32_t dr[4][2 * G];
#pragma unroll
          for (int ch = 0; ch < 4; ++ch)
            tmem_ld_cols<G>(lane_addr + kColQK + uint32_t(64 * (t & 1) + kN * ch), dr[ch]);
          tc_wait_ld();
#pragma unroll
          for (int n = 0; n < 2 * G; ++n)
            dq[n] = (__uint_as_float(dr[0][n]) + __uint_as_float(dr[1][n])) +
                    (__uint_as_float(dr[2][n]) + __uint_as_float(dr[3][n]));
        }
        tc_fence_before();
        mbar_arrive(qk_free + (t & 1));
        const int pi = pbeg + kTilePages * t + pg_in_tile;
        const bool valid = ((mask >> pg_in_tile) & 1u) && pi * kPage + slot < hist;
        const float2 kz = half2_to_float2(ksz), vz = half2_to_float2(vsz);
        float sc[G];
        bool need = false;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          sc[h] = valid ? fmaf(kz.x * (dq[h] + dq[G + h]), uns[h], kz.y * qzh[h]) : -INFINITY;
          need |= sc[h] > m[h] + kRescaleLog2;
        }
        // lazy maximum of this warp; an accumulator that already holds
        // products of an older maximum is rescaled by the V warps
        float f[G];
        bool rescale = false;
#pragma unroll
        for (int h = 0; h < G; ++h) f[h] = 1.f;
        if (__any_sync(kFull, need)) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float wm = sc[h];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(kFull, wm, o));
            const float nm = fmaxf(m[h], wm);
            if (nm != m[h]) {
              rescale |= m[h] != -INFINITY;
              f[h] = exp2f(m[h] - nm);
              l[h] *= f[h];
              z[h] *= f[h];
              m[h] = nm;
            }
          }
        }
        // P operand buffer t % kBpBufs is free once PV of tile t - kBpBufs completed
        const int pb_i = t % kBpBufs;
        if (t >= kBpBufs && !wt.wait(pv_done + pb_i, ((t / kBpBufs) - 1) & 1)) break;
        if (lane == 0) {
          rs_flag[pb_i * 4 + warp] = (rescale && t > 0) ? 1 : 0;
#pragma unroll
          for (int h = 0; h < G; ++h) rs_f[(pb_i * 4 + warp) * G + h] = f[h];
        }
        uint8_t* pb = bp + pb_i * kBBytes;
        const float sv = vz.x * p.sigma_v * pos_scale;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float pr = valid ? exp2f(sc[h] - m[h]) : 0.f;
          l[h] += pr;
          z[h] = valid ? fmaf(pr, vz.y, z[h]) : z[h];
          const float pv = valid ? pr * sv : 0.f;
          const __half hi = __float2half_rn(pv);
          const __half lo = __float2half_rn(pv - __half2float(hi));
          *reinterpret_cast<__half*>(pb + b_offset(h, kslot)) = hi;
          *reinterpret_cast<__half*>(pb + b_offset(G + h, kslot)) = lo;
        }
        fence_proxy_async_smem();
        mbar_arrive(bp_full + pb_i);
      }
      // this warp's statistics
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float lv = l[h], zv = z[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          lv += __shfl_xor_sync(kFull, lv, o);
          zv += __shfl_xor_sync(kFull, zv, o);
        }
        if (lane == 0) {
          st_m[warp * G + h] = m[h];
          st_l[warp * G + h] = lv;
          st_z[warp * G + h] = zv;
        }
      }
    } else {
      // ================= V path (thread c = channel c) and the PV MMAs
      const int c = tid - 128, j = warp - kVWarp0;
      const uint32_t lane_addr = tmem + (uint32_t(j * 32) << 16);
      uint32_t rs_phase = 0;
      // PV MMAs of tile u: rescale requested accumulators first
      auto issue_pv = [&](int u) -> bool {
        const int ub = u % kBpBufs;
        if (!wt.wait(bp_full + ub, (u / kBpBufs) & 1)) return false;
        const int4 fl = *reinterpret_cast<const int4*>(rs_flag + ub * 4);
        if (fl.x | fl.y | fl.z | fl.w) {
          if (u >= 1 && !wt.wait(pv_done + (u - 1) % kBpBufs, ((u - 1) / kBpBufs) & 1)) return false;
          tc_fence_after();
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int fw = w == 0 ? fl.x : w == 1 ? fl.y : w == 2 ? fl.z : fl.w;
            if (fw) {
              const float* fr = rs_f + (ub * 4 + w) * G;
              uint32_t o[2 * G];
              tmem_ld_cols<G>(lane_addr + kColPV + uint32_t(kN * w), o);
              tc_wait_ld();
#pragma unroll
              for (int h = 0; h < G; ++h) {
                o[h] = __float_as_uint(__uint_as_float(o[h]) * fr[h]);
                o[G + h] = __float_as_uint(__uint_as_float(o[G + h]) * fr[h]);
              }
              tmem_st_cols<G>(lane_addr + kColPV + uint32_t(kN * w), o);
            }
          }
          tc_wait_st();
          tc_fence_before();
          mbar_arrive(rsbar);
          if (!wt.wait(rsbar, rs_phase & 1)) return false;
          ++rs_phase;
        }
        int ok = 1;
        if (lane == 0) {
          ok = wt.wait(av_full + u % kAvBufs, (u / kAvBufs) & 1);
          if (ok) {
            tc_fence_after();
            const uint32_t a = tmem + kColAV + 64u * uint32_t(u % kAvBufs);
            const uint32_t bb = smem_addr(bp) + uint32_t(ub) * kBBytes;
#pragma unroll
            for (int kk = 2 * j; kk < 2 * j + 2; ++kk)
              umma_f16_ts(tmem + kColPV + uint32_t(kN * j), a + 8u * kk,
                          smem_desc_kmajor(bb + 512u * kk, 128u, 256u), kIdesc, (u > 0 || (kk & 1)) ? 1u : 0u);
            umma_commit(pv_done + ub);
          }
        }
        return __shfl_sync(kFull, ok, 0) != 0;
      };
      bool ok = true;
      for (int t = 0; t < n_tiles; ++t) {
        const int s = t % kSlots;
        if (!wt.wait(full + s, (t / kSlots) & 1)) { ok = false; break; }
        // A_V buffer t % kAvBufs is free once PV of tile t - kAvBufs completed
        if (t >= kAvBufs && !wt.wait(pv_done + (t - kAvBufs) % kBpBufs, ((t - kAvBufs) / kBpBufs) & 1)) {
          ok = false;
          break;
        }
        const uint8_t* base = stage + s * kTileBytes + kHalfBytes + 4 * c;
        uint32_t wv[kTilePages];
#pragma unroll
        for (int i = 0; i < kTilePages; ++i) wv[i] = *reinterpret_cast<const uint32_t*>(base + i * kBlockBytes);
        codes_to_tmem(lane_addr + kColAV + 64u * uint32_t(t % kAvBufs), wv);
        tc_wait_st();
        mbar_arrive(empty + s);
        tc_fence_before();
        mbar_arrive(av_full + t % kAvBufs);
        if (t >= 1 && !issue_pv(t - 1)) { ok = false; break; }
      }
      if (ok && n_tiles > 0) ok = issue_pv(n_tiles - 1);
      if (lane == 0) umma_commit(fin);
      __syncwarp();
      pv_final = n_tiles > 0 && ok && wt.wait(pv_done + (n_tiles - 1) % kBpBufs, ((n_tiles - 1) / kBpBufs) & 1);
    }
  } else if (warp < kProducerWarp) {
    // ================= K path (thread r = token r) and the QK MMAs
    const int r = tid - 256, j = warp - kKWarp0;
    const uint32_t lane_addr = tmem + (uint32_t(j * 32) << 16);
    const int pg_in_tile = r >> 4, slot = r & 15;
    int ok = 1;
    if (n_tiles > 0 && lane == 0) ok = wt.wait(bqk_ready, 0);
    ok = __shfl_sync(kFull, ok, 0);
    for (int t = 0; ok && t < n_tiles; ++t) {
      const int s = t % kSlots;
      if (!wt.wait(full + s, (t / kSlots) & 1)) break;
      // A_K and D_qk buffers t % 2 are free once the softmax read tile t - 2
      if (t >= 2 && !wt.wait(qk_free + (t & 1), ((t - 2) >> 1) & 1)) break;
      const uint8_t* pg = stage + s * kTileBytes + pg_in_tile * kBlockBytes + 32 * slot;
      const uint4 a0 = *reinterpret_cast<const uint4*>(pg);
      const uint4 a1 = *reinterpret_cast<const uint4*>(pg + 16);
      const uint32_t wv[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      codes_to_tmem(lane_addr + kColAK + 64u * uint32_t(t & 1), wv);
      tc_wait_st();
      mbar_arrive(empty + s);
      tc_fence_before();
      mbar_arrive(ak_full + (t & 1));
      if (lane == 0) {
        ok = wt.wait(ak_full + (t & 1), (t >> 1) & 1);
        if (ok) {
          tc_fence_after();
          const uint32_t a = tmem + kColAK + 64u * uint32_t(t & 1);
          const uint32_t d = tmem + kColQK + uint32_t(64 * (t & 1) + kN * j);
          const uint32_t bq = smem_addr(bqk);
#pragma unroll
          for (int kk = 2 * j; kk < 2 * j + 2; ++kk)
            umma_f16_ts(d, a + 8u * kk, smem_desc_kmajor(bq + 512u * kk, 128u, 256u), kIdesc, kk & 1);
          umma_commit(qk_done + (t & 1));
        }
      }
      ok = __shfl_sync(kFull, ok, 0);
    }
    if (lane == 0) umma_commit(fin);
    __syncwarp();
  } else if (warp == kProducerWarp) {
    // ================= producer: 8 page blocks per tile, one lane per page
    int win_base = -1, win_pid = -1, issued = 0;
    for (int t = 0; t < n_tiles; ++t) {
      const int s = t % kSlots;
      int ok = 1;
      if (t >= kSlots && lane == 0) ok = wt.wait(empty + s, ((t / kSlots) - 1) & 1);
      if (!__shfl_sync(kFull, ok, 0)) break;
      const int wb = (kTilePages * t) & ~31;
      if (wb != win_base) {
        win_base = wb;
        const int pi = pbeg + wb + lane;
        win_pid = pi < pend ? __ldg(ptab + pi) : -1;
      }
      const int pid = __shfl_sync(kFull, win_pid, (kTilePages * t + (lane & 7)) & 31);
      const int pi = pbeg + kTilePages * t + lane;
      const bool in_range = lane < kTilePages && pi < pend;
      const bool good = in_range && pid >= 0 && pid < p.n_pages;
      if (in_range && !good) flag(p.dev_status, 0x1);
      const uint32_t mask = __ballot_sync(kFull, good);
      if (lane == 0) {
        tile_mask[s] = mask;
        if (mask)
          mbar_arrive_expect_tx(full + s, uint32_t(__popc(mask)) * kBlockBytes);
        else
          mbar_arrive(full + s);
      }
      __syncwarp();
      if (good)
        bulk_copy_g2s(stage + s * kTileBytes + lane * kBlockBytes, pool + int64_t(pid) * page_stride,
                      kBlockBytes, full + s);
      issued = t + 1;
    }
    // the copies of the last tiles land before the CTA may end
    if (lane == 0)
      for (int t = max(0, issued - kSlots); t < issued; ++t)
        mbar_wait_bounded(full + t % kSlots, (t / kSlots) & 1, kWaitLimitNs);
    __syncwarp();
  } else if (warp >= kBf16Warp) {
    // ================= BF16 sink / recent tokens (warps 14, 15)
    constexpr int NTQ = Gm::NTQ;
    const int bw = warp - kBf16Warp;
    int sink_len = p.sink_len[b], rec_len = p.recent_len[b];
    const int rec_start = p.recent_start[b];
    if (sink_len < 0 || sink_len > p.sink_cap || rec_len < 0 || rec_len > p.recent_cap ||
        rec_start < 0 || rec_start >= max(p.recent_cap, 1)) {
      if (lane == 0 && bw == 0) flag(p.dev_status, 0x2);
      sink_len = max(0, min(sink_len, p.sink_cap));
      rec_len = max(0, min(rec_len, p.recent_cap));
    }
    const int start = min(max(rec_start, 0), max(p.recent_cap - 1, 0));
    const int n_vp = p.sink_cap / kPage + p.recent_cap / kPage;
    const int64_t hstride = int64_t(p.n_kv) * kHeadDim;
    WarpState<G> st;
    st.init();
    // virtual page vp goes to CTA vp % n_splits, warp (vp / n_splits) % 2
    const int mine = split + bw * n_splits;
    if (mine < n_vp) {
      uint32_t qf[NTQ][8][2];
#pragma unroll
      for (int nt = 0; nt < NTQ; ++nt) {
        const int h = (8 * nt + gid) % G;
        const uint16_t* qrow = p.q + (int64_t(b) * p.n_kv * G + hkv * G + h) * kHeadDim + 32 * tig;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(qrow + 8 * u));
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
      for (int vp = mine; vp < n_vp; vp += 2 * n_splits) {
        const int u0 = vp * kPage;
        bool kok[2], vok[4];
        const uint16_t* krow[2] = {row_of(u0 + gid, false, kok[0]), row_of(u0 + gid + 8, false, kok[1])};
        const uint16_t* vrow[4] = {row_of(u0 + 2 * tig, true, vok[0]), row_of(u0 + 2 * tig + 1, true, vok[1]),
                                   row_of(u0 + 2 * tig + 8, true, vok[2]),
                                   row_of(u0 + 2 * tig + 9, true, vok[3])};
        bf16_page<G>(krow, vrow, kok, vok, gid, tig, qf, st);
      }
    }
    store_warp_state<G>(st, st_bf16 + bw * G * kPartStride, gid, tig);
  }

  // ================= all roles done
  tc_fence_before();
  __syncthreads();

  float* part = p.partials + (int64_t(pair) * n_splits + split) * 2 * G * kPartStride;
  float* os = qscratch;                  // [G][128] o~ without zeta (history, rotated basis)
  float* hz = qscratch + G * kHeadDim;   // [G][4]: zeta, BF16 weights f0, f1
  // history: the 4 softmax warps' accumulators merged with their maxima
  if (warp >= kVWarp0 && warp < kKWarp0) {
    const int c = tid - 128;
    const uint32_t lane_addr = tmem + (uint32_t((warp - kVWarp0) * 32) << 16);
    float o[G];
#pragma unroll
    for (int h = 0; h < G; ++h) o[h] = 0.f;
    if (pv_final) {
      tc_fence_after();
      uint32_t d[4][2 * G];
#pragma unroll
      for (int w = 0; w < 4; ++w) tmem_ld_cols<G>(lane_addr + kColPV + uint32_t(kN * w), d[w]);
      tc_wait_ld();
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w)
          if (st_l[w * G + h] > 0.f) mx = fmaxf(mx, st_m[w * G + h]);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float e = st_l[w * G + h] > 0.f ? exp2f(st_m[w * G + h] - mx) : 0.f;
          o[h] = fmaf(e, __uint_as_float(d[w][h]) + __uint_as_float(d[w][G + h]), o[h]);
        }
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) os[h * kHeadDim + c] = o[h] * p.pv_unscale;
    tc_fence_before();
  }
  // history statistics and the BF16 partial's (m, l)
  if (tid < G) {
    const int h = tid;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w)
      if (st_l[w * G + h] > 0.f) mx = fmaxf(mx, st_m[w * G + h]);
    float lsum = 0.f, zsum = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float e = st_l[w * G + h] > 0.f ? exp2f(st_m[w * G + h] - mx) : 0.f;
      lsum = fmaf(e, st_l[w * G + h], lsum);
      zsum = fmaf(e, st_z[w * G + h], zsum);
    }
    const bool any = n_tiles > 0 && lsum > 0.f;
    part[h * kPartStride + 0] = any ? mx : -INFINITY;
    part[h * kPartStride + 1] = any ? lsum : 0.f;
    hz[h * 4 + 0] = any ? zsum : 0.f;
    const float* s0 = st_bf16 + h * kPartStride;
    const float* s1 = st_bf16 + (G + h) * kPartStride;
    const float m0 = s0[0], l0 = s0[1], m1 = s1[0], l1 = s1[1];
    const float bx = l1 > 0.f ? (l0 > 0.f ? fmaxf(m0, m1) : m1) : m0;
    const float f0 = l0 > 0.f ? exp2f(m0 - bx) : 0.f, f1 = l1 > 0.f ? exp2f(m1 - bx) : 0.f;
    hz[h * 4 + 1] = f0;
    hz[h * 4 + 2] = f1;
    part[(G + h) * kPartStride + 0] = bx;
    part[(G + h) * kPartStride + 1] = fmaf(l0, f0, l1 * f1);
  }
  __syncthreads();
  if (warp == kTmemWarp) {
    tc_fence_after();
    if (lane == 0 && !mbar_wait_bounded(fin, 0, kWaitLimitNs)) flag(p.dev_status, 0x4);
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
  // BF16 partial: merge of the two warps
  for (int idx = tid; idx < G * kHeadDim; idx += T) {
    const int h = idx / kHeadDim, c = idx % kHeadDim;
    part[(G + h) * kPartStride + 4 + c] =
        fmaf(hz[h * 4 + 1], st_bf16[h * kPartStride + 4 + c], hz[h * 4 + 2] * st_bf16[(G + h) * kPartStride + 4 + c]);
  }
  if (n_tiles > 0) {
    if (!mbar_wait_bounded(vbar, 0, kWaitLimitNs) && tid == 0) flag(p.dev_status, 0x4);
    // history partial back in the original basis:
    // o[c] = sum_j (o~[j] + zeta) R_V[c][j]; thread (row c, quarter qq), chunk
    // order rotated by the lane so the 32 lanes of a load hit all 32 banks
    const float* rvs = rks;
    for (int task = tid; task < 4 * kHeadDim; task += T) {
      const int c = task >> 2, qq = task & 3;
      const int rot = lane & 7;
      const float* rrow = rvs + c * kHeadDim + 32 * qq;
      float4 rv[8];
      float rsum = 0.f;
#pragma unroll
      for (int k4 = 0; k4 < 8; ++k4) {
        rv[k4] = reinterpret_cast<const float4*>(rrow)[(k4 + rot) & 7];
        rsum += (rv[k4].x + rv[k4].y) + (rv[k4].z + rv[k4].w);
      }
#pragma unroll 1
      for (int h = 0; h < G; ++h) {
        const float4* o = reinterpret_cast<const float4*>(os + h * kHeadDim + 32 * qq);
        float d = 0.f;
#pragma unroll
        for (int k4 = 0; k4 < 8; ++k4) {
          const float4 ov = o[(k4 + rot) & 7];
          d = fmaf(ov.x, rv[k4].x, fmaf(ov.y, rv[k4].y, fmaf(ov.z, rv[k4].z, fmaf(ov.w, rv[k4].w, d))));
        }
        d = fmaf(hz[h * 4 + 0], rsum, d);
        d += __shfl_xor_sync(kFull, d, 1);
        d += __shfl_xor_sync(kFull, d, 2);
        if (qq == 0) part[h * kPartStride + 4 + c] = d;
      }
    }
  } else {
    for (int idx = tid; idx < G * kHeadDim; idx += T)
      part[(idx / kHeadDim) * kPartStride + 4 + idx % kHeadDim] = 0.f;
  }

  // ---------------- ticket: the last CTA of this (request, KV head) merges
  __syncthreads();
  if (tid == 0) {
    fence_acq_rel_gpu();
    const unsigned tk = atomicAdd(p.counters + pair, 1u);
    *s_last = (tk == unsigned(n_splits - 1)) ? 1 : 0;
  }
  __syncthreads();
  if (!*s_last) return;
  fence_acq_rel_gpu();

  constexpr int W = kWarps;
  const float* pp = p.partials + int64_t(pair) * n_splits * 2 * G * kPartStride;
  const int NP = 2 * n_splits;                        // partials per head
  float* ml = reinterpret_cast<float*>(stage);        // [G][2] (max, 1 / L)
  float* wts = ml + 2 * G;                            // [G][2 * kMaxSplits] weights
  float* oh = wts + G * 2 * kMaxSplits;               // [2][G][128] half sums
  // weights per head over its 2 n_splits partials (split-major, type-minor)
  for (int h = warp; h < G; h += W) {
    float mx = -INFINITY;
    for (int i = lane; i < NP; i += 32) {
      const float* r = pp + int64_t(i * G + h) * kPartStride;
      if (__ldcg(r + 1) > 0.f) mx = fmaxf(mx, __ldcg(r));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    float lsum = 0.f;
    for (int i = lane; i < NP; i += 32) {
      const float* r = pp + int64_t(i * G + h) * kPartStride;
      const float l = __ldcg(r + 1);
      const float f = l > 0.f ? exp2f(__ldcg(r) - mx) : 0.f;
      wts[h * 2 * kMaxSplits + i] = f;
      lsum = fmaf(l, f, lsum);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(kFull, lsum, o);
    if (lane == 0) ml[h * 2 + 1] = lsum > 0.f ? 1.f / lsum : 0.f;
  }
  __syncthreads();
  // weighted sums: one warp per (half, head), lanes over channels (float4),
  // loads of a batch issued together
  for (int task = warp; task < 2 * G; task += W) {
    const int half = task / G, h = task % G;
    const int i0 = half ? NP / 2 : 0, i1 = half ? NP : NP / 2;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int ib = i0; ib < i1; ib += 8) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (ib + u < i1)
          v[u] = __ldcg(reinterpret_cast<const float4*>(pp + int64_t((ib + u) * G + h) * kPartStride + 4) + lane);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (ib + u < i1) {
          const float f = wts[h * 2 * kMaxSplits + ib + u];
          a.x = fmaf(f, v[u].x, a.x);
          a.y = fmaf(f, v[u].y, a.y);
          a.z = fmaf(f, v[u].z, a.z);
          a.w = fmaf(f, v[u].w, a.w);
        }
    }
    reinterpret_cast<float4*>(oh + (half * G + h) * kHeadDim)[lane] = a;
  }
  __syncthreads();
  for (int idx = tid; idx < G * kHeadDim; idx += T) {
    const int h = idx / kHeadDim;
    p.out[(int64_t(b) * p.n_kv * G + int64_t(hkv) * G) * kHeadDim + idx] =
        (oh[idx] + oh[G * kHeadDim + idx]) * ml[h * 2 + 1];
  }
  if (tid == 0) p.counters[pair] = 0u;   // ready for the next call
}

template <int G>
int occupancy() {
  int occ = 0;
  cudaFuncSetAttribute(split_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(Geo<G>::kSmem));
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, split_kernel<G>, kThreads, Geo<G>::kSmem) !=
      cudaSuccess)
    return 0;
  return occ;
}

template <int G>
cudaError_t launch_g(const DecodeParams& p, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(split_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(Geo<G>::kSmem));
  if (e != cudaSuccess) return e;
  split_kernel<G><<<dim3(p.n_splits, p.n_kv, p.batch), kThreads, Geo<G>::kSmem, stream>>>(p);
  return cudaGetLastError();
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

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
  const int64_t slots = int64_t(sms) * occ;
  const int64_t pairs = int64_t(batch) * n_kv;
  const int pages_max = (max_hist + kPage - 1) / kPage;
  // one wave when every (request, KV head) can get whole SMs and each CTA
  // then streams at most 512 tiles; otherwise 32 tiles per CTA and several
  // waves balanced by the block scheduler
  int pps;
  const int64_t per_pair = slots / pairs;
  if (per_pair >= 1 && (pages_max + per_pair - 1) / per_pair <= 512 * kTilePages) {
    pps = int((pages_max + per_pair - 1) / per_pair);
  } else {
    pps = 32 * kTilePages;
  }
  pps = max(pps, 1);
  pps = (pps + kTilePages - 1) / kTilePages * kTilePages;
  int n_splits = max(1, (pages_max + pps - 1) / pps);
  if (n_splits > kMaxSplits) {
    pps = (pages_max + kMaxSplits - 1) / kMaxSplits;
    pps = (pps + kTilePages - 1) / kTilePages * kTilePages;
    n_splits = (pages_max + pps - 1) / pps;
  }
  plan->n_splits = n_splits;
  plan->pages_per_split = pps;
  size_t off = 0;
  plan->off_counters = off;
  off = align256(off + size_t(pairs) * 4);
  plan->off_partials = off;
  off = align256(off + size_t(pairs) * n_splits * 2 * group * kPartStride * 4);
  plan->total_bytes = off;
  *err = cudaSuccess;
  return occ;
}

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
  if (p.group == 4) return launch_g<4>(p, stream);
  if (p.group == 8) return launch_g<8>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace oscar
