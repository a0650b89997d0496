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
// One launch; CTA (split, KV head, request) of 12 warps, one CTA per SM, owns
// a contiguous range of INT2 pages of one (request, KV head) and a share of
// its BF16 sink/recent tokens.  The INT2 pages are processed in tiles of 8
// pages (128 tokens) by a warp-specialised tcgen05 pipeline:
//   warp 8      producer: 1-D TMA bulk copies of the tile's 8 page blocks into
//               a ring of tile slots (mbarrier transaction counts);
//   warps 0-3   K path, thread = token: unpack the token's 128 K codes into
//               fp16 and store them in tensor memory (A of QK); after the QK
//               MMA, read the scores back (one token, all heads per thread),
//               online softmax, write p s_V (hi | lo fp16) to shared memory
//               (B of PV);
//   warps 4-7   V path, thread = channel: unpack the channel's codes of the
//               tile's 128 tokens into fp16 in tensor memory (A of PV);
//   warp 9      owns tensor memory and issues the MMAs from one lane:
//               QK: D[token][col] = codes[token][k] . B_qk[k][col]
//               PV: O[channel][col] += codes^T[channel][token] . P[token][col]
//               (M = 128, N = 16, K = 16 per instruction, fp32 accumulate in
//               tensor memory), completion signalled by tcgen05.commit;
//   warps 10-11 the BF16 sink/recent tokens (mma.sync, bf16), concurrently.
// The columns of B are the GQA heads' hi parts then lo parts (fp16 hi + lo
// split of an fp32 value), so each MMA carries about fp32 precision.
// A 2-bit code c at bit offset 2k of a 16-bit half is read as the fp16
// subnormal c * 4^k * 2^-24 by one AND; the 4^k factors go into B and 2^-24
// into the output scale.  The online-softmax maximum is raised lazily (only
// when a score exceeds it by 2^8), and then the O accumulator in tensor
// memory is rescaled in place.
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
constexpr float kRescaleLog2 = 8.0f;          // lazy rescale threshold (p <= 2^8)
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr uint32_t kFull = 0xffffffffu;
constexpr int kMaxSplits = 128;               // bounds the last CTA's merge scratch

constexpr int kTilePages = 8;
constexpr int kTileTokens = kTilePages * kPage;           // 128
constexpr int kTileBytes = kTilePages * kBlockBytes;      // 9216
constexpr int kSlots = OSCAR_TILE_SLOTS;
constexpr int kWarps = 12;
constexpr int kThreads = kWarps * 32;
constexpr int kProducerWarp = 8, kMmaWarp = 9, kBf16Warp = 10;
constexpr int kN = 16;                                      // MMA N: hi | lo columns
constexpr uint32_t kIdesc = idesc_f16_f32(128, kN);
// tensor-memory columns
constexpr uint32_t kColAK = 0, kColAV = 128, kColQK = 256, kColPV = 288, kTmemCols = 512;
constexpr int kBBytes = kN * kTileTokens * 2;               // one B operand tile (K = 128)

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
  static constexpr int kBars = 2 * kSlots + 2 * 5 + 4;   // full, empty | ak qk bp av pv | x rk rv fin
  static constexpr size_t kBarBytes = (kBars * 8 + 127) / 128 * 128;
  static constexpr size_t kMiscBytes = 1024;
  static constexpr size_t oStage = 0;
  static constexpr size_t oBqk = oStage + kStageBytes;
  static constexpr size_t oBp = oBqk + kBBytes;
  static constexpr size_t oUni = oBp + 2 * kBBytes;
  static constexpr size_t oBf16 = oUni + kUnion;
  static constexpr size_t oBars = (oBf16 + kBf16State + 127) / 128 * 128;
  static constexpr size_t oMisc = oBars + kBarBytes;
  static constexpr size_t kSmem = oMisc + kMiscBytes;
  static_assert(kStageBytes % 128 == 0 && oBqk % 128 == 0 && oUni % 128 == 0, "TMA / UMMA operands aligned");
  static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
  // CTA merge scratch after R_V in the union; last-CTA scratch in the ring
  static_assert((G * kHeadDim + 4 * G) * 4 <= kQFloats * 4, "CTA merge scratch");
  static_assert((2 * G + 2 * G * 128 + 2 * G * kHeadDim) * 4 <= kStageBytes, "merge scratch");
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

// Bounded mbarrier wait that also ends early once another role aborted.
struct Waiter {
  volatile int* abort_flag;
  int32_t* dev_status;
  __device__ __forceinline__ bool wait(uint64_t* bar, uint32_t parity) {
    if (*abort_flag) return false;
    if (mbar_try_wait_sleep(bar, parity, 1000000u)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
      if (mbar_try_wait_sleep(bar, parity, 1000000u)) return true;
      if (*abort_flag) return false;
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
                             int32_t* dev_status) {
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
  uint64_t* bp_full = qk_done + 2;
  uint64_t* av_full = bp_full + 2;
  uint64_t* pv_done = av_full + 2;
  uint64_t* xbar = pv_done + 2;
  uint64_t* rbar = xbar + 1;
  uint64_t* vbar = rbar + 1;
  uint64_t* fin = vbar + 1;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Gm::oMisc);
  uint32_t* tmem_slot = misc;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  int* s_last = reinterpret_cast<int*>(misc + 2);
  constexpr int kMaskWords = (kSlots + 3) / 4 * 4;
  uint32_t* tile_mask = misc + 4;                                    // [kSlots]
  float* xchg = reinterpret_cast<float*>(misc + 4 + kMaskWords);     // [2][4 + 4G], 16-byte aligned
  float* red_lz = xchg + 2 * (4 + 4 * G);                            // [4][2G] (l | zeta)
  float* s_m = red_lz + 8 * G;                                       // [G]
  static_assert(4 + kMaskWords + 2 * (4 + 4 * G) + 8 * G + G <= int(Gm::kMiscBytes / 4), "misc fits");

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
      mbar_init(empty + s, 256);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(ak_full + i, 128);
      mbar_init(qk_done + i, 1);
      mbar_init(bp_full + i, 128);
      mbar_init(av_full + i, 128);
      mbar_init(pv_done + i, 1);
    }
    mbar_init(xbar, 128);
    mbar_init(rbar, 1);
    mbar_init(vbar, 1);
    mbar_init(fin, 1);
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
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, kTmemCols);
  if (warp < 8 && pbeg < p.max_pages) {
    const uint16_t* qg = p.q + (int64_t(b) * p.n_kv * G + int64_t(hkv) * G) * kHeadDim;
    for (int i = tid; i < G * kHeadDim; i += kPrologueThreads)
      qscratch[QScratch<G>::kQs + i] = __uint_as_float(uint32_t(qg[i]) << 16);
    // P operand buffers: rows >= 2G stay zero
    for (int i = tid; i < 2 * kBBytes / 16; i += kPrologueThreads)
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

  if (warp < 8) {
    // ================= prologue: q~ and the QK operand (warps 0-7)
    float uns[G], qzh[G];
    if (n_tiles > 0) {
      rotate_query<G>(rks, rbar, qscratch, bqk, p.dev_status);
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
      // ================= K path and softmax: thread r = token r of a tile
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
      uint32_t ksz_n = 0, vsz_n = 0, mask_n = 0;   // of the tile converted last
      // K codes of tile t -> A_K[t % 2]; keeps the tile's scales for its softmax
      auto convert = [&](int t) -> bool {
        const int s = t % kSlots;
        if (!wt.wait(full + s, (t / kSlots) & 1)) return false;
        const uint8_t* pg = stage + s * kTileBytes + pg_in_tile * kBlockBytes;
        const uint4 a0 = *reinterpret_cast<const uint4*>(pg + 32 * slot);
        const uint4 a1 = *reinterpret_cast<const uint4*>(pg + 32 * slot + 16);
        ksz_n = *reinterpret_cast<const uint32_t*>(pg + 512 + 4 * slot);
        vsz_n = *reinterpret_cast<const uint32_t*>(pg + kHalfBytes + 512 + 4 * slot);
        mask_n = tile_mask[s];
        const uint32_t wv[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint32_t col0 = lane_addr + kColAK + 64u * uint32_t(t & 1);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t rr[32];
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {
            const uint32_t w = wv[4 * half + wi], wsh = w >> 6;
#pragma unroll
            for (int j = 0; j < 8; ++j) rr[8 * wi + j] = code_pair(w, wsh, j);
          }
          tmem_st32(col0 + 32u * half, rr);
        }
        tc_wait_st();
        mbar_arrive(empty + s);
        tc_fence_before();
        mbar_arrive(ak_full + (t & 1));
        return true;
      };
      auto softmax = [&](int t, uint32_t ksz, uint32_t vsz, uint32_t mask) -> bool {
        if (!wt.wait(qk_done + (t & 1), (t >> 1) & 1)) return false;
        tc_fence_after();
        uint32_t dr[16];
        tmem_ld16(lane_addr + kColQK + 16u * uint32_t(t & 1), dr);
        tc_wait_ld();
        const int pi = pbeg + kTilePages * t + pg_in_tile;
        const bool valid = ((mask >> pg_in_tile) & 1u) && pi * kPage + slot < hist;
        const float2 kz = half2_to_float2(ksz), vz = half2_to_float2(vsz);
        float sc[G];
        bool need = false;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float full_d = __uint_as_float(dr[h]) + __uint_as_float(dr[G + h]);
          sc[h] = valid ? fmaf(kz.x * full_d, uns[h], kz.y * qzh[h]) : -INFINITY;
          need |= sc[h] > m[h] + kRescaleLog2;
        }
        // lazy maximum: the 4 warps agree through one exchange per tile
        float* xv = xchg + (t & 1) * (4 + 4 * G);
        const bool vote = __any_sync(kFull, need);
        if (lane == 0) reinterpret_cast<int*>(xv)[warp] = vote ? 1 : 0;
        if (vote) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float wm = sc[h];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(kFull, wm, o));
            if (lane == h) xv[4 + warp * G + h] = wm;
          }
        }
        mbar_arrive(xbar);
        if (!wt.wait(xbar, t & 1)) return false;
        const int4 votes = *reinterpret_cast<const int4*>(xv);
        if (votes.x | votes.y | votes.z | votes.w) {
          float f[G];
          bool any_f = false;
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float nm = m[h];
            if (votes.x) nm = fmaxf(nm, xv[4 + 0 * G + h]);
            if (votes.y) nm = fmaxf(nm, xv[4 + 1 * G + h]);
            if (votes.z) nm = fmaxf(nm, xv[4 + 2 * G + h]);
            if (votes.w) nm = fmaxf(nm, xv[4 + 3 * G + h]);
            f[h] = nm == m[h] ? 1.f : exp2f(m[h] - nm);
            any_f |= nm != m[h];
            m[h] = nm;
            l[h] *= f[h];
            z[h] *= f[h];
          }
          if (any_f && t > 0) {
            // rescale O (row r) once every earlier PV product has landed
            if (!wt.wait(pv_done + ((t - 1) & 1), ((t - 1) >> 1) & 1)) return false;
            tc_fence_after();
            uint32_t orow[16];
            tmem_ld16(lane_addr + kColPV, orow);
            tc_wait_ld();
#pragma unroll
            for (int h = 0; h < G; ++h) {
              orow[h] = __float_as_uint(__uint_as_float(orow[h]) * f[h]);
              orow[G + h] = __float_as_uint(__uint_as_float(orow[G + h]) * f[h]);
            }
            tmem_st16(lane_addr + kColPV, orow);
            tc_wait_st();
          }
        }
        // probabilities -> P operand (hi | lo), K index of this token
        if (t >= 2 && !wt.wait(pv_done + (t & 1), ((t - 2) >> 1) & 1)) return false;
        uint8_t* pb = bp + (t & 1) * kBBytes;
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
        tc_fence_before();
        mbar_arrive(bp_full + (t & 1));
        return true;
      };
      bool ok = n_tiles > 0 ? convert(0) : true;
      for (int t = 0; ok && t < n_tiles; ++t) {
        const uint32_t ksz = ksz_n, vsz = vsz_n, mask = mask_n;
        if (t + 1 < n_tiles && !convert(t + 1)) break;
        ok = softmax(t, ksz, vsz, mask);
      }
      // per-warp sums of l and zeta
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float lv = l[h], zv = z[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          lv += __shfl_xor_sync(kFull, lv, o);
          zv += __shfl_xor_sync(kFull, zv, o);
        }
        if (lane == h) {
          red_lz[warp * 2 * G + h] = lv;
          red_lz[warp * 2 * G + G + h] = zv;
        }
        if (tid == 0) s_m[h] = m[h];
      }
    } else {
      // ================= V path: thread c = channel c
      const int c = tid - 128;
      const uint32_t lane_addr = tmem + (uint32_t((warp & 3) * 32) << 16);
      bool ok = true;
      for (int t = 0; t < n_tiles; ++t) {
        const int s = t % kSlots;
        if (!wt.wait(full + s, (t / kSlots) & 1)) { ok = false; break; }
        if (t >= 2 && !wt.wait(pv_done + (t & 1), ((t - 2) >> 1) & 1)) { ok = false; break; }
        const uint8_t* base = stage + s * kTileBytes + kHalfBytes + 4 * c;
        uint32_t wv[kTilePages];
#pragma unroll
        for (int i = 0; i < kTilePages; ++i) wv[i] = *reinterpret_cast<const uint32_t*>(base + i * kBlockBytes);
        const uint32_t col0 = lane_addr + kColAV + 64u * uint32_t(t & 1);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t rr[32];
#pragma unroll
          for (int ii = 0; ii < 4; ++ii) {
            const uint32_t w = wv[4 * half + ii], wsh = w >> 6;
#pragma unroll
            for (int j = 0; j < 8; ++j) rr[8 * ii + j] = code_pair(w, wsh, j);
          }
          tmem_st32(col0 + 32u * half, rr);
        }
        tc_wait_st();
        mbar_arrive(empty + s);
        tc_fence_before();
        mbar_arrive(av_full + (t & 1));
      }
      // O row c: o~_h[c] = (hi + lo) * 2^24 / sigma_v (zeta added later)
      float* os = qscratch;   // [G][128], read after the role barrier
      if (n_tiles > 0 && ok &&
          wt.wait(pv_done + ((n_tiles - 1) & 1), ((n_tiles - 1) >> 1) & 1)) {
        tc_fence_after();
        uint32_t orow[16];
        tmem_ld16(lane_addr + kColPV, orow);
        tc_wait_ld();
#pragma unroll
        for (int h = 0; h < G; ++h)
          os[h * kHeadDim + c] = (__uint_as_float(orow[h]) + __uint_as_float(orow[G + h])) * p.pv_unscale;
      } else {
#pragma unroll
        for (int h = 0; h < G; ++h) os[h * kHeadDim + c] = 0.f;
      }
    }
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
  } else if (warp == kMmaWarp) {
    // ================= MMA issue (one lane)
    if (lane == 0) {
      const uint32_t idesc = kIdesc;
      const uint32_t bqk_addr = smem_addr(bqk), bp_addr = smem_addr(bp);
      for (int t = 0; t <= n_tiles; ++t) {
        if (t < n_tiles) {
          if (!wt.wait(ak_full + (t & 1), (t >> 1) & 1)) break;
          tc_fence_after();
          const uint32_t a = tmem + kColAK + 64u * uint32_t(t & 1);
          const uint32_t d = tmem + kColQK + 16u * uint32_t(t & 1);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_f16_ts(d, a + 8u * kk, smem_desc_kmajor(bqk_addr + 512u * kk, 128u, 256u), idesc, kk > 0);
          umma_commit(qk_done + (t & 1));
        }
        if (t >= 1) {
          const int u = t - 1;
          if (!wt.wait(av_full + (u & 1), (u >> 1) & 1)) break;
          if (!wt.wait(bp_full + (u & 1), (u >> 1) & 1)) break;
          tc_fence_after();
          const uint32_t a = tmem + kColAV + 64u * uint32_t(u & 1);
          const uint32_t bb = bp_addr + uint32_t(u & 1) * kBBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_f16_ts(tmem + kColPV, a + 8u * kk, smem_desc_kmajor(bb + 512u * kk, 128u, 256u), idesc,
                        (u > 0 || kk > 0) ? 1u : 0u);
          umma_commit(pv_done + (u & 1));
        }
      }
      // every MMA issued has completed before tensor memory is released
      umma_commit(fin);
      mbar_wait_bounded(fin, 0, kWaitLimitNs);
    }
    __syncwarp();
  } else {
    // ================= BF16 sink / recent tokens (warps 10, 11)
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
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }

  float* part = p.partials + (int64_t(pair) * n_splits + split) * 2 * G * kPartStride;
  float* os = qscratch;                  // [G][128] o~ without zeta (history, rotated basis)
  float* hz = qscratch + G * kHeadDim;   // [G][4]: m, l, zeta
  // BF16 partial: merge of the two warps; history statistics
  if (tid < G) {
    const int h = tid;
    const float* s0 = st_bf16 + h * kPartStride;
    const float* s1 = st_bf16 + (G + h) * kPartStride;
    const float m0 = s0[0], l0 = s0[1], m1 = s1[0], l1 = s1[1];
    const float mx = l1 > 0.f ? (l0 > 0.f ? fmaxf(m0, m1) : m1) : m0;
    const float f0 = l0 > 0.f ? exp2f(m0 - mx) : 0.f, f1 = l1 > 0.f ? exp2f(m1 - mx) : 0.f;
    hz[G * 4 + h * 4 + 0] = f0;
    hz[G * 4 + h * 4 + 1] = f1;
    part[(G + h) * kPartStride + 0] = mx;
    part[(G + h) * kPartStride + 1] = fmaf(l0, f0, l1 * f1);
    float lsum = 0.f, zsum = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      lsum += red_lz[w * 2 * G + h];
      zsum += red_lz[w * 2 * G + G + h];
    }
    const bool any = n_tiles > 0 && lsum > 0.f;
    part[h * kPartStride + 0] = any ? s_m[h] : -INFINITY;
    part[h * kPartStride + 1] = any ? lsum : 0.f;
    hz[h * 4 + 2] = any ? zsum : 0.f;
  }
  __syncthreads();
  for (int idx = tid; idx < G * kHeadDim; idx += T) {
    const int h = idx / kHeadDim, c = idx % kHeadDim;
    part[(G + h) * kPartStride + 4 + c] =
        fmaf(hz[G * 4 + h * 4 + 0], st_bf16[h * kPartStride + 4 + c],
             hz[G * 4 + h * 4 + 1] * st_bf16[(G + h) * kPartStride + 4 + c]);
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
        d = fmaf(hz[h * 4 + 2], rsum, d);
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
