// Bulk demotion on the tensor cores: rotate -> clip -> quantise -> pack ->
// place, for many tokens at once (a prefill moved into INT2 history).
//
// gist.science "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV
// Cache Quantization", Technical summary 2.2 A (fixed R = U.H.P, per-layer
// clip thresholds) and 2.2 B (paged cache); myzaker.com OSCAR article, part
// "从离线校准到在线推理的 pipeline" (rotate, clip, quantise with scale/zero
// point, pack 4 codes per byte).
//
// The rotation of 128 tokens is one 128 x 128 x 128 contraction,
// D[token][j] = sum_i x[token][i] R[i][j], on tcgen05 (M = N = 128, K = 16
// per instruction, fp32 accumulators in tensor memory).  x is bf16 and is
// the A operand as it is (exact at any magnitude); R is scaled by 16 and
// split into three bf16 parts, 16 R = r1 + r2 + r3 with r1 = bf16(16 R),
// r2 = bf16(16 R - r1), r3 = bf16(16 R - r1 - r2) (about 24 significant
// bits), so D = x.r3 + x.r2 + x.r1 (products exact in fp32, the smallest
// parts first) and x~ = D / 16.
//
// CTA (tile stride, KV head, K|V) of 14 warps, one CTA per SM:
//   warps 8-11 look up each token's page; with gathered rows each thread
//              also loads its token's row into the A operand (with
//              contiguous rows 16 2-D TMA copies, 8 columns x 128 rows each,
//              one K column of 8 x 16-byte core matrices, put it there);
//   warp 12    issues the 24 MMAs of a tile from one lane;
//   warp 13    starts the tile copies (contiguous rows) as buffers free up;
//   warps 0-7  read half a token's 128 rotated values from tensor memory
//              (warps w and w + 4 share the lane quadrant w % 4; thread =
//              token = TMEM lane), meet on its min/max through shared memory,
//              form the fp16 scale and zero point, and pack and store 16
//              bytes of codes each.
// Operand, accumulator and metadata buffers are threefold, so loading, MMA
// and the epilogue of consecutive tiles overlap.  Every wait is bounded (1 s).
#include <cudaTypedefs.h>

#include "kernels.h"
#include "ptx.cuh"

namespace oscar {
namespace {

constexpr int kTile = 128;                          // tokens per tile (MMA M)
constexpr int kEpiWarps = 8, kLoadWarps = 4;     // epilogue: two warps per TMEM lane quadrant
constexpr int kMmaWarp = kEpiWarps + kLoadWarps;    // warp 12
constexpr int kTmaWarp = kMmaWarp + 1;               // warp 13: source tile copies
constexpr int kThreads = (kTmaWarp + 1) * 32;
constexpr int kOpBytes = kTile * kHeadDim * 2;      // one bf16 128 x 128 operand
constexpr float kRScale = 16.f;
constexpr int kBParts = 3;                          // bf16 parts of 16 R
constexpr int kBufs = 3;                            // operand / accumulator / metadata buffers
constexpr size_t oB = 0, oA = size_t(kBParts) * kOpBytes;
constexpr size_t oMeta = oA + size_t(kBufs) * kOpBytes;
constexpr size_t oXchg = oMeta + size_t(kBufs) * kTile * sizeof(int2);   // [2][2][128][NG] (min, max)
constexpr size_t oBars = oXchg + 2 * 2 * kTile * 4 * sizeof(float2);   // up to 4 groups
constexpr size_t kSmem = oBars + (4 * kBufs + 10) * 8 + 16;
constexpr uint32_t kCols = 512;                     // allocation (a power of two) for D[kBufs] x 128
static_assert(128 * kBufs <= kCols, "tensor memory columns");
static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
constexpr uint32_t kIdesc = idesc_bf16_f32(128, 128);
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// byte offset of (row, k) in a 128 x 128 fp16 operand, canonical K-major
// layout without swizzle: 8 x 16-byte core matrices, 128 bytes between the
// two K halves of a 16-wide K step (LBO), 256 bytes between 8-row groups
// (SBO), 4096 bytes per K step (the B operand)
__device__ __forceinline__ int op_offset(int row, int k) {
  return (k >> 4) * 4096 + (row >> 3) * 256 + ((k >> 3) & 1) * 128 + (row & 7) * 16 + (k & 7) * 2;
}

// the A operand: one 2 KB column of core matrices per 8 K values (the box
// of one TMA copy), rows 16 bytes apart: LBO 2048, SBO 128, 4096 bytes per
// K step
__device__ __forceinline__ int a_offset(int row, int k) { return (k >> 3) * 2048 + row * 16 + (k & 7) * 2; }

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
        if (dev_status) atomicOr(dev_status, 0x4);
        return false;
      }
    }
  }
};

// Epilogue of one token-half: v[i] = 16 x~ at code position 64 hh + i, whose
// quantisation group is ((64 hh + i) & 7) / (8 / NG) in the page format (K
// and V alike).  The two halves of a token meet on each group's (min, max)
// through shared memory; then the group's fp16 scale and zero point and the
// codes.  kLevels (codebook): the code is the number of the thresholds thr
// strictly below u = (x - zero) / scale, u formed with the reciprocal of the
// scale.  Returns false when the exchange wait expired.
template <int NG, bool kLevels>
__device__ __forceinline__ bool epi_finish(const DemoteParams& p, float (&v)[kHeadDim / 2], float2* xchg,
                                           uint64_t* xfull, Waiter& wt, int k, int hh, int j, int2 m, float tau,
                                           int which, int head, const float* thr) {
  constexpr int kSpan = 8 / NG;   // consecutive positions (mod 8) per group
  const int slot = m.y;
  // clipping moves only the extremes: min and max of the clipped values
  // are the clipped min and max, and a value beyond +-tau gets the code
  // of the clipped extreme (0 or 3) through the final clamp
  float mn[NG], mx[NG];
#pragma unroll
  for (int q = 0; q < NG; ++q) {
    mn[q] = v[q * kSpan];
    mx[q] = v[q * kSpan];
  }
#pragma unroll
  for (int i = 0; i < kHeadDim / 2; ++i) {
    const int q = (i & 7) / kSpan;
    mn[q] = fminf(mn[q], v[i]);
    mx[q] = fmaxf(mx[q], v[i]);
  }
  float2* xs = xchg + (k & 1) * 2 * kTile * NG;
#pragma unroll
  for (int q = 0; q < NG; ++q) xs[(hh * kTile + j) * NG + q] = make_float2(mn[q], mx[q]);
  mbar_arrive(xfull + (k & 1));
  if (!wt.wait(xfull + (k & 1), (k >> 1) & 1)) return false;   // (the quadrant's two warps)
#pragma unroll
  for (int q = 0; q < NG; ++q) {
    const float2 other = xs[((1 - hh) * kTile + j) * NG + q];
    mn[q] = fminf(mn[q], other.x);
    mx[q] = fmaxf(mx[q], other.y);
  }
  // code = clamp(rint((x - z) / s), 0, 3) with x = D / 16: one saturating
  // FMA gives (x - z) / (3 s) clamped to [0, 1]; a second FMA scales by 3
  // and adds 1.5 * 2^23, which rounds to an integer held in the float's
  // low bits (0x4B400000 + code); the bits are accumulated as bits * 4^i
  // (mod 2^32) and the constant part of the sum removed once per word
  __half s16[NG], z16[NG];
  float a48[NG], nzi3[NG], a16[NG], nzi[NG];
#pragma unroll
  for (int q = 0; q < NG; ++q) {
    const float lo = fminf(fmaxf(mn[q] * (1.f / kRScale), -tau), tau);
    const float hi = fminf(fmaxf(mx[q] * (1.f / kRScale), -tau), tau);
    s16[q] = __float2half_rn(__fdiv_rn(hi - lo, 3.0f));
    z16[q] = __float2half_rn(lo);
    const float s = __half2float(s16[q]), z = __half2float(z16[q]);
    const float inv = s > 0.f ? __frcp_rn(s) : 0.f;
    a48[q] = inv * (1.f / (3.f * kRScale));
    nzi3[q] = -z * inv * (1.f / 3.f);
    a16[q] = inv * (1.f / kRScale);
    nzi[q] = -z * inv;
  }
  const float kMagic = 12582912.f;
  constexpr uint32_t kBitsSum = 0x4B400000u * 0x55555555u;   // 0x4B400000 * sum_i 4^i (mod 2^32)
  uint32_t w[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    uint32_t word = 0u;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int q = (i & 7) / kSpan;
      if constexpr (kLevels) {
        // (scale 0: a16 = nzi = 0, so u = 0 and the code is 0)
        const float un = fmaf(v[16 * u + i], a16[q], nzi[q]);
        word |= (uint32_t(un > thr[0]) + uint32_t(un > thr[1]) + uint32_t(un > thr[2])) << (2 * i);
      } else {
        const float t = __saturatef(fmaf(v[16 * u + i], a48[q], nzi3[q]));
        word += __float_as_uint(fmaf(t, 3.f, kMagic)) << (2 * i);
      }
    }
    w[u] = kLevels ? word : word - kBitsSum;
  }
  // V rows interleave the two tokens of a slot pair by 16-bit halves.  When
  // the neighbouring lane (token j ^ 1 of the tile, same half hh) holds the
  // other token of this token's slot pair in the same page - consecutive
  // positions from an even one, as in a prefill - the two lanes trade half
  // their codes and each stores 16 bytes of whole words; otherwise each
  // lane stores its eight halves 4 bytes apart.  (Every lane takes part in
  // the exchange, stored or not; lanes run in step here.)
  const unsigned am = __activemask();
  const int lane = int(threadIdx.x & 31);
  const bool odd = lane & 1;
  const int ppage = __shfl_xor_sync(am, m.x, 1), pslot = __shfl_xor_sync(am, slot, 1);
  const bool paired = which == 1 && ((am >> (lane ^ 1)) & 1u) && m.x >= 0 && ppage == m.x &&
                      (slot & 1) == int(odd) && (pslot ^ 1) == slot;
  const uint32_t r0 = __shfl_xor_sync(am, odd ? w[0] : w[2], 1);
  const uint32_t r1 = __shfl_xor_sync(am, odd ? w[1] : w[3], 1);
  if (m.x < 0) return true;
  uint8_t* blk = p.pages + (int64_t(m.x) * p.n_kv + head) * block_bytes(p.ng_k, p.ng_v);
  if (which == 0) {
    *reinterpret_cast<uint4*>(blk + 32 * slot + 16 * hh) = make_uint4(w[0], w[1], w[2], w[3]);
  } else if (paired) {
    // word i of the pair's row = (even token's half i | odd token's half i);
    // the even lane stores words 8 hh .. 8 hh + 3, the odd lane the next four
    const uint4 v = odd ? make_uint4(prmt(r0, w[2], 0x5410), prmt(r0, w[2], 0x7632), prmt(r1, w[3], 0x5410),
                                     prmt(r1, w[3], 0x7632))
                        : make_uint4(prmt(w[0], r0, 0x5410), prmt(w[0], r0, 0x7632), prmt(w[1], r1, 0x5410),
                                     prmt(w[1], r1, 0x7632));
    *reinterpret_cast<uint4*>(blk + v_code_byte(slot & ~1, 16 * hh) + (odd ? 16 : 0)) = v;
  } else {
    // the eight halves 8 hh .. 8 hh + 7 of this token go 4 bytes apart
    uint16_t* dst = reinterpret_cast<uint16_t*>(blk + v_code_byte(slot, 16 * hh));
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      dst[4 * u] = uint16_t(w[u] & 0xFFFFu);
      dst[4 * u + 2] = uint16_t(w[u] >> 16);
    }
  }
  if (hh == 0) {
    uint32_t sz[NG];
#pragma unroll
    for (int q = 0; q < NG; ++q)
      sz[q] = uint32_t(__half_as_ushort(s16[q])) | (uint32_t(__half_as_ushort(z16[q])) << 16);
    // (4-byte stores: with K and V pairs side by side a token's pairs are
    // only 4-byte aligned in general)
    uint32_t* dst = reinterpret_cast<uint32_t*>(blk + pair_byte(p.ng_k, p.ng_v, slot, which, 0));
#pragma unroll
    for (int q = 0; q < NG; ++q) dst[q] = sz[q];
  }
  return true;
}

__global__ void __launch_bounds__(kThreads, 1) bulk_demote_kernel(const __grid_constant__ DemoteParams p) {
  pdl_wait();                 // the previous kernel's writes are visible
  pdl_launch_dependents();
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* bparts = smem + oB;   // [kBParts] bf16 parts of (16 R)^T
  uint8_t* abuf = smem + oA;
  int2* meta = reinterpret_cast<int2*>(smem + oMeta);          // [kBufs][128] (page, slot)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + oBars);
  uint64_t* a_full = bars;                // [kBufs] loaders
  uint64_t* mma_done = bars + kBufs;      // [kBufs] commit
  uint64_t* d_free = bars + 2 * kBufs;    // [kBufs] epilogue
  uint64_t* tma_full = bars + 3 * kBufs; // [kBufs] source tile copies
  uint64_t* xfull = bars + 4 * kBufs;    // [4 quadrants][2] epilogue halves' (min, max) exchange
  uint64_t* fin = bars + 4 * kBufs + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 4 * kBufs + 9);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 4 * kBufs + 9) + 1;
  float2* xchg = reinterpret_cast<float2*>(smem + oXchg);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int which = int(blockIdx.y & 1), head = int(blockIdx.y >> 1);
  const int n_tiles = (p.n + kTile - 1) / kTile;
  const int my_tiles = int(blockIdx.x) < n_tiles ? (n_tiles - int(blockIdx.x) + int(gridDim.x) - 1) / int(gridDim.x) : 0;

  if (tid == 0) {
    for (int i = 0; i < kBufs; ++i) {
      mbar_init(a_full + i, kLoadWarps * 32);
      mbar_init(mma_done + i, 1);
      mbar_init(d_free + i, kEpiWarps * 32);
      mbar_init(tma_full + i, 1);
    }
    for (int i = 0; i < 8; ++i) mbar_init(xfull + i, 2 * 32);   // warps w and w + 4
    mbar_init(fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, kCols);
  // B = (16 R)^T split into three bf16 parts: B[n][k] = 16 R[k][n] = r1 +
  // r2 + r3, each part the bf16 rounding of what the previous ones leave
  // (exact differences in fp32); thread (n, half of k) writes 8 16-byte
  // chunks of each part (column n of the product is code position n of the
  // page format, so B takes column storage_channel(n) of R)
  if (tid < 2 * kTile) {
    const int n = tid & (kTile - 1), k0 = (tid >> 7) * 64;
    const int ng = which ? p.ng_v : p.ng_k;
    const int cn = which ? storage_channel_v(ng, n) : storage_channel_k(ng, n);
    const float* rg = (which ? p.r_v : p.r_k) + int64_t(head) * kHeadDim * kHeadDim + cn;
#pragma unroll 2
    for (int kc = 0; kc < 8; ++kc) {
      const int k = k0 + 8 * kc;
      uint32_t part[kBParts][4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float r0 = __ldg(rg + (k + 2 * e) * kHeadDim) * kRScale;
        float r1 = __ldg(rg + (k + 2 * e + 1) * kHeadDim) * kRScale;
#pragma unroll
        for (int t = 0; t < kBParts; ++t) {
          part[t][e] = pack_bf162(r0, r1);
          r0 -= bf16_lo(part[t][e]);
          r1 -= bf16_hi(part[t][e]);
        }
      }
#pragma unroll
      for (int t = 0; t < kBParts; ++t)
        *reinterpret_cast<uint4*>(bparts + t * kOpBytes + op_offset(n, k)) =
            make_uint4(part[t][0], part[t][1], part[t][2], part[t][3]);
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  Waiter wt{abort_flag, p.dev_status};
  const float tau = which ? p.tau_v : p.tau_k;

  if (warp < kEpiWarps) {
    // ================= epilogue: thread (token j = TMEM lane j, half hh):
    // warps w and w + 4 read the lane quadrant w % 4, columns 64 hh .. 64 hh
    // + 63 each, and meet on the token's min and max through shared memory
    const int quad = warp & 3, hh = warp >> 2;
    const int j = 32 * quad + lane;
    const uint32_t lane_addr = tmem + (uint32_t(32 * quad) << 16);
    for (int k = 0; k < my_tiles; ++k) {
      const int buf = k % kBufs;
      const uint32_t par = (k / kBufs) & 1;
      if (!wt.wait(a_full + buf, par)) break;        // the loaders' page lookups
      if (!wt.wait(mma_done + buf, par)) break;
      tc_fence_after();
      const int2 m = meta[buf * kTile + j];
      // D = 16 x~ (the operand scale), two 32-column loads behind one wait
      float v[kHeadDim / 2];
      {
        uint32_t r[2][32];
#pragma unroll
        for (int c = 0; c < 2; ++c) tmem_ld32(lane_addr + uint32_t(buf * 128 + 64 * hh + 32 * c), r[c]);
        tc_wait_ld();
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) v[32 * c + i] = __uint_as_float(r[c][i]);
      }
      tc_fence_before();
      mbar_arrive(d_free + buf);
      const int ngw = which ? p.ng_v : p.ng_k;
      const float* thr = which ? p.thr_v : p.thr_k;
      uint64_t* xq = xfull + 2 * quad;   // this quadrant's exchange barriers
      const bool ok =
          p.codebook ? epi_finish<1, true>(p, v, xchg, xq, wt, k, hh, j, m, tau, which, head, thr)
          : ngw == 4 ? epi_finish<4, false>(p, v, xchg, xq, wt, k, hh, j, m, tau, which, head, thr)
          : ngw == 2 ? epi_finish<2, false>(p, v, xchg, xq, wt, k, hh, j, m, tau, which, head, thr)
                     : epi_finish<1, false>(p, v, xchg, xq, wt, k, hh, j, m, tau, which, head, thr);
      if (!ok) break;
    }
  } else if (warp < kMmaWarp) {
    // ================= loaders: thread j = token j of the tile
    const int j = tid - kEpiWarps * 32;
    // the token's indices (source row, request, position) are requested two
    // tiles ahead and its page id one tile ahead, so neither dependent load
    // waits in the tile loop
    struct Idx {
      bool live;
      int64_t row;
      int bq, pos;
    };
    auto load_idx = [&](int kt) {
      const int item = (int(blockIdx.x) + kt * int(gridDim.x)) * kTile + j;
      Idx r{item < p.n, 0, 0, 0};
      if (r.live) {
        r.row = p.src_index ? int64_t(p.src_index[item]) : int64_t(item);
        r.bq = p.dst_req[item];
        r.pos = p.dst_pos[item];
      }
      return r;
    };
    auto check_and_look_up = [&](Idx& r) {
      if (r.live && (r.row < 0 || r.row >= p.src_rows || r.bq < 0 || r.bq >= p.batch || r.pos < 0 ||
                     r.pos / kPage >= p.max_pages)) {
        if (p.dev_status) atomicOr(p.dev_status, 0x2);
        r.live = false;
      }
      return r.live ? p.page_table[int64_t(r.bq) * p.max_pages + r.pos / kPage] : -1;
    };
    Idx nxt = my_tiles > 0 ? load_idx(0) : Idx{false, 0, 0, 0};
    Idx nxt2 = my_tiles > 1 ? load_idx(1) : Idx{false, 0, 0, 0};
    int nxt_pid = check_and_look_up(nxt);
    for (int k = 0; k < my_tiles; ++k) {
      const int buf = k % kBufs;
      // (TMA path: the copy warp waited for the buffer before its copies;
      // here operand, accumulator and metadata of buffer k % kBufs are free
      // once the epilogue of tile k - kBufs has read them)
      if (!p.use_tma && k >= kBufs && !wt.wait(d_free + buf, ((k - kBufs) / kBufs) & 1)) break;
      // this tile's token, then the pipeline moves on by one tile
      bool live = nxt.live;
      const int64_t row = nxt.row;
      const int pos = nxt.pos;
      const int pid = nxt_pid;
      if (k + 1 < my_tiles) {
        nxt = nxt2;
        nxt_pid = check_and_look_up(nxt);
      }
      if (k + 2 < my_tiles) nxt2 = load_idx(k + 2);
      int page = -1;
      if (live) {
        if (pid < 0 || pid >= p.n_pages) {
          if (p.dev_status) atomicOr(p.dev_status, 0x1);
          live = false;
        } else {
          page = pid;
        }
      }
      uint8_t* a = abuf + buf * kOpBytes;
      if (p.use_tma) {
        // the tile copies put the bf16 rows in place: the operand is ready
        // once they have landed
        if (!wt.wait(tma_full + buf, (k / kBufs) & 1)) break;
      } else {
        const uint16_t* src = (which ? p.v_src : p.k_src) + row * p.row_stride + int64_t(head) * kHeadDim;
        uint4 raw[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          raw[c] = live ? __ldg(reinterpret_cast<const uint4*>(src + 8 * c)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int c = 0; c < 16; ++c) *reinterpret_cast<uint4*>(a + a_offset(j, 8 * c)) = raw[c];
      }
      // (page, slot): the epilogue's store target
      meta[buf * kTile + j] = make_int2(live ? page : -1, pos % kPage);
      fence_proxy_async_smem();
      mbar_arrive(a_full + buf);
    }
  } else if (warp == kTmaWarp) {
    // ================= source tile copies (TMA path): the 16 copies of
    // tile k (one per 8 columns, lane c copies columns 8c .. 8c + 7) go out
    // as soon as buffer k % kBufs is free
    if (p.use_tma) {
      for (int k = 0; k < my_tiles; ++k) {
        const int b = k % kBufs;
        if (k >= kBufs && !wt.wait(d_free + b, ((k - kBufs) / kBufs) & 1)) break;
        if (lane == 0) mbar_arrive_expect_tx(tma_full + b, uint32_t(kOpBytes));
        __syncwarp();
        if (lane < kHeadDim / 8) {
          const int row0 = (int(blockIdx.x) + k * int(gridDim.x)) * kTile;
          tma_load_2d(abuf + b * kOpBytes + lane * 2048, &p.tm_src[which], head * kHeadDim + 8 * lane, row0,
                      tma_full + b);
        }
      }
    }
  } else {
    // ================= MMA issue (one lane)
    if (lane == 0) {
      const uint32_t bb = smem_addr(bparts);
      for (int k = 0; k < my_tiles; ++k) {
        const int buf = k % kBufs;
        if (!wt.wait(a_full + buf, (k / kBufs) & 1)) break;
        tc_fence_after();
        const uint32_t aa = smem_addr(abuf + buf * kOpBytes);
        const uint32_t d = tmem + uint32_t(buf * 128);
        // the smallest part first: x.r3, then x.r2, then x.r1
#pragma unroll
        for (int t = kBParts - 1; t >= 0; --t)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_f16_ss(d, smem_desc_kmajor(aa + 4096u * kk, 2048u, 128u),
                        smem_desc_kmajor(bb + uint32_t(t * kOpBytes) + 4096u * kk, 128u, 256u), kIdesc,
                        (t < kBParts - 1 || kk > 0) ? 1u : 0u);
        umma_commit(mma_done + buf);
      }
      // every MMA issued has completed before tensor memory is released
      umma_commit(fin);
      mbar_wait_bounded(fin, 0, kWaitLimitNs);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

}  // namespace

// 2-D bf16 tensor maps over k_src / v_src (n_kv * 128 columns x src_rows
// rows, row_stride elements apart) for the tile copies; false (gathered
// rows instead) when the rows are indexed, the row pitch is not a multiple
// of 16 bytes or the driver refuses
bool encode_src_maps(DemoteParams* p) {
  p->use_tma = 0;
  if (p->src_index || (p->row_stride * 2) % 16 != 0 || p->src_rows < 1 || p->src_rows > (int64_t(1) << 31)) return false;
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
  const cuuint64_t dims[2] = {cuuint64_t(p->n_kv) * kHeadDim, cuuint64_t(p->src_rows)};
  const cuuint64_t strides[1] = {cuuint64_t(p->row_stride) * 2};
  const cuuint32_t box[2] = {8, cuuint32_t(kTile)};
  const cuuint32_t estr[2] = {1, 1};
  const uint16_t* srcs[2] = {p->k_src, p->v_src};
  for (int w = 0; w < 2; ++w)
    if (encode(&p->tm_src[w], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(srcs[w]), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  p->use_tma = 1;
  return true;
}

cudaError_t launch_demote_bulk(const DemoteParams& p_in, cudaStream_t stream) {
  DemoteParams p = p_in;
  encode_src_maps(&p);
  const int64_t n_tiles = (int64_t(p.n) + kTile - 1) / kTile;
  if (n_tiles == 0) return cudaSuccess;
  if (int64_t(p.n_kv) * 2 > 65535) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = set_smem_limit<bulk_demote_kernel>(int(kSmem));
  if (e != cudaSuccess) return e;
  // one CTA per SM shared out over the (KV head, K|V) pairs
  const int64_t per_pair = int64_t(sms) / (2 * p.n_kv);
  const int64_t gx = per_pair < n_tiles ? (per_pair > 0 ? per_pair : 1) : n_tiles;
  return launch_pdl(bulk_demote_kernel, dim3(unsigned(gx), unsigned(p.n_kv * 2)), dim3(kThreads), kSmem,
                    stream, p);
}

}  // namespace oscar
