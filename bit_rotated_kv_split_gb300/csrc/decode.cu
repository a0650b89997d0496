// Decode attention over BF16 sink | INT2 history | BF16 recent window.
//
// myzaker.com OSCAR article, part "从离线校准到在线推理的 pipeline": the INT2
// kernel unpacks, dequantises with scale/zero point and accumulates in float;
// a BF16 kernel handles sink and recent; an online-softmax merge joins them.
// gist.science "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV
// Cache Quantization", Technical summary 2.2 B: the inverse rotation is fused
// into the attention kernel with no extra memory traffic.  Here it is applied
// as q~ = q . R_K once per query head (prep kernel) and one o . R_V^T per head
// after the history partials are merged, instead of rotating every token.
//
// Launch 1 (prep, one CTA per (request, KV head)): q~ = q . R_K in fp32, split
//   into fp16 hi + lo with a power-of-two scale and laid out as the B fragments
//   of the QK tensor-core MMA; zeroes the merge tickets.
// Launch 2 (split kernel, programmatic dependent launch): CTA (split, kv, b).
//   Splits < n_hist_splits scan a range of INT2 pages; the rest scan the BF16
//   sink/recent tokens.  Each of the 4 warps streams its own pages through a
//   6-stage shared-memory ring filled by 1-D TMA bulk copies (one 1152-byte
//   page block per stage, mbarrier completion, bounded waits) and keeps its
//   own online-softmax state; the CTA merges its warps and writes one partial
//   (m, l, o) per query head.  The last CTA of a (request, KV head) to finish
//   (atomic ticket, no waiting) merges all partials, applies . R_V^T to the
//   history part and writes the normalised output.
//
// INT2 arithmetic on the tensor cores (mma.sync m16n8k16, fp32 accumulate):
//   QK: A = codes of 16 tokens x 128 channels, B = q~ (hi | lo columns), so
//       q~ . k^ = s (q~ . c) + z sum(q~).
//   PV: A = codes^T (128 channels x 16 tokens), B = p s_V (hi | lo columns),
//       so o~ = sum p (s_V c + z_V) = (p s_V) . c + sum(p z_V).
//   A 2-bit code c at bit offset 2k of a 16-bit half is taken as the fp16
//   subnormal c * 4^k * 2^-24 by a single AND (no conversion); the 4^k and
//   2^-24 factors are folded into the B operand (QK) or the output (PV).
//   The contraction order of channels is free, so B is permuted to match.
#include <cfloat>

#include "kernels.h"
#include "ptx.cuh"

namespace oscar {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 6;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;          // lazy rescale threshold (p <= 2^8)
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr uint32_t kFull = 0xffffffffu;

template <int G>
struct Geo {
  static constexpr int NT = (2 * G + 7) / 8;          // column tiles holding hi | lo parts
  static constexpr int HS = G >= 8 ? G / 4 : 2;       // head slots per lane
  static constexpr int NTQ = (G + 7) / 8;             // BF16 QK column tiles
  static constexpr size_t kStageBytes = size_t(kWarps) * kStages * kBlockBytes;
  static constexpr size_t kBarBytes = size_t(kWarps) * kStages * 8;
  static constexpr size_t kStateBytes = size_t(kWarps) * G * kPartStride * 4;
  static constexpr size_t kSmem = kStageBytes + kBarBytes + kStateBytes + 16;
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

__device__ __forceinline__ void flag(int32_t* st, int bit) {
  if (st) atomicOr(st, bit);
}

// ------------------------------------------------------------------ prep kernel

template <int G>
__global__ void __launch_bounds__(kThreads) prep_kernel(DecodeParams p) {
  pdl_launch_dependents();
  constexpr int NT = Geo<G>::NT;
  __shared__ float qs[G][kHeadDim];
  __shared__ float qt[G][kHeadDim];
  __shared__ float red_max[G][kWarps], red_sum[G][kWarps];
  __shared__ float sigma[G];
  const int hkv = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int pair = b * p.n_kv + hkv;
  const int lane = tid & 31, warp = tid >> 5;

  for (int h = 0; h < G; ++h) {
    const uint16_t v = p.q[(int64_t(b) * p.n_kv * G + hkv * G + h) * kHeadDim + tid];
    qs[h][tid] = __uint_as_float(uint32_t(v) << 16);
  }
  if (tid == 0) p.counters[pair] = 0u;
  __syncthreads();

  // q~[h][j] = sum_i q[h][i] R_K[i][j]  (thread j, i ascending)
  const float* r = p.r_k + int64_t(hkv) * kHeadDim * kHeadDim + tid;
  float acc[G];
#pragma unroll
  for (int h = 0; h < G; ++h) acc[h] = 0.f;
  for (int i = 0; i < kHeadDim; ++i) {
    const float rij = __ldg(r + i * kHeadDim);
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = fmaf(qs[h][i], rij, acc[h]);
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    qt[h][tid] = acc[h];
    float mx = fabsf(acc[h]), sm = acc[h];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
      sm += __shfl_xor_sync(kFull, sm, o);
    }
    if (lane == 0) {
      red_max[h][warp] = mx;
      red_sum[h][warp] = sm;
    }
  }
  __syncthreads();
  if (tid < G) {
    float mx = 0.f, sm = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      mx = fmaxf(mx, red_max[tid][w]);
      sm += red_sum[tid][w];
    }
    // power-of-two scale putting max|q~| in [2^13, 2^14): keeps the fp16 hi
    // part normal and the lo part precise
    int e = 0;
    if (mx > 0.f) {
      frexpf(mx, &e);            // mx in [2^(e-1), 2^e)
      e = 14 - e;
      e = max(-100, min(100, e));
    }
    const float sg = ldexpf(1.f, e);
    sigma[tid] = sg;
    const float scale = kLog2e * rsqrtf(float(kHeadDim));
    p.qaux[(pair * G + tid) * 2 + 0] = ldexpf(1.f, 24 - e) * scale;  // 2^24/sigma * log2e/sqrt(d)
    p.qaux[(pair * G + tid) * 2 + 1] = sm * scale;
  }
  __syncthreads();

  // B fragments: [nt][j][lane][r]; column n = 8nt + gid is head n (hi part)
  // for n < G, head n-G (lo part) for n < 2G, zero otherwise.  r = 0 holds
  // channels (32tig + j, 32tig + j + 8), r = 1 (32tig + 16 + j, 32tig + 24 + j),
  // each scaled by sigma * 4^-pos(j).
  for (int idx = tid; idx < NT * 8 * 32; idx += kThreads) {
    const int ln = idx & 31, j = (idx >> 5) & 7, nt = idx >> 8;
    const int gid = ln >> 2, tig = ln & 3;
    const int col = 8 * nt + gid;
    uint32_t out[2] = {0u, 0u};
    if (col < 2 * G) {
      const int h = col < G ? col : col - G;
      const bool lo = col >= G;
      const float f = sigma[h] * ldexpf(1.f, -2 * code_pos(j));
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int c0 = 32 * tig + 16 * rr + j;
        float v0 = qt[h][c0] * f, v1 = qt[h][c0 + 8] * f;
        if (lo) {
          v0 = split_lo(v0);
          v1 = split_lo(v1);
        }
        out[rr] = pack_half2(v0, v1);
      }
    }
    reinterpret_cast<uint2*>(p.qfrag)[(int64_t(pair) * NT * 8 + nt * 8 + j) * 32 + ln] =
        make_uint2(out[0], out[1]);
  }
}

// ------------------------------------------------------------------ INT2 page

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

template <int G>
__device__ __forceinline__ void int2_page(const uint8_t* __restrict__ pg, int ntok, int gid,
                                          int tig, const uint32_t (&qb)[Geo<G>::NT][8][2],
                                          const float (&unscale)[Geo<G>::HS],
                                          const float (&qz)[Geo<G>::HS], float sigma_v,
                                          WarpState<G>& st) {
  constexpr int NT = Geo<G>::NT, HS = Geo<G>::HS;
  const uint2 kw0 = *reinterpret_cast<const uint2*>(pg + 32 * gid + 8 * tig);
  const uint2 kw1 = *reinterpret_cast<const uint2*>(pg + 32 * (gid + 8) + 8 * tig);
  const uint32_t ksz0 = *reinterpret_cast<const uint32_t*>(pg + 512 + 4 * gid);
  const uint32_t ksz1 = *reinterpret_cast<const uint32_t*>(pg + 512 + 4 * (gid + 8));
  const uint8_t* pv = pg + kHalfBytes;
  const uint32_t va = *reinterpret_cast<const uint32_t*>(pv + 64 * tig + 4 * gid);
  const uint32_t vb = *reinterpret_cast<const uint32_t*>(pv + 64 * tig + 32 + 4 * gid);
  const uint32_t vc = *reinterpret_cast<const uint32_t*>(pv + 64 * tig + 256 + 4 * gid);
  const uint32_t vd = *reinterpret_cast<const uint32_t*>(pv + 64 * tig + 288 + 4 * gid);
  const uint32_t vsz0 = *reinterpret_cast<const uint32_t*>(pv + 512 + 4 * gid);
  const uint32_t vsz1 = *reinterpret_cast<const uint32_t*>(pv + 512 + 4 * (gid + 8));

  // ---- scores: D[token][col] = 2^-24 sigma (q~ . c)
  float d[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
  {
    const uint32_t w00 = kw0.x, w01 = kw0.y, w10 = kw1.x, w11 = kw1.y;
    const uint32_t s00 = w00 >> 6, s01 = w01 >> 6, s10 = w10 >> 6, s11 = w11 >> 6;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t a0 = code_pair(w00, s00, j), a1 = code_pair(w10, s10, j);
      const uint32_t a2 = code_pair(w01, s01, j), a3 = code_pair(w11, s11, j);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_f16(d[nt], a0, a1, a2, a3, qb[nt][j][0], qb[nt][j][1]);
    }
  }
  float full[HS][2];
  if (G <= 4) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
      full[c & 1][c >> 1] = d[0][c] + __shfl_xor_sync(kFull, d[0][c], G / 2);
  } else {
#pragma unroll
    for (int nt = 0; nt < NT / 2; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) full[2 * nt + (c & 1)][c >> 1] = d[nt][c] + d[nt + NT / 2][c];
  }
  const float2 kz0 = half2_to_float2(ksz0), kz1 = half2_to_float2(ksz1);
  const bool ok0 = gid < ntok, ok1 = gid + 8 < ntok;
  float sc[HS][2];
#pragma unroll
  for (int hs = 0; hs < HS; ++hs) {
    sc[hs][0] = ok0 ? fmaf(kz0.x * full[hs][0], unscale[hs], kz0.y * qz[hs]) : -INFINITY;
    sc[hs][1] = ok1 ? fmaf(kz1.x * full[hs][1], unscale[hs], kz1.y * qz[hs]) : -INFINITY;
  }
  st.update_max(sc);

  // ---- probabilities
  const float2 vz0 = half2_to_float2(vsz0), vz1 = half2_to_float2(vsz1);
  float pp[HS][2];
#pragma unroll
  for (int hs = 0; hs < HS; ++hs) {
    const float p0 = ok0 ? exp2f(sc[hs][0] - st.m[hs]) : 0.f;
    const float p1 = ok1 ? exp2f(sc[hs][1] - st.m[hs]) : 0.f;
    st.l[hs] += p0 + p1;
    st.z[hs] += (ok0 ? p0 * vz0.y : 0.f) + (ok1 ? p1 * vz1.y : 0.f);
    pp[hs][0] = ok0 ? p0 * vz0.x * sigma_v : 0.f;
    pp[hs][1] = ok1 ? p1 * vz1.x * sigma_v : 0.f;
  }
  uint32_t pb[NT][2];
  st.template pv_operand<true>(pp, tig, pb);

  // ---- values: acc[ch][col] += codes^T . (p s_V)
  const uint32_t x0l = prmt(va, vb, 0x5410), x0h = prmt(va, vb, 0x7632);
  const uint32_t x8l = prmt(vc, vd, 0x5410), x8h = prmt(vc, vd, 0x7632);
  const uint32_t y0l = x0l >> 6, y0h = x0h >> 6, y8l = x8l >> 6, y8h = x8h >> 6;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const uint32_t a0 = code_pair(x0l, y0l, mt), a1 = code_pair(x0h, y0h, mt);
    const uint32_t a2 = code_pair(x8l, y8l, mt), a3 = code_pair(x8h, y8h, mt);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mma_f16(st.acc[nt][mt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
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
// 2^24 4^-pos(mt) / sigma_v plus the zero-point term; BF16: 16gid + 2mt (+1).
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

// ------------------------------------------------------------------ split kernel

template <int G>
__global__ void __launch_bounds__(kThreads) split_kernel(DecodeParams p) {
  constexpr int NT = Geo<G>::NT, HS = Geo<G>::HS, NTQ = Geo<G>::NTQ;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stage = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Geo<G>::kStageBytes);
  float* wstate = reinterpret_cast<float*>(smem + Geo<G>::kStageBytes + Geo<G>::kBarBytes);
  int* s_last = reinterpret_cast<int*>(smem + Geo<G>::kStageBytes + Geo<G>::kBarBytes +
                                       Geo<G>::kStateBytes);

  const int split = blockIdx.x, hkv = blockIdx.y, b = blockIdx.z;
  const int pair = b * p.n_kv + hkv;
  const int n_splits = p.n_hist_splits + p.n_bf16_splits;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gid = lane >> 2, tig = lane & 3;

  WarpState<G> st;
  st.init();
  float* ws = wstate + warp * G * kPartStride;

  if (split < p.n_hist_splits) {
    // ---------------- INT2 history pages [pbeg, pend)
    int hist = p.hist_len[b];
    if (hist < 0 || hist > p.max_pages * kPage) {
      if (tid == 0) flag(p.dev_status, 0x2);
      hist = max(0, min(hist, p.max_pages * kPage));
    }
    const int n_pg = (hist + kPage - 1) / kPage;
    if (n_pg > p.n_hist_splits * p.pages_per_split && split == 0 && tid == 0)
      flag(p.dev_status, 0x2);  // longer than the host bound max_hist: tail not read
    const int pbeg = split * p.pages_per_split;
    const int pend = min(pbeg + p.pages_per_split, n_pg);
    const int first = pbeg + warp;
    const int count = pend > first ? (pend - first + kWarps - 1) / kWarps : 0;
    uint8_t* ring = stage + size_t(warp) * kStages * kBlockBytes;
    uint64_t* bar = bars + warp * kStages;
    const int32_t* ptab = p.page_table + int64_t(b) * p.max_pages;
    const uint8_t* pool = p.pages + int64_t(hkv) * kBlockBytes;
    const int64_t page_stride = int64_t(p.n_kv) * kBlockBytes;

    if (lane == 0) {
      for (int s = 0; s < kStages; ++s) mbar_init(bar + s, 1);
      fence_mbar_init();
    }
    __syncwarp();
    auto issue = [&](int k) {  // lane 0 only
      const int pi = first + k * kWarps;
      const int pid = ptab[pi];
      const int s = k % kStages;
      if (pid < 0 || pid >= p.n_pages) {
        // no copy: complete the stage's phase without bytes so the ring stays in step
        flag(p.dev_status, 0x1);
        mbar_arrive(bar + s);
        return;
      }
      mbar_arrive_expect_tx(bar + s, kBlockBytes);
      bulk_copy_g2s(ring + s * kBlockBytes, pool + int64_t(pid) * page_stride, kBlockBytes, bar + s);
    };
    if (lane == 0)
      for (int k = 0; k < min(count, kStages); ++k) issue(k);

    pdl_wait();  // q~ fragments and tickets come from the prep kernel
    uint32_t qb[NT][8][2];
    {
      const uint2* src = reinterpret_cast<const uint2*>(p.qfrag) + int64_t(pair) * NT * 8 * 32;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint2 v = src[(nt * 8 + j) * 32 + lane];
          qb[nt][j][0] = v.x;
          qb[nt][j][1] = v.y;
        }
    }
    float unscale[HS], qz[HS];
#pragma unroll
    for (int hs = 0; hs < HS; ++hs) {
      const int h = slot_head<G>(tig, hs);
      unscale[hs] = p.qaux[(pair * G + h) * 2 + 0];
      qz[hs] = p.qaux[(pair * G + h) * 2 + 1];
    }

    bool timed_out = false;
    int k = 0;
    for (; k < count; ++k) {
      const int pi = first + k * kWarps;
      const int pid = ptab[pi];
      const bool valid = pid >= 0 && pid < p.n_pages;
      const int s = k % kStages;
      if (!mbar_wait_bounded(bar + s, (k / kStages) & 1, kWaitLimitNs)) {
        timed_out = true;
        break;
      }
      if (valid) {
        const int ntok = min(kPage, hist - pi * kPage);
        int2_page<G>(ring + s * kBlockBytes, ntok, gid, tig, qb, unscale, qz, p.sigma_v, st);
      }
      __syncwarp();
      if (lane == 0 && k + kStages < count) issue(k + kStages);
    }
    if (timed_out) {
      if (lane == 0) flag(p.dev_status, 0x4);
      // let copies still in flight land before the CTA (and its shared
      // memory) goes away; each wait is bounded
      for (int kk = k; kk < min(count, k + kStages); ++kk)
        mbar_wait_bounded(bar + kk % kStages, (kk / kStages) & 1, kWaitLimitNs);
    }
    store_warp_state<G, true>(st, ws, gid, tig, p.pv_unscale);
  } else {
    // ---------------- BF16 sink and recent tokens
    pdl_wait();
    const int bs = split - p.n_hist_splits;
    int sink_len = p.sink_len[b], rec_len = p.recent_len[b];
    const int rec_start = p.recent_start[b];
    if (sink_len < 0 || sink_len > p.sink_cap || rec_len < 0 || rec_len > p.recent_cap ||
        rec_start < 0 || rec_start >= max(p.recent_cap, 1)) {
      if (tid == 0) flag(p.dev_status, 0x2);
      sink_len = max(0, min(sink_len, p.sink_cap));
      rec_len = max(0, min(rec_len, p.recent_cap));
    }
    const int start = min(max(rec_start, 0), max(p.recent_cap - 1, 0));
    const int sink_pages = p.sink_cap / kPage;
    const int n_vp = sink_pages + p.recent_cap / kPage;
    const int vbeg = bs * p.vpages_per_split;
    const int vend = min(vbeg + p.vpages_per_split, n_vp);
    const int64_t hstride = int64_t(p.n_kv) * kHeadDim;

    uint32_t qf[NTQ][8][2];
    {
      // B operand: column n is head n % G (heads duplicated when G < 8);
      // r = 0 holds channels (32tig + 4j, +1), r = 1 (32tig + 4j + 2, +3)
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
    for (int vp = vbeg + warp; vp < vend; vp += kWarps) {
      const int u0 = vp * kPage;
      bool kok[2], vok[4];
      const uint16_t* krow[2] = {row_of(u0 + gid, false, kok[0]), row_of(u0 + gid + 8, false, kok[1])};
      const uint16_t* vrow[4] = {row_of(u0 + 2 * tig, true, vok[0]), row_of(u0 + 2 * tig + 1, true, vok[1]),
                                 row_of(u0 + 2 * tig + 8, true, vok[2]),
                                 row_of(u0 + 2 * tig + 9, true, vok[3])};
      bf16_page<G>(krow, vrow, kok, vok, gid, tig, qf, st);
    }
    store_warp_state<G, false>(st, ws, gid, tig, 1.f);
  }
  __syncthreads();

  // ---------------- CTA merge of the warps' states -> one partial per head
  float* part = p.partials + (int64_t(pair) * n_splits + split) * G * kPartStride;
  for (int h = 0; h < G; ++h) {
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
      if (wstate[(w * G + h) * kPartStride + 1] > 0.f) mx = fmaxf(mx, wstate[(w * G + h) * kPartStride]);
    float lsum = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float* s = wstate + (w * G + h) * kPartStride;
      if (s[1] > 0.f) {
        const float f = exp2f(s[0] - mx);
        lsum = fmaf(s[1], f, lsum);
        o = fmaf(s[4 + tid], f, o);
      }
    }
    part[h * kPartStride + 4 + tid] = o;
    if (tid == 0) {
      part[h * kPartStride + 0] = mx;
      part[h * kPartStride + 1] = lsum;
    }
  }

  // ---------------- ticket: the last CTA of this (request, KV head) merges
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned t = atomicAdd(p.counters + pair, 1u);
    *s_last = (t == unsigned(n_splits - 1)) ? 1 : 0;
  }
  __syncthreads();
  if (!*s_last) return;
  __threadfence();

  const float* pp = p.partials + int64_t(pair) * n_splits * G * kPartStride;
  float* oh = wstate;  // [G][128] merged history partial (rotated domain)
  float mh[G], lh[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float mx = -INFINITY;
    for (int s = 0; s < p.n_hist_splits; ++s) {
      const float* q = pp + (s * G + h) * kPartStride;
      if (__ldcg(q + 1) > 0.f) mx = fmaxf(mx, __ldcg(q));
    }
    float lsum = 0.f, o = 0.f;
    for (int s = 0; s < p.n_hist_splits; ++s) {
      const float* q = pp + (s * G + h) * kPartStride;
      const float l = __ldcg(q + 1);
      if (l > 0.f) {
        const float f = exp2f(__ldcg(q) - mx);
        lsum = fmaf(l, f, lsum);
        o = fmaf(__ldcg(q + 4 + tid), f, o);
      }
    }
    mh[h] = mx;
    lh[h] = lsum;
    oh[h * kHeadDim + tid] = o;
  }
  __syncthreads();
  // history output back in the original basis: o[c] = sum_j o~[j] R_V[c][j]
  float orot[G];
#pragma unroll
  for (int h = 0; h < G; ++h) orot[h] = 0.f;
  {
    const float4* rrow = reinterpret_cast<const float4*>(p.r_v + (int64_t(hkv) * kHeadDim + tid) * kHeadDim);
#pragma unroll 4
    for (int j4 = 0; j4 < kHeadDim / 4; ++j4) {
      const float4 r = __ldg(rrow + j4);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float* o = oh + h * kHeadDim + 4 * j4;
        orot[h] = fmaf(o[0], r.x, fmaf(o[1], r.y, fmaf(o[2], r.z, fmaf(o[3], r.w, orot[h]))));
      }
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float mx = lh[h] > 0.f ? mh[h] : -INFINITY;
    for (int s = p.n_hist_splits; s < n_splits; ++s) {
      const float* q = pp + (s * G + h) * kPartStride;
      if (__ldcg(q + 1) > 0.f) mx = fmaxf(mx, __ldcg(q));
    }
    float lsum = 0.f, o = 0.f;
    if (lh[h] > 0.f) {
      const float f = exp2f(mh[h] - mx);
      lsum = lh[h] * f;
      o = orot[h] * f;
    }
    for (int s = p.n_hist_splits; s < n_splits; ++s) {
      const float* q = pp + (s * G + h) * kPartStride;
      const float l = __ldcg(q + 1);
      if (l > 0.f) {
        const float f = exp2f(__ldcg(q) - mx);
        lsum = fmaf(l, f, lsum);
        o = fmaf(__ldcg(q + 4 + tid), f, o);
      }
    }
    p.out[(int64_t(b) * p.n_kv * G + hkv * G + h) * kHeadDim + tid] = lsum > 0.f ? o / lsum : 0.f;
  }
}

template <int G>
int occupancy() {
  int occ = 0;
  cudaFuncSetAttribute(split_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       int(Geo<G>::kSmem));
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, split_kernel<G>, kThreads,
                                                    Geo<G>::kSmem) != cudaSuccess)
    return 0;
  return occ;
}

template <int G>
cudaError_t launch_g(const DecodeParams& p, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(split_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(Geo<G>::kSmem));
  if (e != cudaSuccess) return e;
  prep_kernel<G><<<dim3(p.n_kv, p.batch), kThreads, 0, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_hist_splits + p.n_bf16_splits, p.n_kv, p.batch);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Geo<G>::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, split_kernel<G>, p);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

int plan_decode(int batch, int n_kv, int group, int sink_cap, int recent_cap, int max_hist,
                DecodePlan* plan, cudaError_t* err) {
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
  const int n_vp = sink_cap / kPage + recent_cap / kPage;
  int n_bf16 = (n_vp == 0) ? 0 : (pairs * 2 <= slots ? 2 : 1);
  n_bf16 = min(n_bf16, n_vp);
  int n_hist = 1, pps = max(pages_max, 1);
  const int64_t avail = slots - pairs * n_bf16;
  const int kOneWaveCap = 256;
  if (avail >= pairs && pages_max > 0) {
    const int per_pair = int(avail / pairs < 4096 ? avail / pairs : 4096);
    const int p1 = (pages_max + per_pair - 1) / per_pair;
    if (p1 <= kOneWaveCap) pps = max(p1, 1);
    else pps = 128;
  } else {
    pps = 128;
  }
  n_hist = max(1, (pages_max + pps - 1) / pps);
  plan->n_hist_splits = n_hist;
  plan->n_bf16_splits = n_bf16;
  plan->pages_per_split = pps;
  plan->vpages_per_split = n_bf16 ? (n_vp + n_bf16 - 1) / n_bf16 : 0;
  const int nt = (2 * group + 7) / 8;
  const int n_splits = n_hist + n_bf16;
  size_t off = 0;
  plan->off_counters = off;
  off = align256(off + size_t(pairs) * 4);
  plan->off_qfrag = off;
  off = align256(off + size_t(pairs) * nt * 8 * 32 * 8);
  plan->off_qaux = off;
  off = align256(off + size_t(pairs) * group * 2 * 4);
  plan->off_partials = off;
  off = align256(off + size_t(pairs) * n_splits * group * kPartStride * 4);
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
