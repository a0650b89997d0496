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
// per instruction, fp32 accumulators in tensor memory).  x is bf16, exact in
// fp16 within the fp16 range (larger magnitudes saturate at 65504); R is
// scaled by 16 and split into fp16 hi + lo parts (about 22 significant
// bits), so D = x.(16 R)_hi + x.(16 R)_lo and x~ = D / 16.
//
// CTA (tile stride, KV head, K|V) of 9 warps, one CTA per SM:
//   warps 4-7  load the next tile's 128 source rows (thread = token), convert
//              to fp16 into the canonical K-major operand layout in shared
//              memory, and look up each token's page;
//   warp 8     issues the 16 MMAs of a tile from one lane;
//   warps 0-3  read one token's 128 rotated values from tensor memory
//              (thread = token = TMEM lane), clip, min/max, fp16 scale and
//              zero point, codes, pack 32 bytes and store them in the page.
// Operand, accumulator and metadata buffers are fourfold, so loading, MMA
// and the epilogue of consecutive tiles overlap.  Every wait is bounded (1 s).
#include "kernels.h"
#include "ptx.cuh"

namespace oscar {
namespace {

constexpr int kTile = 128;                          // tokens per tile (MMA M)
constexpr int kEpiWarps = 4, kLoadWarps = 4;
constexpr int kMmaWarp = kEpiWarps + kLoadWarps;    // warp 8
constexpr int kThreads = (kMmaWarp + 1) * 32;
constexpr int kOpBytes = kTile * kHeadDim * 2;      // one fp16 128 x 128 operand
constexpr float kRScale = 16.f;
constexpr int kBufs = 4;                            // operand / accumulator / metadata buffers
constexpr size_t oBhi = 0, oBlo = kOpBytes, oA = 2 * size_t(kOpBytes);
constexpr size_t oMeta = oA + size_t(kBufs) * kOpBytes;
constexpr size_t oBars = oMeta + size_t(kBufs) * kTile * sizeof(int2);
constexpr size_t kSmem = oBars + (3 * kBufs + 2) * 8 + 16;
constexpr uint32_t kCols = 128 * kBufs;             // D[kBufs] x 128 columns
static_assert(kCols <= 512, "tensor memory columns");
static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
constexpr uint32_t kIdesc = idesc_f16_f32(128, 128);
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr uint32_t kFull = 0xffffffffu;

// byte offset of (row, k) in a 128 x 128 fp16 operand, canonical K-major
// layout without swizzle: 8 x 16-byte core matrices, 128 bytes between the
// two K halves of a 16-wide K step (LBO), 256 bytes between 8-row groups
// (SBO), 4096 bytes per K step
__device__ __forceinline__ int op_offset(int row, int k) {
  return (k >> 4) * 4096 + (row >> 3) * 256 + ((k >> 3) & 1) * 128 + (row & 7) * 16 + (k & 7) * 2;
}

__device__ __forceinline__ uint32_t f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float sat16(float x) { return fminf(fmaxf(x, -65504.f), 65504.f); }

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

__global__ void __launch_bounds__(kThreads, 1) bulk_demote_kernel(DemoteParams p) {
  pdl_wait();                 // the previous kernel's writes are visible
  pdl_launch_dependents();
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* bhi = smem + oBhi;
  uint8_t* blo = smem + oBlo;
  uint8_t* abuf = smem + oA;
  int2* meta = reinterpret_cast<int2*>(smem + oMeta);          // [kBufs][128] (page, slot)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + oBars);
  uint64_t* a_full = bars;                // [kBufs] loaders
  uint64_t* mma_done = bars + kBufs;      // [kBufs] commit
  uint64_t* d_free = bars + 2 * kBufs;    // [kBufs] epilogue
  uint64_t* fin = bars + 3 * kBufs;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * kBufs + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 3 * kBufs + 1) + 1;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int which = int(blockIdx.y & 1), head = int(blockIdx.y >> 1);
  const int n_tiles = (p.n + kTile - 1) / kTile;
  const int my_tiles = int(blockIdx.x) < n_tiles ? (n_tiles - int(blockIdx.x) + int(gridDim.x) - 1) / int(gridDim.x) : 0;

  if (tid == 0) {
    for (int i = 0; i < kBufs; ++i) {
      mbar_init(a_full + i, kLoadWarps * 32);
      mbar_init(mma_done + i, 1);
      mbar_init(d_free + i, kEpiWarps * 32);
    }
    mbar_init(fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, kCols);
  // B = (16 R)^T split into fp16 hi + lo: B[n][k] = 16 R[k][n]; thread (n,
  // half of k) writes 8 16-byte chunks of each part
  if (tid < 2 * kTile) {
    const int n = tid & (kTile - 1), k0 = (tid >> 7) * 64;
    const float* rg = (which ? p.r_v : p.r_k) + int64_t(head) * kHeadDim * kHeadDim;
#pragma unroll 2
    for (int kc = 0; kc < 8; ++kc) {
      const int k = k0 + 8 * kc;
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float r0 = __ldg(rg + (k + 2 * e) * kHeadDim + n) * kRScale;
        const float r1 = __ldg(rg + (k + 2 * e + 1) * kHeadDim + n) * kRScale;
        const __half h0 = __float2half_rn(r0), h1 = __float2half_rn(r1);
        hi[e] = uint32_t(__half_as_ushort(h0)) | (uint32_t(__half_as_ushort(h1)) << 16);
        lo[e] = f16x2(r0 - __half2float(h0), r1 - __half2float(h1));
      }
      *reinterpret_cast<uint4*>(bhi + op_offset(n, k)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(blo + op_offset(n, k)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
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
    // ================= epilogue: thread j = token j of the tile = TMEM lane j
    const int j = tid;
    const uint32_t lane_addr = tmem + (uint32_t(warp * 32) << 16);
    for (int k = 0; k < my_tiles; ++k) {
      const int buf = k % kBufs;
      const uint32_t par = (k / kBufs) & 1;
      if (!wt.wait(a_full + buf, par)) break;        // the loaders' page lookups
      if (!wt.wait(mma_done + buf, par)) break;
      tc_fence_after();
      const int2 m = meta[buf * kTile + j];
      // D = 16 x~ (the operand scale), read as four 32-column loads behind one wait
      float v[kHeadDim];
      {
        uint32_t r[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(lane_addr + uint32_t(buf * 128 + 32 * c), r[c]);
        tc_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) v[32 * c + i] = __uint_as_float(r[c][i]);
      }
      tc_fence_before();
      mbar_arrive(d_free + buf);
      if (m.x < 0) continue;
      // clipping moves only the extremes: min and max of the clipped values
      // are the clipped min and max, and a value beyond +-tau gets the code
      // of the clipped extreme (0 or 3) through the final clamp
      float mn = v[0], mx = v[0];
#pragma unroll
      for (int i = 1; i < kHeadDim; ++i) {
        mn = fminf(mn, v[i]);
        mx = fmaxf(mx, v[i]);
      }
      mn = fminf(fmaxf(mn * (1.f / kRScale), -tau), tau);
      mx = fminf(fmaxf(mx * (1.f / kRScale), -tau), tau);
      const __half s16 = __float2half_rn(__fdiv_rn(mx - mn, 3.0f));
      const __half z16 = __float2half_rn(mn);
      const float s = __half2float(s16), z = __half2float(z16);
      // code = clamp(rint((x - z) / s), 0, 3) with x = D / 16: (x - z) / s by
      // one FMA, clamped to [0, 3]; adding 1.5 * 2^23 rounds it to an
      // integer held in the float's low bits (0x4B400000 + code), which are
      // accumulated as bits * 4^i (mod 2^32) with the constant part of the
      // sum removed once per word
      const float inv = s > 0.f ? __frcp_rn(s) : 0.f;
      const float a16 = inv * (1.f / kRScale), nzi = -z * inv;
      const float kMagic = 12582912.f;
      constexpr uint32_t kBitsSum = 0x4B400000u * 0x55555555u;   // 0x4B400000 * sum_i 4^i (mod 2^32)
      uint32_t w[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        uint32_t word = 0u;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float t = fminf(fmaxf(fmaf(v[16 * q + i], a16, nzi), 0.f), 3.f);
          word += __float_as_uint(t + kMagic) << (2 * i);
        }
        w[q] = word - kBitsSum;
      }
      uint8_t* blk = p.pages + (int64_t(m.x) * p.n_kv + head) * kBlockBytes + which * kHalfBytes;
      *reinterpret_cast<uint4*>(blk + 32 * m.y) = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4*>(blk + 32 * m.y + 16) = make_uint4(w[4], w[5], w[6], w[7]);
      __half2 sz = __halves2half2(s16, z16);
      *reinterpret_cast<__half2*>(blk + 32 * kPage + 4 * m.y) = sz;
    }
  } else if (warp < kMmaWarp) {
    // ================= loaders: thread j = token j of the next tile
    const int j = tid - kEpiWarps * 32;
    for (int k = 0; k < my_tiles; ++k) {
      const int buf = k % kBufs;
      // operand, accumulator and metadata of buffer k % kBufs are free once
      // the epilogue of tile k - kBufs has read them
      if (k >= kBufs && !wt.wait(d_free + buf, ((k - kBufs) / kBufs) & 1)) break;
      const int item = (int(blockIdx.x) + k * int(gridDim.x)) * kTile + j;
      bool live = item < p.n;
      int64_t row = 0;
      int bq = 0, pos = 0;
      int page = -1;
      if (live) {
        row = p.src_index ? int64_t(p.src_index[item]) : int64_t(item);
        bq = p.dst_req[item];
        pos = p.dst_pos[item];
        if (row < 0 || row >= p.src_rows || bq < 0 || bq >= p.batch || pos < 0 || pos / kPage >= p.max_pages) {
          if (p.dev_status) atomicOr(p.dev_status, 0x2);
          live = false;
        }
      }
      if (live) {
        const int pid = p.page_table[int64_t(bq) * p.max_pages + pos / kPage];
        if (pid < 0 || pid >= p.n_pages) {
          if (p.dev_status) atomicOr(p.dev_status, 0x1);
          live = false;
        } else {
          page = pid;
        }
      }
      uint8_t* a = abuf + buf * kOpBytes;
      const uint16_t* src = (which ? p.v_src : p.k_src) + row * p.row_stride + int64_t(head) * kHeadDim;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint4 raw[8];
#pragma unroll
        for (int c = 0; c < 8; ++c)
          raw[c] = live ? __ldg(reinterpret_cast<const uint4*>(src + 64 * half + 8 * c)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t wv[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
          uint32_t h[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) h[e] = f16x2(sat16(bf16_lo(wv[e])), sat16(bf16_hi(wv[e])));
          *reinterpret_cast<uint4*>(a + op_offset(j, 64 * half + 8 * c)) = make_uint4(h[0], h[1], h[2], h[3]);
        }
      }
      meta[buf * kTile + j] = make_int2(live ? page : -1, pos % kPage);
      fence_proxy_async_smem();
      mbar_arrive(a_full + buf);
    }
  } else {
    // ================= MMA issue (one lane)
    if (lane == 0) {
      const uint32_t bh = smem_addr(bhi), bl = smem_addr(blo);
      for (int k = 0; k < my_tiles; ++k) {
        const int buf = k % kBufs;
        if (!wt.wait(a_full + buf, (k / kBufs) & 1)) break;
        tc_fence_after();
        const uint32_t aa = smem_addr(abuf + buf * kOpBytes);
        const uint32_t d = tmem + uint32_t(buf * 128);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_f16_ss(d, smem_desc_kmajor(aa + 4096u * kk, 128u, 256u), smem_desc_kmajor(bh + 4096u * kk, 128u, 256u),
                      kIdesc, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_f16_ss(d, smem_desc_kmajor(aa + 4096u * kk, 128u, 256u), smem_desc_kmajor(bl + 4096u * kk, 128u, 256u),
                      kIdesc, 1u);
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

cudaError_t launch_demote_bulk(const DemoteParams& p, cudaStream_t stream) {
  const int64_t n_tiles = (int64_t(p.n) + kTile - 1) / kTile;
  if (n_tiles == 0) return cudaSuccess;
  if (int64_t(p.n_kv) * 2 > 65535) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(bulk_demote_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmem));
  if (e != cudaSuccess) return e;
  // one CTA per SM shared out over the (KV head, K|V) pairs
  const int64_t per_pair = int64_t(sms) / (2 * p.n_kv);
  const int64_t gx = per_pair < n_tiles ? (per_pair > 0 ? per_pair : 1) : n_tiles;
  return launch_pdl(bulk_demote_kernel, dim3(unsigned(gx), unsigned(p.n_kv * 2)), dim3(kThreads), kSmem,
                    stream, p);
}

}  // namespace oscar
