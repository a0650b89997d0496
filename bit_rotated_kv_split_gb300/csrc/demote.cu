// Fused demotion kernel: rotate -> clip -> quantise -> pack -> place in page.
//
// myzaker.com OSCAR article, part "从离线校准到在线推理的 pipeline": the oldest
// recent-window token is rotated, clipped, quantised and packed (4 codes per
// byte, scale/zero point) and moved into INT2 history.  gist.science "OSCAR:
// Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache Quantization",
// Technical summary 2.2 A (fixed R = U.H.P, per-layer clip thresholds) and
// 2.2 B (paged cache).
//
// One CTA per (KV head, K|V, group of 4 items): the head's rotation R (64 KB)
// is staged into shared memory by one TMA bulk copy, then each warp demotes
// one item: lane l owns rotated channels 4l..4l+3 (one code byte),
// x~_j = sum_i x_i R[i][j] in fp32 with i ascending, read from shared memory.
#include "kernels.h"
#include "ptx.cuh"

namespace oscar {
namespace {

constexpr int kWarps = 4;
constexpr uint32_t kRotBytes = kHeadDim * kHeadDim * 4;
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr size_t kSmem = kRotBytes + 16;

__global__ void __launch_bounds__(kWarps * 32) demote_kernel(DemoteParams p) {
  pdl_wait();                 // the previous kernel's writes are visible
  pdl_launch_dependents();
  extern __shared__ __align__(128) uint8_t smem[];
  float* rs = reinterpret_cast<float*>(smem);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kRotBytes);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int which = int(blockIdx.y & 1);     // 0 = K, 1 = V
  const int head = int(blockIdx.y >> 1);
  const int item = int(blockIdx.x) * kWarps + warp;
  const float* rg = (which ? p.r_v : p.r_k) + int64_t(head) * kHeadDim * kHeadDim;
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, kRotBytes);
#pragma unroll
    for (int c = 0; c < 4; ++c)
      bulk_copy_g2s(smem + c * (kRotBytes / 4), rg + c * (kRotBytes / 16), kRotBytes / 4, bar);
  }
  __syncthreads();

  // indices first, then the source row and the destination page (two
  // levels of independent loads, overlapping the R transfer)
  bool live = item < p.n;
  int64_t row = 0;
  int bq = 0, pos = 0;
  if (live) {
    row = p.src_index ? int64_t(p.src_index[item]) : int64_t(item);
    bq = p.dst_req[item];
    pos = p.dst_pos[item];
    if (row < 0 || row >= p.src_rows || bq < 0 || bq >= p.batch || pos < 0 || pos / kPage >= p.max_pages) {
      if (lane == 0 && p.dev_status) atomicOr(p.dev_status, 0x2);
      live = false;
    }
  }
  uint16_t* src = (which ? p.v_src : p.k_src) + row * p.row_stride + int64_t(head) * kHeadDim;
  float xv[4] = {0.f, 0.f, 0.f, 0.f};
  int64_t page = -1;
  if (live) {
    const uint2 raw = *reinterpret_cast<const uint2*>(src + 4 * lane);
    page = p.page_table[int64_t(bq) * p.max_pages + pos / kPage];
    xv[0] = bf16_lo(raw.x);
    xv[1] = bf16_hi(raw.x);
    xv[2] = bf16_lo(raw.y);
    xv[3] = bf16_hi(raw.y);
  }
  // the source row may be overwritten by the new token only after every
  // lane has read it
  __syncwarp();
  const uint16_t* fresh = which ? p.new_v : p.new_k;
  if (live && fresh) {
    const uint2 nw = *reinterpret_cast<const uint2*>(
        fresh + (int64_t(item) * p.n_kv + head) * kHeadDim + 4 * lane);
    *reinterpret_cast<uint2*>(src + 4 * lane) = nw;
  }

  const bool ready = mbar_wait_bounded(bar, 0, kWaitLimitNs);
  if (!ready) {
    if (threadIdx.x == 0 && p.dev_status) atomicOr(p.dev_status, 0x4);
    return;
  }
  if (!live) return;
  float a[4] = {0.f, 0.f, 0.f, 0.f};
  const float4* r4 = reinterpret_cast<const float4*>(rs) + lane;
#pragma unroll 8
  for (int i = 0; i < kHeadDim; ++i) {
    const float xi = __shfl_sync(0xffffffffu, xv[i & 3], i >> 2);
    const float4 rr = r4[i * (kHeadDim / 4)];
    a[0] = fmaf(xi, rr.x, a[0]);
    a[1] = fmaf(xi, rr.y, a[1]);
    a[2] = fmaf(xi, rr.z, a[2]);
    a[3] = fmaf(xi, rr.w, a[3]);
  }

  const float tau = which ? p.tau_v : p.tau_k;
  float mn = INFINITY, mx = -INFINITY;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    a[c] = fminf(fmaxf(a[c], -tau), tau);
    mn = fminf(mn, a[c]);
    mx = fmaxf(mx, a[c]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  const __half s16 = __float2half_rn(__fdiv_rn(mx - mn, 3.0f));
  const __half z16 = __float2half_rn(mn);
  const float s = __half2float(s16);
  const float z = __half2float(z16);
  uint32_t byte = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float code = 0.f;
    if (s > 0.f) code = fminf(fmaxf(rintf(__fdiv_rn(a[c] - z, s)), 0.f), 3.f);
    byte |= uint32_t(code) << (2 * c);
  }

  if (page < 0 || page >= p.n_pages) {
    if (lane == 0 && p.dev_status) atomicOr(p.dev_status, 0x1);
    return;
  }
  uint8_t* blk = p.pages + (page * p.n_kv + head) * kBlockBytes + which * kHalfBytes;
  const int slot = pos % kPage;
  blk[32 * slot + lane] = uint8_t(byte);
  if (lane == 0) {
    __half2 sz = __halves2half2(s16, z16);
    *reinterpret_cast<__half2*>(blk + 32 * kPage + 4 * slot) = sz;
  }
}

}  // namespace

cudaError_t launch_demote(const DemoteParams& p, cudaStream_t stream) {
  const int64_t chunks = (int64_t(p.n) + kWarps - 1) / kWarps;
  if (chunks == 0) return cudaSuccess;
  if (chunks > 0x7fffffff || int64_t(p.n_kv) * 2 > 65535) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(demote_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmem));
  if (e != cudaSuccess) return e;
  return launch_pdl(demote_kernel, dim3(unsigned(chunks), unsigned(p.n_kv * 2)), dim3(kWarps * 32), kSmem,
                    stream, p);
}

}  // namespace oscar
