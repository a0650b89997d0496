// Fused demotion kernel: rotate -> clip -> quantise -> pack -> place in page.
//
// myzaker.com OSCAR article, part "从离线校准到在线推理的 pipeline": the oldest
// recent-window token is rotated, clipped, quantised and packed (4 codes per
// byte, scale/zero point) and moved into INT2 history.  gist.science "OSCAR:
// Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache Quantization",
// Technical summary 2.2 A (fixed R = U.H.P, per-layer clip thresholds) and
// 2.2 B (paged cache).
//
// One warp handles one (item, KV head, K|V) vector of 128 channels: lane l
// owns rotated channels 4l..4l+3, i.e. exactly code byte l of the token.
// x~_j = sum_i x_i R[i][j] in fp32, i ascending; R rows are read as 512-byte
// coalesced lines (R of a head, 64 KB, stays in L2 across items).
#include "kernels.h"
#include "ptx.cuh"

namespace oscar {
namespace {

constexpr int kWarps = 4;

__global__ void __launch_bounds__(kWarps * 32) demote_kernel(DemoteParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t idx = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t total = int64_t(p.n) * p.n_kv * 2;
  if (idx >= total) return;
  const int which = int(idx & 1);            // 0 = K, 1 = V
  const int head = int((idx >> 1) % p.n_kv);
  const int item = int((idx >> 1) / p.n_kv);

  const int64_t row = p.src_index ? int64_t(p.src_index[item]) : int64_t(item);
  if (row < 0 || row >= p.src_rows) {
    if (lane == 0 && p.dev_status) atomicOr(p.dev_status, 0x2);
    return;
  }
  uint16_t* src = (which ? p.v_src : p.k_src) + row * p.row_stride + int64_t(head) * kHeadDim;
  const uint2 raw = *reinterpret_cast<const uint2*>(src + 4 * lane);
  float xv[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};

  const float* r = (which ? p.r_v : p.r_k) + int64_t(head) * kHeadDim * kHeadDim + 4 * lane;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
  for (int i = 0; i < kHeadDim; ++i) {
    const float xi = __shfl_sync(0xffffffffu, xv[i & 3], i >> 2);
    const float4 rr = __ldg(reinterpret_cast<const float4*>(r + i * kHeadDim));
    acc[0] = fmaf(xi, rr.x, acc[0]);
    acc[1] = fmaf(xi, rr.y, acc[1]);
    acc[2] = fmaf(xi, rr.z, acc[2]);
    acc[3] = fmaf(xi, rr.w, acc[3]);
  }

  // the source row may be overwritten by the new token only after every lane
  // has read it
  __syncwarp();
  const uint16_t* fresh = which ? p.new_v : p.new_k;
  if (fresh) {
    const uint2 nw = *reinterpret_cast<const uint2*>(
        fresh + (int64_t(item) * p.n_kv + head) * kHeadDim + 4 * lane);
    *reinterpret_cast<uint2*>(src + 4 * lane) = nw;
  }

  const float tau = which ? p.tau_v : p.tau_k;
  float mn = INFINITY, mx = -INFINITY;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    acc[c] = fminf(fmaxf(acc[c], -tau), tau);
    mn = fminf(mn, acc[c]);
    mx = fmaxf(mx, acc[c]);
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
    if (s > 0.f) code = fminf(fmaxf(rintf(__fdiv_rn(acc[c] - z, s)), 0.f), 3.f);
    byte |= uint32_t(code) << (2 * c);
  }

  const int b = p.dst_req[item];
  const int pos = p.dst_pos[item];
  if (b < 0 || b >= p.batch || pos < 0 || pos / kPage >= p.max_pages) {
    if (lane == 0 && p.dev_status) atomicOr(p.dev_status, 0x2);
    return;
  }
  const int64_t page = p.page_table[int64_t(b) * p.max_pages + pos / kPage];
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
  const int64_t warps = int64_t(p.n) * p.n_kv * 2;
  const int64_t blocks = (warps + kWarps - 1) / kWarps;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  demote_kernel<<<unsigned(blocks), kWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace oscar
