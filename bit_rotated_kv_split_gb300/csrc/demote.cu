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
// is staged into shared memory by four TMA bulk copies (one barrier per
// quarter of its rows), then the CTA demotes its items one after another,
// all four warps on each: warp w sums the inputs i in [32 w, 32 w + 32)
// for every output, lane l owning rotated channels 4l..4l+3; the four
// partial sums meet in shared memory, and warp 0 clips, quantises (per
// quantisation group) and packs, lane l forming code byte l of the page
// format.  Splitting the inputs over the warps shortens the
// dependent chain of a lone item (a decode step demotes one token per
// request) from 128 to 32 steps.
#include "demote_math.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace oscar {
namespace {

constexpr int kWarps = 4;
constexpr int kItems = 4;                    // items per CTA
constexpr uint32_t kRotBytes = kHeadDim * kHeadDim * 4;
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr size_t kRedBytes = size_t(kWarps) * kHeadDim * 4;   // partial sums of one item
constexpr size_t kSmem = kRotBytes + kRedBytes + 4 * 8;

// Clip, quantise, pack and store one item from the four warps' partial sums
// red[w][channel] (warp 0): lane l owns code byte l of the token row, i.e.
// code positions 4 l + c (c < 4), which hold the rotated channels of the
// page format's order for NG groups per token-head.  The group of position
// 4 l + c is (4 (l & 1) + c) / (8 / NG) for K and V alike, so with c a
// compile-time constant each code picks between two fixed groups by the
// lane's parity.  Each group's (min, max) is reduced over the warp and
// gives its fp16 (scale, zero).  kLevels: the code is the number of the
// codebook thresholds `thr` strictly below u = (x - zero) / scale instead of
// rint(u) clamped to [0, 3].
// (finish_codes forms lane l's code byte and, for lane q < NG, group q's
// (scale, zero) pair; store_codes writes them to the page.)
template <int NG, bool kLevels>
__device__ __forceinline__ uint32_t finish_codes(const float* red, int which, float tau, int lane, const float* thr,
                                                 uint32_t& pair) {
  float v[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int ch = which ? storage_channel_v(NG, 4 * lane + c) : storage_channel_k(NG, 4 * lane + c);
    v[c] = (red[ch] + red[kHeadDim + ch]) + (red[2 * kHeadDim + ch] + red[3 * kHeadDim + ch]);
    v[c] = fminf(fmaxf(v[c], -tau), tau);
  }
  __half s16[NG], z16[NG];
  const uint32_t byte = quantize_lane<NG, kLevels>(v, lane, thr, s16, z16);
  __half2 sz = __halves2half2(s16[0], z16[0]);
#pragma unroll
  for (int q = 1; q < NG; ++q)
    if (lane == q) sz = __halves2half2(s16[q], z16[q]);
  pair = *reinterpret_cast<uint32_t*>(&sz);
  return byte;
}

__device__ __forceinline__ void store_codes(const DemoteParams& p, int ng, int which, int head, int64_t page,
                                            int slot, int lane, uint32_t byte, uint32_t pair) {
  if (page < 0 || page >= p.n_pages) {
    if (lane == 0 && p.dev_status) atomicOr(p.dev_status, 0x1);
    return;
  }
  uint8_t* blk = p.pages + (page * p.n_kv + head) * block_bytes(p.ng_k, p.ng_v);
  blk[which ? v_code_byte(slot, lane) : 32 * slot + lane] = uint8_t(byte);
  if (lane < ng) *reinterpret_cast<uint32_t*>(blk + pair_byte(p.ng_k, p.ng_v, slot, which, lane)) = pair;
}

// NGK / NGV: quantisation groups per token-head of K and V (template
// arguments, so a kernel holds only the finishing code it uses).
// kEarly (DemoteParams::early): the caller guarantees that the kernels that
// may still run (the one just before on the stream, and the ones it lets
// start early) write none of the rotation, the index arrays, the page table
// and the source rows, so everything up to the codes runs before the wait
// for that kernel; only the stores (the codes, and the new tokens into the
// source rows) follow it, and the loads of the new tokens unless
// DemoteParams::early_rows says that kernel does not write them either.  The
// next kernel may start at once: it waits for this one before it reads
// anything this one writes.
template <int NGK, int NGV, bool kLevels, bool kEarly = false>
__global__ void __launch_bounds__(kWarps * 32) demote_kernel(DemoteParams p) {
  if constexpr (kEarly) pdl_launch_dependents();
  {
    // L2 prefetch of this CTA's rotation (a hint that reads nothing, so it
    // may precede the wait for the previous kernel)
    const char* rg = reinterpret_cast<const char*>((blockIdx.y & 1 ? p.r_v : p.r_k) +
                                                   int64_t(blockIdx.y >> 1) * kHeadDim * kHeadDim);
    for (int i = threadIdx.x; i < int(kRotBytes / 128); i += kWarps * 32)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(rg + 128 * i));
    // and the lines of this CTA's item indices (the first level of its
    // dependent loads)
    const int it0 = int(blockIdx.x) * kItems;
    if (threadIdx.x < 3 && it0 < p.n) {
      const int32_t* idx = threadIdx.x == 0 ? p.dst_req : threadIdx.x == 1 ? p.dst_pos : p.src_index;
      if (idx) asm volatile("prefetch.global.L2 [%0];" ::"l"(idx + it0));
    }
  }
  if constexpr (!kEarly) {
    pdl_wait();                 // the previous kernel's writes are visible
    pdl_launch_dependents();
  }
  extern __shared__ __align__(128) uint8_t smem[];
  float* rs = reinterpret_cast<float*>(smem);
  float* red = reinterpret_cast<float*>(smem + kRotBytes);       // [kWarps][128]
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kRotBytes + kRedBytes);   // [4] R quarters
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int which = int(blockIdx.y & 1);     // 0 = K, 1 = V
  const int head = int(blockIdx.y >> 1);
  const float* rg = (which ? p.r_v : p.r_k) + int64_t(head) * kHeadDim * kHeadDim;
  if (threadIdx.x == 0) {
    for (int c = 0; c < 4; ++c) mbar_init(bar + c, 1);
    fence_mbar_init();
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      mbar_arrive_expect_tx(bar + c, kRotBytes / 4);
      bulk_copy_g2s(smem + c * (kRotBytes / 4), rg + c * (kRotBytes / 16), kRotBytes / 4, bar + c);
    }
  }
  __syncthreads();

  // every warp reads the items' indices and its quarter of each source row
  // (two levels of independent loads, overlapping the R transfer)
  const int item0 = int(blockIdx.x) * kItems;
  bool live[kItems];
  int64_t page[kItems];
  int64_t srow[kItems];        // the item's source row (the new token goes there)
  int slot[kItems];
  float xv[kItems];            // x_i, i = 32 warp + lane
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    const int item = item0 + it;
    live[it] = item < p.n;
    page[it] = -1;
    srow[it] = 0;
    slot[it] = 0;
    xv[it] = 0.f;
    if (!live[it]) continue;
    // (the step's inputs may sit in pinned host memory, read over the
    // CPU-GPU link: cache-volatile loads fetch them anew on every call)
    const int64_t row = p.src_index ? int64_t(__ldcv(p.src_index + item)) : int64_t(item);
    const int bq = __ldcv(p.dst_req + item), pos = __ldcv(p.dst_pos + item);
    if (row < 0 || row >= p.src_rows || bq < 0 || bq >= p.batch || pos < 0 || pos / kPage >= p.max_pages) {
      if (warp == 0 && lane == 0 && p.dev_status) atomicOr(p.dev_status, 0x2);
      live[it] = false;
      continue;
    }
    srow[it] = row;
    const uint16_t* src = (which ? p.v_src : p.k_src) + row * p.row_stride + int64_t(head) * kHeadDim;
    xv[it] = bf16_lo(uint32_t(src[32 * warp + lane]));
    page[it] = p.page_table[int64_t(bq) * p.max_pages + pos / kPage];
    slot[it] = pos % kPage;
  }
  // the source rows may be overwritten by the new tokens only after every
  // warp has read its part of them
  __syncthreads();
  const uint16_t* fresh = which ? p.new_v : p.new_k;
  uint16_t nv[kItems];         // the new tokens' elements 32 warp + lane
  auto load_new_tokens = [&]() {
#pragma unroll
    for (int it = 0; it < kItems; ++it)
      nv[it] = fresh && live[it]
                   ? __ldcv(reinterpret_cast<const unsigned short*>(fresh) +
                            (int64_t(item0 + it) * p.n_kv + head) * kHeadDim + 32 * warp + lane)
                   : uint16_t(0);
  };
  auto store_new_tokens = [&]() {
    if (!fresh) return;
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
      uint16_t* dst = (which ? p.v_src : p.k_src) + srow[it] * p.row_stride + int64_t(head) * kHeadDim;
      if (live[it]) dst[32 * warp + lane] = nv[it];
    }
  };
  if constexpr (!kEarly) {
    load_new_tokens();
    store_new_tokens();
  } else if (p.early_rows) {
    load_new_tokens();         // the caller's rows are final already
  }

  // warp w needs the rows 32 w .. 32 w + 31 of R: quarter w of the copy;
  // on an expired wait the whole CTA leaves (after waiting, bounded, for
  // the other quarters so that no copy lands after exit)
  if (!__syncthreads_and(mbar_wait_bounded(bar + warp, 0, kWaitLimitNs))) {
    if (threadIdx.x == 0 && p.dev_status) atomicOr(p.dev_status, 0x4);
    for (int c = 0; c < 4; ++c) mbar_wait_bounded(bar + c, 0, kWaitLimitNs);
    if constexpr (kEarly) pdl_wait();   // the next kernel still follows the previous one
    return;
  }
  const float tau = which ? p.tau_v : p.tau_k;
  const float4* r4 = reinterpret_cast<const float4*>(rs) + lane;
  const int ng = which ? NGV : NGK;
  uint32_t code_byte[kItems], code_pair[kItems];   // warp 0 (kEarly: stored after the wait)
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    if (!__syncthreads_or(live[it])) continue;   // uniform over the CTA
    float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int k = 0; k < 32; ++k) {
      const int i = 32 * warp + k;
      const float xi = __shfl_sync(0xffffffffu, xv[it], k);
      const float4 rr = r4[i * (kHeadDim / 4)];
      a[0] = fmaf(xi, rr.x, a[0]);
      a[1] = fmaf(xi, rr.y, a[1]);
      a[2] = fmaf(xi, rr.z, a[2]);
      a[3] = fmaf(xi, rr.w, a[3]);
    }
    *reinterpret_cast<float4*>(red + warp * kHeadDim + 4 * lane) = make_float4(a[0], a[1], a[2], a[3]);
    __syncthreads();
    code_byte[it] = code_pair[it] = 0u;
    if (warp == 0 && live[it]) {
      const float* thr = which ? p.thr_v : p.thr_k;
      if constexpr (NGK == NGV) {
        code_byte[it] = finish_codes<NGK, kLevels>(red, which, tau, lane, thr, code_pair[it]);
      } else if (which) {
        code_byte[it] = finish_codes<NGV, kLevels>(red, which, tau, lane, thr, code_pair[it]);
      } else {
        code_byte[it] = finish_codes<NGK, kLevels>(red, which, tau, lane, thr, code_pair[it]);
      }
      if constexpr (!kEarly) store_codes(p, ng, which, head, page[it], slot[it], lane, code_byte[it], code_pair[it]);
    }
    __syncthreads();   // red is reused by the next item
  }
  if constexpr (kEarly) {
    pdl_wait();                 // the previous kernel is done: the stores may start
    if (!p.early_rows) load_new_tokens();
    store_new_tokens();
    if (warp == 0) {
#pragma unroll
      for (int it = 0; it < kItems; ++it)
        if (live[it]) store_codes(p, ng, which, head, page[it], slot[it], lane, code_byte[it], code_pair[it]);
    }
  }
}

}  // namespace

namespace {

template <int NGK, int NGV, bool kLevels = false, bool kEarly = false>
cudaError_t launch_ng(const DemoteParams& p, int64_t chunks, cudaStream_t stream) {
  if constexpr (!kEarly) {
    if (p.early) return launch_ng<NGK, NGV, kLevels, true>(p, chunks, stream);
  }
  cudaError_t e = set_smem_limit<demote_kernel<NGK, NGV, kLevels, kEarly>>(int(kSmem));
  if (e != cudaSuccess) return e;
  return launch_pdl(demote_kernel<NGK, NGV, kLevels, kEarly>, dim3(unsigned(chunks), unsigned(p.n_kv * 2)),
                    dim3(kWarps * 32), kSmem, stream, p);
}

template <int NGK>
cudaError_t launch_ngk(const DemoteParams& p, int64_t chunks, cudaStream_t stream) {
  if (p.ng_v == 1) return launch_ng<NGK, 1>(p, chunks, stream);
  if (p.ng_v == 2) return launch_ng<NGK, 2>(p, chunks, stream);
  if (p.ng_v == 4) return launch_ng<NGK, 4>(p, chunks, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_demote(const DemoteParams& p, cudaStream_t stream) {
  const int64_t chunks = (int64_t(p.n) + kItems - 1) / kItems;
  if (chunks == 0) return cudaSuccess;
  if (chunks > 0x7fffffff || int64_t(p.n_kv) * 2 > 65535) return cudaErrorInvalidValue;
  if (p.codebook) {   // one group per vector (checked by the caller)
    return p.ng_k == 1 && p.ng_v == 1 ? launch_ng<1, 1, true>(p, chunks, stream) : cudaErrorInvalidValue;
  }
  if (p.ng_k == 1) return launch_ngk<1>(p, chunks, stream);
  if (p.ng_k == 2) return launch_ngk<2>(p, chunks, stream);
  if (p.ng_k == 4) return launch_ngk<4>(p, chunks, stream);
  return cudaErrorInvalidValue;
}

}  // namespace oscar
