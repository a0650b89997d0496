// Internal interface between the C-ABI layer (oscar_api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace oscar {

constexpr int kHeadDim = 128;
constexpr int kPage = 16;
// Page block of one (physical page, KV head) with ng_k / ng_v quantisation
// groups per K / V vector:
//   [0, 512)     K code rows: token slot t, code byte l at 32 t + l;
//   [512, 1024)  V code rows interleaved by token pair: token slot t, code
//                byte l at 512 + 64 (t / 2) + 4 (l / 2) + 2 (t % 2) + l % 2,
//                so the 32-bit word at 512 + 64 a + 4 h holds 16-bit half h
//                (code positions 8h .. 8h+7) of slots 2a (low) and 2a + 1;
//   [1024, ...)  per token slot t, its ng_k K (scale, zero) fp16 pairs and
//                then its ng_v V pairs, at 1024 + 4 (ng_k + ng_v) t.
constexpr int kCodeBytes = 512;   // 16 token rows of 32 code bytes (K, and V)
constexpr int kVCodes = 512;      // offset of the V code rows
constexpr int kPairs = 1024;      // offset of the (scale, zero) pairs
constexpr int block_bytes(int ng_k, int ng_v) { return kPairs + 64 * (ng_k + ng_v); }
constexpr int kBlockBytes = block_bytes(1, 1);   // 1152: one group per token-head
__host__ __device__ constexpr int v_code_byte(int t, int l) {
  return kVCodes + 64 * (t >> 1) + 4 * (l >> 1) + 2 * (t & 1) + (l & 1);
}
__host__ __device__ constexpr int pair_byte(int ng_k, int ng_v, int t, int which, int q) {
  return kPairs + 4 * (ng_k + ng_v) * t + 4 * (which ? ng_k : 0) + 4 * q;
}

// Rotated channel held by code position c of a token row with ng groups
// (ng = 1: c itself).  K: c = 32 t + 8 e + j holds (j / J) g + (j % J) 16 +
// 4 t + e; V: c = 16 a + 8 e + m holds (m / M) g + (m % M) 16 + 2 a + e, with
// J = M = 8 / ng and g = 128 / ng, so one tensor-core K step (K) or one
// 16-row tile (V) of the decode kernel reads one group.
__host__ __device__ constexpr int storage_channel_k(int ng, int c) {
  return ng == 1 ? c
                 : ((c & 7) / (8 / ng)) * (kHeadDim / ng) + ((c & 7) % (8 / ng)) * 16 + 4 * (c >> 5) + ((c >> 3) & 3);
}
__host__ __device__ constexpr int storage_channel_v(int ng, int c) {
  return ng == 1 ? c
                 : ((c & 7) / (8 / ng)) * (kHeadDim / ng) + ((c & 7) % (8 / ng)) * 16 + 2 * (c >> 4) + ((c >> 3) & 1);
}
// Bounded waits: the default limit of every wait and the limit of the
// waits that let copies already issued land before a CTA exits.
constexpr uint64_t kDefaultWaitNs = 1000000000ull;
constexpr uint64_t kDrainWaitNs = 1000000000ull;
constexpr int kPartStride = 132;  // floats per (split, head) partial: m, l, pad, pad, o[128]

// Lazy online-softmax maximum: a running maximum m is raised only when a
// score (log2 units) exceeds it by more than this, so p = 2^(s - m) <= 2^this.
#ifndef OSCAR_RESCALE_LOG2
#define OSCAR_RESCALE_LOG2 8
#endif
constexpr int kRescaleLog2 = OSCAR_RESCALE_LOG2;

// Every kernel launches with programmatic stream serialisation: its CTAs may
// become resident while the kernel before it on the stream drains, and its
// first instruction (griddepcontrol.wait) holds them until that kernel has
// completed and its writes are visible, so results are those of plain stream
// order; each kernel also allows the kernel after it to launch at once.
template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// The kernel's dynamic shared-memory limit, set through the runtime once per
// kernel and device (a call per launch would cost host time on every step).
template <auto Kernel>
inline cudaError_t set_smem_limit(int bytes) {
  static int done[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev] >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = bytes;
  return e;
}

// ---------------------------------------------------------------- demotion
struct DemoteParams {
  uint8_t* pages;
  const int32_t* page_table;
  int32_t* dev_status;
  uint16_t* k_src;
  uint16_t* v_src;
  int64_t src_rows;
  int64_t row_stride;
  const int32_t* src_index;
  const int32_t* dst_req;
  const int32_t* dst_pos;
  const uint16_t* new_k;
  const uint16_t* new_v;
  const float* r_k;
  const float* r_v;
  float tau_k, tau_v;
  int32_t n, batch, n_kv, max_pages;
  int64_t n_pages;
  int32_t ng_k, ng_v;   // quantisation groups per token-head (1, 2 or 4)
  // codebook 1: code = number of thresholds (midpoints of adjacent levels)
  // strictly below u = (x - zero) / scale; K then V
  int32_t codebook;
  float thr_k[3], thr_v[3];
  // bulk path with contiguous source rows (no src_index): k_src / v_src as
  // 2-D bf16 tensors (n_kv * 128 columns x src_rows rows) read in boxes of 8
  // columns x 128 rows; use_tma = 0 means the rows are gathered by threads
  CUtensorMap tm_src[2];
  int32_t use_tma;
  // per-token path: 1 = everything before the stores runs ahead of the wait
  // for the previous kernel on the stream (that kernel writes nothing the
  // demotion reads before it); early_rows: the new rows are read ahead of it
  // too (that kernel does not write them either)
  int32_t early, early_rows;
};

cudaError_t launch_demote(const DemoteParams& p, cudaStream_t stream);

// Tensor-core bulk path (128 tokens per MMA tile); used for at least
// kBulkDemoteMin items without a new-token write.
constexpr int kBulkDemoteMin = 1024;
cudaError_t launch_demote_bulk(const DemoteParams& p, cudaStream_t stream);

// ---------------------------------------------------------------- decode
struct DecodeParams {
  // cache
  const uint8_t* pages;
  const int32_t* page_table;
  const int32_t* hist_len;
  const uint16_t* sink_k;
  const uint16_t* sink_v;
  const int32_t* sink_len;
  const uint16_t* recent_k;
  const uint16_t* recent_v;
  const int32_t* recent_len;
  const int32_t* recent_start;
  const float* r_k;
  const float* r_v;
  int32_t* dev_status;
  // io
  const uint16_t* q;
  float* out;
  // optional second copy of the output in pinned host memory (16-byte
  // aligned), written by the same stores that write `out`
  float* out_host;
  // workspace views
  uint32_t* counters;   // [pairs] merge tickets (zero between calls)
  float* partials;      // [pairs][n_splits][G][kPartStride]
  // dims
  int32_t batch, n_kv, group, sink_cap, recent_cap, max_pages;
  int32_t ng_k, ng_v;   // quantisation groups per token-head (1, 2 or 4)
  // codebook 1: a code's level is l[c] = l_0 + d1 c + a2 (2 b1) + b (b0 b1)
  // over its bits c = b0 + 2 b1 (d1 = l_1 - l_0, a2 = (l_2 - 2 l_1 + l_0) / 2,
  // b = l_3 - l_2 - l_1 + l_0); coef = {l_0, d1, a2, b} for K and for V
  int32_t codebook;
  float coef_k[4], coef_v[4];
  int64_t n_pages;
  int32_t max_hist;
  // split plan
  int32_t n_splits, pages_per_split;
  // time budget of a warp's page scan, and the limit of each wait for a page
  // copy: past either the warp gives up the rest of its pages
  // (OSCAR_DEV_TIMEOUT); copies already issued are still waited for, each up
  // to kDrainWaitNs, before the CTA exits
  uint64_t page_wait_ns;
  // the PV B operand is p s_V 2^pv_log2 (an integer pv_log2 keeps it in the
  // fp16 range): the INT2 states carry that factor in every term and keep
  // their maximum lowered by pv_log2; pv_unscale = 2^24 undoes the codes'
  // subnormal scale
  float pv_log2, pv_unscale;
  // R_V as a 2-D tensor (128 columns x n_kv * 128 rows of fp32) read in
  // boxes of 32 columns x 128 rows with the 128-byte swizzle
  CUtensorMap tm_rv;
};

// Fills p->tm_rv for p->r_v and p->n_kv; false if the driver refuses.
bool encode_rv_map(DecodeParams* p);

struct DecodePlan {
  int32_t n_splits, pages_per_split;
  size_t off_counters, off_partials, total_bytes;
};

// Split plan and workspace layout for the current device; returns the
// number of CTAs per SM the split kernel reaches, or <= 0 on a CUDA error.
int plan_decode(int batch, int n_kv, int group, int sink_cap, int recent_cap, int max_hist,
                DecodePlan* plan, cudaError_t* err);

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream);

// ---------------------------------------------------------------- staging
// Copies `bytes` from src to dst by a kernel in the launch chain; either side
// may be pinned host memory that the device addresses directly.
cudaError_t launch_stage(const void* src, void* dst, size_t bytes, cudaStream_t stream);

// ---------------------------------------------------------------- calibration
// C = X^T X / n over n bf16 rows of 128 values (ld elements apart), split
// over the rows into partials in `workspace`, added in a fixed order.
size_t covariance_workspace_bytes(int64_t n);
cudaError_t launch_covariance(const uint16_t* x, int64_t n, int64_t ld, float* c, void* workspace,
                              cudaStream_t stream);

// C_S = (S V)^T (S V) / n_q, S = row-softmax(Q K^T / sqrt(128)), over bf16
// rows of q [n_q], k and v [n_k] (ld elements apart): the fp32 rows of S V,
// then their covariance (partials added in a fixed order).
size_t value_covariance_workspace_bytes(int64_t n_q);
cudaError_t launch_value_covariance(const uint16_t* q, int64_t n_q, const uint16_t* k, const uint16_t* v,
                                    int64_t n_k, int64_t ld, float* c, void* workspace, cudaStream_t stream);

}  // namespace oscar
