// C-ABI entry points: host validation, split planning and kernel launches.
// Every check runs before any launch; a rejected call launches nothing.
#include <atomic>
#include <cmath>
#include <cstdint>

#include <cuda_fp16.h>

#include "kernels.h"
#include "oscar.h"
#include "trace.h"

namespace {

// limit of the decode kernel's waits for page copies (oscar_set_page_wait_limit)
std::atomic<int64_t> g_page_wait_ns{int64_t(oscar::kDefaultWaitNs)};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// codebook levels: fp16 values, 0 <= l_0 < l_1 < l_2 < l_3 <= 3
bool levels_ok(const float* l) {
  for (int k = 0; k < 4; ++k) {
    if (!std::isfinite(l[k]) || __half2float(__float2half_rn(l[k])) != l[k]) return false;
    if (k > 0 && !(l[k] > l[k - 1])) return false;
  }
  return l[0] >= 0.f && l[3] <= 3.f;
}

int groups_of(int32_t g);

// pinned host memory that the current device addresses at the same pointer
bool device_addressable_host(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();   // clear the error of an unregistered pointer
    return false;
  }
  return a.type == cudaMemoryTypeHost && a.devicePointer == p;
}

// the codebook form of a descriptor needs one quantisation group per vector
bool codebook_supported(const oscar_layer_desc* d) {
  return d->codebook == 0 || (groups_of(d->quant_group_k) == 1 && groups_of(d->quant_group_v) == 1);
}

// level coefficients {l_0, d1, a2, b} of l[c] = l_0 + d1 c + a2 (2 b1) + b b0 b1
void level_coef(const float* l, float* c) {
  c[0] = l[0];
  c[1] = l[1] - l[0];
  c[2] = (l[2] - 2.f * l[1] + l[0]) * 0.5f;
  c[3] = l[3] - l[2] - l[1] + l[0];
}

// groups per token-head for a quantisation group size (0 = 128); 0 if invalid
int groups_of(int32_t g) {
  if (g == 0 || g == 128) return 1;
  if (g == 64) return 2;
  if (g == 32) return 4;
  return 0;
}

oscar_status check_desc(const oscar_layer_desc* d, bool need_cache_segments) {
  if (!d) return OSCAR_ERR_INVALID_ARG;
  if (d->batch < 1 || d->n_kv_heads < 1 || d->n_q_heads < 1 || d->head_dim != OSCAR_HEAD_DIM)
    return OSCAR_ERR_INVALID_ARG;
  if (d->n_q_heads % d->n_kv_heads) return OSCAR_ERR_INVALID_ARG;
  if (d->sink_cap < 0 || d->recent_cap < 0 || d->sink_cap % OSCAR_PAGE_TOKENS ||
      d->recent_cap % OSCAR_PAGE_TOKENS)
    return OSCAR_ERR_INVALID_ARG;
  if (d->max_pages_per_seq < 1 || d->n_pages < 1 || d->n_pages > INT32_MAX) return OSCAR_ERR_INVALID_ARG;
  if (d->max_hist < 0 || int64_t(d->max_hist) > int64_t(d->max_pages_per_seq) * OSCAR_PAGE_TOKENS)
    return OSCAR_ERR_INVALID_ARG;
  // 2 tau / 3 must fit fp16 for the stored scale; tau > 0 and finite
  if (!(d->tau_k > 0.f) || !(d->tau_v > 0.f) || !(d->tau_k <= 65504.f) || !(d->tau_v <= 65504.f))
    return OSCAR_ERR_INVALID_ARG;
  if (!d->pages || !d->page_table || !d->r_k || !d->r_v) return OSCAR_ERR_INVALID_ARG;
  if (!groups_of(d->quant_group_k) || !groups_of(d->quant_group_v)) return OSCAR_ERR_INVALID_ARG;
  if (d->codebook != 0 && d->codebook != 1) return OSCAR_ERR_INVALID_ARG;
  if (d->codebook == 1 && (!levels_ok(d->levels_k) || !levels_ok(d->levels_v))) return OSCAR_ERR_INVALID_ARG;
  if (!aligned(d->pages, 128) || !aligned(d->r_k, 16) || !aligned(d->r_v, 16) ||
      !aligned(d->page_table, 4))
    return OSCAR_ERR_ALIGNMENT;
  if (need_cache_segments) {
    if (!d->hist_len || !d->sink_len || !d->recent_len || !d->recent_start)
      return OSCAR_ERR_INVALID_ARG;
    if ((d->sink_cap > 0 && (!d->sink_k || !d->sink_v)) ||
        (d->recent_cap > 0 && (!d->recent_k || !d->recent_v)))
      return OSCAR_ERR_INVALID_ARG;
    if (!aligned(d->sink_k, 16) || !aligned(d->sink_v, 16) || !aligned(d->recent_k, 16) ||
        !aligned(d->recent_v, 16))
      return OSCAR_ERR_ALIGNMENT;
  }
  return OSCAR_OK;
}

}  // namespace

extern "C" const char* oscar_status_string(oscar_status s) {
  switch (s) {
    case OSCAR_OK: return "ok";
    case OSCAR_ERR_INVALID_ARG: return "invalid argument";
    case OSCAR_ERR_ALIGNMENT: return "misaligned pointer";
    case OSCAR_ERR_WORKSPACE: return "workspace missing or too small";
    case OSCAR_ERR_CUDA: return "CUDA error";
    case OSCAR_ERR_NO_CONVERGENCE: return "eigensolver did not converge";
    case OSCAR_ERR_UNSUPPORTED: return "unsupported configuration";
    case OSCAR_ERR_FILE: return "file missing, unreadable, truncated or damaged";
    default: return "unknown status";
  }
}

extern "C" int32_t oscar_abi_version(void) { return OSCAR_ABI_VERSION; }

extern "C" int64_t oscar_set_page_wait_limit(int64_t limit_ns) {
  return g_page_wait_ns.exchange(limit_ns > 0 ? limit_ns : int64_t(oscar::kDefaultWaitNs));
}

extern "C" int64_t oscar_block_bytes(int32_t quant_group_k, int32_t quant_group_v) {
  const int gk = groups_of(quant_group_k), gv = groups_of(quant_group_v);
  return gk && gv ? int64_t(oscar::block_bytes(gk, gv)) : 0;
}

namespace {

// Validates an append and fills its kernel parameters (no launch).  *empty:
// n == 0, nothing to launch.
oscar_status prepare_append(const oscar_layer_desc* desc, uint16_t* k_src, uint16_t* v_src, int64_t src_rows,
                            int64_t row_stride, const int32_t* src_index, const int32_t* dst_req,
                            const int32_t* dst_pos, int32_t n, const uint16_t* new_k, const uint16_t* new_v,
                            oscar::DemoteParams* out, bool* empty) {
  *empty = false;
  oscar_status st = check_desc(desc, false);
  if (st != OSCAR_OK) return st;
  if (n < 0) return OSCAR_ERR_INVALID_ARG;
  if (n == 0) {
    *empty = true;
    return OSCAR_OK;
  }
  if (!k_src || !v_src || !dst_req || !dst_pos || src_rows < 1) return OSCAR_ERR_INVALID_ARG;
  if (!src_index && src_rows < n) return OSCAR_ERR_INVALID_ARG;
  if ((new_k == nullptr) != (new_v == nullptr)) return OSCAR_ERR_INVALID_ARG;
  if (row_stride < int64_t(desc->n_kv_heads) * OSCAR_HEAD_DIM || row_stride % 8)
    return OSCAR_ERR_INVALID_ARG;
  if (!aligned(k_src, 16) || !aligned(v_src, 16) || !aligned(new_k, 16) || !aligned(new_v, 16) ||
      !aligned(src_index, 4) || !aligned(dst_req, 4) || !aligned(dst_pos, 4))
    return OSCAR_ERR_ALIGNMENT;
  oscar::DemoteParams p{};
  p.pages = desc->pages;
  p.page_table = desc->page_table;
  p.dev_status = desc->dev_status;
  p.k_src = k_src;
  p.v_src = v_src;
  p.src_rows = src_rows;
  p.row_stride = row_stride;
  p.src_index = src_index;
  p.dst_req = dst_req;
  p.dst_pos = dst_pos;
  p.new_k = new_k;
  p.new_v = new_v;
  p.r_k = desc->r_k;
  p.r_v = desc->r_v;
  p.tau_k = desc->tau_k;
  p.tau_v = desc->tau_v;
  p.n = n;
  p.batch = desc->batch;
  p.n_kv = desc->n_kv_heads;
  p.max_pages = desc->max_pages_per_seq;
  p.n_pages = desc->n_pages;
  p.ng_k = groups_of(desc->quant_group_k);
  p.ng_v = groups_of(desc->quant_group_v);
  if (!codebook_supported(desc)) return OSCAR_ERR_UNSUPPORTED;
  p.codebook = desc->codebook;
  if (p.codebook) {
    for (int k = 0; k < 3; ++k) {
      p.thr_k[k] = (desc->levels_k[k] + desc->levels_k[k + 1]) * 0.5f;   // exact: fp16 inputs
      p.thr_v[k] = (desc->levels_v[k] + desc->levels_v[k + 1]) * 0.5f;
    }
  }
  *out = p;
  return OSCAR_OK;
}

cudaError_t launch_append(const oscar::DemoteParams& p, cudaStream_t stream) {
  const bool bulk = p.n >= oscar::kBulkDemoteMin && !p.new_k && !p.new_v;
  return bulk ? oscar::launch_demote_bulk(p, stream) : oscar::launch_demote(p, stream);
}

// Validates a decode call and fills its kernel parameters (no launch).
// *size_only: workspace was NULL and *workspace_bytes now holds the size.
oscar_status prepare_decode(const oscar_layer_desc* desc, const uint16_t* q, float* out, void* workspace,
                            size_t* workspace_bytes, oscar::DecodeParams* pout, bool* size_only) {
  *size_only = false;
  oscar_status st = check_desc(desc, true);
  if (st != OSCAR_OK) return st;
  const int group = desc->n_q_heads / desc->n_kv_heads;
  if (group != 4 && group != 8) return OSCAR_ERR_UNSUPPORTED;
  if (!workspace_bytes) return OSCAR_ERR_INVALID_ARG;
  oscar::DecodePlan plan{};
  cudaError_t err = cudaSuccess;
  if (oscar::plan_decode(desc->batch, desc->n_kv_heads, group, desc->sink_cap, desc->recent_cap,
                         desc->max_hist, &plan, &err) <= 0)
    return OSCAR_ERR_CUDA;
  if (!workspace) {
    *workspace_bytes = plan.total_bytes;
    *size_only = true;
    return OSCAR_OK;
  }
  if (*workspace_bytes < plan.total_bytes) return OSCAR_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return OSCAR_ERR_ALIGNMENT;
  if (!q || !out) return OSCAR_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16)) return OSCAR_ERR_ALIGNMENT;
  if (int64_t(desc->batch) * desc->n_kv_heads > 65535 * 65535LL || desc->batch > 65535 ||
      desc->n_kv_heads > 65535)
    return OSCAR_ERR_UNSUPPORTED;

  oscar::DecodeParams p{};
  p.pages = desc->pages;
  p.page_table = desc->page_table;
  p.hist_len = desc->hist_len;
  p.sink_k = desc->sink_k;
  p.sink_v = desc->sink_v;
  p.sink_len = desc->sink_len;
  p.recent_k = desc->recent_k;
  p.recent_v = desc->recent_v;
  p.recent_len = desc->recent_len;
  p.recent_start = desc->recent_start;
  p.r_k = desc->r_k;
  p.r_v = desc->r_v;
  p.dev_status = desc->dev_status;
  p.q = q;
  p.out = out;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.counters = reinterpret_cast<uint32_t*>(ws + plan.off_counters);
  p.partials = reinterpret_cast<float*>(ws + plan.off_partials);
  p.batch = desc->batch;
  p.n_kv = desc->n_kv_heads;
  p.group = group;
  p.sink_cap = desc->sink_cap;
  p.recent_cap = desc->recent_cap;
  p.max_pages = desc->max_pages_per_seq;
  p.n_pages = desc->n_pages;
  p.max_hist = desc->max_hist;
  p.ng_k = groups_of(desc->quant_group_k);
  p.ng_v = groups_of(desc->quant_group_v);
  if (!codebook_supported(desc)) return OSCAR_ERR_UNSUPPORTED;
  p.codebook = desc->codebook;
  if (p.codebook) {
    level_coef(desc->levels_k, p.coef_k);
    level_coef(desc->levels_v, p.coef_v);
  }
  p.n_splits = plan.n_splits;
  p.pages_per_split = plan.pages_per_split;
  p.page_wait_ns = uint64_t(g_page_wait_ns.load());
  // PV operand scale: p <= 2^kRescaleLog2 and s_V <= 2 tau_v / 3 (x2 margin
  // for fp16 rounding), so p s_V 2^pv_log2 stays below 2^14 in fp16
  int e = 0;
  std::frexp(std::ldexp(double(desc->tau_v) * (2.0 / 3.0) * 2.0, oscar::kRescaleLog2), &e);
  // (codebook 1: the PV operands are p s_V times level coefficients of
  // magnitude up to 3, so the scale is 8 times smaller)
  const int sig_exp = 14 - e - (desc->codebook ? 3 : 0);
  p.pv_log2 = float(sig_exp);
  p.pv_unscale = std::ldexp(1.0f, 24);
  if (!oscar::encode_rv_map(&p)) return OSCAR_ERR_CUDA;
  *pout = p;
  return OSCAR_OK;
}

}  // namespace

extern "C" oscar_status oscar_quantize_append(const oscar_layer_desc* desc, uint16_t* k_src,
                                              uint16_t* v_src, int64_t src_rows,
                                              int64_t row_stride,
                                              const int32_t* src_index, const int32_t* dst_req,
                                              const int32_t* dst_pos, int32_t n,
                                              const uint16_t* new_k, const uint16_t* new_v,
                                              void* stream) {
  OSCAR_TRACE_CALL();
  oscar::DemoteParams p{};
  bool empty = false;
  const oscar_status st = prepare_append(desc, k_src, v_src, src_rows, row_stride, src_index, dst_req, dst_pos, n,
                                         new_k, new_v, &p, &empty);
  if (st != OSCAR_OK || empty) return st;
  return launch_append(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

extern "C" oscar_status oscar_quantize_append_overlapped(const oscar_layer_desc* desc, uint16_t* k_src,
                                                         uint16_t* v_src, int64_t src_rows, int64_t row_stride,
                                                         const int32_t* src_index, const int32_t* dst_req,
                                                         const int32_t* dst_pos, int32_t n, const uint16_t* new_k,
                                                         const uint16_t* new_v, void* stream) {
  OSCAR_TRACE_CALL();
  oscar::DemoteParams p{};
  bool empty = false;
  const oscar_status st = prepare_append(desc, k_src, v_src, src_rows, row_stride, src_index, dst_req, dst_pos, n,
                                         new_k, new_v, &p, &empty);
  if (st != OSCAR_OK || empty) return st;
  p.early = 1;   // the tensor-core path ignores it and waits first
  return launch_append(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

extern "C" oscar_status oscar_decode_attention(const oscar_layer_desc* desc, const uint16_t* q,
                                               float* out, void* workspace,
                                               size_t* workspace_bytes, void* stream) {
  OSCAR_TRACE_CALL();
  oscar::DecodeParams p{};
  bool size_only = false;
  const oscar_status st = prepare_decode(desc, q, out, workspace, workspace_bytes, &p, &size_only);
  if (st != OSCAR_OK || size_only) return st;
  return oscar::launch_decode(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

extern "C" oscar_status oscar_decode_step(const oscar_layer_desc* desc, const void* host_in, void* dev_in,
                                          size_t in_bytes, uint16_t* k_src, uint16_t* v_src, int64_t src_rows,
                                          int64_t row_stride, const int32_t* src_index, const int32_t* dst_req,
                                          const int32_t* dst_pos, int32_t n, const uint16_t* new_k,
                                          const uint16_t* new_v, const uint16_t* q, float* out, void* workspace,
                                          size_t workspace_bytes, float* host_out, uint32_t flags,
                                          void* stream) {
  OSCAR_TRACE_CALL();
  if ((flags & ~OSCAR_STEP_OVERLAP_PREVIOUS) != 0) return OSCAR_ERR_INVALID_ARG;
  if ((in_bytes > 0) != (host_in != nullptr && dev_in != nullptr)) return OSCAR_ERR_INVALID_ARG;
  if (!workspace) return OSCAR_ERR_WORKSPACE;
  if ((in_bytes > 0 && !device_addressable_host(host_in)) || (host_out && !device_addressable_host(host_out)))
    return OSCAR_ERR_INVALID_ARG;
  oscar::DemoteParams pa{};
  bool empty = false;
  oscar_status st = prepare_append(desc, k_src, v_src, src_rows, row_stride, src_index, dst_req, dst_pos, n, new_k,
                                   new_v, &pa, &empty);
  if (st != OSCAR_OK) return st;
  oscar::DecodeParams pd{};
  bool size_only = false;
  size_t ws_bytes = workspace_bytes;
  st = prepare_decode(desc, q, out, workspace, &ws_bytes, &pd, &size_only);
  if (st != OSCAR_OK) return st;
  // The step's inputs that lie in the staging range [dev_in, dev_in +
  // in_bytes) are read by the kernels straight from the same offsets of
  // host_in (cache-volatile loads over the CPU-GPU link), when the two
  // buffers share their alignment modulo 16 bytes, the per-token demotion
  // kernel runs, and the demotion's source rows lie outside the range;
  // otherwise a copy kernel fills dev_in first.  Both run in the launch chain.
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uintptr_t lo = reinterpret_cast<uintptr_t>(dev_in), hi = lo + in_bytes;
  auto inside = [&](const void* ptr) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(ptr);
    return ptr != nullptr && a >= lo && a < hi;
  };
  auto to_host = [&](const void* ptr) -> const void* {
    return inside(ptr) ? static_cast<const uint8_t*>(host_in) + (reinterpret_cast<uintptr_t>(ptr) - lo) : ptr;
  };
  const bool bulk = !empty && pa.n >= oscar::kBulkDemoteMin && !pa.new_k && !pa.new_v;
  const bool any_in = inside(q) || (!empty && (inside(pa.src_index) || inside(pa.dst_req) || inside(pa.dst_pos) ||
                                               inside(pa.new_k) || inside(pa.new_v)));
  const bool direct_in = in_bytes > 0 && any_in && ((lo ^ reinterpret_cast<uintptr_t>(host_in)) & 15) == 0 &&
                         !bulk && !inside(pa.k_src) && !inside(pa.v_src);
  if (direct_in) {
    pd.q = static_cast<const uint16_t*>(to_host(pd.q));
    pa.src_index = static_cast<const int32_t*>(to_host(pa.src_index));
    pa.dst_req = static_cast<const int32_t*>(to_host(pa.dst_req));
    pa.dst_pos = static_cast<const int32_t*>(to_host(pa.dst_pos));
    pa.new_k = static_cast<const uint16_t*>(to_host(pa.new_k));
    pa.new_v = static_cast<const uint16_t*>(to_host(pa.new_v));
  } else if (in_bytes > 0 && oscar::launch_stage(host_in, dev_in, in_bytes, s) != cudaSuccess) {
    return OSCAR_ERR_CUDA;
  }
  // after a copy kernel of this call the demotion reads what it wrote: it
  // waits first; otherwise the caller may let it overlap the kernel before
  const bool staged = in_bytes > 0 && !direct_in;
  if ((flags & OSCAR_STEP_OVERLAP_PREVIOUS) && !staged) pa.early = pa.early_rows = 1;
  if (!empty && launch_append(pa, s) != cudaSuccess) return OSCAR_ERR_CUDA;
  // a 16-byte aligned host_out is written by the decode kernel itself, with
  // the same stores as `out`; otherwise a copy kernel follows it
  const bool direct_out = host_out && aligned(host_out, 16);
  if (direct_out) pd.out_host = host_out;
  if (oscar::launch_decode(pd, s) != cudaSuccess) return OSCAR_ERR_CUDA;
  if (host_out && !direct_out) {
    const size_t out_bytes = size_t(desc->batch) * desc->n_q_heads * OSCAR_HEAD_DIM * sizeof(float);
    if (oscar::launch_stage(out, host_out, out_bytes, s) != cudaSuccess) return OSCAR_ERR_CUDA;
  }
  return OSCAR_OK;
}

// [GIST] 2.1 / 2.2 A: C_Q and C_S as one contraction over calibration rows.
extern "C" oscar_status oscar_covariance(const uint16_t* x, int64_t n, int32_t d, int64_t ld, float* c_out,
                                         void* workspace, size_t* workspace_bytes, void* stream) {
  OSCAR_TRACE_CALL();
  if (!workspace_bytes || n < 1 || d != 128 || ld < d) return OSCAR_ERR_INVALID_ARG;
  const size_t need = oscar::covariance_workspace_bytes(n);
  if (!workspace) {
    *workspace_bytes = need;
    return OSCAR_OK;
  }
  if (*workspace_bytes < need) return OSCAR_ERR_WORKSPACE;
  if (!x || !c_out) return OSCAR_ERR_INVALID_ARG;
  if (!aligned(x, 16) || (ld % 8) != 0 || !aligned(c_out, 16) || !aligned(workspace, 256)) return OSCAR_ERR_ALIGNMENT;
  const cudaError_t err = oscar::launch_covariance(x, n, ld, c_out, workspace, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

// [GIST] 2.1 / 2.2 A: C_S from calibration queries, keys and values.
extern "C" oscar_status oscar_value_covariance(const uint16_t* q, int64_t n_q, const uint16_t* k, const uint16_t* v,
                                               int64_t n_k, int32_t d, int64_t ld, float* c_out, void* workspace,
                                               size_t* workspace_bytes, void* stream) {
  OSCAR_TRACE_CALL();
  if (!workspace_bytes || n_q < 1 || n_k < 1 || d != 128 || ld < d) return OSCAR_ERR_INVALID_ARG;
  const size_t need = oscar::value_covariance_workspace_bytes(n_q);
  if (!workspace) {
    *workspace_bytes = need;
    return OSCAR_OK;
  }
  if (*workspace_bytes < need) return OSCAR_ERR_WORKSPACE;
  if (!q || !k || !v || !c_out) return OSCAR_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || (ld % 8) != 0 || !aligned(c_out, 16) ||
      !aligned(workspace, 256))
    return OSCAR_ERR_ALIGNMENT;
  const cudaError_t err =
      oscar::launch_value_covariance(q, n_q, k, v, n_k, ld, c_out, workspace, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}
