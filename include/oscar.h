/*
 * oscar.h - C ABI of the OSCAR two-bit rotated KV-cache decode path for GB300
 * (sm_103a).
 *
 * Method (three web pages about one paper, cited by title and section):
 *   [GIST]  gist.science, "OSCAR: Offline Spectral Covariance-Aware Rotation
 *           for 2-bit KV Cache Quantization", Technical summary 2.1, 2.2 A
 *           (offline calibration), 2.2 B (online serving).
 *   [ZAKER] myzaker.com OSCAR article, parts "OSCAR 把旋转对准 attention"
 *           (rotation) and "从离线校准到在线推理的 pipeline" (token pool,
 *           demotion kernel, INT2 decode, online-softmax merge).
 *
 * Conventions shared by every call:
 *   - Row vectors: a rotated key is k~ = k . R with R = U . H_Had . P_br.
 *   - head_dim d = 128, 16 tokens per page; a (token, KV head, K|V) vector
 *     of 128 rotated channels is quantised in groups of g consecutive
 *     channels (g = 128 by default; 64 or 32 per layer, for K and V apart,
 *     see quant_group_k / quant_group_v), each with an fp16 scale and zero.
 *     Smaller groups are where the bit-reversal P_br of R matters: it
 *     interleaves high- and low-variance channels across the groups
 *     ([GIST] 2.2 A; [ZAKER] "OSCAR 把旋转对准 attention").
 *   - bfloat16 data is passed as uint16_t bit patterns.
 *   - All device memory is allocated and freed by the caller.  The library
 *     keeps no state besides cached device attributes; calls on different
 *     streams may run concurrently when they touch disjoint memory.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Device
 *     calls are asynchronous; every argument is validated on the host before
 *     any launch, and a rejected call launches nothing.
 *   - Device-side faults the host cannot see in advance (page ids outside the
 *     pool, lengths above their capacity, an expired bounded wait) never trap:
 *     the kernel skips the offending access and ORs a bit into the optional
 *     device status word `dev_status` (see OSCAR_DEV_*).
 *   - No C++ exception crosses this boundary.
 *
 * Page pool layout (this library's format; the pages fix only "paged KV",
 * "4 codes per byte" and "scale/zero point"), with G_K = 128 / g_K and
 * G_V = 128 / g_V groups per vector.  A block of one (page p, KV head h)
 * has 1024 + 64 (G_K + G_V) bytes (1152 with one group each,
 * OSCAR_BLOCK_BYTES) and sits at byte (p * n_kv_heads + h) * block:
 *   [0, 512)     K code rows: token slot t, code byte l at 32 t + l;
 *   [512, 1024)  V code rows, the two tokens of a slot pair interleaved by
 *                16-bit halves: token slot t, code byte l at
 *                512 + 64 (t / 2) + 4 (l / 2) + 2 (t % 2) + (l % 2);
 *   [1024, ...)  token slot t: its G_K K (scale, zero) fp16 pairs, then its
 *                G_V V pairs, at 1024 + 4 (G_K + G_V) t.
 *   Code byte l of a token row holds code positions 4l .. 4l+3 (bits
 *   2 (c % 4)); position c holds rotated channel c when G = 1.  When G > 1
 *   it holds channel
 *     K: c = 32 t + 8 e + j (t, e < 4, j < 8):  (j / J) g + (j % J) 16 + 4 t + e,
 *     V: c = 16 a + 8 e + m (a < 8, e < 2, m < 8): (m / M) g + (m % M) 16 + 2 a + e,
 *   with J = M = 8 / G, so that each tensor-core operand tile of the decode
 *   kernel draws on one group.  Group q is rotated channels [q g, (q+1) g).
 *   Logical history position x of request b lives in page
 *   page_table[b][x / 16], slot x % 16.
 */
#ifndef OSCAR_H_
#define OSCAR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define OSCAR_ABI_VERSION 4

#define OSCAR_HEAD_DIM 128
#define OSCAR_PAGE_TOKENS 16
#define OSCAR_BLOCK_BYTES 1152

typedef int32_t oscar_status;
enum {
  OSCAR_OK = 0,
  OSCAR_ERR_INVALID_ARG = 1,     /* null pointer, bad dimension or length     */
  OSCAR_ERR_ALIGNMENT = 2,       /* a pointer misses its required alignment  */
  OSCAR_ERR_WORKSPACE = 3,       /* workspace missing or too small            */
  OSCAR_ERR_CUDA = 4,            /* a CUDA runtime call or launch failed      */
  OSCAR_ERR_NO_CONVERGENCE = 5,  /* the host eigensolver did not converge     */
  OSCAR_ERR_UNSUPPORTED = 6,     /* a valid but unimplemented configuration   */
  OSCAR_ERR_FILE = 7             /* a file missing, unreadable, truncated or   */
                                 /* failing its format or checksum check       */
};

/* Bits a kernel ORs into *dev_status (never cleared by the library). */
#define OSCAR_DEV_PAGE_BOUNDS 0x1   /* a page id outside [0, n_pages): skipped  */
#define OSCAR_DEV_LENGTH 0x2        /* a length above its capacity: clamped     */
#define OSCAR_DEV_TIMEOUT 0x4       /* a bounded wait expired: work abandoned   */

/* Human-readable name of a status code (static string, never NULL). */
const char* oscar_status_string(oscar_status s);

/* OSCAR_ABI_VERSION of the loaded library. */
int32_t oscar_abi_version(void);

/*
 * oscar_set_page_wait_limit - the decode kernel's time budget for a warp's
 * scan of its INT2 pages, which also bounds each wait for a page copy to
 * land.  A warp past it gives up the rest of its pages, sets
 * OSCAR_DEV_TIMEOUT in dev_status, and the call's output must not be used.
 * limit_ns <= 0 restores the default (1 s, far beyond any scan).  Returns
 * the previous limit.  Copies already issued are still waited for (up to
 * 1 s each) before a CTA exits, and the workspace stays ready for the next
 * call.  A stalled copy is the only way this path runs in normal use; a
 * short limit makes it run on purpose (tests of the failure path).
 * Process-wide, read when a decode call is issued.  Host-only.
 */
int64_t oscar_set_page_wait_limit(int64_t limit_ns);

/*
 * One attention layer's cache: a three-segment token pool, BF16 sink (64
 * tokens) | INT2 history (paged) | BF16 recent window (256-slot ring).
 * [ZAKER] pipeline part; [GIST] 2.2 B (hybrid-precision paged layout).
 * Pointers are device pointers unless marked host.  The struct itself is
 * read on the host during the call only; it may be reused or freed after.
 */
typedef struct oscar_layer_desc {
  int32_t batch;              /* B >= 1                                        */
  int32_t n_q_heads;          /* H_q, a multiple of n_kv_heads                */
  int32_t n_kv_heads;         /* H_kv >= 1; GQA group g = H_q / H_kv in {4, 8} */
  int32_t head_dim;           /* must be 128                                   */
  int32_t sink_cap;           /* sink capacity in tokens (64 on the pages)     */
  int32_t recent_cap;         /* recent ring capacity (256 on the pages)       */
  int32_t max_pages_per_seq;  /* row length of page_table                      */
  int32_t max_hist;           /* host upper bound on every hist_len[b]         */
  int64_t n_pages;            /* physical pages in the pool                    */
  float tau_k;                /* clip threshold of this layer's keys, > 0      */
  float tau_v;                /* clip threshold of this layer's values, > 0    */
  uint8_t* pages;             /* pool, 128-byte aligned (layout above)         */
  const int32_t* page_table;  /* [B][max_pages_per_seq] physical page ids      */
  const int32_t* hist_len;    /* [B] INT2 history length of each request       */
  const uint16_t* sink_k;     /* [B][sink_cap][H_kv][d] bf16, 16-byte aligned  */
  const uint16_t* sink_v;     /* same layout                                   */
  const int32_t* sink_len;    /* [B] valid sink tokens (slots 0..len-1)        */
  uint16_t* recent_k;         /* [B][recent_cap][H_kv][d] bf16 ring            */
  uint16_t* recent_v;         /* same layout                                   */
  const int32_t* recent_len;  /* [B] valid recent tokens                       */
  const int32_t* recent_start;/* [B] ring slot of the oldest recent token      */
  const float* r_k;           /* [H_kv][d][d] row-major R_K, k~ = k . R_K      */
  const float* r_v;           /* [H_kv][d][d] row-major R_V                    */
  int32_t* dev_status;        /* optional device word for OSCAR_DEV_* bits     */
  int32_t quant_group_k;      /* K quantisation group g_K: 32, 64 or 128 (0 = 128) */
  int32_t quant_group_v;      /* V quantisation group g_V: 32, 64 or 128 (0 = 128) */
  int32_t codebook;           /* 0: uniform levels 0..3; 1: levels_k / levels_v  */
  float levels_k[4];          /* codebook 1: K levels l_0 < .. < l_3 (fp16 values) */
  float levels_v[4];          /* codebook 1: V levels                          */
} oscar_layer_desc;

/*
 * Codebook levels (desc->levels_k / levels_v, used when desc->codebook = 1):
 * four fp16 values 0 <= l_0 < l_1 < l_2 < l_3 <= 3 in the normalised domain
 * u = (x - zero) / scale, where the group's (scale, zero) are those of the
 * uniform codec; a value dequantises to zero + scale * l[code].  Levels that
 * are not fp16 values, not increasing or outside [0, 3] are rejected with
 * OSCAR_ERR_INVALID_ARG.  Levels 0, 1, 2, 3 give the uniform codes except
 * at exact ties u = 1.5 (lower level here, round-half-even there).
 */

/* Bytes of one (page, KV head) block for groups g_k, g_v (0 = 128); 0 for
 * any other value.  Host-only. */
int64_t oscar_block_bytes(int32_t quant_group_k, int32_t quant_group_v);

/*
 * oscar_build_rotation - the fixed rotation of one (layer, KV head) from
 * calibration rows.  [GIST] 2.1 and 2.2 A; [ZAKER] "OSCAR 把旋转对准 attention".
 *
 *   C = x^T x / n over the n rows of x (host, row-major [n][d], float64):
 *   post-RoPE queries of the KV head's query group for R_K (C_Q), or rows of
 *   S.V (see oscar_score_weighted_rows) for R_V (C_S).  U = eigenvectors of C
 *   by descending eigenvalue, each column's largest-|entry| made positive
 *   (ties: lowest index).  r_out = U . H . P_br with the orthonormal Sylvester
 *   Hadamard H and the bit-reversal permutation P_br.
 *
 *   d must be a power of two in [2, 1024]; n >= 1.  r_out (host, [d][d]
 *   row-major) is written; eigvals_out (host, [d], nullable) receives the
 *   eigenvalues in the same order.  Host-only, synchronous, thread-safe.
 *   Returns OSCAR_ERR_NO_CONVERGENCE if the eigensolver does not converge.
 */
oscar_status oscar_build_rotation(const double* x, int64_t n, int32_t d,
                                  double* r_out, double* eigvals_out);

/*
 * oscar_build_canalized_rotation - the block-diagonal rotation of the OScaR
 * variant.  [CSDN] section 四.2 (channels split into groups, each rotated
 * within the group; no inversion, no iteration).
 *
 *   r_out (host, [d][d] row-major, float64) = I_(d/block) (x) H_block, with
 *   H_block the orthonormal Sylvester Hadamard of size block.  The variant's
 *   per-token scaling is carried by the per-token (scale, zero) of this
 *   codec, so the rotation is the whole difference; the demotion and decode
 *   calls take it like any R.  d and block powers of two, 1 <= block <= d
 *   <= 1024.  Host-only, synchronous, thread-safe.
 */
oscar_status oscar_build_canalized_rotation(int32_t d, int32_t block, double* r_out);

/*
 * oscar_build_rotation_from_covariance - as oscar_build_rotation, from a
 * covariance computed elsewhere (for instance by oscar_covariance on the
 * device): c (host, [d][d] row-major, float64) is symmetrised as
 * (c + c^T) / 2 and decomposed; r_out = U . H . P_br, eigvals_out (nullable)
 * as in oscar_build_rotation.  OSCAR_ERR_INVALID_ARG for non-finite entries.
 * Host-only, synchronous, thread-safe.
 */
oscar_status oscar_build_rotation_from_covariance(const double* c, int32_t d, double* r_out,
                                                  double* eigvals_out);

/*
 * oscar_covariance - calibration covariance on the device.  [GIST] 2.1 and
 * 2.2 A (C_Q = Q^T Q over calibration queries for R_K, C_S = (S V)^T (S V)
 * for R_V, both divided by the number of rows).
 *
 *   c_out (device, [d][d] row-major, fp32) = X^T X / n over the n rows of x
 *   (device, bf16, row r at x + r * ld, d = 128 values each).  Products of
 *   bf16 values are exact in fp32; sums are fp32 over at most 2048 rows,
 *   then over those partials in a fixed order (the result does not depend
 *   on scheduling).  If workspace is NULL the required size is written to
 *   *workspace_bytes and nothing runs; otherwise the call is asynchronous on
 *   `stream`.  x 16-byte aligned, ld a multiple of 8, c_out 16-byte and the
 *   workspace 256-byte aligned (OSCAR_ERR_ALIGNMENT); d must be 128.
 */
oscar_status oscar_covariance(const uint16_t* x, int64_t n, int32_t d, int64_t ld, float* c_out,
                              void* workspace, size_t* workspace_bytes, void* stream);

/*
 * oscar_value_covariance - the score-weighted value covariance on the
 * device.  [GIST] 2.1 and 2.2 A (C_S = (1/N) V^T S^T S V, S = row-softmax of
 * the calibration scores).
 *
 *   c_out (device, [d][d] row-major, fp32) = (S V)^T (S V) / n_q with
 *   S = row-softmax(q k^T / sqrt(d)), over device bf16 rows q [n_q], k and
 *   v [n_k] (row r at base + r * ld, d = 128 values each).  The rows of S V
 *   are formed in fp32 (exact bf16 products in Q K^T, an fp32 softmax, P
 *   split into two bf16 parts against the bf16 values), then their
 *   covariance as fp32 partials of 256 rows added in a fixed order.  If
 *   workspace is NULL the required size is written to *workspace_bytes and
 *   nothing runs; otherwise asynchronous on `stream`.  q, k, v 16-byte
 *   aligned, ld a multiple of 8, c_out 16-byte and workspace 256-byte
 *   aligned (OSCAR_ERR_ALIGNMENT); n_q, n_k >= 1 and d = 128.
 */
oscar_status oscar_value_covariance(const uint16_t* q, int64_t n_q, const uint16_t* k, const uint16_t* v,
                                    int64_t n_k, int32_t d, int64_t ld, float* c_out, void* workspace,
                                    size_t* workspace_bytes, void* stream);

/*
 * oscar_score_weighted_rows - rows of S.V for the value covariance
 * C_S = (1/N) V^T S^T S V.  [GIST] 2.1 and 2.2 A.
 *
 *   S = row-softmax(q k^T * scale) with q [n_q][d], k and v [n_k][d] (host,
 *   row-major, float64); out [n_q][d] = S . v.  scale is normally 1/sqrt(d).
 *   Host-only, synchronous.
 */
oscar_status oscar_score_weighted_rows(const double* q, int64_t n_q, const double* k,
                                       const double* v, int64_t n_k, int32_t d,
                                       double scale, double* out);

/*
 * oscar_clip_threshold - per-layer clip threshold from rotated calibration
 * activations.  [GIST] 2.2 A (thresholds estimated from the rotated
 * calibration activations); the estimator is this library's choice:
 *
 *   tau = nearest-rank `quantile` of |acts[h] . r[h]| over every element of
 *   every head h < n_heads (acts [n_heads][rows][d], r [n_heads][d][d], host,
 *   float64).  0 < quantile <= 1.  Writes *tau_out.  Host-only.
 */
oscar_status oscar_clip_threshold(const double* acts, int64_t rows, int32_t n_heads,
                                  int32_t d, const double* r, double quantile,
                                  double* tau_out);

/*
 * oscar_fit_codebook - the Lloyd-Max codebook of one layer's K or V from
 * calibration rows.  [ZAKER] "OSCAR 把旋转对准 attention", closing part (the
 * code repo combines the rotation with a Lloyd-Max codebook); the fit is this
 * library's reading:
 *
 *   For every row of x [n][d] (host float64, d = 128) and its head's
 *   rotation r [d][d]: x~ = clamp(x . r, -tau, tau); scale = fp16((max -
 *   min) / 3), zero = fp16(min) (round to nearest even); rows with scale 0
 *   are skipped; u = (x~ - zero) / scale for each channel.  Lloyd's iteration
 *   over all u from levels {0, 1, 2, 3}: thresholds at the midpoints of
 *   adjacent levels, each level the mean of the u in its cell (u <= t_1, t_1
 *   < u <= t_2, ...; an empty cell keeps its level), at most `iters` rounds
 *   or until no level moves.  levels_out[4] = the levels clamped to [0, 3]
 *   and rounded to fp16 (as float).  OSCAR_ERR_INVALID_ARG for bad sizes, tau <= 0, iters < 1, no
 *   usable row, or fitted levels that are not strictly increasing in fp16.
 *   Host-only, synchronous.
 */
oscar_status oscar_fit_codebook(const double* x, int64_t n, int32_t d, const double* r, double tau,
                                int32_t iters, float* levels_out);

/*
 * Rotation files: a model's fixed rotations and clip thresholds, computed
 * once offline, stored for serving start-up.  [ZAKER] closing part (the
 * release ships a zoo of precomputed per-layer rotations); [GIST] 2.2 A
 * (R and the thresholds are fixed per layer after calibration).
 *
 *   Layout (little-endian): "OSCARROT", u32 version 1, u32 n_layers, u32
 *   n_kv_heads, u32 d; per layer f32 tau_k, f32 tau_v, R_K [n_kv][d][d] f32,
 *   R_V [n_kv][d][d] f32; then the 64-bit FNV-1a hash of all bytes before it.
 *   r_k / r_v (host) are [n_layers][n_kv][d][d] row-major, tau_k / tau_v
 *   (host) [n_layers].  write creates or replaces the file; info reads the
 *   dimensions; read checks the magic, version, dimensions (the caller's
 *   must equal the file's, else OSCAR_ERR_INVALID_ARG), size and hash before
 *   it writes any output.  OSCAR_ERR_FILE for an unreadable, truncated or
 *   damaged file.  Host-only, synchronous.
 */
oscar_status oscar_rotation_file_write(const char* path, int32_t n_layers, int32_t n_kv_heads, int32_t d,
                                       const float* r_k, const float* r_v, const float* tau_k,
                                       const float* tau_v);
oscar_status oscar_rotation_file_info(const char* path, int32_t* n_layers, int32_t* n_kv_heads, int32_t* d);
oscar_status oscar_rotation_file_read(const char* path, int32_t n_layers, int32_t n_kv_heads, int32_t d,
                                      float* r_k, float* r_v, float* tau_k, float* tau_v);

/*
 * oscar_quantize_append - the fused demotion kernel: rotate, clip, quantise
 * and pack tokens into INT2 history pages.  [ZAKER] pipeline part (the
 * oldest recent token is rotated, clipped, quantised and packed into INT2
 * history; 4 codes per byte; scale/zero point); [GIST] 2.2 B.
 *
 *   For item i < n and every KV head h: x = src row src_index[i] (identity if
 *   src_index is NULL) of k_src / v_src, viewed as [src_rows][row_stride]
 *   bf16 with head h at elements h*d .. h*d+d-1.  A source row outside
 *   [0, src_rows), a request outside the batch or a position beyond the page
 *   table skips the item and sets OSCAR_DEV_LENGTH; a page id outside the
 *   pool skips it and sets OSCAR_DEV_PAGE_BOUNDS.  x~ = x . R[h] (fp32 accumulate),
 *   clamped to [-tau, tau]; per group of g consecutive channels (g =
 *   quant_group_k for K, quant_group_v for V) scale = fp16((max - min) / 3),
 *   zero = fp16(min) over the group; code = clamp(rint((x~ - zero) / scale),
 *   0, 3) (0 if scale is 0).  With desc->codebook == 1 (Lloyd-Max levels;
 *   one group per vector only, else OSCAR_ERR_UNSUPPORTED) the code is
 *   instead the number of thresholds (l_(k-1) + l_k) / 2 of levels_k / levels_v
 *   strictly below u = (x~ - zero) / scale (the nearest level, ties to the
 *   lower), 0 if scale is 0.  The codes and (scale, zero) pairs go to history
 *   position dst_pos[i] of request dst_req[i] through desc->page_table, in the
 *   pool layout above.  K and V are both written.
 *
 *   Any finite bf16 row is accepted at any magnitude: calls of n >= 1024
 *   items (the tensor-core path) multiply the bf16 rows as they are by R
 *   held as three bf16 parts (about 24 significant bits), with exact
 *   products and fp32 sums, like the per-token path's fp32 arithmetic.
 *   Rows holding an infinity or a NaN give unspecified codes.
 *
 *   new_k / new_v (nullable, both or neither): [n][H_kv][d] bf16 rows that
 *   replace the demoted source rows after they have been read - the decode
 *   step's "write the new token into the freed ring slot".  k_src / v_src
 *   are written only then.
 *
 *   src_index, dst_req, dst_pos: device int32 [n].  k_src, v_src, new_k,
 *   new_v: 16-byte aligned; row_stride a multiple of 8 and >= H_kv * d.
 *   The caller owns lengths and page allocation: writing into a page that
 *   another request also references is a caller error.  Items must name
 *   distinct (request, position) pairs.  n = 0 is a no-op.  Async.
 */
oscar_status oscar_quantize_append(const oscar_layer_desc* desc,
                                   uint16_t* k_src, uint16_t* v_src,
                                   int64_t src_rows, int64_t row_stride,
                                   const int32_t* src_index,
                                   const int32_t* dst_req, const int32_t* dst_pos,
                                   int32_t n, const uint16_t* new_k,
                                   const uint16_t* new_v, void* stream);

/*
 * oscar_quantize_append_overlapped - oscar_quantize_append whose reads and
 * arithmetic run while the kernel before it on `stream` is still running.
 * [ZAKER] pipeline part (demote the oldest recent token, write the new one):
 * the same operation, the same arguments, bit for bit the same results.
 *
 *   The per-token kernel reads the rotations, the index arrays, the page
 *   table and the source rows, rotates and quantises, and only then waits
 *   for the previous kernel on the stream to finish; the code stores and
 *   the new-token writes into k_src / v_src (new_k / new_v are read only
 *   then) follow the wait.  This is for a decode loop in which that previous
 *   kernel is the projection that produces new_k / new_v, or the attention
 *   of the layer before (oscar_decode_attention reads, never writes, the
 *   cache).  Precondition (the caller's): no kernel that may still be
 *   running when this one starts writes desc->r_k / r_v, desc->page_table,
 *   src_index, dst_req, dst_pos or the source rows src_index names; new_k /
 *   new_v and anything else may be written.  Those kernels are the one
 *   issued on `stream` just before this call and, if that one lets its
 *   successor start early, the ones still running at that point.  The other
 *   kernels of this library let a successor start only after their own
 *   wait, so after one of them only that kernel counts.  This kernel lets
 *   its successor start at once (the successor's own wait still covers
 *   everything this kernel and its predecessor write), so for a call after
 *   it that reads before its wait, this call's predecessor counts too.
 *   Calls that take the tensor-core path (n >= 1024,
 *   no new rows) wait first, like oscar_quantize_append.  Argument checks
 *   and error codes are those of oscar_quantize_append.  Async.
 */
oscar_status oscar_quantize_append_overlapped(const oscar_layer_desc* desc,
                                              uint16_t* k_src, uint16_t* v_src,
                                              int64_t src_rows, int64_t row_stride,
                                              const int32_t* src_index,
                                              const int32_t* dst_req, const int32_t* dst_pos,
                                              int32_t n, const uint16_t* new_k,
                                              const uint16_t* new_v, void* stream);

/*
 * oscar_decode_attention - one decode step of attention for every request of
 * the batch over BF16 sink | INT2 history | BF16 recent.  [ZAKER] pipeline
 * part (INT2 kernel: unpack, scale/zero dequantisation, float accumulation;
 * BF16 kernel for sink/recent; online-softmax merge); [GIST] 2.2 B (inverse
 * rotation fused into the kernel with no extra memory traffic); [CSDN] the
 * aicoding.csdn.net explainer, section 三.1 (load INT2, rotate back, attend).
 *
 *   q: [B][H_q][d] bf16 (16-byte aligned); out: [B][H_q][d] float32
 *   (16-byte aligned), normalised softmax(q K^T / sqrt(d)) V over the valid
 *   tokens of all three segments; query head j reads KV head j / g.
 *   History keys/values are c * s + z (codebook 0) or l[c] * s + z
 *   (codebook 1) rotated back with R^T; the kernel
 *   computes this as (q . R_K) against c * s + z and one output rotation
 *   . R_V^T per head, which is the same quantity.  A request with no valid
 *   token gets zeros.
 *
 *   Workspace: call with workspace == NULL to receive the required size in
 *   *workspace_bytes (depends on desc dims and the current device) and
 *   return.  Otherwise workspace must be 256-byte aligned device memory of
 *   at least that size, zero-filled before its first use (cudaMemset); each
 *   call leaves it ready for the next one.  It holds per-call merge tickets
 *   and split partials, so two calls in flight at the same time need two
 *   workspaces.  Async.
 */
oscar_status oscar_decode_attention(const oscar_layer_desc* desc, const uint16_t* q,
                                    float* out, void* workspace, size_t* workspace_bytes,
                                    void* stream);

/*
 * oscar_decode_step - one decode step of a layer in one call, for a serving
 * loop that holds the step's inputs in host memory: [ZAKER] pipeline part
 * (demote the oldest recent token, write the new one, attend).
 *
 *   On `stream`, in this order: (1) if in_bytes > 0, bring in_bytes from
 *   host_in (pinned host memory) to dev_in (device), the staging range that
 *   q, new_k / new_v and the index arrays may point into; (2)
 *   oscar_quantize_append with the given arguments (nothing when n = 0);
 *   (3) oscar_decode_attention(desc, q, out, workspace, workspace_bytes);
 *   (4) if host_out is not NULL, copy out ([B][H_q][d] float32) to host_out
 *   (pinned host memory): when host_out is 16-byte aligned the decode kernel
 *   of step (3) writes it with the same stores as `out`, else a copy kernel
 *   follows.  The results are those of the separate calls.
 *   Step (1) is not a copy when it need not be: if q or an argument of (2)
 *   lies inside [dev_in, dev_in + in_bytes), host_in and dev_in are equal
 *   modulo 16 bytes, the per-token demotion kernel runs (new rows given, or
 *   n < 1024) and k_src / v_src lie outside that range, the kernels of (2)
 *   and (3) read those inputs straight from the same offsets of host_in
 *   and dev_in is left unwritten; otherwise a copy kernel fills dev_in.
 *   The copies run in the same launch chain as kernels: the GPU reads
 *   host_in and writes host_out directly (GB300's coherent CPU-GPU link), so
 *   both must be pinned host memory the device addresses at the same pointer
 *   (cudaHostAlloc / cudaMallocHost on a system with unified addressing);
 *   otherwise OSCAR_ERR_INVALID_ARG.  host_in is read anew on every call.
 *   Every argument of (2) and (3) is validated before (1) is issued: a
 *   rejected call copies and launches nothing.  in_bytes > 0 requires
 *   host_in and dev_in (OSCAR_ERR_INVALID_ARG otherwise); workspace must be
 *   given (OSCAR_ERR_WORKSPACE).  Async: host_in must not change until the
 *   stream has passed step (3), and host_out holds the output once the
 *   stream has passed step (4).
 *
 *   flags: 0, or OSCAR_STEP_OVERLAP_PREVIOUS: when no copy kernel of step
 *   (1) runs, step (2) is oscar_quantize_append_overlapped (its reads and
 *   arithmetic overlap the kernel before the call on `stream`), under that
 *   function's precondition on that kernel, which here covers new_k / new_v
 *   too (they are read before the wait as well); in a loop of
 *   oscar_decode_step calls that kernel is the previous call's decode (or
 *   its output copy), which qualifies as long as host_out and out overlap
 *   none of the inputs.
 *   Other bits: OSCAR_ERR_INVALID_ARG.
 */
#define OSCAR_STEP_OVERLAP_PREVIOUS 1u
oscar_status oscar_decode_step(const oscar_layer_desc* desc, const void* host_in, void* dev_in,
                               size_t in_bytes, uint16_t* k_src, uint16_t* v_src, int64_t src_rows,
                               int64_t row_stride, const int32_t* src_index, const int32_t* dst_req,
                               const int32_t* dst_pos, int32_t n, const uint16_t* new_k,
                               const uint16_t* new_v, const uint16_t* q, float* out,
                               void* workspace, size_t workspace_bytes, float* host_out,
                               uint32_t flags, void* stream);

/*
 * oscar_decode_attention_static - oscar_decode_attention for callers that
 * cannot allocate device memory.  The paper has no counterpart: this is a
 * deployment convenience of this library.
 *
 *   Some callers have no way to call cudaMalloc or to hand the library a
 *   workspace: code embedded in a host framework that owns every device
 *   allocation, or a latency-critical serving loop that forbids allocation
 *   after start-up.  This entry point computes exactly what
 *   oscar_decode_attention computes, but its workspace is a fixed array of
 *   OSCAR_STATIC_WORKSPACE_BYTES inside the library, reserved on every GPU
 *   that loads the library until the process exits.  It allocates nothing.
 *
 *   q, out and the cache are the caller's, as for oscar_decode_attention.
 *   Returns OSCAR_ERR_WORKSPACE when the problem needs more workspace than
 *   the fixed array holds (the size oscar_decode_attention reports for a
 *   NULL workspace must not exceed OSCAR_STATIC_WORKSPACE_BYTES; about 0.65
 *   MB for one 100k-token request with 8 KV heads and GQA 4).
 *
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current, and so does the first
 *   call after the device's context was replaced (cudaDeviceReset); make
 *   those calls before any stream capture.  Each call clears the part of the array that
 *   must start at zero, on `stream`, then launches.  Every call shares the
 *   one array and it keeps the last call's contents: calls whose work
 *   overlaps on the GPU (different streams, or concurrent host threads
 *   without stream ordering) race on it and must not be issued.
 */
#define OSCAR_STATIC_WORKSPACE_BYTES (8u << 20)

oscar_status oscar_decode_attention_static(const oscar_layer_desc* desc, const uint16_t* q,
                                           float* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* OSCAR_H_ */
