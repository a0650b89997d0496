// Score-weighted value covariance on the device: C_S = (S V)^T (S V) / N with
// S = row-softmax(Q K^T / sqrt(d)).
//
// gist.science "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV
// Cache Quantization", Technical summary 2.1 and 2.2 A: the value rotation
// is the eigenbasis of the covariance of the attention-weighted values S V
// over calibration queries, keys and values.
//
// Two steps.  (1) sv_rows_kernel: the rows of S V, one CTA per 64 queries
// (four warps of 16), keys in tiles of 64 staged in shared memory.  Q K^T on
// the tensor cores (bf16 in: the products are exact; fp32 accumulate), an
// online softmax in fp32 per query row, and P V on the tensor cores with P
// split into bf16 hi + lo parts (about 16 bits) against the bf16 values; the
// rows are normalised and written in fp32.  (2) sv_covariance_kernel: fp32
// partials of (S V)^T (S V) over chunks of 256 rows, each thread an 8 x 8
// block of the 128 x 128 result; the partials are then added in chunk order
// (the result does not depend on scheduling) and divided by N.
#include <cfloat>

#include "kernels.h"
#include "ptx.cuh"

namespace oscar {
namespace {

constexpr int kSvRows = 64;       // queries per CTA (4 warps x 16)
constexpr int kSvKeys = 64;       // keys per staged tile
constexpr int kSvPitch = 272;     // bytes between staged rows (256 + 16: ldmatrix rows in 8 bank groups)
constexpr int kCovChunk = 256;    // rows per covariance partial
constexpr int kCovStage = 32;     // rows staged per pass

__device__ __forceinline__ uint32_t bf16x2_of(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(128) sv_rows_kernel(const uint16_t* __restrict__ q, int64_t n_q,
                                                      const uint16_t* __restrict__ k,
                                                      const uint16_t* __restrict__ v, int64_t n_k, int64_t ld,
                                                      float scale_log2, float* __restrict__ sv) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ __align__(128) uint8_t ks[kSvKeys * kSvPitch];
  __shared__ __align__(128) uint8_t vs[kSvKeys * kSvPitch];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const int64_t row0 = int64_t(blockIdx.x) * kSvRows + 16 * warp;
  const int64_t ra = row0 + gid, rb = row0 + gid + 8;
  // A fragments of the warp's 16 query rows, 8 K-steps of 16 dims
  uint32_t qa[8][4];
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const int c = 16 * kk + 2 * tig;
    qa[kk][0] = ra < n_q ? *reinterpret_cast<const uint32_t*>(q + ra * ld + c) : 0u;
    qa[kk][1] = rb < n_q ? *reinterpret_cast<const uint32_t*>(q + rb * ld + c) : 0u;
    qa[kk][2] = ra < n_q ? *reinterpret_cast<const uint32_t*>(q + ra * ld + c + 8) : 0u;
    qa[kk][3] = rb < n_q ? *reinterpret_cast<const uint32_t*>(q + rb * ld + c + 8) : 0u;
  }
  float o[16][4];
#pragma unroll
  for (int t = 0; t < 16; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};   // rows gid, gid + 8
  const int mm = lane >> 3, mr = lane & 7;                   // ldmatrix matrix / row
  for (int64_t k0 = 0; k0 < n_k; k0 += kSvKeys) {
    __syncthreads();   // the previous tile's reads are done
    // 64 keys x 16 chunks of 8 bf16, for K and V: 8 + 8 per thread; zero
    // past the last key
#pragma unroll
    for (int u = 0; u < kSvKeys * 16 / 128; ++u) {
      const int idx = tid + 128 * u, row = idx >> 4, ch = idx & 15;
      uint4 kv = make_uint4(0u, 0u, 0u, 0u), vv = kv;
      if (k0 + row < n_k) {
        kv = __ldg(reinterpret_cast<const uint4*>(k + (k0 + row) * ld) + ch);
        vv = __ldg(reinterpret_cast<const uint4*>(v + (k0 + row) * ld) + ch);
      }
      *reinterpret_cast<uint4*>(ks + row * kSvPitch + ch * 16) = kv;
      *reinterpret_cast<uint4*>(vs + row * kSvPitch + ch * 16) = vv;
    }
    __syncthreads();
    // S = Q K^T for 64 keys: n-tile t holds keys 8 t .. 8 t + 7 (B = K rows,
    // read untransposed: lane t holds K[key gid][dims 2 tig, 2 tig + 1])
    float s[8][4];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
      const uint8_t* krow = ks + (8 * t + gid) * kSvPitch + 4 * tig;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(krow + 32 * kk);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(krow + 32 * kk + 16);
        mma_bf16(s[t], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
      }
    }
    // scores in log2 units; keys past the end get -inf
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int t = 0; t < 8; ++t) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int64_t key = k0 + 8 * t + 2 * tig + (c & 1);
        s[t][c] = key < n_k ? s[t][c] * scale_log2 : -INFINITY;
        tmax[c >> 1] = fmaxf(tmax[c >> 1], s[t][c]);
      }
    }
    float f[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 1));
      tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 2));
      const float mn = fmaxf(m[r], tmax[r]);
      f[r] = m[r] == -INFINITY ? 0.f : exp2f(m[r] - mn);
      m[r] = mn;
      l[r] *= f[r];
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      o[t][0] *= f[0];
      o[t][1] *= f[0];
      o[t][2] *= f[1];
      o[t][3] *= f[1];
    }
    // P = 2^(s - m), summed per row; as A fragments of the P V contraction
    // (K-step j: keys 16 j .. 16 j + 15 = n-tiles 2 j, 2 j + 1), each a
    // bf16 hi part and the bf16 rounding of the remainder
    uint32_t ph[4][4], pl[4][4];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      float p[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        p[c] = s[t][c] == -INFINITY ? 0.f : exp2f(s[t][c] - m[c >> 1]);
        l[c >> 1] += p[c];
      }
      const uint32_t h01 = bf16x2_of(p[0], p[1]), h23 = bf16x2_of(p[2], p[3]);
      const uint32_t l01 = bf16x2_of(p[0] - bf16_lo(h01), p[1] - bf16_hi(h01));
      const uint32_t l23 = bf16x2_of(p[2] - bf16_lo(h23), p[3] - bf16_hi(h23));
      const int j = t >> 1, e = t & 1;
      ph[j][2 * e] = h01;       // row gid (a0 | a2)
      ph[j][2 * e + 1] = h23;   // row gid + 8 (a1 | a3)
      pl[j][2 * e] = l01;
      pl[j][2 * e + 1] = l23;
    }
    // O += P V: B = V rows transposed by ldmatrix (lane t: rows 2 tig, +1
    // of output column gid); n-tile pair np covers dims 16 np .. 16 np + 15
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        uint32_t b[4];
        ldmatrix_x4_trans(b, vs + (16 * j + 8 * (mm & 1) + mr) * kSvPitch + (16 * np + 8 * (mm >> 1)) * 2);
        mma_bf16(o[2 * np], ph[j][0], ph[j][1], ph[j][2], ph[j][3], b[0], b[1]);
        mma_bf16(o[2 * np], pl[j][0], pl[j][1], pl[j][2], pl[j][3], b[0], b[1]);
        mma_bf16(o[2 * np + 1], ph[j][0], ph[j][1], ph[j][2], ph[j][3], b[2], b[3]);
        mma_bf16(o[2 * np + 1], pl[j][0], pl[j][1], pl[j][2], pl[j][3], b[2], b[3]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
  }
  const float ia = l[0] > 0.f ? 1.f / l[0] : 0.f, ib = l[1] > 0.f ? 1.f / l[1] : 0.f;
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    const int c = 8 * t + 2 * tig;
    if (ra < n_q) *reinterpret_cast<float2*>(sv + ra * kHeadDim + c) = make_float2(o[t][0] * ia, o[t][1] * ia);
    if (rb < n_q) *reinterpret_cast<float2*>(sv + rb * kHeadDim + c) = make_float2(o[t][2] * ib, o[t][3] * ib);
  }
}

// Partial (S V)^T (S V) of rows [c kCovChunk, (c + 1) kCovChunk): thread
// (bi, bj) accumulates the 8 x 8 block rows 8 bi .., columns 8 bj .. in fp32
// over the rows in order.
__global__ void __launch_bounds__(256) sv_covariance_kernel(const float* __restrict__ x, int64_t n,
                                                            float* __restrict__ part) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ __align__(16) float xs[kCovStage][kHeadDim];
  const int tid = threadIdx.x, bi = tid >> 4, bj = tid & 15;
  const int64_t r_begin = int64_t(blockIdx.x) * kCovChunk;
  const int64_t r_end = min(r_begin + kCovChunk, n);
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  for (int64_t r0 = r_begin; r0 < r_end; r0 += kCovStage) {
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kCovStage * kHeadDim / 4 / 256; ++u) {
      const int idx = tid + 256 * u, row = idx / (kHeadDim / 4), c4 = idx % (kHeadDim / 4);
      float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r0 + row < r_end) val = reinterpret_cast<const float4*>(x + (r0 + row) * kHeadDim)[c4];
      reinterpret_cast<float4*>(xs[row])[c4] = val;
    }
    __syncthreads();
    const int64_t left = r_end - r0;
    const int rows = left < kCovStage ? int(left) : kCovStage;
    for (int r = 0; r < rows; ++r) {
      const float4 a0 = reinterpret_cast<const float4*>(xs[r] + 8 * bi)[0];
      const float4 a1 = reinterpret_cast<const float4*>(xs[r] + 8 * bi)[1];
      const float4 b0 = reinterpret_cast<const float4*>(xs[r] + 8 * bj)[0];
      const float4 b1 = reinterpret_cast<const float4*>(xs[r] + 8 * bj)[1];
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
    }
  }
  float* pc = part + int64_t(blockIdx.x) * kHeadDim * kHeadDim;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float4* dst = reinterpret_cast<float4*>(pc + (8 * bi + i) * kHeadDim + 8 * bj);
    dst[0] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    dst[1] = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
  }
}

__global__ void sv_reduce_kernel(const float* part, int chunks, double inv_n, float* c) {
  pdl_wait();
  pdl_launch_dependents();
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= kHeadDim * kHeadDim) return;
  float s = 0.f;
  for (int k = 0; k < chunks; ++k) s += part[int64_t(k) * kHeadDim * kHeadDim + e];
  c[e] = float(double(s) * inv_n);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

size_t value_covariance_workspace_bytes(int64_t n_q) {
  const int64_t chunks = (n_q + kCovChunk - 1) / kCovChunk;
  return align256(size_t(n_q) * kHeadDim * sizeof(float)) + size_t(chunks) * kHeadDim * kHeadDim * sizeof(float);
}

cudaError_t launch_value_covariance(const uint16_t* q, int64_t n_q, const uint16_t* k, const uint16_t* v,
                                    int64_t n_k, int64_t ld, float* c, void* workspace, cudaStream_t stream) {
  const int64_t blocks = (n_q + kSvRows - 1) / kSvRows;
  const int64_t chunks = (n_q + kCovChunk - 1) / kCovChunk;
  if (blocks < 1 || blocks > 0x7fffffff || chunks > 0x7fffffff) return cudaErrorInvalidValue;
  float* sv = static_cast<float*>(workspace);
  float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                         align256(size_t(n_q) * kHeadDim * sizeof(float)));
  const float scale_log2 = 1.4426950408889634f / sqrtf(float(kHeadDim));
  cudaError_t e = launch_pdl(sv_rows_kernel, dim3(unsigned(blocks)), dim3(128), 0, stream, q, n_q, k, v, n_k, ld,
                             scale_log2, sv);
  if (e != cudaSuccess) return e;
  e = launch_pdl(sv_covariance_kernel, dim3(unsigned(chunks)), dim3(256), 0, stream,
                 static_cast<const float*>(sv), n_q, part);
  if (e != cudaSuccess) return e;
  return launch_pdl(sv_reduce_kernel, dim3((kHeadDim * kHeadDim + 255) / 256), dim3(256), 0, stream,
                    static_cast<const float*>(part), int(chunks), 1.0 / double(n_q), c);
}

}  // namespace oscar
