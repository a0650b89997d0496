// Calibration covariance on the device: C = X^T X / n over bf16 rows.
//
// gist.science "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV
// Cache Quantization", Technical summary 2.1 and 2.2 A: the key rotation
// comes from the query covariance C_Q = Q^T Q and the value rotation from
// the score-weighted value covariance C_S = (S V)^T (S V); both are sums of
// outer products of calibration rows, i.e. one contraction over the rows.
//
// Split over the rows: CTA c takes rows [c R, (c + 1) R) and accumulates its
// 128 x 128 partial with mma.sync (bf16 in, fp32 accumulate; the products of
// bf16 values are exact), warp w holding output rows 16 w .. 16 w + 15.  Rows
// are staged 64 at a time in shared memory with a 272-byte pitch so that the
// eight row addresses of an ldmatrix hit eight bank groups, through a ring of
// four stages filled by cp.async (three passes in flight while one is
// computed).  A second kernel adds the partials in a fixed order and divides
// by n, so the result does not depend on scheduling.
#include "kernels.h"
#include "ptx.cuh"

namespace oscar {
namespace {

constexpr int kCovRows = 2048;        // rows per CTA
constexpr int kStageRows = 64;        // rows staged per pass
constexpr int kPitch = 272;           // bytes between staged rows (256 + 16)
constexpr int kCovWarps = 8;
constexpr int kCovStages = 4;         // passes in flight (cp.async ring)
constexpr int kStageBytes = kStageRows * kPitch;
constexpr int kCovSmem = kCovStages * kStageBytes;

__global__ void __launch_bounds__(kCovWarps * 32) covariance_partial_kernel(const uint16_t* __restrict__ x,
                                                                           int64_t n, int64_t ld, float* part) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ __align__(128) uint8_t xs[];   // kCovStages x [kStageRows][kPitch]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const int64_t r_begin = int64_t(blockIdx.x) * kCovRows;
  const int64_t r_end = min(r_begin + kCovRows, n);
  const int n_pass = int((r_end - r_begin + kStageRows - 1) / kStageRows);
  // pass k's 64 rows x 16 chunks of 8 bf16 into stage k % kCovStages: four
  // 16-byte copies per thread, zeros past the end; every thread commits one
  // group per pass (empty past the last), so the group counts stay aligned
  auto issue = [&](int k) {
    if (k < n_pass) {
      const int64_t r0 = r_begin + int64_t(k) * kStageRows;
      uint8_t* buf = xs + (k % kCovStages) * kStageBytes;
#pragma unroll
      for (int u = 0; u < kStageRows * 16 / (kCovWarps * 32); ++u) {
        const int idx = tid + u * kCovWarps * 32;
        const int row = idx >> 4, ch = idx & 15;
        const bool ok = r0 + row < r_end;
        const uint16_t* src = x + (ok ? (r0 + row) * ld : 0) + 8 * ch;
        cp_async16(buf + row * kPitch + ch * 16, src, ok ? 16u : 0u);
      }
    }
    cp_async_commit();
  };
  float acc[16][4];
#pragma unroll
  for (int t = 0; t < 16; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
  // ldmatrix row addresses: matrix m = lane / 8, row lane % 8
  const int m = lane >> 3, mr = lane & 7;
#pragma unroll
  for (int k = 0; k < kCovStages - 1; ++k) issue(k);
  for (int k = 0; k < n_pass; ++k) {
    cp_async_wait<kCovStages - 2>();   // this thread's copies of pass k have landed
    __syncthreads();                   // everyone's have; pass k - 1 is computed by all warps
    issue(k + kCovStages - 1);         // into the stage pass k - 1 used
    const uint8_t* st = xs + (k % kCovStages) * kStageBytes;
#pragma unroll
    for (int k0 = 0; k0 < kStageRows; k0 += 16) {
      // A = (X block)^T for output rows 16 warp ..: matrices (i block, r
      // block) = (m & 1, m >> 1), read transposed from X rows
      uint32_t a[4];
      ldmatrix_x4_trans(a, st + (k0 + 8 * (m >> 1) + mr) * kPitch + (16 * warp + 8 * (m & 1)) * 2);
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        // B for output columns 16 np ..: matrices (r block, n tile) =
        // (m & 1, m >> 1), transposed so lane t holds rows 2 tig, +1
        uint32_t b[4];
        ldmatrix_x4_trans(b, st + (k0 + 8 * (m & 1) + mr) * kPitch + (16 * np + 8 * (m >> 1)) * 2);
        mma_bf16(acc[2 * np], a[0], a[1], a[2], a[3], b[0], b[1]);
        mma_bf16(acc[2 * np + 1], a[0], a[1], a[2], a[3], b[2], b[3]);
      }
    }
  }
  cp_async_wait<0>();   // (only empty groups remain)
  // partial [128][128]: accumulator tile t covers columns 8 t .. 8 t + 7
  float* pc = part + int64_t(blockIdx.x) * kHeadDim * kHeadDim;
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    const int i = 16 * warp + gid, j = 8 * t + 2 * tig;
    *reinterpret_cast<float2*>(pc + i * kHeadDim + j) = make_float2(acc[t][0], acc[t][1]);
    *reinterpret_cast<float2*>(pc + (i + 8) * kHeadDim + j) = make_float2(acc[t][2], acc[t][3]);
  }
}

// Entry e of C: the partials in chunk order, as eight interleaved running
// sums (chunks k = 8 i + j into sum j) added in order at the end, so eight
// loads are in flight at a time; the order is fixed, so the result does not
// depend on scheduling.
__global__ void covariance_reduce_kernel(const float* part, int chunks, double inv_n, float* c) {
  pdl_wait();
  pdl_launch_dependents();
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= kHeadDim * kHeadDim) return;
  float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int k = 0;
  for (; k + 8 <= chunks; k += 8) {
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j] += part[int64_t(k + j) * kHeadDim * kHeadDim + e];
  }
  for (int j = 0; k + j < chunks; ++j) s[j] += part[int64_t(k + j) * kHeadDim * kHeadDim + e];
  const float t = ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
  c[e] = float(double(t) * inv_n);
}

}  // namespace

size_t covariance_workspace_bytes(int64_t n) {
  const int64_t chunks = (n + kCovRows - 1) / kCovRows;
  return size_t(chunks) * kHeadDim * kHeadDim * sizeof(float);
}

cudaError_t launch_covariance(const uint16_t* x, int64_t n, int64_t ld, float* c, void* workspace,
                              cudaStream_t stream) {
  const int64_t chunks = (n + kCovRows - 1) / kCovRows;
  if (chunks < 1 || chunks > 0x7fffffff) return cudaErrorInvalidValue;
  float* part = static_cast<float*>(workspace);
  cudaError_t e = set_smem_limit<covariance_partial_kernel>(kCovSmem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(covariance_partial_kernel, dim3(unsigned(chunks)), dim3(kCovWarps * 32), size_t(kCovSmem), stream, x,
                 n, ld, part);
  if (e != cudaSuccess) return e;
  return launch_pdl(covariance_reduce_kernel, dim3((kHeadDim * kHeadDim + 255) / 256), dim3(256), 0, stream,
                    static_cast<const float*>(part), int(chunks), 1.0 / double(n), c);
}

}  // namespace oscar
