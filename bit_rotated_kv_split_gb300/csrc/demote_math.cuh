// Quantisation of one token-head vector by one warp, shared by the per-token
// demotion kernel and the one-kernel decode step, so that both write the
// same codes and (scale, zero) pairs bit for bit.
//
// myzaker.com OSCAR article, part "从离线校准到在线推理的 pipeline" (scale/zero
// point, four 2-bit codes per byte); gist.science "OSCAR: Offline Spectral
// Covariance-Aware Rotation for 2-bit KV Cache Quantization", Technical
// summary 2.2 A (clip to the per-layer threshold).
#pragma once

#include <cuda_fp16.h>

#include "kernels.h"

namespace oscar {

// Lane l holds the clipped rotated values v[c] of code positions 4 l + c;
// position 4 l + c belongs to quantisation group (4 (l & 1) + c) / (8 / NG).
// Each group's (min, max) is reduced over the warp and gives its fp16
// scale = fp16((max - min) / 3) and zero = fp16(min); the lane's code byte
// holds code c in bits 2 c: rint((v - zero) / scale) clamped to [0, 3], or
// with kLevels the number of codebook thresholds `thr` strictly below
// (v - zero) / scale; 0 when the scale is 0.  Every lane of the warp calls it.
template <int NG, bool kLevels>
__device__ __forceinline__ uint32_t quantize_lane(const float (&v)[4], int lane, const float* thr,
                                                  __half (&s16)[NG], __half (&z16)[NG]) {
  constexpr int kSpan = 8 / NG;
  const bool odd = lane & 1;
  float s[NG], z[NG];
#pragma unroll
  for (int q = 0; q < NG; ++q) {
    float mn = INFINITY, mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const bool in = odd ? ((4 + c) / kSpan == q) : (c / kSpan == q);
      mn = in ? fminf(mn, v[c]) : mn;
      mx = in ? fmaxf(mx, v[c]) : mx;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    s16[q] = __float2half_rn(__fdiv_rn(mx - mn, 3.0f));
    z16[q] = __float2half_rn(mn);
    s[q] = __half2float(s16[q]);
    z[q] = __half2float(z16[q]);
  }
  uint32_t byte = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const float sc = odd ? s[(4 + c) / kSpan] : s[c / kSpan];
    const float zc = odd ? z[(4 + c) / kSpan] : z[c / kSpan];
    uint32_t code = 0u;
    if (sc > 0.f) {
      const float u = __fdiv_rn(v[c] - zc, sc);
      if constexpr (kLevels) {
        code = uint32_t(u > thr[0]) + uint32_t(u > thr[1]) + uint32_t(u > thr[2]);
      } else {
        code = uint32_t(fminf(fmaxf(rintf(u), 0.f), 3.f));
      }
    }
    byte |= code << (2 * c);
  }
  return byte;
}

}  // namespace oscar
