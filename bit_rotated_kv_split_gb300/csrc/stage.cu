// Host <-> device staging of a decode step's inputs and output through the
// SMs (GB300: the GPU addresses pinned host memory directly over the
// coherent CPU-GPU link), so the copies sit in the chain of programmatic
// dependent launches instead of breaking it as copy-engine transfers would.
//
// One launch copies `bytes` from src to dst: 16-byte loads and stores when
// both addresses allow it, bytes for the rest.  Source loads are
// cache-volatile (ld.global.cv), so data in host memory is fetched again on
// every call rather than served from a cached line.
#include "kernels.h"
#include "ptx.cuh"

namespace oscar {
namespace {

constexpr int kStageThreads = 256;

__global__ void __launch_bounds__(kStageThreads) stage_kernel(const uint8_t* src, uint8_t* dst, size_t bytes) {
  pdl_wait();                 // the previous kernel's reads and writes are done
  pdl_launch_dependents();
  const size_t tid = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t nth = size_t(gridDim.x) * blockDim.x;
  const bool vec = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0;
  const size_t n16 = vec ? bytes / 16 : 0;
  for (size_t i = tid; i < n16; i += nth) {
    const uint4 v = __ldcv(reinterpret_cast<const uint4*>(src) + i);
    reinterpret_cast<uint4*>(dst)[i] = v;
  }
  for (size_t i = n16 * 16 + tid; i < bytes; i += nth) dst[i] = __ldcv(src + i);
}

}  // namespace

cudaError_t launch_stage(const void* src, void* dst, size_t bytes, cudaStream_t stream) {
  if (bytes == 0) return cudaSuccess;
  const size_t units = (bytes + 15) / 16;
  const unsigned blocks = unsigned(std::min<size_t>((units + kStageThreads - 1) / kStageThreads, 64));
  return launch_pdl(stage_kernel, dim3(blocks), dim3(kStageThreads), 0, stream,
                    static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), bytes);
}

}  // namespace oscar
