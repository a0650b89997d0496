// NVTX ranges around the library's C-ABI calls: a profiler or tracer that
// attaches through NVTX (Nsight Systems, ncu's NVTX filters) sees each call
// as a named range on the calling thread.  NVTX v3 is header-only; without
// an attached tool a range costs a load and a branch.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace oscar {

struct TraceRange {
  explicit TraceRange(const char* name) { nvtxRangePushA(name); }
  ~TraceRange() { nvtxRangePop(); }
  TraceRange(const TraceRange&) = delete;
  TraceRange& operator=(const TraceRange&) = delete;
};

}  // namespace oscar

// One range covering the enclosing C-ABI function, named after it.
#define OSCAR_TRACE_CALL() ::oscar::TraceRange oscar_trace_range_(__func__)
