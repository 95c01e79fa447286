// zero_trace.h -- NVTX ranges around the library's entry points, so a profiler
// (ncu --nvtx, Nsight Systems) can attribute kernels and host work to the call
// that issued them.  NVTX v3 is header-only: with no tool attached a range costs
// a check of a function pointer.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace zero {

struct TraceRange {
    explicit TraceRange(const char* name) { nvtxRangePushA(name); }
    ~TraceRange() { nvtxRangePop(); }
    TraceRange(const TraceRange&) = delete;
    TraceRange& operator=(const TraceRange&) = delete;
};

}  // namespace zero
