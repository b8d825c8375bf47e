// call_range.h -- a named NVTX range around each call of the C ABI, so that a profiler
// (Nsight Systems, or ncu filtering by NVTX range) shows where a call's host work and launches
// happen.  Header-only NVTX (version 3, shipped with the CUDA toolkit); without an attached tool
// a range costs a few nanoseconds.
#pragma once
#include <nvtx3/nvToolsExt.h>

namespace sinkattn {

struct CallRange {
    explicit CallRange(const char* name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
    CallRange(const CallRange&) = delete;
    CallRange& operator=(const CallRange&) = delete;
};

}  // namespace sinkattn
