// ddp_trace.h -- an NVTX range around every C-ABI call, so that a timeline
// tool (nsys, or ncu's NVTX filters) shows which library call issued which
// kernels.  NVTX v3 is header-only; with no tool attached a range costs a
// function-pointer check.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace ddpk {

struct TraceScope {
    explicit TraceScope(const char* name) { nvtxRangePushA(name); }
    ~TraceScope() { nvtxRangePop(); }
    TraceScope(const TraceScope&) = delete;
    TraceScope& operator=(const TraceScope&) = delete;
};

}  // namespace ddpk

#define DDP_TRACE_CALL() ::ddpk::TraceScope ddp_trace_call_(__func__)
