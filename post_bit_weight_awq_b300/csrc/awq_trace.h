// Tracing: every entry point of the library that enqueues GPU work opens an
// NVTX range named after itself for the duration of the call (host time), so
// a profiler can attribute the kernels it launches to the API call (for ncu:
// --nvtx --nvtx-include "awq_search_layer/"). NVTX costs a branch per call
// when no tool is attached.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace awq {

struct TraceRange {
  explicit TraceRange(const char* name) { nvtxRangePushA(name); }
  ~TraceRange() { nvtxRangePop(); }
  TraceRange(const TraceRange&) = delete;
  TraceRange& operator=(const TraceRange&) = delete;
};

}  // namespace awq

#define AWQ_TRACE(name) ::awq::TraceRange awq_trace_range_(name)
