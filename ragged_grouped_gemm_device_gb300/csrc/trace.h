// Host-side NVTX ranges around the C-ABI entry points: each call opens a range named after the
// entry point for as long as it validates its arguments and enqueues its kernels, so profilers
// (ncu --nvtx, nsys) can attribute every kernel launch to the call that issued it. NVTX is
// header-only; without a tool attached a range costs one check of an initialised flag.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace moe {

struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace moe

#define MOE_TRACE_CALL() ::moe::NvtxRange moe_trace_range_(__func__)
