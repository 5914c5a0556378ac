// Host-side NVTX ranges around the C-ABI entry points: each call opens a range named after the
// entry point for as long as it validates its arguments and enqueues its kernels, so profilers
// (ncu --nvtx, nsys) can attribute every kernel launch to the call that issued it. NVTX is
// header-only; without a tool attached a range costs one check of an initialised flag.
//
// In the debug build (-DMOE_GG_DEBUG) the same scope also waits for the call's stream when the
// entry point returns, unless that stream is being captured, and records a CUDA error found
// then under the call's name (moe_debug_report).
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "../../include/moe_gg.h"

namespace moe {

#ifdef MOE_GG_DEBUG
void dbg_after_call(const char* name, cudaStream_t stream);  // moe_gg.cu
#endif

class CallScope {
 public:
  CallScope(const char* name, moe_stream_t stream) : name_(name), stream_(stream) { nvtxRangePushA(name); }
  ~CallScope() {
    nvtxRangePop();
#ifdef MOE_GG_DEBUG
    dbg_after_call(name_, reinterpret_cast<cudaStream_t>(stream_));
#endif
  }
  CallScope(const CallScope&) = delete;
  CallScope& operator=(const CallScope&) = delete;

 private:
  [[maybe_unused]] const char* name_;
  [[maybe_unused]] moe_stream_t stream_;
};

}  // namespace moe

// every entry point names its stream argument `stream`
#define MOE_TRACE_CALL() ::moe::CallScope moe_trace_scope_(__func__, stream)
