// Bounds checks of the debug build (nvcc -DMOE_GG_DEBUG: libmoe_gg_debug.so).
//
// Each kernel translation unit checks its data-dependent global accesses -- the indices that come
// from offsets, slot maps or tile decoding rather than from the launch shape -- against the extent
// of the buffer they address. A failed check skips the access (or, for a copy whose bytes a
// barrier expects, redirects it to the buffer's first element so that the count still balances)
// and records the site, the index and its bound in the translation unit's debug record, which
// moe_debug_report() reads back. Release builds compile every check to `true`.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "internal.h"  // DbgRecord, DbgSite

namespace moe {

#ifdef MOE_GG_DEBUG

static __device__ DbgRecord g_moe_dbg = {0, -1, 0, 0};

static __device__ __noinline__ bool dbg_fail(int site, long long index, long long limit) {
  atomicOr(&g_moe_dbg.mask, 1 << site);
  if (atomicCAS(&g_moe_dbg.site, -1, site) == -1) {
    g_moe_dbg.index = index;
    g_moe_dbg.limit = limit;
  }
  return false;
}

// true when 0 <= i < lim; else records the failure and yields false
#define MOE_DBG_IN(site, i, lim)                                                              \
  ((static_cast<long long>(i) >= 0 && static_cast<long long>(i) < static_cast<long long>(lim)) || \
   ::moe::dbg_fail((site), static_cast<long long>(i), static_cast<long long>(lim)))

// Host: merge this translation unit's record into *acc (the first failing site recorded wins)
// and clear it when `reset`.
static cudaError_t dbg_collect_here(DbgRecord* acc, bool reset) {
  DbgRecord r;
  cudaError_t e = cudaMemcpyFromSymbol(&r, g_moe_dbg, sizeof(r));
  if (e != cudaSuccess) return e;
  acc->mask |= r.mask;
  if (acc->site < 0 && r.site >= 0) {
    acc->site = r.site;
    acc->index = r.index;
    acc->limit = r.limit;
  }
  if (reset) {
    const DbgRecord z = {0, -1, 0, 0};
    e = cudaMemcpyToSymbol(g_moe_dbg, &z, sizeof(z));
  }
  return e;
}

#define MOE_DBG_DEFINE_COLLECTOR(fn) \
  cudaError_t fn(::moe::DbgRecord* acc, bool reset) { return ::moe::dbg_collect_here(acc, reset); }

#else

#define MOE_DBG_IN(site, i, lim) true
#define MOE_DBG_DEFINE_COLLECTOR(fn) \
  cudaError_t fn(::moe::DbgRecord*, bool) { return cudaSuccess; }

#endif

}  // namespace moe
