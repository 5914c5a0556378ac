// Route histogram, cumulative offsets, stable placement and inverse map, on the device.
//
// "Section 09: Grouped GEMM", Fig. 37 steps 1-2 and §9.3: the route histogram and the int32
// cumulative offsets are produced on the GPU, so no count crosses to the host. "grouped_mm"
// agent doc: rows are sorted by expert into contiguous blocks after dropping ids outside
// [0, E), and an inverse map of sorted positions per (token, slot) replaces the scatter-add.
//
// Three launches, all deterministic (no order-dependent atomics):
//   1. route_hist_kernel    each warp owns a contiguous chunk of 256 slots and counts its
//                           experts with warp match (one leader per expert per 32 slots);
//                           per-warp histograms go to the workspace [W, E].
//   2. route_colscan_kernel per expert, the exclusive prefix of the per-warp counts in warp
//                           order (in place) and the expert's total count.
//   3. route_scatter_kernel every block scans the counts into segment starts (block 0 also
//                           writes the offsets); each warp then walks its chunk again and
//                           places slot i of expert e at start[e] + (earlier warps' count of
//                           e) + (earlier slots of e in this chunk). Slots keep flat-index
//                           order inside a segment.
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "trace.h"

namespace moe {
namespace {

constexpr int CHUNK = 256;          // slots per warp chunk
constexpr int WARPS_PER_BLOCK = 8;  // 256-thread blocks
constexpr int MAX_E = 1024;

__global__ void __launch_bounds__(256) route_hist_kernel(const int32_t* __restrict__ ids, int n,
                                                         int E, int W,
                                                         int32_t* __restrict__ hist) {
  extern __shared__ int32_t sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w = blockIdx.x * WARPS_PER_BLOCK + warp;
  int32_t* hw = sh + warp * E;
  for (int e = lane; e < E; e += 32) hw[e] = 0;
  __syncwarp();
  if (w >= W) return;
  const int base = w * CHUNK;
#pragma unroll 1
  for (int s = 0; s < CHUNK; s += 32) {
    const int i = base + s + lane;
    const int e = (i < n) ? __ldg(ids + i) : -1;
    const bool valid = (e >= 0) && (e < E);
    const int key = valid ? e : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    if (valid && lane == __ffs(peers) - 1) hw[e] += __popc(peers);
    __syncwarp();
  }
  int32_t* out = hist + static_cast<size_t>(w) * E;
  for (int e = lane; e < E; e += 32) out[e] = hw[e];
}

// block: 32 experts (x) by 32 warp groups (y)
__global__ void __launch_bounds__(1024) route_colscan_kernel(int32_t* __restrict__ hist, int W,
                                                             int E, int32_t* __restrict__ counts) {
  __shared__ int32_t part[32][33];
  const int ex = threadIdx.x & 31, wg = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + ex;
  const int per = (W + 31) / 32;
  const int w0 = min(W, wg * per), w1 = min(W, w0 + per);
  int sum = 0;
  if (e < E)
    for (int w = w0; w < w1; ++w) sum += hist[static_cast<size_t>(w) * E + e];
  part[wg][ex] = sum;
  __syncthreads();
  if (wg == 0) {
    int run = 0;
    for (int g = 0; g < 32; ++g) {
      const int v = part[g][ex];
      part[g][ex] = run;
      run += v;
    }
    if (e < E) counts[e] = run;
  }
  __syncthreads();
  int run = part[wg][ex];
  if (e < E)
    for (int w = w0; w < w1; ++w) {
      const size_t at = static_cast<size_t>(w) * E + e;
      const int c = hist[at];
      hist[at] = run;
      run += c;
    }
}

// Exclusive scan of counts[0..E) into start[0..E], start[E] = M (block-wide, E <= 1024).
__device__ void block_scan_counts(const int32_t* counts, int E, int32_t* start) {
  __shared__ int32_t warp_tot[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  int carry = 0;
  for (int base = 0; base < E; base += blockDim.x) {
    const int e = base + threadIdx.x;
    int v = (e < E) ? counts[e] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int nb = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += nb;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int t = (lane < nwarps) ? warp_tot[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int nb = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += nb;
      }
      if (lane < nwarps) warp_tot[lane] = t;  // inclusive over warps
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_tot[warp - 1] : 0);
    if (e < E) start[e] = carry + before + incl - v;
    carry += warp_tot[nwarps - 1];
    __syncthreads();
  }
  if (threadIdx.x == 0) start[E] = carry;
  __syncthreads();
}

__global__ void __launch_bounds__(256) route_scatter_kernel(
    const int32_t* __restrict__ ids, int n, int E, int W, const int32_t* __restrict__ hist,
    const int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ sorted_src, int32_t* __restrict__ inv_map) {
  extern __shared__ int32_t sh[];
  int32_t* start = sh;                 // E + 1
  int32_t* run_all = sh + (E + 1);     // WARPS_PER_BLOCK x E
  block_scan_counts(counts, E, start);
  const int M = start[E];
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e < E; e += blockDim.x) offsets[e] = start[e + 1];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w = blockIdx.x * WARPS_PER_BLOCK + warp;
  if (w < W) {
    int32_t* run = run_all + warp * E;
    const int32_t* hw = hist + static_cast<size_t>(w) * E;
    for (int e = lane; e < E; e += 32) run[e] = start[e] + hw[e];
    __syncwarp();
    const int base = w * CHUNK;
#pragma unroll 1
    for (int s = 0; s < CHUNK; s += 32) {
      const int i = base + s + lane;
      if (base + s >= n) break;  // warp-uniform
      const int e = (i < n) ? __ldg(ids + i) : -1;
      const bool valid = (e >= 0) && (e < E);
      const int key = valid ? e : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, key);
      if (valid) {
        const int pos = run[e] + __popc(peers & ((1u << lane) - 1u));
        if (MOE_DBG_IN(DBG_ROUTE_POS, pos, n)) {
          sorted_src[pos] = i;
          inv_map[i] = pos;
        }
      } else if (i < n) {
        inv_map[i] = -1;
      }
      __syncwarp();
      if (valid && lane == __ffs(peers) - 1) run[e] += __popc(peers);
      __syncwarp();
    }
  }
  // rows past the final offset hold no slot
  const int stride = gridDim.x * blockDim.x;
  for (long long p = M + static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; p < n; p += stride)
    sorted_src[p] = -1;
}

}  // namespace

MOE_DBG_DEFINE_COLLECTOR(dbg_collect_route)

size_t route_workspace_bytes(long long n, int E) {
  const long long W = (n + CHUNK - 1) / CHUNK;
  const size_t bytes = static_cast<size_t>(W) * static_cast<size_t>(E) * sizeof(int32_t);
  return (bytes + 255) & ~static_cast<size_t>(255);
}

moe_status_t launch_route(const int32_t* ids, int n, int E, int32_t* counts, int32_t* offsets,
                          int32_t* sorted_src, int32_t* inv_map, void* ws, cudaStream_t s) {
  if (E < 1 || E > MAX_E) return MOE_ERR_UNSUPPORTED_SHAPE;
  const int W = static_cast<int>((static_cast<long long>(n) + CHUNK - 1) / CHUNK);  // n < 2^31
  int32_t* hist = static_cast<int32_t*>(ws);
  if (W == 0) {
    // no slots: zero counts and offsets
    cudaError_t err = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s);
    if (err == cudaSuccess) err = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * E, s);
    return err == cudaSuccess ? MOE_OK : cuda_fail(err);
  }
  const int blocks = (W + WARPS_PER_BLOCK - 1) / WARPS_PER_BLOCK;
  const size_t sh_hist = sizeof(int32_t) * WARPS_PER_BLOCK * E;
  const size_t sh_scatter = sizeof(int32_t) * ((E + 1) + WARPS_PER_BLOCK * E);
  cudaError_t aerr = ensure_max_dynamic_smem(reinterpret_cast<const void*>(route_hist_kernel),
                                             static_cast<int>(sizeof(int32_t) * WARPS_PER_BLOCK * MAX_E));
  if (aerr == cudaSuccess)
    aerr = ensure_max_dynamic_smem(reinterpret_cast<const void*>(route_scatter_kernel),
                                   static_cast<int>(sizeof(int32_t) * ((MAX_E + 1) + WARPS_PER_BLOCK * MAX_E)));
  if (aerr != cudaSuccess) return cuda_fail(aerr);
  route_hist_kernel<<<blocks, 256, sh_hist, s>>>(ids, n, E, W, hist);
  route_colscan_kernel<<<(E + 31) / 32, 1024, 0, s>>>(hist, W, E, counts);
  route_scatter_kernel<<<blocks, 256, sh_scatter, s>>>(ids, n, E, W, hist, counts, offsets,
                                                      sorted_src, inv_map);
  const cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? MOE_OK : cuda_fail(err);
}

}  // namespace moe

// ---------------------------------------------------------------------------------------------
// moe_route_offsets without a caller workspace, for callers that cannot allocate device memory
// (see include/moe_gg.h). The per-warp histogram scratch is this file-scope device array; its
// name is only a host-side stand-in in host code, so the host looks up its device address once
// per device and passes that address to the kernels.
// ---------------------------------------------------------------------------------------------
namespace moe {
namespace {

constexpr int NOALLOC_MAX_DEVICES = 64;
static __device__ __align__(256) int32_t g_route_scratch[MOE_NOALLOC_ROUTE_SCRATCH_BYTES / sizeof(int32_t)];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry-point query (the library does not link
// libcuda directly)
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

std::mutex g_scratch_mu;
void* g_scratch_addr[NOALLOC_MAX_DEVICES] = {};
CUcontext g_scratch_ctx[NOALLOC_MAX_DEVICES] = {};

// Device address of g_route_scratch on the current device. It is looked up on the first call
// with that device current, and looked up again whenever the device's current context is not
// the one of the last lookup (after cudaDeviceReset the module is loaded again and the array
// may sit at another address).
moe_status_t route_scratch_address(void** addr) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err);
  if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return MOE_ERR_UNSUPPORTED_DEVICE;
  const CtxGetCurrentFn get = ctx_get_current();
  if (get == nullptr) return cuda_fail(cudaErrorNotSupported);
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) ctx = nullptr;  // no context current yet: look up below
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr || ctx == nullptr || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_route_scratch);  // makes the device's context current
    if (err != cudaSuccess) return cuda_fail(err);
    if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cuda_fail(cudaErrorDeviceUninitialized);
    g_scratch_addr[dev] = p;
    g_scratch_ctx[dev] = ctx;
  }
  *addr = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_route_offsets_noalloc(const int32_t* ids, int T, int top_k, int E,
                                                  int32_t* counts, int32_t* offsets,
                                                  int32_t* sorted_src, int32_t* inv_map,
                                                  moe_stream_t stream) {
  using namespace moe;
  MOE_TRACE_CALL();
  if (T < 0 || top_k < 1) return MOE_ERR_INVALID_ARG;
  if (top_k > 32 || E < 1 || E > MAX_E) return MOE_ERR_UNSUPPORTED_SHAPE;
  const long long n = static_cast<long long>(T) * top_k;
  if (n >= (1LL << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (n > 0 && (!ids || !sorted_src || !inv_map)) return MOE_ERR_INVALID_ARG;
  // the one array has a fixed size: larger problems must use moe_route_offsets with a workspace
  if (route_workspace_bytes(n, E) > MOE_NOALLOC_ROUTE_SCRATCH_BYTES) return MOE_ERR_WORKSPACE_TOO_SMALL;
  moe_status_t st = check_device();
  if (st != MOE_OK) return st;
  void* scratch = nullptr;
  if ((st = route_scratch_address(&scratch)) != MOE_OK) return st;
  return launch_route(ids, static_cast<int>(n), E, counts, offsets, sorted_src, inv_map, scratch,
                      reinterpret_cast<cudaStream_t>(stream));
}
