// C-ABI entry points (include/moe_gg.h): argument validation, workspace carving, tensor-map
// construction and stream-ordered launches. No entry point allocates device memory; only
// moe_loop_swiglu_fwd synchronises (by design, it is the host-scheduled comparison variant).
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.h"
#include "trace.h"

namespace moe {

namespace {
thread_local char g_last_error[256] = "no error";
constexpr int MAX_DEVICES = 64;
constexpr int MAX_E = 1024;
constexpr int MAX_TOPK = 32;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

size_t round256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

moe_status_t map_fail(const char* what) {
  std::snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled failed for %s", what);
  return MOE_ERR_CUDA;
}

bool dim_ok(int v) { return v > 0 && v % 8 == 0 && v <= (1 << 20); }

bool shape_ok(int E, int d, int h) { return E >= 1 && E <= MAX_E && dim_ok(d) && dim_ok(h); }

// Widths whose bf16 rows are not 16-byte multiples (TMA needs 16-byte row pitches) are run by
// the composite calls on zero-padded copies of width round8(w); the result is exact (the extra
// columns and rows are zeros, which add nothing to any sum).
int round8(int v) { return (v + 7) & ~7; }
bool any_width_ok(int v) { return v > 0 && v <= (1 << 20); }
bool odd_pitch(int d, int h) { return d % 8 != 0 || h % 8 != 0; }

long long row_tiles_bound(long long rows, int E) { return (rows + 127) / 128 + E; }

GemmArgs base_args(int E, int cap, int32_t* status) {
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.E = E;
  a.single_expert = -1;
  a.cap = cap;
  a.status = status;
  a.timeout_ns = wait_timeout_ns();
  a.drain_ns = std::max(a.timeout_ns, 2000000000LL);
  return a;
}

// saved = low half of P [rows, h] bf16 (P = w*A, or A; the high half is a_save) | U rounded to
// 24 bits in blocks of 32 rows x 16 columns per (row tile, lane quadrant, column chunk). The row
// tiles of any problem list with at most `rows` rows number at most sum_e ceil(M_e / 128) <=
// (rows + 127 E) / 128; each holds 4 quadrants x 2 ceil(h/16) chunks of 1536 bytes.
size_t saved_p_bytes(long long rows, int h) { return round256(static_cast<size_t>(rows) * h * 2); }
long long saved_u_tiles(long long rows, int E) { return (rows + 127LL * E) / 128; }
size_t saved_u_bytes(long long rows, int h, int E) {
  return round256(static_cast<size_t>(saved_u_tiles(rows, E)) * 4 * (2 * ((h + 15) / 16)) * 1536);
}
size_t saved_bytes(long long rows, int h, int E) {
  return saved_p_bytes(rows, h) + saved_u_bytes(rows, h, E);
}
const void* saved_u(const void* saved, long long rows, int h) {
  return static_cast<const uint8_t*>(saved) + saved_p_bytes(rows, h);
}
size_t bwd_ws_half(long long rows, int h) { return round256(static_cast<size_t>(rows) * 2 * h * 2); }
// routing-weight gradient partials: one per (256-column tile, warp half) of the dgrad, per row
int route_grad_parts(int h) { return 2 * ((h + 255) / 256); }
size_t route_grad_part_bytes(long long rows, int h) {
  return round256(static_cast<size_t>(rows) * route_grad_parts(h) * 4);
}
size_t bwd_core_bytes(long long rows, int h) { return 2 * bwd_ws_half(rows, h) + route_grad_part_bytes(rows, h); }

// Workspace of the repacked (odd-pitch) composites: each piece rounded to 256 bytes, in order.
size_t bf16_bytes(long long rows, int cols) { return round256(static_cast<size_t>(rows) * cols * 2); }
size_t f32_bytes(long long rows, int cols) { return round256(static_cast<size_t>(rows) * cols * 4); }
size_t fwd_repack_bytes(long long cap, int E, int d, int h) {
  const int d8 = round8(d), h8 = round8(h);
  return 2 * bf16_bytes(cap, d8) + bf16_bytes(cap, h8) + bf16_bytes(static_cast<long long>(E) * 2 * h8, d8) +
         bf16_bytes(static_cast<long long>(E) * h8, d8);
}
size_t bwd_repack_bytes(long long cap, int E, int d, int h) {
  const int d8 = round8(d), h8 = round8(h);
  return 3 * bf16_bytes(cap, d8) + bf16_bytes(cap, h8) + bf16_bytes(static_cast<long long>(E) * 2 * h8, d8) +
         bf16_bytes(static_cast<long long>(E) * h8, d8) + f32_bytes(static_cast<long long>(E) * 2 * h8, d8) +
         f32_bytes(static_cast<long long>(E) * h8, d8) + bwd_core_bytes(cap, h8);
}

// Takes consecutive 256-byte aligned pieces from a workspace.
struct Carver {
  uint8_t* p;
  void* take(size_t bytes) {
    void* r = p;
    p += bytes;
    return r;
  }
};

// Activation rows [cap, w] <-> [cap, w8] (rows below M only); weights [E*blk rows] with their
// sub-blocks of `sub` rows widened to round8(sub) rows.
moe_status_t pack_rows(const void* src, void* dst, long long cap, int w, const int32_t* offsets, int E,
                       cudaStream_t s) {
  const int c = static_cast<int>(cap);
  return launch_pitch_repack(src, dst, false, cap, w, round8(w), c, c, c, c, true, offsets, E, s);
}
moe_status_t unpack_rows(const void* src, void* dst, long long cap, int w, const int32_t* offsets, int E,
                         cudaStream_t s) {
  const int c = static_cast<int>(cap);
  return launch_pitch_repack(src, dst, false, cap, w, round8(w), c, c, c, c, false, offsets, E, s);
}
moe_status_t repack_weight(const void* src, void* dst, bool fp32, int E, int nsub, int sub, int cols,
                           bool to_wide, cudaStream_t s) {
  const int sub8 = round8(sub);
  const long long rows = static_cast<long long>(E) * nsub * (to_wide ? sub8 : sub);
  return launch_pitch_repack(src, dst, fp32, rows, cols, round8(cols), nsub * sub, sub, nsub * sub8, sub8,
                             to_wide, nullptr, E, s);
}

// ---- one launch per step; `src` carries the problem source (device offsets, uniform rows or
// one expert), `rows` the rows of the row buffers, `tiles_bound` an upper bound of row tiles.

// a6: U = xp W_ug^T, P = w*SwiGLU(U) (w = 1 without row weights) into a_save as bf16; saved
// (nullable) receives U (rounded to 24 bits, blocked) and the low half of P.
moe_status_t run_up_swiglu(const GemmArgs& src, long long rows, long long tiles_bound, int E, int d,
                           int h, const void* xp, const void* w_ug, void* a_save, void* saved,
                           cudaStream_t s) {
  GemmMaps m{};
  if (!make_map_rows2d(&m.a, xp, rows, d, 128)) return map_fail("xp");
  if (!make_map_weight3d(&m.b, w_ug, E, 2LL * h, d, 128)) return map_fail("w_ug");
  GemmArgs a = src;
  a.N = h;
  a.K = d;
  a.h = h;
  a.out = a_save;
  a.ldo = h;
  if (saved != nullptr) {
    a.out2 = const_cast<void*>(saved_u(saved, rows, h));
    a.out3 = saved;
    a.ldo3 = h;
    a.dbg_u_tiles = saved_u_tiles(rows, E);
  }
  a.vec32 = (h % 16 == 0 && aligned32(a_save) && (saved == nullptr || aligned32(saved))) ? 1 : 0;
  return launch_grouped_gemm(MODE_UP_SWIGLU, m, a, tiles_bound * gemm_tiles_n(MODE_UP_SWIGLU, h), s);
}

// a7: y = A W_down.
moe_status_t run_down(const GemmArgs& src, long long rows, long long tiles_bound, int E, int d,
                      int h, const void* a_in, const void* w_down, void* y, cudaStream_t s) {
  GemmMaps m{};
  if (!make_map_rows2d(&m.a, a_in, rows, h, 128)) return map_fail("a");
  if (!make_map_weight3d(&m.b, w_down, E, h, d, 64)) return map_fail("w_down");
  GemmArgs a = src;
  a.N = d;
  a.K = h;
  a.h = h;
  a.out = y;
  a.ldo = d;
  a.vec32 = (d % 16 == 0 && aligned32(y)) ? 1 : 0;
  return launch_grouped_gemm(MODE_PLAIN_BF16, m, a, tiles_bound * gemm_tiles_n(MODE_PLAIN_BF16, d), s);
}

// a10: dA = dy W_down^T with the SwiGLU backward -> dU high and low halves.
moe_status_t run_down_dgrad_swiglu(const GemmArgs& src, long long rows, int E, int d, int h,
                                   const void* dy, const void* saved, const void* w_down,
                                   void* du_hi, void* du_lo, float* dw_part, cudaStream_t s) {
  GemmMaps m{};
  if (!make_map_rows2d(&m.a, dy, rows, d, 128)) return map_fail("dy");
  if (!make_map_weight3d(&m.b, w_down, E, h, d, 256)) return map_fail("w_down");
  GemmArgs a = src;
  a.N = h;
  a.K = d;
  a.h = h;
  a.out = du_hi;
  a.ldo = 2LL * h;
  a.out2 = du_lo;
  a.ldo2 = 2LL * h;
  a.aux = saved_u(saved, rows, h);
  a.dbg_u_tiles = saved_u_tiles(rows, E);
  a.vec32 = (h % 16 == 0 && aligned32(du_hi) && aligned32(du_lo)) ? 1 : 0;
  a.dw_part = dw_part;
  a.dw_np = route_grad_parts(h);
  if (!make_map_rows2d_store(&m.out, du_hi, rows, 2LL * h)) return map_fail("du_hi");
  if (!make_map_rows2d_store(&m.out2, du_lo, rows, 2LL * h)) return map_fail("du_lo");
  return launch_grouped_gemm(MODE_DGRAD_SWIGLU, m, a,
                             row_tiles_bound(rows, src.E) * gemm_tiles_n(MODE_DGRAD_SWIGLU, h), s);
}

// a12: dxp = dU W_ug.
moe_status_t run_up_dgrad(const GemmArgs& src, long long rows, int E, int d, int h,
                          const void* du_hi, const void* w_ug, void* dxp, cudaStream_t s) {
  GemmMaps m{};
  if (!make_map_rows2d(&m.a, du_hi, rows, 2LL * h, 128)) return map_fail("dU");
  if (!make_map_weight3d(&m.b, w_ug, E, 2LL * h, d, 64)) return map_fail("w_ug");
  GemmArgs a = src;
  a.N = d;
  a.K = 2 * h;
  a.h = h;
  a.out = dxp;
  a.ldo = d;
  a.vec32 = (d % 16 == 0 && aligned32(dxp)) ? 1 : 0;
  return launch_grouped_gemm(MODE_PLAIN_BF16, m, a,
                             row_tiles_bound(rows, src.E) * gemm_tiles_n(MODE_PLAIN_BF16, d), s);
}

// One wgrad problem: dW_e = (P_hi + P_lo)_e^T Q_e over each expert's rows (P_lo may be null).
struct WgradProblem {
  const void* p_hi;
  const void* p_lo;
  int p_cols;
  const void* q;
  int q_cols;
  float* dw;
};

// Operand and gradient maps of one problem (with no rows every expert is empty: the maps then
// describe a one-row placeholder).
moe_status_t wgrad_maps(const WgradProblem& w, long long rows, int E, CUtensorMap* a, CUtensorMap* a_lo,
                        CUtensorMap* b, CUtensorMap* out) {
  const long long r = std::max(rows, 1LL);
  if (!make_map_rows2d(a, w.p_hi, r, w.p_cols, 64)) return map_fail("p_hi");
  if (!make_map_rows2d(a_lo, w.p_lo ? w.p_lo : w.p_hi, r, w.p_cols, 64)) return map_fail("p_lo");
  if (!make_map_rows2d(b, w.q, r, w.q_cols, 64)) return map_fail("q");
  if (!make_map_grad3d_f32(out, w.dw, E, w.p_cols, w.q_cols)) return map_fail("dw");
  return MOE_OK;
}

// tiles of one problem: 256 gradient rows (a CTA pair) x 256 columns
long long wgrad_tiles(const WgradProblem& w, int E) {
  return static_cast<long long>(E) * ((w.p_cols + 255) / 256) * ((w.q_cols + 255) / 256);
}

// a11 / a13: one or two wgrad problems over the same experts in one persistent launch (the
// second one's tiles follow the first's). Both must agree on whether P has a low half.
moe_status_t run_wgrad(const GemmArgs& src, long long rows, int E, const WgradProblem& w1,
                       const WgradProblem* w2, cudaStream_t s) {
  GemmMaps m{};
  moe_status_t st = wgrad_maps(w1, rows, E, &m.a, &m.a_lo, &m.b, &m.out);
  if (st != MOE_OK) return st;
  GemmArgs a = src;
  a.N = w1.q_cols;
  a.Mdim = w1.p_cols;
  a.out = w1.dw;
  a.ldo = w1.q_cols;
  a.nprob = 1;
  long long tiles = wgrad_tiles(w1, E);
  if (w2 != nullptr) {
    if ((w2->p_lo == nullptr) != (w1.p_lo == nullptr)) return MOE_ERR_INVALID_ARG;
    st = wgrad_maps(*w2, rows, E, &m.a2, &m.a_lo2, &m.b2, &m.out2);
    if (st != MOE_OK) return st;
    a.nprob = 2;
    a.N2 = w2->q_cols;
    a.Mdim2 = w2->p_cols;
    a.out_b = w2->dw;
    a.ldo_b = w2->q_cols;
    tiles += wgrad_tiles(*w2, E);
  }
  return launch_grouped_gemm(w1.p_lo ? MODE_WGRAD : MODE_WGRAD_BF16, m, a, tiles, s);
}

moe_status_t check_grouped_common(int E, int cap, int d, int h) {
  if (cap < 0 || d <= 0 || h <= 0 || E < 1) return MOE_ERR_INVALID_ARG;
  if (!shape_ok(E, d, h)) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

// The composite calls: any width (odd pitches go through zero-padded copies)
moe_status_t check_grouped_any_width(int E, int cap, int d, int h) {
  if (cap < 0 || d <= 0 || h <= 0 || E < 1) return MOE_ERR_INVALID_ARG;
  if (E > MAX_E || !any_width_ok(d) || !any_width_ok(h)) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

}  // namespace

moe_status_t cuda_fail(cudaError_t err) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s", cudaGetErrorName(err),
                cudaGetErrorString(err));
  return MOE_ERR_CUDA;
}

int device_sm_count() {
  static int cache[MAX_DEVICES] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return 1;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 1;
  }
  return cache[dev];
}

long long wait_timeout_ns() {
  static const long long v = [] {
    const char* s = std::getenv("MOE_GG_WAIT_TIMEOUT_NS");
    const long long t = s ? std::atoll(s) : 0;
    return t > 0 ? t : 2000000000LL;
  }();
  return v;
}

cudaError_t ensure_max_dynamic_smem(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(mu);
  for (const auto& p : done)
    if (p.first == kernel && p.second == dev) return cudaSuccess;
  err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err == cudaSuccess) done.emplace_back(kernel, dev);
  return err;
}

moe_status_t check_device() {
  static int ok_cache[MAX_DEVICES] = {0};  // 0 unknown, 1 ok, -1 unsupported
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err);
  if (dev < 0 || dev >= MAX_DEVICES) return MOE_ERR_UNSUPPORTED_DEVICE;
  if (ok_cache[dev] == 0) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    ok_cache[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  return ok_cache[dev] == 1 ? MOE_OK : MOE_ERR_UNSUPPORTED_DEVICE;
}

#ifdef MOE_GG_DEBUG
namespace {
std::atomic<bool> g_dbg_call_error{false};
}  // namespace

void dbg_after_call(const char* name, cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return;
  const cudaError_t err = cudaStreamSynchronize(stream);
  if (err == cudaSuccess) return;
  g_dbg_call_error = true;
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s: %s", name, cudaGetErrorName(err),
                cudaGetErrorString(err));
}
#endif

}  // namespace moe

using namespace moe;

extern "C" {

int moe_abi_version(void) { return 2; }

int moe_debug_build(void) {
#ifdef MOE_GG_DEBUG
  return 1;
#else
  return 0;
#endif
}

moe_status_t moe_debug_report(int32_t* site_mask, int32_t* first_site, long long* index, long long* limit,
                              int reset) {
  DbgRecord acc = {0, -1, 0, 0};
#ifdef MOE_GG_DEBUG
  cudaError_t err = cudaDeviceSynchronize();
  if (err == cudaSuccess) err = dbg_collect_grouped(&acc, reset != 0);
  if (err == cudaSuccess) err = dbg_collect_permute(&acc, reset != 0);
  if (err == cudaSuccess) err = dbg_collect_route(&acc, reset != 0);
  if (err == cudaSuccess) err = dbg_collect_mx(&acc, reset != 0);
  if (err != cudaSuccess) return cuda_fail(err);
  if (g_dbg_call_error) acc.mask |= 1 << MOE_DEBUG_CALL_ERROR_BIT;
  if (reset) g_dbg_call_error = false;
#else
  (void)reset;
#endif
  if (site_mask) *site_mask = acc.mask;
  if (first_site) *first_site = acc.site;
  if (index) *index = acc.index;
  if (limit) *limit = acc.limit;
  return MOE_OK;
}

const char* moe_debug_site_name(int site) {
  static const char* const names[DBG_SITES] = {
      "grouped: epilogue row", "grouped: saved U row tile", "grouped: row slot",
      "grouped: destination row", "grouped: activation scale tile", "grouped: weight scale tile",
      "grouped: written scale tile", "combine: inverse-map row", "routing-weight grad: inverse-map row",
      "route: placed row", "mxfp8 quantization: scale tile"};
  return (site >= 0 && site < DBG_SITES) ? names[site] : "?";
}

const char* moe_last_cuda_error(void) { return g_last_error; }

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (null, negative or misaligned)";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "a device-side wait timed out";
    case MOE_ERR_UNSUPPORTED_DEVICE: return "current device is not sm_103";
  }
  return "unknown status";
}

size_t moe_workspace_bytes(int op, int T, int top_k, int E, int d, int h, int capacity_C) {
  if (T < 0 || top_k < 1 || top_k > MAX_TOPK || E < 1 || E > MAX_E) return 0;
  const long long n = static_cast<long long>(T) * top_k;
  switch (op) {
    case MOE_OP_ROUTE: return route_workspace_bytes(n, E);
    case MOE_OP_FWD:
      if (!any_width_ok(d) || !any_width_ok(h)) return 0;
      return odd_pitch(d, h) ? fwd_repack_bytes(n, E, d, h) : 0;
    case MOE_OP_BWD:
      if (!any_width_ok(d) || !any_width_ok(h)) return 0;
      return odd_pitch(d, h) ? bwd_repack_bytes(n, E, d, h) : bwd_core_bytes(n, h);
    case MOE_OP_SAVED: return any_width_ok(h) ? saved_bytes(n, round8(h), E) : 0;
    case MOE_OP_PADDED_BMM: {
      if (capacity_C <= 0 || d <= 0 || h <= 0) return 0;
      const size_t rows = static_cast<size_t>(E) * capacity_C;
      return round256(rows * d * 2) * 2 + round256(rows * h * 2);
    }
    case MOE_OP_LOOP: return 0;
    case MOE_OP_MX_WEIGHTS:
    case MOE_OP_MX_FWD:
    case MOE_OP_MX_BWD:
    case MOE_OP_MX_ROW_SCALES: return mx_workspace_bytes(op, n, E, d, h);
  }
  return 0;
}

moe_status_t moe_route_offsets(const int32_t* ids, int T, int top_k, int E, int32_t* counts,
                               int32_t* offsets, int32_t* sorted_src, int32_t* inv_map,
                               void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (T < 0 || top_k < 1) return MOE_ERR_INVALID_ARG;
  if (top_k > MAX_TOPK || E < 1 || E > MAX_E) return MOE_ERR_UNSUPPORTED_SHAPE;
  const long long n = static_cast<long long>(T) * top_k;
  if (n >= (1LL << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (n > 0 && (!ids || !sorted_src || !inv_map)) return MOE_ERR_INVALID_ARG;
  const size_t need = route_workspace_bytes(n, E);
  if (ws_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (need > 0 && !ws) return MOE_ERR_INVALID_ARG;
  moe_status_t st = check_device();
  if (st != MOE_OK) return st;
  return launch_route(ids, static_cast<int>(n), E, counts, offsets, sorted_src, inv_map, ws,
                      reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_permute(const moe_bf16* x, const int32_t* sorted_src, const int32_t* offsets,
                         const float* row_scale, int T, int top_k, int E, int d, moe_bf16* xp,
                         moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (T < 0 || top_k < 1 || d <= 0) return MOE_ERR_INVALID_ARG;
  if (top_k > MAX_TOPK || E < 1 || E > MAX_E || !any_width_ok(d)) return MOE_ERR_UNSUPPORTED_SHAPE;
  const long long n = static_cast<long long>(T) * top_k;
  if (n >= (1LL << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!offsets) return MOE_ERR_INVALID_ARG;
  if (n > 0 && (!x || !sorted_src || !xp)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(xp)) return MOE_ERR_INVALID_ARG;
  moe_status_t st = check_device();
  if (st != MOE_OK) return st;
  return launch_permute(x, sorted_src, offsets, row_scale, static_cast<int>(n), top_k, E, d, xp,
                        reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_unpermute_combine(const moe_bf16* y, const int32_t* inv_map, const float* weights,
                                   int T, int top_k, int d, moe_bf16* out, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (T < 0 || top_k < 1 || d <= 0) return MOE_ERR_INVALID_ARG;
  if (top_k > MAX_TOPK || !any_width_ok(d)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<long long>(T) * top_k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (T > 0 && (!y || !inv_map || !out)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  moe_status_t st = check_device();
  if (st != MOE_OK) return st;
  return launch_combine(y, inv_map, weights, T, top_k, d, out,
                        reinterpret_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------ single grouped kernels
moe_status_t moe_grouped_up_swiglu(const moe_bf16* xp, const int32_t* offsets,
                                   const int32_t* sorted_src, const float* weights, int E, int cap,
                                   int d, int h, const moe_bf16* w_ug, moe_bf16* a_save,
                                   void* saved, int32_t* dev_status, moe_stream_t stream) {
  MOE_TRACE_CALL();
  moe_status_t st = check_grouped_common(E, cap, d, h);
  if (st != MOE_OK) return st;
  if (!xp || !offsets || !w_ug || !a_save || (weights && !sorted_src)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(xp) || !aligned16(w_ug) || !aligned16(a_save) || !aligned16(saved))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_OK || cap == 0) return st;
  GemmArgs src = base_args(E, cap, dev_status);
  src.offsets = offsets;
  src.row_src = sorted_src;
  src.row_weight = weights;
  return run_up_swiglu(src, cap, row_tiles_bound(cap, E), E, d, h, xp, w_ug, a_save, saved,
                       reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_grouped_down(const moe_bf16* a, const int32_t* offsets, int E, int cap, int d,
                              int h, const moe_bf16* w_down, moe_bf16* y, int32_t* dev_status,
                              moe_stream_t stream) {
  MOE_TRACE_CALL();
  moe_status_t st = check_grouped_common(E, cap, d, h);
  if (st != MOE_OK) return st;
  if (!a || !offsets || !w_down || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(w_down) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_OK || cap == 0) return st;
  GemmArgs src = base_args(E, cap, dev_status);
  src.offsets = offsets;
  return run_down(src, cap, row_tiles_bound(cap, E), E, d, h, a, w_down, y,
                  reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_grouped_down_dgrad_swiglu(const moe_bf16* dy, const void* saved,
                                           const int32_t* offsets, const int32_t* sorted_src,
                                           const float* weights, int E, int cap, int d, int h,
                                           const moe_bf16* w_down, moe_bf16* du_hi,
                                           moe_bf16* du_lo, float* dw_part, int32_t* dev_status,
                                           moe_stream_t stream) {
  MOE_TRACE_CALL();
  moe_status_t st = check_grouped_common(E, cap, d, h);
  if (st != MOE_OK) return st;
  if (!dy || !saved || !offsets || !w_down || !du_hi || !du_lo || (weights && !sorted_src))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(dy) || !aligned16(saved) || !aligned16(w_down) || !aligned16(du_hi) ||
      !aligned16(du_lo) || (reinterpret_cast<uintptr_t>(dw_part) & 3u))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_OK || cap == 0) return st;
  GemmArgs src = base_args(E, cap, dev_status);
  src.offsets = offsets;
  src.row_src = sorted_src;
  src.row_weight = weights;
  return run_down_dgrad_swiglu(src, cap, E, d, h, dy, saved, w_down, du_hi, du_lo, dw_part,
                               reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_routing_weight_grad(const float* dw_part, const int32_t* inv_map, int T,
                                     int top_k, int h, float* dw_route, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (T < 0 || top_k < 1 || h <= 0) return MOE_ERR_INVALID_ARG;
  if (top_k > MAX_TOPK) return MOE_ERR_UNSUPPORTED_SHAPE;
  const long long n = static_cast<long long>(T) * top_k;
  if (n > INT32_MAX) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (n == 0) return MOE_OK;
  if (!dw_part || !inv_map || !dw_route) return MOE_ERR_INVALID_ARG;
  moe_status_t st = check_device();
  if (st != MOE_OK) return st;
  return launch_routing_weight_grad(dw_part, route_grad_parts(h), inv_map, static_cast<int>(n),
                                    dw_route, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_grouped_up_dgrad(const moe_bf16* du_hi, const int32_t* offsets, int E, int cap,
                                  int d, int h, const moe_bf16* w_ug, moe_bf16* dxp,
                                  int32_t* dev_status, moe_stream_t stream) {
  MOE_TRACE_CALL();
  moe_status_t st = check_grouped_common(E, cap, d, h);
  if (st != MOE_OK) return st;
  if (!du_hi || !offsets || !w_ug || !dxp) return MOE_ERR_INVALID_ARG;
  if (!aligned16(du_hi) || !aligned16(w_ug) || !aligned16(dxp)) return MOE_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_OK || cap == 0) return st;
  GemmArgs src = base_args(E, cap, dev_status);
  src.offsets = offsets;
  return run_up_dgrad(src, cap, E, d, h, du_hi, w_ug, dxp, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_grouped_wgrad(const moe_bf16* p_hi, const moe_bf16* p_lo, int p_cols,
                               const moe_bf16* q, int q_cols, const int32_t* offsets, int E,
                               int cap, float* dw, int32_t* dev_status, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (cap < 0 || E < 1 || p_cols <= 0 || q_cols <= 0) return MOE_ERR_INVALID_ARG;
  if (E > MAX_E || !dim_ok(p_cols) || !dim_ok(q_cols)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!p_hi || !q || !offsets || !dw) return MOE_ERR_INVALID_ARG;
  if (!aligned16(p_hi) || !aligned16(p_lo) || !aligned16(q) || !aligned16(dw))
    return MOE_ERR_INVALID_ARG;
  moe_status_t st = check_device();
  if (st != MOE_OK) return st;
  GemmArgs src = base_args(E, cap, dev_status);
  src.offsets = offsets;
  const WgradProblem w{p_hi, p_lo, p_cols, q, q_cols, dw};
  return run_wgrad(src, cap, E, w, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_grouped_wgrad_dual(const moe_bf16* p1_hi, const moe_bf16* p1_lo, int p1_cols,
                                    const moe_bf16* q1, int q1_cols, float* dw1,
                                    const moe_bf16* p2_hi, const moe_bf16* p2_lo, int p2_cols,
                                    const moe_bf16* q2, int q2_cols, float* dw2,
                                    const int32_t* offsets, int E, int cap, int32_t* dev_status,
                                    moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (cap < 0 || E < 1 || p1_cols <= 0 || q1_cols <= 0 || p2_cols <= 0 || q2_cols <= 0)
    return MOE_ERR_INVALID_ARG;
  if (E > MAX_E || !dim_ok(p1_cols) || !dim_ok(q1_cols) || !dim_ok(p2_cols) || !dim_ok(q2_cols))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!p1_hi || !q1 || !dw1 || !p2_hi || !q2 || !dw2 || !offsets) return MOE_ERR_INVALID_ARG;
  if ((p1_lo == nullptr) != (p2_lo == nullptr)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(p1_hi) || !aligned16(p1_lo) || !aligned16(q1) || !aligned16(dw1) || !aligned16(p2_hi) ||
      !aligned16(p2_lo) || !aligned16(q2) || !aligned16(dw2))
    return MOE_ERR_INVALID_ARG;
  moe_status_t st = check_device();
  if (st != MOE_OK) return st;
  GemmArgs src = base_args(E, cap, dev_status);
  src.offsets = offsets;
  const WgradProblem w1{p1_hi, p1_lo, p1_cols, q1, q1_cols, dw1};
  const WgradProblem w2{p2_hi, p2_lo, p2_cols, q2, q2_cols, dw2};
  return run_wgrad(src, cap, E, w1, &w2, reinterpret_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------ composite calls
moe_status_t moe_grouped_swiglu_fwd(const moe_bf16* xp, const int32_t* offsets,
                                    const int32_t* sorted_src, const float* weights, int E,
                                    int cap, int d, int h, const moe_bf16* w_ug,
                                    const moe_bf16* w_down, moe_bf16* y, moe_bf16* a_save,
                                    void* saved, void* ws, size_t ws_bytes, int32_t* dev_status,
                                    moe_stream_t stream) {
  MOE_TRACE_CALL();
  moe_status_t st = check_grouped_any_width(E, cap, d, h);
  if (st != MOE_OK) return st;
  if (!xp || !offsets || !w_ug || !w_down || !y || !a_save || (weights && !sorted_src))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(xp) || !aligned16(w_ug) || !aligned16(w_down) || !aligned16(y) ||
      !aligned16(a_save) || !aligned16(saved) || !aligned16(ws))
    return MOE_ERR_INVALID_ARG;
  const bool odd = odd_pitch(d, h);
  if (odd && ws_bytes < fwd_repack_bytes(cap, E, d, h)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if ((st = check_device()) != MOE_OK || cap == 0) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  GemmArgs src = base_args(E, cap, dev_status);
  src.offsets = offsets;
  src.row_src = sorted_src;
  src.row_weight = weights;
  const long long tb = row_tiles_bound(cap, E);
  GemmArgs dsrc = base_args(E, cap, dev_status);  // the weight is already in a_save
  dsrc.offsets = offsets;
  if (!odd) {
    st = run_up_swiglu(src, cap, tb, E, d, h, xp, w_ug, a_save, saved, s);
    if (st != MOE_OK) return st;
    return run_down(dsrc, cap, tb, E, d, h, a_save, w_down, y, s);
  }
  // zero-padded copies of width d8 / h8 (gate and up halves of W_ug widened separately)
  const int d8 = round8(d), h8 = round8(h);
  Carver cv{static_cast<uint8_t*>(ws)};
  void* xp8 = cv.take(bf16_bytes(cap, d8));
  void* y8 = cv.take(bf16_bytes(cap, d8));
  void* a8 = cv.take(bf16_bytes(cap, h8));
  void* wug8 = cv.take(bf16_bytes(static_cast<long long>(E) * 2 * h8, d8));
  void* wdn8 = cv.take(bf16_bytes(static_cast<long long>(E) * h8, d8));
  if ((st = pack_rows(xp, xp8, cap, d, offsets, E, s)) != MOE_OK) return st;
  if ((st = repack_weight(w_ug, wug8, false, E, 2, h, d, true, s)) != MOE_OK) return st;
  if ((st = repack_weight(w_down, wdn8, false, E, 1, h, d, true, s)) != MOE_OK) return st;
  if ((st = run_up_swiglu(src, cap, tb, E, d8, h8, xp8, wug8, a8, saved, s)) != MOE_OK) return st;
  if ((st = run_down(dsrc, cap, tb, E, d8, h8, a8, wdn8, y8, s)) != MOE_OK) return st;
  if ((st = unpack_rows(y8, y, cap, d, offsets, E, s)) != MOE_OK) return st;
  return unpack_rows(a8, a_save, cap, h, offsets, E, s);
}

}  // extern "C"

namespace moe {
namespace {

// The backward on 16-byte row pitches (d, h multiples of 8). ws: dU high and low halves, then
// the routing-gradient partials (used with dw_route).
moe_status_t grouped_bwd_core(const void* dy, const void* xp, const void* a_save, const void* saved,
                              const int32_t* offsets, const int32_t* sorted_src, const float* weights,
                              int E, int cap, int d, int h, const void* w_ug, const void* w_down,
                              void* dxp, float* dw_ug, float* dw_down, const int32_t* inv_map,
                              float* dw_route, void* ws, int32_t* dev_status, cudaStream_t s) {
  const size_t half = bwd_ws_half(cap, h);
  moe_bf16* du_hi = static_cast<moe_bf16*>(ws);
  moe_bf16* du_lo = reinterpret_cast<moe_bf16*>(static_cast<uint8_t*>(ws) + half);
  float* dw_part = dw_route ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + 2 * half) : nullptr;
  // P = w*A (or A): its high half is a_save, its low half is in saved
  const void* p_hi = a_save;
  const void* p_lo = saved;
  GemmArgs src = base_args(E, cap, dev_status);
  src.offsets = offsets;
  moe_status_t st = MOE_OK;
  if (cap > 0) {
    GemmArgs wsrc = src;
    wsrc.row_src = sorted_src;
    wsrc.row_weight = weights;
    st = run_down_dgrad_swiglu(wsrc, cap, E, d, h, dy, saved, w_down, du_hi, du_lo, dw_part, s);
    if (st != MOE_OK) return st;
    if (dw_route) {
      st = launch_routing_weight_grad(dw_part, route_grad_parts(h), inv_map, cap, dw_route, s);
      if (st != MOE_OK) return st;
    }
    st = run_up_dgrad(src, cap, E, d, h, du_hi, w_ug, dxp, s);
    if (st != MOE_OK) return st;
  }
  // both wgrads in one launch; they contract over each expert's rows, empty experts get zeros
  // (with no rows the operands are never read: a_save stands in for the unwritten dU)
  const WgradProblem wd{p_hi, cap > 0 ? p_lo : p_hi, h, dy, d, dw_down};
  const WgradProblem wu{cap > 0 ? du_hi : a_save, cap > 0 ? du_lo : a_save, 2 * h, xp, d, dw_ug};
  return run_wgrad(src, cap, E, wd, &wu, s);
}

}  // namespace
}  // namespace moe

extern "C" {

moe_status_t moe_grouped_bwd(const moe_bf16* dy, const moe_bf16* xp, const moe_bf16* a_save,
                             const void* saved, const int32_t* offsets, const int32_t* sorted_src,
                             const float* weights, int E, int cap, int d, int h,
                             const moe_bf16* w_ug, const moe_bf16* w_down, moe_bf16* dxp,
                             float* dw_ug, float* dw_down, const int32_t* inv_map,
                             float* dw_route, void* ws, size_t ws_bytes, int32_t* dev_status,
                             moe_stream_t stream) {
  MOE_TRACE_CALL();
  moe_status_t st = check_grouped_any_width(E, cap, d, h);
  if (st != MOE_OK) return st;
  if (!dy || !xp || !a_save || !saved || !offsets || !w_ug || !w_down || !dxp || !dw_ug ||
      !dw_down || (weights && !sorted_src) || (dw_route && !inv_map))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(dy) || !aligned16(xp) || !aligned16(a_save) || !aligned16(saved) ||
      !aligned16(w_ug) || !aligned16(w_down) || !aligned16(dxp) || !aligned16(dw_ug) ||
      !aligned16(dw_down) || !aligned16(ws))
    return MOE_ERR_INVALID_ARG;
  const bool odd = odd_pitch(d, h);
  const size_t need = odd ? bwd_repack_bytes(cap, E, d, h)
                          : 2 * bwd_ws_half(cap, h) + (dw_route ? route_grad_part_bytes(cap, h) : 0);
  if (ws_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (need > 0 && !ws) return MOE_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!odd)
    return grouped_bwd_core(dy, xp, a_save, saved, offsets, sorted_src, weights, E, cap, d, h, w_ug,
                            w_down, dxp, dw_ug, dw_down, inv_map, dw_route, ws, dev_status, s);
  // zero-padded copies of width d8 / h8; the gradients come back to the caller's widths
  const int d8 = round8(d), h8 = round8(h);
  Carver cv{static_cast<uint8_t*>(ws)};
  void* dy8 = cv.take(bf16_bytes(cap, d8));
  void* xp8 = cv.take(bf16_bytes(cap, d8));
  void* dxp8 = cv.take(bf16_bytes(cap, d8));
  void* a8 = cv.take(bf16_bytes(cap, h8));
  void* wug8 = cv.take(bf16_bytes(static_cast<long long>(E) * 2 * h8, d8));
  void* wdn8 = cv.take(bf16_bytes(static_cast<long long>(E) * h8, d8));
  float* dwug8 = static_cast<float*>(cv.take(f32_bytes(static_cast<long long>(E) * 2 * h8, d8)));
  float* dwdn8 = static_cast<float*>(cv.take(f32_bytes(static_cast<long long>(E) * h8, d8)));
  void* core_ws = cv.take(bwd_core_bytes(cap, h8));
  (void)core_ws;
  if ((st = pack_rows(dy, dy8, cap, d, offsets, E, s)) != MOE_OK) return st;
  if ((st = pack_rows(xp, xp8, cap, d, offsets, E, s)) != MOE_OK) return st;
  if ((st = pack_rows(a_save, a8, cap, h, offsets, E, s)) != MOE_OK) return st;
  if ((st = repack_weight(w_ug, wug8, false, E, 2, h, d, true, s)) != MOE_OK) return st;
  if ((st = repack_weight(w_down, wdn8, false, E, 1, h, d, true, s)) != MOE_OK) return st;
  st = grouped_bwd_core(dy8, xp8, a8, saved, offsets, sorted_src, weights, E, cap, d8, h8, wug8, wdn8,
                        dxp8, dwug8, dwdn8, inv_map, dw_route, core_ws, dev_status, s);
  if (st != MOE_OK) return st;
  if ((st = unpack_rows(dxp8, dxp, cap, d, offsets, E, s)) != MOE_OK) return st;
  if ((st = repack_weight(dwug8, dw_ug, true, E, 2, h, d, false, s)) != MOE_OK) return st;
  return repack_weight(dwdn8, dw_down, true, E, 1, h, d, false, s);
}

moe_status_t moe_grouped_swiglu_fwd_top1_combine(const moe_bf16* xp, const int32_t* offsets,
                                                 const int32_t* sorted_src, const int32_t* inv_map,
                                                 const float* weights, int E, int T, int d, int h,
                                                 const moe_bf16* w_ug, const moe_bf16* w_down, moe_bf16* out,
                                                 moe_bf16* a_save, void* saved, int32_t* dev_status,
                                                 moe_stream_t stream) {
  MOE_TRACE_CALL();
  moe_status_t st = check_grouped_common(E, T, d, h);
  if (st != MOE_OK) return st;
  if (!xp || !offsets || !sorted_src || !inv_map || !w_ug || !w_down || !out || !a_save) return MOE_ERR_INVALID_ARG;
  if (!aligned16(xp) || !aligned16(w_ug) || !aligned16(w_down) || !aligned16(out) || !aligned16(a_save) ||
      !aligned16(saved))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_OK || T == 0) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int cap = T;  // one slot per token
  // tokens whose only slot was dropped get zero rows; every other row is the down projection's
  if ((st = launch_zero_dropped_rows(inv_map, T, d, out, s)) != MOE_OK) return st;
  GemmArgs src = base_args(E, cap, dev_status);
  src.offsets = offsets;
  src.row_src = sorted_src;
  src.row_weight = weights;
  const long long tb = row_tiles_bound(cap, E);
  if ((st = run_up_swiglu(src, cap, tb, E, d, h, xp, w_ug, a_save, saved, s)) != MOE_OK) return st;
  GemmArgs dsrc = base_args(E, cap, dev_status);  // the weight is already in a_save
  dsrc.offsets = offsets;
  dsrc.row_dst = sorted_src;                      // flat slot = token when top_k = 1
  dsrc.dbg_dst_rows = T;
  return run_down(dsrc, cap, tb, E, d, h, a_save, w_down, out, s);
}

moe_status_t moe_padded_bmm_swiglu_fwd(const moe_bf16* xp, const int32_t* offsets, int E, int cap,
                                       int d, int h, int capacity_C, const moe_bf16* w_ug,
                                       const moe_bf16* w_down, moe_bf16* y, void* ws,
                                       size_t ws_bytes, int32_t* dev_status, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (cap < 0 || d <= 0 || h <= 0 || E < 1 || capacity_C < 1) return MOE_ERR_INVALID_ARG;
  if (!shape_ok(E, d, h)) return MOE_ERR_UNSUPPORTED_SHAPE;
  const long long rows = static_cast<long long>(E) * capacity_C;
  if (rows >= (1LL << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!xp || !offsets || !w_ug || !w_down || !y || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned16(xp) || !aligned16(w_ug) || !aligned16(w_down) || !aligned16(y) || !aligned16(ws))
    return MOE_ERR_INVALID_ARG;
  const size_t bx = round256(static_cast<size_t>(rows) * d * 2);
  const size_t ba = round256(static_cast<size_t>(rows) * h * 2);
  if (ws_bytes < 2 * bx + ba) return MOE_ERR_WORKSPACE_TOO_SMALL;
  moe_status_t st = check_device();
  if (st != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  moe_bf16* xpad = reinterpret_cast<moe_bf16*>(base);
  moe_bf16* ypad = reinterpret_cast<moe_bf16*>(base + bx);
  moe_bf16* apad = reinterpret_cast<moe_bf16*>(base + 2 * bx);
  st = launch_pad_rows(xp, offsets, E, capacity_C, d, xpad, s);
  if (st != MOE_OK) return st;
  GemmArgs src = base_args(E, static_cast<int>(rows), dev_status);
  src.uniform_rows = capacity_C;
  const long long tb = static_cast<long long>(E) * ((capacity_C + 127) / 128);
  st = run_up_swiglu(src, rows, tb, E, d, h, xpad, w_ug, apad, nullptr, s);
  if (st != MOE_OK) return st;
  st = run_down(src, rows, tb, E, d, h, apad, w_down, ypad, s);
  if (st != MOE_OK) return st;
  return launch_unpad_rows(ypad, offsets, E, capacity_C, cap, d, y, s);
}

moe_status_t moe_loop_swiglu_fwd(const moe_bf16* xp, const int32_t* offsets, int E, int cap,
                                 int d, int h, const moe_bf16* w_ug, const moe_bf16* w_down,
                                 moe_bf16* y, moe_bf16* a_save, void* saved,
                                 int32_t* dev_status, moe_stream_t stream) {
  MOE_TRACE_CALL();
  moe_status_t st = check_grouped_common(E, cap, d, h);
  if (st != MOE_OK) return st;
  if (!xp || !offsets || !w_ug || !w_down || !y || !a_save) return MOE_ERR_INVALID_ARG;
  if (!aligned16(xp) || !aligned16(w_ug) || !aligned16(w_down) || !aligned16(y) ||
      !aligned16(a_save) || !aligned16(saved))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // Fig. 36: the counts become host-visible first; the CPU waits for them.
  std::vector<int32_t> off(E);
  cudaError_t err = cudaMemcpyAsync(off.data(), offsets, sizeof(int32_t) * E, cudaMemcpyDeviceToHost, s);
  if (err == cudaSuccess) err = cudaStreamSynchronize(s);
  if (err != cudaSuccess) return cuda_fail(err);
  int prev = 0;
  for (int e = 0; e < E; ++e) {
    if (off[e] < prev || off[e] > cap) return MOE_ERR_INVALID_ARG;
    prev = off[e];
  }
  prev = 0;
  long long tile_base = 0;  // row tiles of the experts before e, as the grouped kernels count
  for (int e = 0; e < E; ++e) {
    const int rows = off[e] - prev;
    if (rows > 0) {
      GemmArgs src = base_args(1, cap, dev_status);
      src.single_expert = e;
      src.single_row0 = prev;
      src.single_rows = rows;
      src.tile_base = tile_base;
      tile_base += (rows + 127) / 128;
      const long long tb = (rows + 127) / 128;
      st = run_up_swiglu(src, cap, tb, E, d, h, xp, w_ug, a_save, saved, s);
      if (st != MOE_OK) return st;
      st = run_down(src, cap, tb, E, d, h, a_save, w_down, y, s);
      if (st != MOE_OK) return st;
    }
    prev = off[e];
  }
  return MOE_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ MXFP8 variant
// "Section 09: Grouped GEMM", §9.5: the routed MXFP8 path runs the forward and the Dgrad as
// scaled grouped GEMMs and keeps the Wgrad in BF16. Operands are quantized along their
// contraction dimension (E4M3 codes, one E8M0 scale per 32 elements; layouts in mx_quant.cu).
namespace moe {
namespace {

bool mx_shape_ok(int E, int d, int h) {
  return E >= 1 && E <= MAX_E && d > 0 && h > 0 && d % 32 == 0 && h % 128 == 0 && d <= (1 << 20) &&
         h <= (1 << 20);
}
size_t mx_codes_bytes(long long rows, int K) { return round256(static_cast<size_t>(rows) * K); }
size_t mx_wsf_bytes(int E, int N, int K) {
  return round256(static_cast<size_t>(E) * mx_ntpad(N) * mx_kc(K) * 512);
}
size_t mx_asf_bytes(long long cap, int E, int K) {
  return round256(static_cast<size_t>(saved_u_tiles(cap, E)) * mx_kc(K) * 512);
}

// The prepared weights: four (codes, scales) pairs, each piece 256-byte aligned, in order.
struct MxWeights {
  const uint8_t *ug_q, *ug_sf;    // W_ug along d:       codes [E, 2h, d]  (up/gate forward)
  const uint8_t *dnT_q, *dnT_sf;  // W_down along h:     codes [E, d, h]   (down forward)
  const uint8_t *dn_q, *dn_sf;    // W_down along d:     codes [E, h, d]   (down dgrad)
  const uint8_t *ugT_q, *ugT_sf;  // W_ug along 2h:      codes [E, d, 2h]  (up/gate dgrad)
};

size_t mx_weights_bytes(int E, int d, int h) {
  const long long e = E;
  return mx_codes_bytes(e * 2 * h, d) + mx_wsf_bytes(E, 2 * h, d) + mx_codes_bytes(e * d, h) +
         mx_wsf_bytes(E, d, h) + mx_codes_bytes(e * h, d) + mx_wsf_bytes(E, h, d) +
         mx_codes_bytes(e * d, 2 * h) + mx_wsf_bytes(E, d, 2 * h);
}

MxWeights carve_mx_weights(const void* base, int E, int d, int h) {
  const uint8_t* p = static_cast<const uint8_t*>(base);
  const long long e = E;
  MxWeights w;
  w.ug_q = p;    p += mx_codes_bytes(e * 2 * h, d);
  w.ug_sf = p;   p += mx_wsf_bytes(E, 2 * h, d);
  w.dnT_q = p;   p += mx_codes_bytes(e * d, h);
  w.dnT_sf = p;  p += mx_wsf_bytes(E, d, h);
  w.dn_q = p;    p += mx_codes_bytes(e * h, d);
  w.dn_sf = p;   p += mx_wsf_bytes(E, h, d);
  w.ugT_q = p;   p += mx_codes_bytes(e * d, 2 * h);
  w.ugT_sf = p;
  return w;
}

size_t mx_fwd_ws_bytes(long long cap, int E, int d, int h) {
  return mx_codes_bytes(cap, d) + mx_asf_bytes(cap, E, d) + mx_codes_bytes(cap, h) + mx_asf_bytes(cap, E, h);
}
size_t mx_bwd_ws_bytes(long long cap, int E, int d, int h) {
  return bwd_core_bytes(cap, h) + mx_codes_bytes(cap, d) + mx_asf_bytes(cap, E, d) + mx_codes_bytes(cap, 2 * h) +
         mx_asf_bytes(cap, E, 2 * h);
}

void set_mx(GemmArgs& a, const void* sfa, const void* sfb, int K, int N_b, long long rows, int E) {
  a.sfa = static_cast<const uint8_t*>(sfa);
  a.sfb = static_cast<const uint8_t*>(sfb);
  a.sf_kc = mx_kc(K);
  a.sfb_ntpad = mx_ntpad(N_b);
  a.dbg_sfa_tiles = saved_u_tiles(rows, E);
  a.dbg_sfb_tiles = static_cast<long long>(E) * mx_ntpad(N_b);
  a.dbg_mxsf_tiles = saved_u_tiles(rows, E);
}

// U = q(xp) q(W_ug)^T with the up/gate epilogue of the BF16 path (a_save, optional saved); the
// epilogue also quantizes bf16(P) into pq / psf, the down projection's A operand.
moe_status_t run_up_swiglu_mx(const GemmArgs& src, long long rows, long long tiles_bound, int E, int d, int h,
                              const void* xq, const void* xsf, const MxWeights& w, void* a_save, void* saved,
                              void* pq, void* psf, cudaStream_t s) {
  GemmMaps m{};
  if (!make_map_u8_rows2d(&m.a, xq, rows, d, 128)) return map_fail("xq");
  if (!make_map_u8_weight3d(&m.b, w.ug_q, E, 2LL * h, d, 128)) return map_fail("w_ug codes");
  GemmArgs a = src;
  a.N = h;
  a.K = d;
  a.h = h;
  a.out = a_save;
  a.ldo = h;
  if (saved != nullptr) {
    a.out2 = const_cast<void*>(saved_u(saved, rows, h));
    a.out3 = saved;
    a.ldo3 = h;
    a.dbg_u_tiles = saved_u_tiles(rows, E);
  }
  a.vec32 = (h % 16 == 0 && aligned32(a_save) && (saved == nullptr || aligned32(saved))) ? 1 : 0;
  set_mx(a, xsf, w.ug_sf, d, 2 * h, rows, E);
  a.mxq = static_cast<uint8_t*>(pq);
  a.mxsf = static_cast<uint8_t*>(psf);
  a.mx_ldq = h;
  a.mx_kc = mx_kc(h);
  return launch_grouped_gemm(MODE_UP_SWIGLU_MX, m, a, tiles_bound * gemm_tiles_n(MODE_UP_SWIGLU_MX, h), s);
}

// out = q(A) q(B)^T for a codes operand A [rows, K] and weight codes B [E, N, K]; bf16 out.
moe_status_t run_plain_mx(const GemmArgs& src, long long rows, long long tiles_bound, int E, int K, int N,
                          const void* aq, const void* asf, const void* bq, const void* bsf, void* out,
                          cudaStream_t s) {
  GemmMaps m{};
  if (!make_map_u8_rows2d(&m.a, aq, rows, K, 128)) return map_fail("a codes");
  if (!make_map_u8_weight3d(&m.b, bq, E, N, K, 256)) return map_fail("b codes");
  GemmArgs a = src;
  a.N = N;
  a.K = K;
  a.out = out;
  a.ldo = N;
  a.vec32 = (N % 16 == 0 && aligned32(out)) ? 1 : 0;
  set_mx(a, asf, bsf, K, N, rows, E);
  return launch_grouped_gemm(MODE_PLAIN_MX, m, a, tiles_bound * gemm_tiles_n(MODE_PLAIN_MX, N), s);
}

// dA = w * q(dy) q(W_down)^T with the SwiGLU backward of the BF16 path (dU high / low); the
// epilogue also quantizes dU's high half into duq / dusf, the up/gate dgrad's A operand.
moe_status_t run_dgrad_mx(const GemmArgs& src, long long rows, int E, int d, int h, const void* dyq,
                          const void* dysf, const void* saved, const MxWeights& w, void* du_hi, void* du_lo,
                          float* dw_part, void* duq, void* dusf, cudaStream_t s) {
  GemmMaps m{};
  if (!make_map_u8_rows2d(&m.a, dyq, rows, d, 128)) return map_fail("dy codes");
  if (!make_map_u8_weight3d(&m.b, w.dn_q, E, h, d, 256)) return map_fail("w_down codes");
  if (!make_map_rows2d_store(&m.out, du_hi, rows, 2LL * h)) return map_fail("du_hi");
  if (!make_map_rows2d_store(&m.out2, du_lo, rows, 2LL * h)) return map_fail("du_lo");
  GemmArgs a = src;
  a.N = h;
  a.K = d;
  a.h = h;
  a.out = du_hi;
  a.ldo = 2LL * h;
  a.out2 = du_lo;
  a.ldo2 = 2LL * h;
  a.aux = saved_u(saved, rows, h);
  a.dbg_u_tiles = saved_u_tiles(rows, E);
  a.vec32 = (h % 16 == 0 && aligned32(du_hi) && aligned32(du_lo)) ? 1 : 0;
  a.dw_part = dw_part;
  a.dw_np = route_grad_parts(h);
  set_mx(a, dysf, w.dn_sf, d, h, rows, E);
  a.mxq = static_cast<uint8_t*>(duq);
  a.mxsf = static_cast<uint8_t*>(dusf);
  a.mx_ldq = 2 * h;
  a.mx_kc = mx_kc(2 * h);
  return launch_grouped_gemm(MODE_DGRAD_SWIGLU_MX, m, a,
                             row_tiles_bound(rows, src.E) * gemm_tiles_n(MODE_DGRAD_SWIGLU_MX, h), s);
}

}  // namespace

size_t mx_workspace_bytes(int op, long long n, int E, int d, int h) {
  if (!mx_shape_ok(E, d, h)) return 0;
  switch (op) {
    case MOE_OP_MX_WEIGHTS: return mx_weights_bytes(E, d, h);
    case MOE_OP_MX_FWD: return mx_fwd_ws_bytes(n, E, d, h);
    case MOE_OP_MX_BWD: return mx_bwd_ws_bytes(n, E, d, h);
    case MOE_OP_MX_ROW_SCALES: return mx_asf_bytes(n, E, d);
  }
  return 0;
}

}  // namespace moe

extern "C" {

moe_status_t moe_mx_prepare_weights(const moe_bf16* w_ug, const moe_bf16* w_down, int E, int d, int h, void* mxw,
                                    size_t mxw_bytes, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (E < 1 || d <= 0 || h <= 0) return MOE_ERR_INVALID_ARG;
  if (!mx_shape_ok(E, d, h)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!w_ug || !w_down || !mxw) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w_ug) || !aligned16(w_down) || (reinterpret_cast<uintptr_t>(mxw) & 255u)) return MOE_ERR_INVALID_ARG;
  if (mxw_bytes < mx_weights_bytes(E, d, h)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  moe_status_t st = check_device();
  if (st != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const MxWeights w = carve_mx_weights(mxw, E, d, h);
  auto mut = [](const uint8_t* p) { return const_cast<uint8_t*>(p); };
  const long long e = E;
  if ((st = launch_mx_quant_rows(w_ug, e * 2 * h, d, nullptr, E, 2 * h, mut(w.ug_q), mut(w.ug_sf), nullptr, s)) !=
      MOE_OK)
    return st;
  if ((st = launch_mx_quant_cols(w_down, E, h, d, mut(w.dnT_q), mut(w.dnT_sf), s)) != MOE_OK) return st;
  if ((st = launch_mx_quant_rows(w_down, e * h, d, nullptr, E, h, mut(w.dn_q), mut(w.dn_sf), nullptr, s)) != MOE_OK)
    return st;
  return launch_mx_quant_cols(w_ug, E, 2 * h, d, mut(w.ugT_q), mut(w.ugT_sf), s);
}

moe_status_t moe_permute_mxfp8(const moe_bf16* x, const int32_t* sorted_src, const int32_t* offsets, int T,
                               int top_k, int E, int d, moe_bf16* xp, uint8_t* q, uint8_t* sf, int32_t* dev_status,
                               moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (T < 0 || top_k < 1 || d <= 0 || E < 1) return MOE_ERR_INVALID_ARG;
  if (top_k > MAX_TOPK || E > MAX_E || d % 32 != 0 || d > (1 << 20)) return MOE_ERR_UNSUPPORTED_SHAPE;
  const long long n = static_cast<long long>(T) * top_k;
  if (n >= (1LL << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!offsets || (n > 0 && (!x || !sorted_src || !q || !sf))) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(xp) || !aligned16(q) || !aligned16(sf)) return MOE_ERR_INVALID_ARG;
  moe_status_t st = check_device();
  if (st != MOE_OK || n == 0) return st;
  return launch_mx_permute_quant(x, sorted_src, offsets, E, static_cast<int>(n), top_k, d, xp, q, sf, dev_status,
                                 reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_mx_quantize_rows(const moe_bf16* x, const int32_t* offsets, int E, int cap, int K, uint8_t* q,
                                  uint8_t* sf, int32_t* dev_status, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (cap < 0 || K <= 0 || E < 1) return MOE_ERR_INVALID_ARG;
  if (E > MAX_E || K % 32 != 0 || K > (1 << 20)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!offsets || (cap > 0 && (!x || !q || !sf))) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || !aligned16(sf)) return MOE_ERR_INVALID_ARG;
  moe_status_t st = check_device();
  if (st != MOE_OK || cap == 0) return st;
  return launch_mx_quant_rows(x, cap, K, offsets, E, 0, q, sf, dev_status, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_grouped_swiglu_fwd_mxfp8(const moe_bf16* xp, const uint8_t* xq, const uint8_t* xsf,
                                          const int32_t* offsets, const int32_t* sorted_src, const float* weights,
                                          int E, int cap, int d, int h, const void* mxw, moe_bf16* y,
                                          moe_bf16* a_save, void* saved, void* ws, size_t ws_bytes,
                                          int32_t* dev_status, moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (cap < 0 || d <= 0 || h <= 0 || E < 1) return MOE_ERR_INVALID_ARG;
  if (!mx_shape_ok(E, d, h)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((!xp && !xq) || (!xq != !xsf) || !offsets || !mxw || !y || !a_save || !ws || (weights && !sorted_src))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(xp) || !aligned16(xq) || !aligned16(xsf) || !aligned16(y) || !aligned16(a_save) || !aligned16(saved) ||
      (reinterpret_cast<uintptr_t>(mxw) & 255u) || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < mx_fwd_ws_bytes(cap, E, d, h)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  moe_status_t st = check_device();
  if (st != MOE_OK || cap == 0) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const MxWeights w = carve_mx_weights(mxw, E, d, h);
  Carver cv{static_cast<uint8_t*>(ws)};
  void* xq_ws = cv.take(mx_codes_bytes(cap, d));
  void* xsf_ws = cv.take(mx_asf_bytes(cap, E, d));
  void* pq = cv.take(mx_codes_bytes(cap, h));
  void* psf = cv.take(mx_asf_bytes(cap, E, h));
  GemmArgs src = base_args(E, cap, dev_status);
  src.offsets = offsets;
  src.row_src = sorted_src;
  src.row_weight = weights;
  GemmArgs dsrc = base_args(E, cap, dev_status);  // the weight is already in a_save
  dsrc.offsets = offsets;
  const long long tb = row_tiles_bound(cap, E);
  if (xq == nullptr) {  // the caller passed bf16 rows: quantize them here
    if ((st = launch_mx_quant_rows(xp, cap, d, offsets, E, 0, xq_ws, xsf_ws, dev_status, s)) != MOE_OK) return st;
    xq = static_cast<const uint8_t*>(xq_ws);
    xsf = static_cast<const uint8_t*>(xsf_ws);
  }
  // the up/gate epilogue quantizes P as the BF16 path stores it (bf16) along h for the down GEMM
  if ((st = run_up_swiglu_mx(src, cap, tb, E, d, h, xq, xsf, w, a_save, saved, pq, psf, s)) != MOE_OK) return st;
  return run_plain_mx(dsrc, cap, tb, E, h, d, pq, psf, w.dnT_q, w.dnT_sf, y, s);
}

moe_status_t moe_grouped_bwd_mxfp8(const moe_bf16* dy, const uint8_t* dyq, const uint8_t* dysf, const moe_bf16* xp,
                                   const moe_bf16* a_save, const void* saved, const int32_t* offsets,
                                   const int32_t* sorted_src,
                                   const float* weights, int E, int cap, int d, int h, const void* mxw,
                                   moe_bf16* dxp, float* dw_ug, float* dw_down, const int32_t* inv_map,
                                   float* dw_route, void* ws, size_t ws_bytes, int32_t* dev_status,
                                   moe_stream_t stream) {
  MOE_TRACE_CALL();
  if (cap < 0 || d <= 0 || h <= 0 || E < 1) return MOE_ERR_INVALID_ARG;
  if (!mx_shape_ok(E, d, h)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!dy || !xp || !a_save || !saved || !offsets || !mxw || !dxp || !dw_ug || !dw_down || !ws ||
      (weights && !sorted_src) || (dw_route && !inv_map) || (!dyq != !dysf))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(dy) || !aligned16(dyq) || !aligned16(dysf) || !aligned16(xp) || !aligned16(a_save) || !aligned16(saved) || !aligned16(dxp) ||
      !aligned16(dw_ug) || !aligned16(dw_down) || (reinterpret_cast<uintptr_t>(mxw) & 255u) ||
      (reinterpret_cast<uintptr_t>(ws) & 255u))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < mx_bwd_ws_bytes(cap, E, d, h)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  moe_status_t st = check_device();
  if (st != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const MxWeights w = carve_mx_weights(mxw, E, d, h);
  Carver cv{static_cast<uint8_t*>(ws)};
  moe_bf16* du_hi = static_cast<moe_bf16*>(cv.take(bwd_ws_half(cap, h)));
  moe_bf16* du_lo = static_cast<moe_bf16*>(cv.take(bwd_ws_half(cap, h)));
  float* dw_part = static_cast<float*>(cv.take(route_grad_part_bytes(cap, h)));
  void* dyq_ws = cv.take(mx_codes_bytes(cap, d));
  void* dysf_ws = cv.take(mx_asf_bytes(cap, E, d));
  void* duq = cv.take(mx_codes_bytes(cap, 2 * h));
  void* dusf = cv.take(mx_asf_bytes(cap, E, 2 * h));
  GemmArgs src = base_args(E, cap, dev_status);
  src.offsets = offsets;
  if (cap > 0) {
    GemmArgs wsrc = src;
    wsrc.row_src = sorted_src;
    wsrc.row_weight = weights;
    const long long tb = row_tiles_bound(cap, E);
    if (dyq == nullptr) {  // the caller passed bf16 rows only: quantize them here
      if ((st = launch_mx_quant_rows(dy, cap, d, offsets, E, 0, dyq_ws, dysf_ws, dev_status, s)) != MOE_OK)
        return st;
      dyq = static_cast<const uint8_t*>(dyq_ws);
      dysf = static_cast<const uint8_t*>(dysf_ws);
    }
    // the dgrad epilogue quantizes dU's high half along 2h for the up/gate dgrad
    if ((st = run_dgrad_mx(wsrc, cap, E, d, h, dyq, dysf, saved, w, du_hi, du_lo, dw_route ? dw_part : nullptr,
                           duq, dusf, s)) != MOE_OK)
      return st;
    if (dw_route) {
      if ((st = launch_routing_weight_grad(dw_part, route_grad_parts(h), inv_map, cap, dw_route, s)) != MOE_OK)
        return st;
    }
    if ((st = run_plain_mx(src, cap, tb, E, 2 * h, d, duq, dusf, w.ugT_q, w.ugT_sf, dxp, s)) != MOE_OK) return st;
  }
  // BF16 wgrads of both projections in one launch (both halves of P and dU)
  const WgradProblem wd{a_save, cap > 0 ? saved : a_save, h, dy, d, dw_down};
  const WgradProblem wu{cap > 0 ? du_hi : a_save, cap > 0 ? du_lo : a_save, 2 * h, xp, d, dw_ug};
  return run_wgrad(src, cap, E, wd, &wu, s);
}

}  // extern "C"
