// Row movement around the grouped GEMM: the permute gather, the atomic-free combine through the
// inverse map, and the pad/unpad pair of the capacity-padded comparison variant.
//
// All of these are HBM-bound copies: one warp per row, 16-byte vector loads and stores,
// grid sized to a multiple of the SM count and striding over rows.
#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;

__device__ __forceinline__ uint4 scale_bf16x8(uint4 q, float s) {
  uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = pack_bf16x2(bf16_lo(w[i]) * s, bf16_hi(w[i]) * s);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// "grouped_mm" agent doc, forward gather x[idx]: xp[p] = x[sorted_src[p] / k] (* scale). The
// rows of xp are written with streaming stores (evict-first), so the T·k written rows do not
// push the T source rows, each read k times, out of L2 (measured 152 -> 139 us on the large
// workload).
__global__ void __launch_bounds__(THREADS) permute_kernel(
    const uint4* __restrict__ x, const int32_t* __restrict__ sorted_src,
    const int32_t* __restrict__ offsets, const float* __restrict__ row_scale, int n, int k, int E,
    int vec, uint4* __restrict__ xp) {
  const int M = min(__ldg(offsets + E - 1), n);
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * WARPS + (threadIdx.x >> 5);
  const int nw = gridDim.x * WARPS;
  for (long long p = gw; p < M; p += nw) {
    const int src = __ldg(sorted_src + p);
    if (src < 0 || src >= n) continue;
    const uint4* xr = x + static_cast<size_t>(src / k) * vec;
    uint4* orow = xp + static_cast<size_t>(p) * vec;
    const float s = (row_scale != nullptr) ? __ldg(row_scale + src) : 1.0f;
    int v = lane;
    // four 16-byte loads in flight per lane before their stores
    for (; v + 96 < vec; v += 128) {
      uint4 q[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) q[i] = __ldg(xr + v + 32 * i);
#pragma unroll
      for (int i = 0; i < 4; ++i) __stcs(orow + v + 32 * i, row_scale ? scale_bf16x8(q[i], s) : q[i]);
    }
    for (; v < vec; v += 32) __stcs(orow + v, row_scale ? scale_bf16x8(__ldg(xr + v), s) : __ldg(xr + v));
  }
}

// out[t] = 0 for every token whose single slot (top_k = 1) was dropped (inv[t] < 0): the rows the
// down projection does not write when it stores straight into the token rows.
__global__ void __launch_bounds__(THREADS) zero_dropped_rows_kernel(const int32_t* __restrict__ inv, int T,
                                                                    int vec, uint4* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * WARPS + (threadIdx.x >> 5);
  const int nw = gridDim.x * WARPS;
  for (long long t = gw; t < T; t += nw) {
    if (__ldg(inv + t) >= 0) continue;  // warp-uniform
    for (int v = lane; v < vec; v += 32) out[static_cast<size_t>(t) * vec + v] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// out[t] = sum_j w[t,j] * y[inv[t,j]] over slots with inv >= 0, fp32 in slot order, one bf16
// rounding (gather + reduction in place of the scatter-add, "grouped_mm" agent doc).
__global__ void __launch_bounds__(THREADS) combine_kernel(const uint4* __restrict__ y,
                                                          const int32_t* __restrict__ inv,
                                                          const float* __restrict__ weights,
                                                          int T, int k, int vec,
                                                          uint4* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * WARPS + (threadIdx.x >> 5);
  const int nw = gridDim.x * WARPS;
  for (long long t = gw; t < T; t += nw) {
    // lane j < k holds slot j's row and weight
    int my_p = -1;
    float my_w = 0.f;
    if (lane < k) {
      my_p = __ldg(inv + static_cast<size_t>(t) * k + lane);
      my_w = weights ? __ldg(weights + static_cast<size_t>(t) * k + lane) : 1.0f;
    }
    // every lane runs the same number of iterations: the shuffles need the whole warp
    for (int v0 = 0; v0 < vec; v0 += 32) {
      const int v = v0 + lane;
      const bool active = v < vec;
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      // up to eight slot rows loaded before they are summed, still in slot order (k <= 32)
      for (int j0 = 0; j0 < k; j0 += 8) {
        uint4 q[8];
        float wj[8];
        bool ok[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int j = j0 + jj;
          const int p = __shfl_sync(0xffffffffu, my_p, j & 31);
          wj[jj] = __shfl_sync(0xffffffffu, my_w, j & 31);
          ok[jj] = active && j < k && p >= 0 && MOE_DBG_IN(DBG_COMBINE_ROW, p, static_cast<long long>(T) * k);
          q[jj] = ok[jj] ? __ldg(y + static_cast<size_t>(p) * vec + v) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          if (!ok[jj]) continue;
          const uint32_t w4[4] = {q[jj].x, q[jj].y, q[jj].z, q[jj].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[2 * i] = fmaf(wj[jj], bf16_lo(w4[i]), acc[2 * i]);
            acc[2 * i + 1] = fmaf(wj[jj], bf16_hi(w4[i]), acc[2 * i + 1]);
          }
        }
      }
      if (active)
        out[static_cast<size_t>(t) * vec + v] =
            make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                       pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    }
  }
}

// Routing-weight gradient of the combine: dw[s] = <dOut[t], y_unweighted[inv[s]]>, assembled
// from the per-row partial sums the dgrad epilogue left (summed in index order, so the result
// does not depend on scheduling); 0 for a dropped slot.
__global__ void __launch_bounds__(THREADS) routing_weight_grad_kernel(
    const float* __restrict__ part, int np, const int32_t* __restrict__ inv, int n_slots,
    float* __restrict__ dw) {
  for (long long sl = static_cast<long long>(blockIdx.x) * THREADS + threadIdx.x; sl < n_slots;
       sl += static_cast<long long>(gridDim.x) * THREADS) {
    const int p = __ldg(inv + sl);
    float acc = 0.f;
    if (p >= 0 && MOE_DBG_IN(DBG_RWG_ROW, p, n_slots))
      for (int i = 0; i < np; ++i) acc += __ldg(part + static_cast<size_t>(p) * np + i);
    dw[sl] = acc;
  }
}

// ---- rows whose pitch is not a multiple of 16 bytes (d % 8 != 0): one bf16 per lane step,
// the same arithmetic as the vector kernels above (scale and rounding, fp32 sums in slot order)
__global__ void __launch_bounds__(THREADS) permute_scalar_kernel(
    const bf16* __restrict__ x, const int32_t* __restrict__ sorted_src,
    const int32_t* __restrict__ offsets, const float* __restrict__ row_scale, int n, int k, int E,
    int d, bf16* __restrict__ xp) {
  const int M = min(__ldg(offsets + E - 1), n);
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * WARPS + (threadIdx.x >> 5);
  const int nw = gridDim.x * WARPS;
  for (long long p = gw; p < M; p += nw) {
    const int src = __ldg(sorted_src + p);
    if (src < 0 || src >= n) continue;
    const bf16* xr = x + static_cast<size_t>(src / k) * d;
    bf16* orow = xp + static_cast<size_t>(p) * d;
    const float s = (row_scale != nullptr) ? __ldg(row_scale + src) : 1.0f;
    for (int c = lane; c < d; c += 32)
      orow[c] = row_scale ? __float2bfloat16_rn(__bfloat162float(xr[c]) * s) : xr[c];
  }
}

__global__ void __launch_bounds__(THREADS) combine_scalar_kernel(const bf16* __restrict__ y,
                                                                 const int32_t* __restrict__ inv,
                                                                 const float* __restrict__ weights,
                                                                 int T, int k, int d,
                                                                 bf16* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * WARPS + (threadIdx.x >> 5);
  const int nw = gridDim.x * WARPS;
  for (long long t = gw; t < T; t += nw) {
    for (int c = lane; c < d; c += 32) {
      float acc = 0.f;
      for (int j = 0; j < k; ++j) {
        const int p = __ldg(inv + static_cast<size_t>(t) * k + j);
        if (p < 0 || !MOE_DBG_IN(DBG_COMBINE_ROW, p, static_cast<long long>(T) * k)) continue;
        const float wj = weights ? __ldg(weights + static_cast<size_t>(t) * k + j) : 1.0f;
        acc = fmaf(wj, __bfloat162float(y[static_cast<size_t>(p) * d + c]), acc);
      }
      out[static_cast<size_t>(t) * d + c] = __float2bfloat16_rn(acc);
    }
  }
}

// Pitch change with a row remap, for shapes whose rows are not 16-byte multiples: the narrow
// layout has rows in blocks of `blk`, split into sub-blocks of `sub` rows; the wide layout has
// blocks of `blk8` rows and sub-blocks of `sub8` >= sub rows (the extra rows and the columns
// past `cols` are zero). Wide row r8 = b*blk8 + s*sub8 + j holds narrow row b*blk + s*sub + j
// when j < sub. to_wide: write every wide row (zero fill); else write every narrow row. With
// `offsets`, only rows below M = offsets[E-1] are written (one block: the activation rows).
template <typename Elem>
__global__ void __launch_bounds__(THREADS) pitch_repack_kernel(
    const Elem* __restrict__ src, Elem* __restrict__ dst, long long rows_out, int cols, int cols8,
    int blk, int sub, int blk8, int sub8, bool to_wide, const int32_t* __restrict__ offsets,
    int E) {
  const long long lim = offsets ? min(rows_out, static_cast<long long>(__ldg(offsets + E - 1))) : rows_out;
  const int lane = threadIdx.x & 31;
  const long long gw = static_cast<long long>(blockIdx.x) * WARPS + (threadIdx.x >> 5);
  const long long nw = static_cast<long long>(gridDim.x) * WARPS;
  for (long long r = gw; r < lim; r += nw) {
    if (to_wide) {
      const long long b = r / blk8;
      const int i = static_cast<int>(r - b * blk8), sb = i / sub8, j = i - sb * sub8;
      const bool has = j < sub;
      const Elem* srow = src + (b * blk + static_cast<long long>(sb) * sub + j) * cols;
      Elem* drow = dst + r * cols8;
      for (int c = lane; c < cols8; c += 32) drow[c] = (has && c < cols) ? srow[c] : Elem(0.0f);
    } else {
      const long long b = r / blk;
      const int i = static_cast<int>(r - b * blk), sb = i / sub, j = i - sb * sub;
      const Elem* srow = src + (b * blk8 + static_cast<long long>(sb) * sub8 + j) * cols8;
      Elem* drow = dst + r * cols;
      for (int c = lane; c < cols; c += 32) drow[c] = srow[c];
    }
  }
}

// Capacity-padded layout (Fig. 35 of "Section 09: Grouped GEMM"): dst[e*C + i] = src row
// offs[e-1] + i for i < min(M_e, C), zero rows for M_e <= i < C.
__global__ void __launch_bounds__(THREADS) pad_rows_kernel(const uint4* __restrict__ src,
                                                           const int32_t* __restrict__ offsets,
                                                           int E, int C, int vec,
                                                           uint4* __restrict__ dst) {
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * WARPS + (threadIdx.x >> 5);
  const int nw = gridDim.x * WARPS;
  const long long rows = static_cast<long long>(E) * C;
  for (long long q = gw; q < rows; q += nw) {
    const int e = static_cast<int>(q / C);
    const int i = static_cast<int>(q - static_cast<long long>(e) * C);
    const int start = e > 0 ? __ldg(offsets + e - 1) : 0;
    const int me = __ldg(offsets + e) - start;
    uint4* d = dst + q * vec;
    if (i < me) {
      const uint4* s = src + static_cast<size_t>(start + i) * vec;
      for (int v = lane; v < vec; v += 32) d[v] = __ldg(s + v);
    } else {
      for (int v = lane; v < vec; v += 32) d[v] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// Back from the padded layout: row p of expert e (i = p - start_e) takes dst[p] = src[e*C + i]
// when i < C; rows beyond the capacity were dropped and get zeros.
__global__ void __launch_bounds__(THREADS) unpad_rows_kernel(const uint4* __restrict__ src,
                                                             const int32_t* __restrict__ offsets,
                                                             int E, int C, int cap, int vec,
                                                             uint4* __restrict__ dst) {
  const int M = min(__ldg(offsets + E - 1), cap);
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * WARPS + (threadIdx.x >> 5);
  const int nw = gridDim.x * WARPS;
  for (long long p = gw; p < M; p += nw) {
    int lo = 0, hi = E - 1;  // first e with offsets[e] > p
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(offsets + mid) > p) hi = mid; else lo = mid + 1;
    }
    const int e = lo;
    const int i = p - (e > 0 ? __ldg(offsets + e - 1) : 0);
    uint4* d = dst + static_cast<size_t>(p) * vec;
    if (i < C) {
      const uint4* s = src + (static_cast<size_t>(e) * C + i) * vec;
      for (int v = lane; v < vec; v += 32) d[v] = __ldg(s + v);
    } else {
      for (int v = lane; v < vec; v += 32) d[v] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// One warp per row, at most one wave: the SM count times the blocks of this kernel that fit on
// an SM at once (the grid strides over the remaining rows).
template <typename Kernel>
int grid_for_rows(Kernel kernel, long long rows) {
  const long long want = (rows + WARPS - 1) / WARPS;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, THREADS, 0) != cudaSuccess ||
      per_sm < 1) {
    (void)cudaGetLastError();
    per_sm = 1;
  }
  const long long cap = static_cast<long long>(device_sm_count()) * per_sm;
  return static_cast<int>(std::max(1LL, std::min(want, cap)));
}

moe_status_t last_launch() {
  const cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? MOE_OK : cuda_fail(err);
}

}  // namespace

MOE_DBG_DEFINE_COLLECTOR(dbg_collect_permute)

moe_status_t launch_permute(const void* x, const int32_t* sorted_src, const int32_t* offsets,
                            const float* row_scale, int n, int k, int E, int d, void* xp,
                            cudaStream_t s) {
  if (n == 0) return MOE_OK;
  if (d % 8 != 0) {
    permute_scalar_kernel<<<grid_for_rows(permute_scalar_kernel, n), THREADS, 0, s>>>(
        static_cast<const bf16*>(x), sorted_src, offsets, row_scale, n, k, E, d, static_cast<bf16*>(xp));
    return last_launch();
  }
  permute_kernel<<<grid_for_rows(permute_kernel, n), THREADS, 0, s>>>(
      static_cast<const uint4*>(x), sorted_src, offsets, row_scale, n, k, E, d / 8,
      static_cast<uint4*>(xp));
  return last_launch();
}

moe_status_t launch_zero_dropped_rows(const int32_t* inv_map, int T, int d, void* out, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  const int blocks = std::max(1, std::min((T + WARPS - 1) / WARPS, 8 * device_sm_count()));
  zero_dropped_rows_kernel<<<blocks, THREADS, 0, s>>>(inv_map, T, d / 8, static_cast<uint4*>(out));
  const cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? MOE_OK : cuda_fail(err);
}

moe_status_t launch_combine(const void* y, const int32_t* inv_map, const float* weights, int T,
                            int k, int d, void* out, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  if (d % 8 != 0) {
    combine_scalar_kernel<<<grid_for_rows(combine_scalar_kernel, T), THREADS, 0, s>>>(
        static_cast<const bf16*>(y), inv_map, weights, T, k, d, static_cast<bf16*>(out));
    return last_launch();
  }
  combine_kernel<<<grid_for_rows(combine_kernel, T), THREADS, 0, s>>>(
      static_cast<const uint4*>(y), inv_map, weights, T, k, d / 8, static_cast<uint4*>(out));
  return last_launch();
}

moe_status_t launch_pitch_repack(const void* src, void* dst, bool fp32, long long rows_out,
                                int cols, int cols8, int blk, int sub, int blk8, int sub8,
                                bool to_wide, const int32_t* offsets, int E, cudaStream_t s) {
  if (rows_out == 0) return MOE_OK;
  if (fp32) {
    pitch_repack_kernel<float><<<grid_for_rows(pitch_repack_kernel<float>, rows_out), THREADS, 0, s>>>(
        static_cast<const float*>(src), static_cast<float*>(dst), rows_out, cols, cols8, blk, sub, blk8,
        sub8, to_wide, offsets, E);
  } else {
    pitch_repack_kernel<bf16><<<grid_for_rows(pitch_repack_kernel<bf16>, rows_out), THREADS, 0, s>>>(
        static_cast<const bf16*>(src), static_cast<bf16*>(dst), rows_out, cols, cols8, blk, sub, blk8,
        sub8, to_wide, offsets, E);
  }
  return last_launch();
}

moe_status_t launch_routing_weight_grad(const float* part, int np, const int32_t* inv_map,
                                        int n_slots, float* dw, cudaStream_t s) {
  if (n_slots == 0) return MOE_OK;
  const int grid = static_cast<int>(std::min<long long>((n_slots + THREADS - 1) / THREADS,
                                                        4LL * device_sm_count()));
  routing_weight_grad_kernel<<<grid, THREADS, 0, s>>>(part, np, inv_map, n_slots, dw);
  return last_launch();
}

moe_status_t launch_pad_rows(const void* src, const int32_t* offsets, int E, int C, int cols,
                             void* dst, cudaStream_t s) {
  const long long rows = static_cast<long long>(E) * C;
  if (rows == 0) return MOE_OK;
  pad_rows_kernel<<<grid_for_rows(pad_rows_kernel, rows), THREADS, 0, s>>>(
      static_cast<const uint4*>(src), offsets, E, C, cols / 8, static_cast<uint4*>(dst));
  return last_launch();
}

moe_status_t launch_unpad_rows(const void* src, const int32_t* offsets, int E, int C, int cap,
                               int cols, void* dst, cudaStream_t s) {
  if (cap == 0) return MOE_OK;
  unpad_rows_kernel<<<grid_for_rows(unpad_rows_kernel, cap), THREADS, 0, s>>>(
      static_cast<const uint4*>(src), offsets, E, C, cap, cols / 8, static_cast<uint4*>(dst));
  return last_launch();
}

}  // namespace moe
