// MXFP8 quantization of bf16 operands ("Section 09: Grouped GEMM", §9.5: the routed MXFP8 path
// runs the forward and the Dgrad as scaled grouped GEMMs).
//
// Format (OCP Microscaling MXFP8): blocks of 32 consecutive elements along the contraction
// dimension share one power-of-two scale X = 2^s stored as E8M0 (s + 127); each element is FP8
// E4M3. s = floor(log2(max |v|)) - 8 (8: the exponent of E4M3's largest normal), clamped to
// [-127, 127], -127 for an all-zero block; elements are v / X rounded to nearest (ties to
// even) with saturation to +-448 (cvt.rn.satfinite). Every input here is bf16, so v / X is
// exact in fp32 and the codes are fully determined by the inputs.
//
// Output layout, chosen for the scaled GEMM's operand loads:
//   codes  [rows, K] bytes, row-major (K-major), read by TMA tiles of 128 rows x 128 bytes.
//   scales blocked by (128-row tile G, 128-column chunk kc): one 512-byte atom per (G, kc),
//          atom index G * KC + kc (KC = ceil(K / 128)), holding the scale of row r (0..127 within
//          the tile) and 32-block kb (0..3 within the chunk) at byte (r % 32) * 16 + (r / 32) * 4
//          + kb. That is the order in which one tcgen05.cp of shape 32x128b with warpx4
//          replication puts 32 lanes x 4 columns of tensor memory: lane r % 32, column r / 32,
//          byte kb, which is where the block-scaled MMA reads the scale of row r for the K-step
//          kb of the chunk.
//   For activations, tiles are the problem list's 128-row tiles (each expert's segment split
//   from its start, as the grouped GEMM walks it): G = (row tiles of the experts before e) +
//   (p - start_e) / 128. For weights [E, N, K], tile G = e * NTpad + n / 128 with NTpad the
//   expert's 128-row tiles rounded up to even (a 256-row B tile always has two atoms).
//   The scales of 32-blocks past K inside the last chunk are written as 2^0 (their codes are
//   TMA zero fill), so every scale a valid output reads is defined.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int MXB = 32;        // elements per scale block
constexpr int MAX_E = 1024;

// Quantize 32 fp32 values (already loaded) into 32 codes; returns the scale code.
__device__ __forceinline__ uint8_t mx_block(const float (&v)[MXB], uint32_t (&codes)[8]) {
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < MXB; ++j) amax = fmaxf(amax, fabsf(v[j]));
  const int s = mx_exponent(amax);
  const float inv = mx_inv_scale(s);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t lo = e4m3x2(v[4 * j] * inv, v[4 * j + 1] * inv);
    const uint32_t hi = e4m3x2(v[4 * j + 2] * inv, v[4 * j + 3] * inv);
    codes[j] = lo | (hi << 16);
  }
  return static_cast<uint8_t>(s + 127);
}

// After the last block of a row: scales of the chunk's 32-blocks past K are 2^0.
__device__ __forceinline__ void fill_chunk_tail(uint8_t* sf, long long G, int KC, int nb, int r) {
  for (int kb = nb; kb < ((nb + 3) & ~3); ++kb) sf[atom_byte(G, KC, kb, r)] = 127;
}

// The problem list as the grouped GEMM derives it from the offsets: s_end[e] = inclusive end of
// expert e's rows, s_pre[e] = 128-row tiles of the experts before e (block-wide scan, 256
// threads). Offsets that decrease or end past `rows` would place rows outside the scale atoms:
// they are flagged (MOE_DEV_BAD_OFFSETS) and the function returns false in every thread.
__device__ bool load_problem_tiles(const int32_t* __restrict__ offsets, int E, long long rows, int* s_end,
                                   int* s_pre, int32_t* status) {
  __shared__ int s_carry;
  __shared__ int wsum[8];
  if (threadIdx.x == 0) s_carry = 0;
  __syncthreads();
  for (int base = 0; base < E; base += blockDim.x) {
    const int e = base + threadIdx.x;
    int tiles = 0;
    if (e < E) {
      const int end = __ldg(offsets + e);
      const int start = e > 0 ? __ldg(offsets + e - 1) : 0;
      s_end[e] = end;
      tiles = (end - start + 127) / 128;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = tiles;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int nb = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += nb;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int before = s_carry;
    for (int w = 0; w < warp; ++w) before += wsum[w];
    if (e < E) s_pre[e] = before + incl - tiles;
    __syncthreads();
    if (threadIdx.x == 0) {
      int tot = 0;
      for (int w = 0; w < 8; ++w) tot += wsum[w];
      s_carry += tot;
    }
    __syncthreads();
  }
  bool bad = false;
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    bad |= (s_end[e] < (e > 0 ? s_end[e - 1] : 0)) || (e == E - 1 && s_end[e] > rows);
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0 && blockIdx.x == 0) record_status(status, MOE_DEV_BAD_OFFSETS);
    return false;
  }
  return true;
}

// Tile (G) and row within the tile (r) of row p of the problem list.
__device__ __forceinline__ void row_tile(const int* s_end, const int* s_pre, int E, long long p, long long& G,
                                         int& r) {
  int lo = 0, hi = E - 1;  // first expert whose segment ends after p
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (s_end[mid] > p) hi = mid; else lo = mid + 1;
  }
  const long long start = lo > 0 ? s_end[lo - 1] : 0;
  G = s_pre[lo] + (p - start) / 128;
  r = static_cast<int>((p - start) % 128);
}

// Rows along K (the contraction), one thread per (row, 32-block). With offsets: rows p < M of a
// problem list (activations); else `rows` rows of E weights of `per_expert` rows each.
__global__ void __launch_bounds__(256) mx_quant_rows_kernel(const bf16* __restrict__ src, long long rows,
                                                            int K, const int32_t* __restrict__ offsets,
                                                            int E, int per_expert, int ntpad,
                                                            uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                                            long long sf_tiles, int32_t* status) {
  __shared__ int s_end[MAX_E];   // inclusive offsets
  __shared__ int s_pre[MAX_E];   // 128-row tiles of the experts before e
  const bool act = offsets != nullptr;
  if (act && !load_problem_tiles(offsets, E, rows, s_end, s_pre, status)) return;
  const int nb = K / MXB;
  const int KC = (K + 127) / 128;
  const long long M = act ? s_end[E - 1] : rows;
  const long long items = M * nb;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < items;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long p = i / nb;
    const int b = static_cast<int>(i - p * nb);
    long long G;
    int r;
    if (act) {
      row_tile(s_end, s_pre, E, p, G, r);
    } else {
      const long long e = p / per_expert, n = p - e * per_expert;
      G = e * ntpad + n / 128;
      r = static_cast<int>(n % 128);
    }
    const uint4* s4 = reinterpret_cast<const uint4*>(src + p * K + b * MXB);
    float v[MXB];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 w = __ldg(s4 + j);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        v[8 * j + 2 * t] = bf16_lo(ww[t]);
        v[8 * j + 2 * t + 1] = bf16_hi(ww[t]);
      }
    }
    uint32_t c[8];
    const uint8_t code = mx_block(v, c);
    uint4* d4 = reinterpret_cast<uint4*>(q + p * K + b * MXB);
    d4[0] = make_uint4(c[0], c[1], c[2], c[3]);
    d4[1] = make_uint4(c[4], c[5], c[6], c[7]);
    if (!MOE_DBG_IN(DBG_MX_TILE, G, sf_tiles)) continue;
    sf[atom_byte(G, KC, b, r)] = code;
    if (b == nb - 1) fill_chunk_tail(sf, G, KC, nb, r);
  }
}

// The gather of the permute (xp[p] = x[sorted_src[p] / k]) and the quantization of the gathered
// row along d in one pass: one warp per row p < M; lane l moves 16-byte pieces l, l + 32, ...
// (8 elements each), four consecutive lanes hold one 32-element block and agree on its scale
// by two shuffles. Optionally also writes the bf16 row (the BF16 wgrad's operand).
__global__ void __launch_bounds__(256) mx_permute_quant_kernel(const uint4* __restrict__ x,
                                                               const int32_t* __restrict__ sorted_src,
                                                               const int32_t* __restrict__ offsets, int E,
                                                               int n, int k, int d, uint4* __restrict__ xp,
                                                               uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                                               long long sf_tiles, int32_t* status) {
  __shared__ int s_end[MAX_E];
  __shared__ int s_pre[MAX_E];
  if (!load_problem_tiles(offsets, E, n, s_end, s_pre, status)) return;
  const int M = s_end[E - 1];
  const int vec = d / 8, nb = d / MXB, KC = (d + 127) / 128;
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int nw = gridDim.x * 8;
  for (long long p = gw; p < M; p += nw) {
    const int src = __ldg(sorted_src + p);
    if (src < 0 || src >= n) continue;  // warp-uniform
    long long G;
    int r;
    row_tile(s_end, s_pre, E, p, G, r);
    const uint4* xr = x + static_cast<size_t>(src / k) * vec;
    for (int v0 = 0; v0 < vec; v0 += 32) {  // every lane runs every pass: the shuffles need the warp
      const int v = v0 + lane;
      const bool act = v < vec;                // vec % 4 == 0: a block's four lanes agree
      const uint4 w4 = act ? __ldg(xr + v) : make_uint4(0u, 0u, 0u, 0u);
      if (act && xp != nullptr) __stcs(xp + static_cast<size_t>(p) * vec + v, w4);
      const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
      float f[8];
      float amax = 0.f;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        f[2 * t] = bf16_lo(ww[t]);
        f[2 * t + 1] = bf16_hi(ww[t]);
        amax = fmaxf(amax, fmaxf(fabsf(f[2 * t]), fabsf(f[2 * t + 1])));
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      const int e8 = mx_exponent(amax);
      const float inv = mx_inv_scale(e8);
      if (act) {
        const uint32_t lo = e4m3x2(f[0] * inv, f[1] * inv) | (e4m3x2(f[2] * inv, f[3] * inv) << 16);
        const uint32_t hi = e4m3x2(f[4] * inv, f[5] * inv) | (e4m3x2(f[6] * inv, f[7] * inv) << 16);
        *reinterpret_cast<uint2*>(q + static_cast<size_t>(p) * d + v * 8) = make_uint2(lo, hi);
        if ((lane & 3) == 0 && MOE_DBG_IN(DBG_MX_TILE, G, sf_tiles)) {
          const int b = v >> 2;
          sf[atom_byte(G, KC, b, r)] = static_cast<uint8_t>(e8 + 127);
          if (b == nb - 1) fill_chunk_tail(sf, G, KC, nb, r);
        }
      }
    }
  }
}

// A weight [E, R, C] quantized along R (its rows): output [E, C, R] codes (K = R contiguous),
// scale atoms per (expert, 128-column tile of C, chunk of R). One thread per (e, 32-block of R,
// column c), c fastest: the 32 strided reads of a thread are coalesced across the warp.
__global__ void __launch_bounds__(256) mx_quant_cols_kernel(const bf16* __restrict__ w, int E, int R, int C,
                                                            int ntpad, uint8_t* __restrict__ q,
                                                            uint8_t* __restrict__ sf) {
  const int nb = R / MXB;
  const int KC = (R + 127) / 128;
  const long long items = static_cast<long long>(E) * nb * C;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < items;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i % C);
    const long long rest = i / C;
    const int b = static_cast<int>(rest % nb);
    const int e = static_cast<int>(rest / nb);
    const bf16* col = w + (static_cast<long long>(e) * R + static_cast<long long>(b) * MXB) * C + c;
    float v[MXB];
#pragma unroll
    for (int j = 0; j < MXB; ++j) v[j] = __bfloat162float(col[static_cast<long long>(j) * C]);
    uint32_t cd[8];
    const uint8_t code = mx_block(v, cd);
    uint4* d4 = reinterpret_cast<uint4*>(q + (static_cast<long long>(e) * C + c) * R + b * MXB);
    d4[0] = make_uint4(cd[0], cd[1], cd[2], cd[3]);
    d4[1] = make_uint4(cd[4], cd[5], cd[6], cd[7]);
    const long long G = static_cast<long long>(e) * ntpad + c / 128;
    if (!MOE_DBG_IN(DBG_MX_TILE, G, static_cast<long long>(E) * ntpad)) continue;
    sf[atom_byte(G, KC, b, c % 128)] = code;
    if (b == nb - 1) fill_chunk_tail(sf, G, KC, nb, c % 128);
  }
}

int grid_for(long long items) {
  const long long blocks = (items + 255) / 256;
  return static_cast<int>(std::max(1LL, std::min<long long>(blocks, 16LL * device_sm_count())));
}

// scale-atom tiles of a problem list of at most `rows` rows over E experts (each expert's segment
// starts a tile): the size the activation scale buffers are given
long long activation_sf_tiles(long long rows, int E) { return (rows + 127LL * E) / 128; }

}  // namespace

MOE_DBG_DEFINE_COLLECTOR(dbg_collect_mx)

int mx_ntpad(int N) { return 2 * ((((N + 127) / 128) + 1) / 2); }
int mx_kc(int K) { return (K + 127) / 128; }

moe_status_t launch_mx_quant_rows(const void* src, long long rows, int K, const int32_t* offsets, int E,
                                  int per_expert, void* q, void* sf, int32_t* status, cudaStream_t s) {
  if (K % MXB != 0 || E < 1 || E > MAX_E) return MOE_ERR_UNSUPPORTED_SHAPE;
  const long long items = rows * (K / MXB);
  if (items == 0) return MOE_OK;
  const int ntpad = offsets ? 0 : mx_ntpad(per_expert);
  const long long sf_tiles = offsets ? activation_sf_tiles(rows, E) : (rows / per_expert) * ntpad;
  mx_quant_rows_kernel<<<grid_for(items), 256, 0, s>>>(static_cast<const bf16*>(src), rows, K, offsets, E,
                                                       per_expert, ntpad, static_cast<uint8_t*>(q),
                                                       static_cast<uint8_t*>(sf), sf_tiles, status);
  const cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? MOE_OK : cuda_fail(err);
}

moe_status_t launch_mx_permute_quant(const void* x, const int32_t* sorted_src, const int32_t* offsets, int E,
                                    int n, int k, int d, void* xp, void* q, void* sf, int32_t* status,
                                    cudaStream_t s) {
  if (d % MXB != 0 || E < 1 || E > MAX_E) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (n == 0) return MOE_OK;
  const int blocks = static_cast<int>(std::max(1LL, std::min((static_cast<long long>(n) + 7) / 8,
                                                            8LL * device_sm_count())));
  mx_permute_quant_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint4*>(x), sorted_src, offsets, E, n, k, d,
                                                 static_cast<uint4*>(xp), static_cast<uint8_t*>(q),
                                                 static_cast<uint8_t*>(sf), activation_sf_tiles(n, E), status);
  const cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? MOE_OK : cuda_fail(err);
}

moe_status_t launch_mx_quant_cols(const void* w, int E, int R, int C, void* q, void* sf, cudaStream_t s) {
  if (R % MXB != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  const long long items = static_cast<long long>(E) * (R / MXB) * C;
  if (items == 0) return MOE_OK;
  mx_quant_cols_kernel<<<grid_for(items), 256, 0, s>>>(static_cast<const bf16*>(w), E, R, C, mx_ntpad(C),
                                                       static_cast<uint8_t*>(q), static_cast<uint8_t*>(sf));
  const cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? MOE_OK : cuda_fail(err);
}

}  // namespace moe
