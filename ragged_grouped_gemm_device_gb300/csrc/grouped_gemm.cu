// Persistent, device-scheduled grouped GEMM on the 5th-generation tensor cores (sm_103a).
//
// "Section 09: Grouped GEMM" (Fig. 37): the cumulative expert offsets stay on the GPU, a
// preparation step derives the problem list, and one grouped kernel schedules tiles across it.
// Here the preparation is the kernel's own prologue: every CTA reads the E offsets into shared
// memory, derives each expert's row segment and 128-row tile count, and prefix-sums the tile
// counts; a tile index then maps to (expert, row block, column block) by binary search. The
// grid is one CTA per SM; CTA c takes tiles c, c + grid, ... ("thread blocks take tiles in
// turn"). The host never learns M. A wgrad launch may carry two independent gradients over the
// same experts (the down and the up/gate projection's): the second one's tiles follow the
// first's in the same tile sequence, so one persistent launch covers both.
//
// Roles (384 threads, warp-specialised):
//   warp 0      TMA producer of the A operand: 128B-swizzled tiles into a 4-stage
//               shared-memory ring (the wgrad's stages hold A high, A low and half of B).
//   warp 10     TMA producer of the B operand into the same stages.
//   warp 1      tensor-memory allocator and MMA issuer: tcgen05.mma 128x256x16 (bf16 in, fp32
//               accumulate) into one of two 256-column TMEM accumulators, so the epilogue of a
//               tile overlaps the main loop of the next. A contraction longer than SEG_KB K
//               blocks takes both: its later segments go to the second one.
//   warps 2..9  epilogue, two warps per TMEM lane quadrant (each takes half of the tile's
//               columns): tcgen05.ld of the accumulator, fused SwiGLU (forward or backward),
//               conversion and row/column-masked stores. A tile that runs past its expert's
//               segment still multiplies the neighbouring rows (rows of a product are
//               independent) but never stores them. For a segmented contraction they first
//               add each later segment into the tile's accumulator (fp32, tcgen05.st).
//   warp 11     wgrad: zeroes the rows of the next expert in each expert's last K block.
// The wgrad modes contract over the M_e rows of an expert (Table 15) with MN-major operands.
// They run as pairs of CTAs (clusters of two, tcgen05 cta_group::2) on 256 x 256 gradient
// tiles: each CTA stages its 128 gradient rows of A and 128 of the tile's 256 B rows, the even
// CTA issues M = 256 MMAs that read both CTAs' stages and write each CTA's 128 accumulator rows
// into its own tensor memory, and each CTA stores its rows. Per SM that moves 48 KB of
// operands per 64-deep K block instead of 64 KB for the same MMA work. The odd CTA's copies
// complete on the even CTA's barriers; the even CTA's MMAs release both CTAs' stages. An
// expert's last K block runs only the 16-row K steps that hold its rows, and the rows of the
// next expert inside the last of them are zeroed in both CTAs' stages by warp 11 before the MMA
// issuer sees the stage as full. The A operand comes as a bf16 high/low pair (the activation
// and its rounding remainder); both halves are multiplied with the same B tile into one fp32
// accumulator, which keeps about 16 significant bits of the activations in the weight
// gradient.
#include <algorithm>
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int BM = 128;          // UMMA M: accumulator rows = TMEM lanes
constexpr int BN = 256;          // UMMA N: accumulator columns
constexpr int BK = 64;           // one 128-byte swizzle atom of bf16 along K
constexpr int UK = 16;           // K of one tcgen05.mma kind::f16
constexpr int STAGES = 4;                     // ring depth of the row-grouped modes
constexpr int MAX_STAGES = 6;                 // deepest ring of any mode (bf16-only wgrad)
constexpr int A_BYTES = BM * BK * 2;          // 16 KB
constexpr int B_BYTES = BN * BK * 2;          // 32 KB
constexpr int RING_BYTES = STAGES * (A_BYTES + B_BYTES);  // 192 KB, shared by every mode
constexpr int ATOM_BYTES = 64 * BK * 2;       // one MN-major 64x64 box: 8 KB
constexpr int EPI_WARPS = 8;                 // epilogue warps: 2 per TMEM lane quadrant
constexpr int PRODUCER_B_WARP = 2 + EPI_WARPS;  // second TMA producer (B operand)
constexpr int ZERO_WARP = PRODUCER_B_WARP + 1;   // wgrad: zeroes the rows of the next expert
constexpr int THREADS = 32 * (ZERO_WARP + 1);
constexpr int TMEM_COLS = 512;                // two 256-column accumulators
constexpr int MAX_E = 1024;
constexpr int RASTER_M = 16;                  // row tiles per raster group (see decode_tile)
constexpr int CTL_BYTES = 256;
// The tensor core adds each MMA's products into the fp32 accumulator without rounding to
// nearest: measured on GB300, the error of one accumulator grows with the number of K steps
// like truncation (an rms error of 1.2 on sums of rms 990 after 2^20 products, against 0.005
// for round-to-nearest fp32). A tile whose contraction is longer than SEG_KB K blocks therefore
// accumulates in segments of SEG_KB blocks: the first into its own accumulator R, each later one
// into the other tensor-memory buffer P, which the epilogue adds into R in fp32 (round to
// nearest) before the next segment starts. Shorter contractions (every K up to 8192 here) keep
// the double-buffered pipeline unchanged.
constexpr int SEG_KB = 128;
// per epilogue warp, one 32-row x 16-column fp32 chunk staged for a TMA store (wgrad), or two
// 32-row x 16-column bf16 boxes (dgrad)
constexpr int STAGE_OUT_BYTES = 32 * 16 * 4;
constexpr int STAGING_BYTES = EPI_WARPS * STAGE_OUT_BYTES;
// MXFP8 modes: per stage, the scale atoms of A (512 bytes) and of B's two 128-row halves
// (2 x 512); in tensor memory each stage's scales take 12 columns of a 16-column slot after
// the (single) accumulator
constexpr int SF_STAGE_BYTES = 1536;
constexpr int SF_RING_BYTES = STAGES * SF_STAGE_BYTES;
constexpr int SF_TMEM_COL = 256;
constexpr int MX_BK = 128;                    // K elements per MXFP8 stage (128 bytes of E4M3)
constexpr int MX_UK = 32;                     // K of one block-scaled MMA

struct Ctl {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tail_full[MAX_STAGES];  // wgrad: the stage of an expert's last K block has landed
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t done;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Ctl) <= CTL_BYTES, "control block too large");

constexpr size_t smem_bytes_for(int E) {
  return 1024 + static_cast<size_t>(RING_BYTES) + SF_RING_BYTES + STAGING_BYTES + CTL_BYTES +
         2 * sizeof(int) * static_cast<size_t>(E + 2);
}

// Segments of a tile's contraction: one unless the tile is longer than SEG_KB K blocks and the
// mode has two accumulators (the MXFP8 modes hold their scales in the second half of tensor
// memory and keep one accumulator).
template <int NACC>
__device__ __forceinline__ int num_segments(int kblocks) {
  return (NACC == 2 && kblocks > SEG_KB) ? (kblocks + SEG_KB - 1) / SEG_KB : 1;
}

template <int MODE>
struct ModeTraits {
  static constexpr bool mx = MODE >= MODE_UP_SWIGLU_MX;
  // the bf16 mode whose tile shape and epilogue this mode has
  static constexpr int epi = mx ? MODE - MODE_UP_SWIGLU_MX : MODE;
  static constexpr bool wgrad = (MODE == MODE_WGRAD || MODE == MODE_WGRAD_BF16);
  static constexpr bool a_mn = wgrad;
  static constexpr bool b_mn = (MODE == MODE_PLAIN_BF16 || wgrad);
  static constexpr int out_cols_per_tile = (epi == MODE_UP_SWIGLU) ? 128 : BN;
  // accumulators in tensor memory: two (a tile's epilogue overlaps the next tile's main loop),
  // one in the MXFP8 modes, whose scale slots take the other half of the 512 columns
  static constexpr int nacc = mx ? 1 : 2;
  static constexpr int bk = mx ? MX_BK : BK;  // K elements per stage
  // The wgrad modes run as pairs of CTAs (clusters of two) on 256-row gradient tiles: each CTA
  // stages its 128 rows of A and half (128) of the tile's 256 B rows, and the even CTA of the
  // pair issues M = 256 MMAs (cta_group::2) that read both CTAs' shared memory and write each
  // CTA's 128 accumulator rows into its own tensor memory. Per SM that is 48 KB of operands
  // (hi/lo) per 64-deep K block instead of 64 KB for the same MMA work.
  static constexpr bool pair = wgrad;
  static constexpr int cg = pair ? 2 : 1;              // CTA group of every tcgen05 instruction
  static constexpr int tile_m = pair ? 2 * BM : BM;    // wgrad: gradient rows per tile
  static constexpr int b_rows = pair ? BN / 2 : BN;    // B rows staged by this CTA
  // MODE_WGRAD stages hold A high, A low and this CTA's half of B: 48 KB, four of them; the
  // bf16-only wgrad 32 KB, six; the row-grouped modes 48 KB, four
  static constexpr int a_parts = (MODE == MODE_WGRAD) ? 2 : 1;
  static constexpr int stage_bytes = a_parts * A_BYTES + b_rows * BK * 2;
  static constexpr int stages = RING_BYTES / stage_bytes;
  static_assert(stages <= MAX_STAGES, "ring deeper than the control block's barriers");
  static_assert(tile_m % BM == 0 && out_cols_per_tile % 16 == 0 && bk % UK == 0, "tile shape");
  static_assert(!wgrad || pair, "the wgrad modes run as CTA pairs");
  // A and B parts of each stage loaded by two producer threads (see the producer role)
  static constexpr bool split_producer = true;
};

struct Tile {
  int e;        // expert index within the problem list
  int g;        // row-grouped: row tile index over the whole problem list
  int row0;     // first row of the tile (row-grouped) or of the expert segment (wgrad)
  int rows;     // valid rows of the tile (row-grouped)
  int m0;       // wgrad: first output row
  int n0;       // first output column
  int kblocks;  // K blocks of 64
  int kvalid;   // wgrad: contraction length M_e
  int prob;     // wgrad: 0 for the first gradient of the launch, 1 for the second
};

struct Sched {
  const int* offs;  // offs[e] = first row of expert e, offs[E] = end (E+1 entries)
  const int* pre;   // row-grouped: prefix of 128-row tiles, E+1 entries
  int E;
  int nt;           // column tiles per problem (wgrad: of the first gradient)
  int mt;           // wgrad: row tiles per expert gradient (first gradient)
  int nt2, mt2;     // wgrad: the same for the second gradient (0 without one)
  int total0;       // wgrad: tiles of the first gradient
  int kblocks;      // row-grouped: K blocks
  int total;        // tiles
};

template <int MODE>
__device__ __forceinline__ Tile decode_tile(const Sched& s, int t) {
  Tile ti;
  ti.prob = 0;
  if constexpr (ModeTraits<MODE>::wgrad) {
    // the first gradient's tiles, then the second's; within a gradient (expert, row tile,
    // column tile), column tile fastest: the CTAs in flight share an expert's A column slice
    // and its rows of B, which stay in L2
    int tt = t;
    if (tt >= s.total0) {
      tt -= s.total0;
      ti.prob = 1;
    }
    const int nt = ti.prob ? s.nt2 : s.nt;
    const int per = (ti.prob ? s.mt2 : s.mt) * nt;
    ti.e = tt / per;
    const int r = tt - ti.e * per;
    const int mi = r / nt;
    ti.m0 = mi * ModeTraits<MODE>::tile_m;
    ti.n0 = (r - mi * nt) * BN;
    ti.row0 = s.offs[ti.e];
    ti.kvalid = s.offs[ti.e + 1] - ti.row0;
    ti.kblocks = (ti.kvalid + BK - 1) / BK;
    ti.rows = 0;
    ti.g = 0;
  } else {
    // expert e owns tiles [pre[e]*nt, pre[e+1]*nt): largest e with pre[e] <= t/nt (experts
    // without tiles have pre[e] == pre[e+1]); pre counts 128-row tiles
    const int nt = s.nt;
    const int gq = t / nt;
    int lo = 0, hi = s.E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s.pre[mid] <= gq) lo = mid; else hi = mid;
    }
    ti.e = lo;
    // Inside the expert, groups of up to RASTER_M row tiles are walked column tile by column
    // tile (row tile fastest): the CTAs in flight then share a few column slices of the weight
    // and a few row tiles of the input, which stay in L2 even when the expert's weight does not
    // (a weight of 8192 x 20480 columns would otherwise be re-read for every row tile).
    const int mt_e = s.pre[lo + 1] - s.pre[lo];
    const int l = t - s.pre[lo] * nt;
    const int grp = l / (RASTER_M * nt);
    const int gm = min(RASTER_M, mt_e - grp * RASTER_M);
    const int within = l - grp * RASTER_M * nt;
    const int m_local = grp * RASTER_M + within % gm;
    const int n = within / gm;
    ti.g = s.pre[lo] + m_local;
    ti.row0 = s.offs[lo] + m_local * BM;
    ti.rows = min(BM, s.offs[lo + 1] - ti.row0);
    ti.n0 = n * ModeTraits<MODE>::out_cols_per_tile;
    ti.m0 = 0;
    ti.kblocks = s.kblocks;
    ti.kvalid = 0;
  }
  return ti;
}

__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

// x / (1 + e^-x) and 1 / (1 + e^-x) with the approximate division (an infinite denominator
// gives 0, the limit)
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }
__device__ __forceinline__ float sigmoid_f(float g) { return __fdividef(1.0f, 1.0f + __expf(-g)); }

// The saved U, blocked the way the epilogue holds it: for row tile G (of the problem list), TMEM
// lane quadrant q and 16-column chunk ci (ci < H16 = ceil(h/16): gate columns 16ci.., else up
// columns 16(ci - H16)..), one 1536-byte block of three 512-byte planes, lane l's 16 bytes of
// plane p at byte p * 512 + l * 16. Each value is the fp32 U rounded to nearest even at 24 bits
// (sign, 8 exponent and 15 mantissa bits: 16 significant bits); plane 0 holds the upper 16 bits
// of columns 0..7 of the chunk, plane 1 those of columns 8..15 and plane 2 the lower 8 bits of
// all 16. A warp's store or load of one plane is one contiguous 512 bytes, and the chunks of one
// (G, q) are contiguous. Each row tile owns its blocks; the slots of its rows past the expert's
// segment are neither written nor read.
constexpr int U_BLOCK_BYTES = 1536;

__device__ __forceinline__ uint4* u_block(const void* base, long long G, int q, int ci, int c2) {
  return const_cast<uint4*>(reinterpret_cast<const uint4*>(base)) + ((G * 4 + q) * c2 + ci) * (U_BLOCK_BYTES / 16);
}

// 16 fp32 values (as bits) -> the three 16-byte planes of this lane
__device__ __forceinline__ void u24_pack(const uint32_t (&x)[16], uint4& p0, uint4& p1, uint4& p2) {
  uint32_t v[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = (x[j] + 0x7Fu + ((x[j] >> 8) & 1u)) >> 8;  // 24 bits, to nearest even
  p0 = make_uint4((v[0] >> 8) | ((v[1] >> 8) << 16), (v[2] >> 8) | ((v[3] >> 8) << 16),
                  (v[4] >> 8) | ((v[5] >> 8) << 16), (v[6] >> 8) | ((v[7] >> 8) << 16));
  p1 = make_uint4((v[8] >> 8) | ((v[9] >> 8) << 16), (v[10] >> 8) | ((v[11] >> 8) << 16),
                  (v[12] >> 8) | ((v[13] >> 8) << 16), (v[14] >> 8) | ((v[15] >> 8) << 16));
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    w[k] = (v[4 * k] & 0xFFu) | ((v[4 * k + 1] & 0xFFu) << 8) | ((v[4 * k + 2] & 0xFFu) << 16) |
           ((v[4 * k + 3] & 0xFFu) << 24);
  p2 = make_uint4(w[0], w[1], w[2], w[3]);
}

// the three planes of one lane -> its 16 values (all-zero planes give +0)
__device__ __forceinline__ void u24_unpack(const uint4 (&p)[3], float (&f)[16]) {
  const uint32_t hi[8] = {p[0].x, p[0].y, p[0].z, p[0].w, p[1].x, p[1].y, p[1].z, p[1].w};
  const uint32_t lo[4] = {p[2].x, p[2].y, p[2].z, p[2].w};
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint32_t h16 = (j & 1) ? (hi[j >> 1] >> 16) : (hi[j >> 1] & 0xFFFFu);
    const uint32_t l8 = (lo[j >> 2] >> (8 * (j & 3))) & 0xFFu;
    f[j] = __uint_as_float((h16 << 16) | (l8 << 8));
  }
}

// 32-byte store (sm_100+ global vector width); the address must be 32-byte aligned
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* v) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

__device__ __forceinline__ void st_global_v4(void* p, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  *reinterpret_cast<uint4*>(p) = make_uint4(a, b, c, d);
}

// Contraction rows [r0, r1) of every 64x64 box of a wgrad stage (SB bytes at sp) belong to the
// next expert: zero them, in this CTA's stage and in the odd CTA's copy of it (same offsets). The
// swizzle only permutes 16-byte pieces inside a 128-byte row, so those rows are the contiguous
// bytes [r0 * 128, r1 * 128) of each box. One warp; the zeros are made visible to the tensor
// cores' reads of both CTAs' shared memory.
template <int SB>
__device__ __forceinline__ void zero_stage_rows(uint8_t* sp, int r0, int r1, int lane) {
  const int pieces = (r1 - r0) * 8;
  const uint32_t peer = cluster_addr(smem_u32(sp), 1u);
#pragma unroll
  for (int atom = 0; atom < SB / ATOM_BYTES; ++atom) {
    const int off = atom * ATOM_BYTES + r0 * 128;
    uint4* base = reinterpret_cast<uint4*>(sp + off);
    for (int c = lane; c < pieces; c += 32) {
      base[c] = make_uint4(0u, 0u, 0u, 0u);
      st_cluster_zero16(peer + off + c * 16);
    }
  }
  fence_proxy_async_smem();
  fence_proxy_async_cluster();
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs args) {
  constexpr int NST = ModeTraits<MODE>::stages;
  constexpr int SB = ModeTraits<MODE>::stage_bytes;
  constexpr int APARTS = ModeTraits<MODE>::a_parts;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem;
  uint8_t* sf_ring = smem + RING_BYTES;  // MXFP8 scale atoms, one slot per stage
  uint8_t* staging = smem + RING_BYTES + SF_RING_BYTES;
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + RING_BYTES + SF_RING_BYTES + STAGING_BYTES);
  int* offs = reinterpret_cast<int*>(smem + RING_BYTES + SF_RING_BYTES + STAGING_BYTES + CTL_BYTES);
  constexpr int EPI = ModeTraits<MODE>::epi;
  constexpr int NACC = ModeTraits<MODE>::nacc;
  constexpr bool MX = ModeTraits<MODE>::mx;
  constexpr bool PAIR = ModeTraits<MODE>::pair;
  constexpr int CG = ModeTraits<MODE>::cg;
  constexpr uint32_t B_STAGE = ModeTraits<MODE>::b_rows * BK * 2;  // B bytes this CTA stages
  const int E = args.E;
  int* pre = offs + (E + 1);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // CTA pairs: rank 0 issues the MMAs of the pair; both CTAs load, stage and store their halves
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;

  // ---- problem list: row segments of the experts (the preparation step, in-kernel)
  const bool single = args.single_expert >= 0;
  const int expert_base = single ? args.single_expert : 0;
  for (int i = tid; i <= E; i += THREADS) {
    int v;
    if (single) v = args.single_row0 + (i > 0 ? args.single_rows : 0);
    else if (args.uniform_rows > 0) v = i * args.uniform_rows;
    else v = (i == 0) ? 0 : __ldg(args.offsets + i - 1);
    offs[i] = v;
  }
  __syncthreads();
  bool bad = false;
  for (int i = tid; i < E; i += THREADS) bad |= (offs[i + 1] < offs[i]) || (offs[i] < 0);
  if (tid == 0) bad |= offs[E] > args.cap;
  if (__syncthreads_or(bad)) {
    if (tid == 0 && blockIdx.x == 0) record_status(args.status, MOE_DEV_BAD_OFFSETS);
    return;  // uniform across the CTA, before any barrier or tensor memory exists
  }

  Sched sc;
  sc.offs = offs;
  sc.pre = pre;
  sc.E = E;
  if constexpr (ModeTraits<MODE>::wgrad) {
    constexpr int TM = ModeTraits<MODE>::tile_m;
    sc.mt = (args.Mdim + TM - 1) / TM;
    sc.nt = (args.N + BN - 1) / BN;
    const bool two = args.nprob == 2;
    sc.mt2 = two ? (args.Mdim2 + TM - 1) / TM : 0;
    sc.nt2 = two ? (args.N2 + BN - 1) / BN : 0;
    sc.kblocks = 0;
    sc.total0 = E * sc.mt * sc.nt;
    sc.total = sc.total0 + E * sc.mt2 * sc.nt2;
  } else {
    sc.mt = 0;
    sc.mt2 = sc.nt2 = sc.total0 = 0;
    sc.nt = (args.N + ModeTraits<MODE>::out_cols_per_tile - 1) / ModeTraits<MODE>::out_cols_per_tile;
    sc.kblocks = (args.K + ModeTraits<MODE>::bk - 1) / ModeTraits<MODE>::bk;
    if (warp == 0) {
      int carry = 0;
      if (lane == 0) pre[0] = 0;
      for (int base = 0; base < E; base += 32) {
        const int e = base + lane;
        const int mt_e = (e < E) ? (offs[e + 1] - offs[e] + BM - 1) / BM : 0;
        int v = mt_e;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int nb = __shfl_up_sync(0xffffffffu, v, o);
          if (lane >= o) v += nb;
        }
        if (e < E) pre[e + 1] = carry + v;
        carry += __shfl_sync(0xffffffffu, v, 31);
      }
    }
  }

  // ---- barriers and tensor memory
  if (tid == 0) {
    // full: this CTA's producers (with pairs the even CTA's expect the odd CTA's bytes too, and
    // the odd CTA's are unused); tempty: every epilogue thread, or with pairs (on the even CTA
    // only) one arrival per epilogue warp of both CTAs
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), ModeTraits<MODE>::split_producer ? 2 : 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
      mbar_init(smem_u32(&ctl->tail_full[s]), ModeTraits<MODE>::split_producer ? 2 : 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctl->tfull[b]), 1);
      mbar_init(smem_u32(&ctl->tempty[b]), PAIR ? 2 * EPI_WARPS : 32 * EPI_WARPS);
    }
    mbar_init(smem_u32(&ctl->done), 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&maps.a);
    if (APARTS == 2) prefetch_tmap(&maps.a_lo);
    prefetch_tmap(&maps.b);
    if (ModeTraits<MODE>::wgrad && args.nprob == 2) {
      prefetch_tmap(&maps.a2);
      if (APARTS == 2) prefetch_tmap(&maps.a_lo2);
      prefetch_tmap(&maps.b2);
    }
  }
  if (warp == 1) {
    tmem_alloc<CG>(smem_u32(&ctl->tmem_base), TMEM_COLS);
    tmem_relinquish<CG>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the peer's barriers must be initialised before any arrival or commit can reach them
  if constexpr (PAIR) cluster_sync_all();
  if constexpr (!ModeTraits<MODE>::wgrad) sc.total = pre[E] * sc.nt;
  // CTA pairs take tiles in turn by cluster, single CTAs by block
  const int t_first = PAIR ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int t_step = PAIR ? static_cast<int>(nclusters_x()) : static_cast<int>(gridDim.x);
  const uint32_t tmem_base = ctl->tmem_base;
  volatile int* abort_flag = &ctl->abort_flag;
  const long long tmo = args.timeout_ns;
  int32_t* status = args.status;
  const uint32_t stage0 = smem_u32(stages);
  const uint32_t sf0 = smem_u32(sf_ring);

  // Two producer threads fill each stage: lane 0 of warp 0 loads the A part, lane 0 of the last
  // warp the B part. Each arrives on the stage's full barrier (count 2) with the bytes it will
  // deliver, so the phase completes when both have arrived and every byte has landed, in
  // whatever order. One instruction stream per part halves the serial issue latency per stage
  // (the MN-major B part alone is four boxes). With CTA pairs the even CTA's producers expect
  // the bytes of both CTAs' parts and the odd CTA's copies complete on the even CTA's barrier
  // (the odd CTA only loads after its own empty barrier, released by the even CTA's MMAs of
  // the stage's previous use, so its bytes always count towards the current phase).
  constexpr bool SPLIT = ModeTraits<MODE>::split_producer;
  const int prole = (warp == 0) ? 0 : (SPLIT && warp == PRODUCER_B_WARP) ? 1 : -1;
  if (prole >= 0) {
    // =========================================================== TMA producers
    if (lane == 0) {
      const bool do_a = prole == 0, do_b = !SPLIT || prole == 1;
      uint32_t it = 0;
      bool ok = true;
      for (int t = t_first; t < sc.total && ok; t += t_step) {
        const Tile ti = decode_tile<MODE>(sc, t);
        const int eg = ti.e + expert_base;
        constexpr uint32_t A_SF = MX ? 512u : 0u, B_SF = MX ? 1024u : 0u;
        const uint32_t bytes = ((do_a ? static_cast<uint32_t>(APARTS * A_BYTES) + A_SF : 0u) +
                                (do_b ? B_STAGE + B_SF : 0u)) * (PAIR ? 2u : 1u);
        for (int kb = 0; kb < ti.kblocks; ++kb, ++it) {
          const int s = it % NST;
          const uint32_t ph = (it / NST) & 1u;
          if (!mbar_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag, status, tmo)) {
            ok = false;
            break;
          }
          // wgrad: the last K block of an expert whose rows end inside a 16-row K step completes
          // on the stage's tail_full barrier instead; the zeroing warp completes full after it
          // has zeroed the next expert's rows
          bool ztail = false;
          if constexpr (ModeTraits<MODE>::wgrad) ztail = kb == ti.kblocks - 1 && (ti.kvalid % UK) != 0;
          const uint32_t fl = smem_u32(ztail ? &ctl->tail_full[s] : &ctl->full[s]);
          const uint32_t fb = (PAIR && rank != 0) ? cluster_addr(fl, 0u) : fl;
          if (!(PAIR && rank != 0)) mbar_arrive_expect_tx(fb, bytes);
          const uint32_t sa = stage0 + s * SB;
          const uint32_t sb = sa + APARTS * A_BYTES;
          const int k0 = kb * BK;
          // A: this CTA's rows; B: the whole tile. The issue path is kept straight-line: it is
          // on the critical path of the MN-major modes.
          if constexpr (MX) {
            // E4M3 codes, 128 bytes of K per row, and the scale atoms of this K chunk: A's by the
            // row tile of the problem list, B's by expert and 128-row tile (gate and up halves
            // of W_ug for the up/gate product, else two consecutive tiles of N)
            const int kc = kb;
            const int m0 = kb * MX_BK;
            const uint32_t sfs = sf0 + s * SF_STAGE_BYTES;
            if (do_a) {
              tma_load_2d(sa, &maps.a, m0, ti.row0, fb);
              long long ta = args.tile_base + ti.g;
              if (!MOE_DBG_IN(DBG_GG_SFA, ta, args.dbg_sfa_tiles)) ta = 0;
              bulk_load(sfs, args.sfa + (ta * args.sf_kc + kc) * 512, 512, fb);
            }
            if (do_b) {
              const long long eb = static_cast<long long>(eg) * args.sfb_ntpad;
              int nt0, nt1;
              if constexpr (EPI == MODE_UP_SWIGLU) {
                tma_load_3d(sb, &maps.b, m0, ti.n0, eg, fb);
                tma_load_3d(sb + B_BYTES / 2, &maps.b, m0, args.h + ti.n0, eg, fb);
                nt0 = ti.n0 / 128;
                nt1 = (args.h + ti.n0) / 128;
              } else {
                tma_load_3d(sb, &maps.b, m0, ti.n0, eg, fb);  // 256 rows of B in one box
                nt0 = ti.n0 / 128;
                nt1 = nt0 + 1;
              }
              long long tb0 = eb + nt0, tb1 = eb + nt1;
              if (!MOE_DBG_IN(DBG_GG_SFB, tb0, args.dbg_sfb_tiles)) tb0 = 0;
              if (!MOE_DBG_IN(DBG_GG_SFB, tb1, args.dbg_sfb_tiles)) tb1 = 0;
              bulk_load(sfs + 512, args.sfb + (tb0 * args.sf_kc + kc) * 512, 512, fb);
              bulk_load(sfs + 1024, args.sfb + (tb1 * args.sf_kc + kc) * 512, 512, fb);
            }
          } else if constexpr (!ModeTraits<MODE>::wgrad) {
            if (do_a) tma_load_2d(sa, &maps.a, k0, ti.row0, fb);
          }
          if constexpr (MX) {
          } else if constexpr (MODE == MODE_UP_SWIGLU) {
            if (do_b) {
              tma_load_3d(sb, &maps.b, k0, ti.n0, eg, fb);                            // gate rows
              tma_load_3d(sb + B_BYTES / 2, &maps.b, k0, args.h + ti.n0, eg, fb);     // up rows
            }
          } else if constexpr (MODE == MODE_PLAIN_BF16) {
            if (do_b) {
#pragma unroll
              for (int i = 0; i < BN / 64; ++i)
                tma_load_3d(sb + i * ATOM_BYTES, &maps.b, ti.n0 + 64 * i, k0, eg, fb);
            }
          } else if constexpr (MODE == MODE_DGRAD_SWIGLU) {
            if (do_b) tma_load_3d(sb, &maps.b, k0, ti.n0, eg, fb);  // 256 rows of W_down in one box
          } else {
            // MN-major 64 x 64 boxes from the operands of this tile's gradient: this CTA's 128
            // rows of the 256-row tile (two boxes of A and two of its low half) and its 128 of
            // the tile's 256 B rows (two boxes). Rows past the gradient read as zeros.
            const int rk = ti.row0 + k0;  // first contraction row of this K block
            auto load = [&](uint32_t dst, const CUtensorMap* map, int c0) {
              if (rank != 0) tma_load_2d_peer(dst, map, c0, rk, fb);
              else tma_load_2d(dst, map, c0, rk, fb);
            };
            if (do_a) {
              const CUtensorMap* ma = ti.prob ? &maps.a2 : &maps.a;
              const int am = ti.m0 + static_cast<int>(rank) * BM;
#pragma unroll
              for (int i = 0; i < BM / 64; ++i) load(sa + i * ATOM_BYTES, ma, am + 64 * i);
              if constexpr (APARTS == 2) {
                const CUtensorMap* ml = ti.prob ? &maps.a_lo2 : &maps.a_lo;
#pragma unroll
                for (int i = 0; i < BM / 64; ++i) load(sa + A_BYTES + i * ATOM_BYTES, ml, am + 64 * i);
              }
            }
            if (do_b) {
              const CUtensorMap* mb = ti.prob ? &maps.b2 : &maps.b;
              constexpr int BR = ModeTraits<MODE>::b_rows;
              const int bn = ti.n0 + static_cast<int>(rank) * BR;
#pragma unroll
              for (int i = 0; i < BR / 64; ++i) load(sb + i * ATOM_BYTES, mb, bn + 64 * i);
            }
          }
        }
      }
      // drain: the copies this thread issued into each stage must land before the CTA can exit.
      // After an abort a stage may lack the other producer's part and never complete; the first
      // wait that runs out (drain_ns, seconds) has outlasted every copy issued here, so stop.
      // The odd CTA of a pair cannot wait on the even CTA's barriers: its copies have landed
      // once the even CTA's MMAs consumed them (the pair leaves together, after the even CTA's
      // last MMA); after an abort it gives them a bounded 200 us instead.
      if (PAIR && rank != 0) {
        if (!ok) {
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 200000ull) __nanosleep(1000);
        }
      } else {
        const uint32_t first = it > NST ? it - NST : 0u;
        for (uint32_t j = first; j < it; ++j)
          if (!mbar_wait(smem_u32(&ctl->full[j % NST]), (j / NST) & 1u, abort_flag, status, args.drain_ns, false))
            break;
      }
    }
  } else if (warp == 1 && rank == 0) {
    // =========================================================== MMA issuer
    // (with CTA pairs, on the even CTA only: M = 256 over both CTAs' stages)
    constexpr uint32_t idesc =
        idesc_bf16_f32(PAIR ? 2 * BM : BM, BN, ModeTraits<MODE>::a_mn, ModeTraits<MODE>::b_mn);
    // barriers of the odd CTA that this CTA's commits also arrive on (pairs)
    [[maybe_unused]] const uint32_t peer_empty0 = PAIR ? cluster_addr(smem_u32(&ctl->empty[0]), 1u) : 0u;
    [[maybe_unused]] const uint32_t peer_tfull0 = PAIR ? cluster_addr(smem_u32(&ctl->tfull[0]), 1u) : 0u;
    uint32_t it = 0, turn = 0;
    uint32_t use0 = 0, use1 = 0;  // completed uses of accumulator buffers 0 and 1 (registers)
    bool ok = true;
    for (int t = t_first; t < sc.total && ok; t += t_step) {
      const Tile ti = decode_tile<MODE>(sc, t);
      if (ti.kblocks == 0) continue;
      // segment 0 into this tile's buffer (turn), later segments into the other one (SEG_KB)
      const int nseg = num_segments<NACC>(ti.kblocks);
      const int seg_len = nseg == 1 ? ti.kblocks : SEG_KB;
      for (int sg = 0; sg < nseg && ok; ++sg) {
        const uint32_t buf = sg == 0 ? turn : (turn ^ 1u);
        ok = warp_all(mbar_wait(smem_u32(&ctl->tempty[buf]), ((buf ? use1 : use0) & 1u) ^ 1u, abort_flag,
                                      status, tmo));
        if (!ok) break;
        tc_fence_after();
        const uint32_t dtm = tmem_base + buf * BN;
        const int kb0 = sg * seg_len, kb1 = min(ti.kblocks, kb0 + seg_len);
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % NST;
          const uint32_t ph = (it / NST) & 1u;
          ok = warp_all(mbar_wait(smem_u32(&ctl->full[s]), ph, abort_flag, status, tmo));
          if (!ok) break;
          tc_fence_after();
          // wgrad: the last K block of an expert runs only the 16-row K steps that hold its
          // rows (kq of them); the rows of the next expert inside the last of those have been
          // zeroed by the zeroing warp before it completed the stage's full barrier
          [[maybe_unused]] int kq = BK / UK;
          if constexpr (ModeTraits<MODE>::wgrad) {
            const int valid = ti.kvalid - kb * BK;
            if (valid < BK) kq = (valid + UK - 1) / UK;
          }
          if constexpr (MX) {
            if (lane == 0) {
              // the stage's scale atoms into this stage's tensor-memory slot (A: 4 columns, B: 8),
              // then four block-scaled MMAs of K = 32, each reading byte ks of the scale words;
              // tcgen05.cp and tcgen05.mma from one thread execute in issue order
              const uint32_t sa = stage0 + s * SB;
              const uint32_t sb = sa + A_BYTES;
              const uint32_t sfs = sf0 + s * SF_STAGE_BYTES;
              const uint32_t sft = tmem_base + SF_TMEM_COL + s * 16;
              tmem_cp_32x128b_x4(sft, smem_desc_rows16(sfs));
              tmem_cp_32x128b_x4(sft + 4, smem_desc_rows16(sfs + 512));
              tmem_cp_32x128b_x4(sft + 8, smem_desc_rows16(sfs + 1024));
              constexpr uint32_t idesc_mx = idesc_mxf8_e4m3(BM, BN);
#pragma unroll
              for (int ks = 0; ks < MX_BK / MX_UK; ++ks) {
                const uint64_t ad = smem_desc_sw128(sa + ks * MX_UK, 16, 1024);
                const uint64_t bd = smem_desc_sw128(sb + ks * MX_UK, 16, 1024);
                mma_mxf8_ss(dtm, ad, bd, idesc_mx | idesc_sf_ids(static_cast<uint32_t>(ks)), sft, sft + 4,
                            ((kb - kb0) | ks) != 0 ? 1u : 0u);
              }
              mma_commit(smem_u32(&ctl->empty[s]));
            }
            __syncwarp();
            continue;
          }
          if (lane == 0) {
            const uint32_t sa = stage0 + s * SB;
            const uint32_t sb = sa + APARTS * A_BYTES;
#pragma unroll
            for (int part = 0; part < APARTS; ++part) {
#pragma unroll
              for (int ks = 0; ks < BK / UK; ++ks) {
                if (ks >= kq) break;
                const uint32_t ap = sa + part * A_BYTES;
                const uint64_t ad = ModeTraits<MODE>::a_mn
                                        ? smem_desc_sw128(ap + ks * (UK * 128), ATOM_BYTES, 1024)
                                        : smem_desc_sw128(ap + ks * (UK * 2), 16, 1024);
                const uint64_t bd = ModeTraits<MODE>::b_mn
                                        ? smem_desc_sw128(sb + ks * (UK * 128), ATOM_BYTES, 1024)
                                        : smem_desc_sw128(sb + ks * (UK * 2), 16, 1024);
                mma_bf16_ss<CG>(dtm, ad, bd, idesc, ((kb - kb0) | ks | part) != 0 ? 1u : 0u);
              }
            }
            // release the stage to the producers (of both CTAs of a pair) once these MMAs have
            // read it
            mma_commit<CG>(smem_u32(&ctl->empty[s]));
            if constexpr (PAIR) mma_commit<CG>(peer_empty0 + s * static_cast<uint32_t>(sizeof(uint64_t)));
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) {
          mma_commit<CG>(smem_u32(&ctl->tfull[buf]));
          if constexpr (PAIR) mma_commit<CG>(peer_tfull0 + buf * static_cast<uint32_t>(sizeof(uint64_t)));
        }
        __syncwarp();
        if (buf) ++use1; else ++use0;
      }
      if (!ok) break;
      if constexpr (NACC == 2) turn ^= 1u;
    }
    // every MMA this thread issued must finish before tensor memory is released
    if (lane == 0) mma_commit<CG>(smem_u32(&ctl->done));
    __syncwarp();
    mbar_wait(smem_u32(&ctl->done), 0u, abort_flag, status, args.drain_ns, false);
  } else if (ModeTraits<MODE>::wgrad && warp == ZERO_WARP && rank == 0) {
    // =========================================================== tail zeroing (wgrad, even CTA)
    // For each expert whose rows end inside a 16-row K step: once its last K block has landed in
    // both CTAs (tail_full), zero the next expert's rows of that K step in both CTAs' copies of
    // the stage, then complete the stage's full barrier for the MMA issuer. tail_full's phases
    // advance only at these blocks, and a stage's next one cannot land before the MMAs have
    // consumed this one, so each wait is for the barrier's current phase.
    uint32_t it = 0, tpar = 0;
    for (int t = t_first; t < sc.total; t += t_step) {
      const Tile ti = decode_tile<MODE>(sc, t);
      it += static_cast<uint32_t>(ti.kblocks);
      if (ti.kblocks == 0 || (ti.kvalid % UK) == 0) continue;
      const int sl = static_cast<int>((it - 1u) % NST);
      if (!warp_all(mbar_wait(smem_u32(&ctl->tail_full[sl]), (tpar >> sl) & 1u, abort_flag, status, tmo))) break;
      tpar ^= 1u << sl;
      const int valid = ti.kvalid - (ti.kblocks - 1) * BK;
      zero_stage_rows<SB>(stages + sl * SB, valid, ((valid + UK - 1) / UK) * UK, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive_count(smem_u32(&ctl->full[sl]), ModeTraits<MODE>::split_producer ? 2u : 1u);
    }
  } else if (warp >= 2 && warp < 2 + EPI_WARPS) {
    // =========================================================== epilogue (warps 2..9)
    const int q = warp & 3;           // TMEM lane quadrant this warp may access
    const int half = (warp - 2) >> 2; // which half of the tile's columns this warp stores
    const int r_in = q * 32 + lane;   // accumulator row = TMEM lane
    uint32_t turn = 0;
    uint32_t use0 = 0, use1 = 0;      // completed uses of accumulator buffers 0 and 1
    uint32_t box_ctr = 0;             // dgrad: staging boxes this warp has stored
    // hand accumulator buffer b back to the MMA issuer: with CTA pairs one arrival per warp on
    // the even CTA's barrier (the odd CTA's accumulator rows are written by the even CTA's MMAs)
    [[maybe_unused]] const uint32_t tempty0 = PAIR ? cluster_addr(smem_u32(&ctl->tempty[0]), 0u) : 0u;
    auto release_acc = [&](uint32_t b) {
      tc_fence_before();
      if constexpr (PAIR) {
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(tempty0 + b * static_cast<uint32_t>(sizeof(uint64_t)));
      } else {
        mbar_arrive(smem_u32(&ctl->tempty[b]));
      }
    };
    for (int t = t_first; t < sc.total; t += t_step) {
      const Tile ti = decode_tile<MODE>(sc, t);
      // wgrad: the gradient this tile belongs to
      [[maybe_unused]] const int gN = ti.prob ? args.N2 : args.N;
      [[maybe_unused]] const int gM = ti.prob ? args.Mdim2 : args.Mdim;
      if constexpr (ModeTraits<MODE>::wgrad) {
        if (ti.kblocks == 0) {
          // empty expert: its gradient is zero (this CTA's 128 rows of the tile)
          const int mrow = ti.m0 + static_cast<int>(rank) * BM + r_in;
          if (mrow < gM) {
            float* dst = reinterpret_cast<float*>(ti.prob ? args.out_b : args.out) +
                         (static_cast<long long>(ti.e + expert_base) * gM + mrow) * (ti.prob ? args.ldo_b : args.ldo);
            for (int c = ti.n0 + half * (BN / 2); c < min(ti.n0 + (half + 1) * (BN / 2), gN); c += 4)
              *reinterpret_cast<float4*>(dst + c) = make_float4(0.f, 0.f, 0.f, 0.f);
          }
          continue;
        }
      }
      // dgrad: the saved U does not depend on the accumulator, so this warp requests its first
      // chunk before waiting for the tile. (An L2 prefetch of the next tile's U measured slower.)
      uint4 gcur[3], ucur[3];  // the three planes of this lane's gate and up values (u_block)
      if constexpr (EPI == MODE_DGRAD_SWIGLU) {
        const int h16 = (args.h + 15) >> 4;
        const int cw = BN / 32;  // 16-column chunks per warp
        const int c0 = (ti.n0 >> 4) + half * cw;
#pragma unroll
        for (int j = 0; j < 3; ++j) {
          gcur[j] = make_uint4(0u, 0u, 0u, 0u);
          ucur[j] = gcur[j];
        }
        if (r_in < ti.rows && c0 < h16 && MOE_DBG_IN(DBG_GG_TILE, args.tile_base + ti.g, args.dbg_u_tiles)) {
          const uint4* bg = u_block(args.aux, args.tile_base + ti.g, q, c0, 2 * h16);
          const uint4* bu = u_block(args.aux, args.tile_base + ti.g, q, h16 + c0, 2 * h16);
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            gcur[j] = __ldg(bg + j * 32 + lane);
            ucur[j] = __ldg(bu + j * 32 + lane);
          }
        }
      }
      const uint32_t buf = turn;
      if (!warp_all(mbar_wait(smem_u32(&ctl->tfull[buf]), (buf ? use1 : use0) & 1u, abort_flag, status, tmo)))
        break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * BN;
      const int nseg = num_segments<NACC>(ti.kblocks);
      if (nseg > 1) {
        // a segmented contraction (SEG_KB): add each later segment's partial sums (the other
        // buffer) into this tile's accumulator, fp32 round to nearest, over exactly the columns
        // this warp reads below, then hand the buffer back for the next segment
        const uint32_t pb = turn ^ 1u;
        const uint32_t tp = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + pb * BN;
        bool seg_ok = true;
        for (int sg = 1; sg < nseg; ++sg) {
          if (!warp_all(mbar_wait(smem_u32(&ctl->tfull[pb]), (pb ? use1 : use0) & 1u, abort_flag, status, tmo))) {
            seg_ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int i = 0; i < 8; ++i) {
            // UP_SWIGLU: gate chunks half*4.. and the matching up chunks 128 columns on; else
            // chunks half*8..half*8+7
            const int col = (EPI == MODE_UP_SWIGLU) ? (i < 4 ? (half * 4 + i) * 16 : 128 + (half * 4 + i - 4) * 16)
                                                    : (half * 8 + i) * 16;
            uint32_t vr[16], vp[16];
            tmem_ld16(tb + col, vr);
            tmem_ld16(tp + col, vp);
            tmem_ld_wait2(vr, vp);
#pragma unroll
            for (int j = 0; j < 16; ++j) vr[j] = __float_as_uint(__uint_as_float(vr[j]) + __uint_as_float(vp[j]));
            tmem_st16(tb + col, vr);
          }
          tmem_st_wait();
          release_acc(pb);
          if (pb) ++use1; else ++use0;
        }
        if (!seg_ok) break;
      }

      if constexpr (EPI == MODE_UP_SWIGLU) {
        bool rv = r_in < ti.rows;
        const long long row = ti.row0 + r_in;
        if (rv && !MOE_DBG_IN(DBG_GG_ROW, row, args.cap)) rv = false;
        const int h = args.h;
        bf16* arow = reinterpret_cast<bf16*>(args.out) + row * args.ldo;
        bf16* lrow = args.out3 ? reinterpret_cast<bf16*>(args.out3) + row * args.ldo3 : nullptr;
        const long long G = args.tile_base + ti.g;
        const bool u_out = args.out2 != nullptr && MOE_DBG_IN(DBG_GG_TILE, G, args.dbg_u_tiles);
        const int h16 = (h + 15) >> 4;
        // P = w*A with the row's routing weight (else P = A): bf16(P) is the down projection's
        // input, P - bf16(P) its low half for the down wgrad
        float wrow = 1.0f;
        if (args.row_weight != nullptr && rv) {
          const int slot = __ldg(args.row_src + row);
          if (MOE_DBG_IN(DBG_GG_SLOT, slot, args.cap)) wrow = __ldg(args.row_weight + slot);
        }
        // chunk c's gate and up columns: U (blocked), then bf16(P) and its low half; bf16(P) is
        // also left in pout for the MXFP8 quantization of the pair of chunks
        auto process = [&](int c, const uint32_t (&g)[16], const uint32_t (&u)[16], uint32_t (&pout)[8]) {
          const int col = ti.n0 + c * 16;
          if (!rv || col >= h) return;
          if (u_out) {
            // U in its blocked 24-bit layout: 512 contiguous bytes per warp-wide store
            uint4* bg = u_block(args.out2, G, q, col >> 4, 2 * h16);
            uint4* bu = u_block(args.out2, G, q, h16 + (col >> 4), 2 * h16);
            uint4 p0, p1, p2;
            u24_pack(g, p0, p1, p2);
            bg[lane] = p0;
            bg[32 + lane] = p1;
            bg[64 + lane] = p2;
            u24_pack(u, p0, p1, p2);
            bu[lane] = p0;
            bu[32 + lane] = p1;
            bu[64 + lane] = p2;
          }
          uint32_t pa[8], pl[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float p0 = wrow * (silu_f(__uint_as_float(g[2 * j])) * __uint_as_float(u[2 * j]));
            const float p1 = wrow * (silu_f(__uint_as_float(g[2 * j + 1])) * __uint_as_float(u[2 * j + 1]));
            pa[j] = pack_bf16x2(p0, p1);
            pl[j] = pack_bf16x2(p0 - bf16_lo(pa[j]), p1 - bf16_hi(pa[j]));
            pout[j] = pa[j];
          }
          const bool two = col + 16 <= h;
          if (args.vec32) {
            st_global_v8(arow + col, pa);
            if (lrow) st_global_v8(lrow + col, pl);
          } else {
            st_global_v4(arow + col, pa[0], pa[1], pa[2], pa[3]);
            if (two) st_global_v4(arow + col + 8, pa[4], pa[5], pa[6], pa[7]);
            if (lrow) {
              st_global_v4(lrow + col, pl[0], pl[1], pl[2], pl[3]);
              if (two) st_global_v4(lrow + col + 8, pl[4], pl[5], pl[6], pl[7]);
            }
          }
        };
        // four chunks per warp; chunk c+1's accumulator columns are in flight while chunk c is
        // processed
        const int cb = half * 4;
        uint32_t ga[16], ua[16], gb[16], ub[16];
        uint32_t pq0[8], pq1[8];
        tmem_ld16(tb + cb * 16, ga);
        tmem_ld16(tb + 128 + cb * 16, ua);
        tmem_ld_wait2(ga, ua);
#pragma unroll 1
        for (int c = cb; c < cb + 4; c += 2) {
          tmem_ld16(tb + (c + 1) * 16, gb);
          tmem_ld16(tb + 128 + (c + 1) * 16, ub);
          process(c, ga, ua, pq0);
          tmem_ld_wait2(gb, ub);
          const bool more = c + 2 < cb + 4;
          if (more) {
            tmem_ld16(tb + (c + 2) * 16, ga);
            tmem_ld16(tb + 128 + (c + 2) * 16, ua);
          }
          process(c + 1, gb, ub, pq1);
          if constexpr (MX) {
            // the down projection's A operand: bf16(P) of these 32 columns as one MXFP8 block
            const int col = ti.n0 + c * 16;
            if (args.mxq != nullptr && rv && col < h && MOE_DBG_IN(DBG_GG_MXSF, G, args.dbg_mxsf_tiles)) {
              uint32_t codes[8];
              const uint8_t sc = mx_block_bf16(pq0, pq1, codes);
              st_global_v8(args.mxq + row * args.mx_ldq + col, codes);
              args.mxsf[atom_byte(G, args.mx_kc, col >> 5, r_in)] = sc;
            }
          }
          if (more) tmem_ld_wait2(ga, ua);
        }
      } else if constexpr (EPI == MODE_PLAIN_BF16) {
        bool rv = r_in < ti.rows;
        const long long row = ti.row0 + r_in;
        if (rv && !MOE_DBG_IN(DBG_GG_ROW, row, args.cap)) rv = false;
        long long orow_idx = row;
        if (args.row_dst != nullptr && rv) {
          orow_idx = __ldg(args.row_dst + row);
          if (!MOE_DBG_IN(DBG_GG_DST, orow_idx, args.dbg_dst_rows)) rv = false;
        }
        bf16* orow = reinterpret_cast<bf16*>(args.out) + orow_idx * args.ldo;
        // 32 columns (two 16-column chunks) at a time; the next pair's accumulator columns are
        // in flight while this pair is converted and stored
        auto store_pair = [&](int c, const uint32_t (&v0)[16], const uint32_t (&v1)[16]) {
          const int col = ti.n0 + c * 16;
          if (!rv) return;
          uint32_t p[16];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            p[j] = pack_bf16x2(__uint_as_float(v0[2 * j]), __uint_as_float(v0[2 * j + 1]));
            p[8 + j] = pack_bf16x2(__uint_as_float(v1[2 * j]), __uint_as_float(v1[2 * j + 1]));
          }
          if (args.vec32 && col + 32 <= args.N) {
            st_global_v8(orow + col, p);
            st_global_v8(orow + col + 16, p + 8);
            return;
          }
#pragma unroll
          for (int hq = 0; hq < 4; ++hq)
            if (col + hq * 8 < args.N)
              st_global_v4(orow + col + hq * 8, p[4 * hq], p[4 * hq + 1], p[4 * hq + 2], p[4 * hq + 3]);
        };
        const int cb = half * (BN / 32), ce = cb + BN / 32;  // four pairs of chunks
        uint32_t va[16], vb[16], vc[16], vd[16];
        tmem_ld16(tb + cb * 16, va);
        tmem_ld16(tb + (cb + 1) * 16, vb);
        tmem_ld_wait2(va, vb);
#pragma unroll 1
        for (int c = cb; c < ce; c += 4) {
          tmem_ld16(tb + (c + 2) * 16, vc);
          tmem_ld16(tb + (c + 3) * 16, vd);
          store_pair(c, va, vb);
          tmem_ld_wait2(vc, vd);
          const bool more = c + 4 < ce;
          if (more) {
            tmem_ld16(tb + (c + 4) * 16, va);
            tmem_ld16(tb + (c + 5) * 16, vb);
          }
          store_pair(c + 2, vc, vd);
          if (more) tmem_ld_wait2(va, vb);
        }
      } else if constexpr (EPI == MODE_DGRAD_SWIGLU) {
        bool rv = r_in < ti.rows;
        const long long row = ti.row0 + r_in;
        if (rv && !MOE_DBG_IN(DBG_GG_ROW, row, args.cap)) rv = false;
        const int h = args.h;
        const int h16 = (h + 15) >> 4;
        const long long G = args.tile_base + ti.g;
        const bool u_in = MOE_DBG_IN(DBG_GG_TILE, G, args.dbg_u_tiles);
        bf16* hrow = reinterpret_cast<bf16*>(args.out) + row * args.ldo;
        bf16* lrow = reinterpret_cast<bf16*>(args.out2) + row * args.ldo2;
        float wrow = 1.0f;
        if (args.row_weight != nullptr && rv) {
          const int slot = __ldg(args.row_src + row);
          if (MOE_DBG_IN(DBG_GG_SLOT, slot, args.cap)) wrow = __ldg(args.row_weight + slot);
        }
        // A warp whose 32 rows all belong to the tile's expert sends whole 16-column chunks out
        // through two 1 KB staging boxes (32-byte swizzle: lane r's 16-byte piece j at piece
        // j ^ ((r >> 2) & 1), conflict-free) and TMA tensor stores: full sectors from the copy
        // engine instead of 32 rows of 16-byte stores per instruction. A box never crosses into
        // the up half or past the slab, so rows of the next expert are never written.
        const bool slab_full = q * 32 + 32 <= ti.rows;  // warp-uniform
        const int y0 = static_cast<int>(ti.row0) + q * 32;
        auto stage_store = [&](const uint32_t (&w)[8], const CUtensorMap* map, int x) {
          uint8_t* sbuf = staging + (warp - 2) * STAGE_OUT_BYTES + (box_ctr & 1u) * 1024;
          if (lane == 0) bulk_wait_group_read1();  // this buffer's previous box has been read
          __syncwarp();
          const int sw = (lane >> 2) & 1;
          *reinterpret_cast<uint4*>(sbuf + lane * 32 + (sw << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4*>(sbuf + lane * 32 + ((sw ^ 1) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(map, smem_u32(sbuf), x, y0);
            bulk_commit_group();
          }
          ++box_ctr;
        };
        // saved U of chunk c (zeros past the last column chunk): this lane's three planes of
        // the gate and of the up values, each load one coalesced 512 bytes per warp
        auto load_u = [&](int c, uint4 (&gq)[3], uint4 (&uq)[3]) {
          const int ci = (ti.n0 >> 4) + c;
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            gq[j] = make_uint4(0u, 0u, 0u, 0u);
            uq[j] = gq[j];
          }
          if (rv && ci < h16 && u_in) {
            const uint4* bg = u_block(args.aux, G, q, ci, 2 * h16);
            const uint4* bu = u_block(args.aux, G, q, h16 + ci, 2 * h16);
#pragma unroll
            for (int j = 0; j < 3; ++j) {
              gq[j] = __ldg(bg + j * 32 + lane);
              uq[j] = __ldg(bu + j * 32 + lane);
            }
          }
        };
        // dA = w * acc; dgate = dA * up * s * (1 + gate * (1 - s)), dup = dA * silu(gate), as
        // bf16 high and low halves. With dw_part: this lane's share of <A, acc> for the
        // routing-weight gradient, A = silu(gate) * up unweighted and acc = dy W_down^T before w
        // (<A, dy W_down^T> = <A W_down, dy>: the unweighted expert output against dOut).
        float dw_acc = 0.f;
        auto process = [&](int c, const uint32_t (&v)[16], uint32_t (&gout)[8], uint32_t (&uout)[8]) {
          const int col = ti.n0 + c * 16;
          if (!rv || col >= h) return;
          const bool two = col + 16 <= h;
          float gv[16], uv[16];
          u24_unpack(gcur, gv);
          u24_unpack(ucur, uv);
          uint32_t gh[8], gl[8], uh[8], ul[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float dg[2], du[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const float g = gv[2 * j + hh], uu = uv[2 * j + hh];
              const float acc_raw = __uint_as_float(v[2 * j + hh]);
              const float da = wrow * acc_raw;
              const float sg = sigmoid_f(g);
              dg[hh] = da * uu * sg * (1.0f + g * (1.0f - sg));
              du[hh] = da * g * sg;
              if (two || j < 4) dw_acc = fmaf(g * sg * uu, acc_raw, dw_acc);  // columns < h
            }
            gh[j] = pack_bf16x2(dg[0], dg[1]);
            uh[j] = pack_bf16x2(du[0], du[1]);
            gl[j] = pack_bf16x2(dg[0] - bf16_lo(gh[j]), dg[1] - bf16_hi(gh[j]));
            ul[j] = pack_bf16x2(du[0] - bf16_lo(uh[j]), du[1] - bf16_hi(uh[j]));
            if constexpr (MX) {
              gout[j] = gh[j];
              uout[j] = uh[j];
            }
          }
          if (slab_full && two) {
            stage_store(gh, &maps.out, col);
            stage_store(uh, &maps.out, h + col);
            stage_store(gl, &maps.out2, col);
            stage_store(ul, &maps.out2, h + col);
            return;
          }
          if (args.vec32) {
            // whole 16-column chunks (h % 16 == 0), 32-byte aligned rows: one full sector a row
            st_global_v8(hrow + col, gh);
            st_global_v8(hrow + h + col, uh);
            st_global_v8(lrow + col, gl);
            st_global_v8(lrow + h + col, ul);
            return;
          }
          st_global_v4(hrow + col, gh[0], gh[1], gh[2], gh[3]);
          st_global_v4(hrow + h + col, uh[0], uh[1], uh[2], uh[3]);
          st_global_v4(lrow + col, gl[0], gl[1], gl[2], gl[3]);
          st_global_v4(lrow + h + col, ul[0], ul[1], ul[2], ul[3]);
          if (two) {
            st_global_v4(hrow + col + 8, gh[4], gh[5], gh[6], gh[7]);
            st_global_v4(hrow + h + col + 8, uh[4], uh[5], uh[6], uh[7]);
            st_global_v4(lrow + col + 8, gl[4], gl[5], gl[6], gl[7]);
            st_global_v4(lrow + h + col + 8, ul[4], ul[5], ul[6], ul[7]);
          }
        };
        const int cb = half * (BN / 32), ce = cb + BN / 32;  // an even number of chunks
        uint4 gnxt[3], unxt[3];
        uint32_t v0[16], v1[16];
        // MXFP8 dgrad: dU's high half of a pair of chunks, kept for its quantization
        [[maybe_unused]] uint32_t qg0[8], qu0[8], qg1[8], qu1[8];
        tmem_ld16(tb + cb * 16, v0);
        tmem_ld_wait(v0);
        // two chunks per iteration: the accumulator columns and saved U of the next chunk are
        // in flight while the current one is processed
#pragma unroll 1
        for (int c = cb; c < ce; c += 2) {
          tmem_ld16(tb + (c + 1) * 16, v1);
          load_u(c + 1, gnxt, unxt);
          process(c, v0, qg0, qu0);
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            gcur[j] = gnxt[j];
            ucur[j] = unxt[j];
          }
          tmem_ld_wait(v1);
          const bool more = c + 2 < ce;
          if (more) {
            tmem_ld16(tb + (c + 2) * 16, v0);
            load_u(c + 2, gnxt, unxt);
          }
          process(c + 1, v1, qg1, qu1);
          if constexpr (MX) {
            // the up/gate dgrad's A operand: dU's high half of these 32 gate and 32 up columns
            // as two MXFP8 blocks along 2h
            const int col = ti.n0 + c * 16;
            if (args.mxq != nullptr && rv && col < h && MOE_DBG_IN(DBG_GG_MXSF, G, args.dbg_mxsf_tiles)) {
              uint32_t codes[8];
              uint8_t* qrow = args.mxq + row * args.mx_ldq;
              uint8_t sc = mx_block_bf16(qg0, qg1, codes);
              st_global_v8(qrow + col, codes);
              args.mxsf[atom_byte(G, args.mx_kc, col >> 5, r_in)] = sc;
              sc = mx_block_bf16(qu0, qu1, codes);
              st_global_v8(qrow + h + col, codes);
              args.mxsf[atom_byte(G, args.mx_kc, (h + col) >> 5, r_in)] = sc;
            }
          }
          if (more) {
#pragma unroll
            for (int j = 0; j < 3; ++j) {
              gcur[j] = gnxt[j];
              ucur[j] = unxt[j];
            }
            tmem_ld_wait(v0);
          }
        }
        // every (row, column tile, half) slot is written once, zero when it has no column < h
        if (args.dw_part != nullptr && rv)
          args.dw_part[row * args.dw_np + (ti.n0 / BN) * 2 + half] = dw_acc;
      } else {  // wgrad modes
        // Each 32-row x 16-column fp32 chunk goes through this warp's staging buffer (64-byte
        // swizzle: lane r writes its row's 16-byte piece j at piece j ^ ((r >> 1) & 3), which
        // keeps the shared-memory writes conflict-free) and out by a TMA tensor store, which
        // writes whole lines and clips at the gradient's row and column bounds.
        uint8_t* sbuf = staging + (warp - 2) * STAGE_OUT_BYTES;
        const uint32_t sbuf_addr = smem_u32(sbuf);
        const int sw = (lane >> 1) & 3;
        const int m_cta = ti.m0 + static_cast<int>(rank) * BM;  // this CTA's rows of the tile
        const bool rows_in = m_cta + q * 32 < gM;  // warp-uniform
        const CUtensorMap* mo = ti.prob ? &maps.out2 : &maps.out;
#pragma unroll 1
        for (int c = half * (BN / 32); c < (half + 1) * (BN / 32); ++c) {
          uint32_t v[16];
          tmem_ld16(tb + c * 16, v);
          tmem_ld_wait(v);
          // a box that would start past the gradient's last row or column is not stored
          if (!rows_in || ti.n0 + c * 16 >= gN) continue;
          if (lane == 0) bulk_wait_group_read0();  // the previous chunk has left the buffer
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(sbuf + lane * 64 + ((j ^ sw) << 4)) =
                make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(mo, sbuf_addr, ti.n0 + c * 16, m_cta + q * 32, ti.e + expert_base);
            bulk_commit_group();
          }
        }
      }
      release_acc(buf);
      if (buf) ++use1; else ++use0;
      if constexpr (NACC == 2) turn ^= 1u;
    }
  }

  // ---- teardown: every role has finished (or given up); release tensor memory
  if ((ModeTraits<MODE>::wgrad || ModeTraits<MODE>::epi == MODE_DGRAD_SWIGLU) && warp >= 2 && lane == 0)
    bulk_wait_group0();
  tc_fence_before();
  __syncthreads();
  // with CTA pairs the even CTA's MMAs write this CTA's tensor memory and read its shared memory:
  // neither CTA releases (or exits) before both are done
  if constexpr (PAIR) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<CG>(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

template <int MODE>
moe_status_t launch_mode(const GemmMaps& maps, const GemmArgs& args, long long max_tiles,
                         cudaStream_t stream) {
  const size_t smem = smem_bytes_for(args.E);
  const cudaError_t attr_err = ensure_max_dynamic_smem(
      reinterpret_cast<const void*>(grouped_gemm_kernel<MODE>), static_cast<int>(smem_bytes_for(MAX_E)));
  if (attr_err != cudaSuccess) return cuda_fail(attr_err);
  const long long sms = device_sm_count();
  if constexpr (ModeTraits<MODE>::pair) {
    // clusters of two CTAs (one per SM), as many as can be resident at once; max_tiles counts
    // the 256-row pair tiles
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(std::max(2LL, sms & ~1LL)));
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, grouped_gemm_kernel<MODE>, &cfg) != cudaSuccess || clusters < 1) {
      cudaGetLastError();
      clusters = static_cast<int>(std::max(1LL, sms / 2));
    }
    const long long pairs = std::max(1LL, std::min<long long>(clusters, max_tiles));
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
    const cudaError_t lerr = cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<MODE>, maps, args);
    if (lerr != cudaSuccess) return cuda_fail(lerr);
  } else {
    const int grid = static_cast<int>(std::max(1LL, std::min(sms, max_tiles)));
    grouped_gemm_kernel<MODE><<<grid, THREADS, smem, stream>>>(maps, args);
  }
  const cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? MOE_OK : cuda_fail(err);
}

}  // namespace

MOE_DBG_DEFINE_COLLECTOR(dbg_collect_grouped)

int gemm_tiles_n(int mode, int N) {
  const int w = (mode == MODE_UP_SWIGLU || mode == MODE_UP_SWIGLU_MX) ? 128 : BN;
  return (N + w - 1) / w;
}

bool make_map_rows2d(CUtensorMap* map, const void* ptr, long long rows, long long cols,
                     int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows <= 0 || cols <= 0) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_grad3d_f32(CUtensorMap* map, const void* ptr, long long E, long long R, long long C) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || E <= 0 || R <= 0 || C <= 0) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(R),
                              static_cast<cuuint64_t>(E)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(C) * 4,
                                 static_cast<cuuint64_t>(R) * static_cast<cuuint64_t>(C) * 4};
  const cuuint32_t box[3] = {16u, 32u, 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_rows2d_store(CUtensorMap* map, const void* ptr, long long rows, long long cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows <= 0 || cols <= 0) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {16u, 32u};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_weight3d(CUtensorMap* map, const void* ptr, long long E, long long R, long long C,
                       int box_r) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || E <= 0 || R <= 0 || C <= 0) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(R),
                              static_cast<cuuint64_t>(E)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(C) * 2,
                                 static_cast<cuuint64_t>(R) * static_cast<cuuint64_t>(C) * 2};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_r), 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_u8_rows2d(CUtensorMap* map, const void* ptr, long long rows, long long cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows <= 0 || cols <= 0) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
  const cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_u8_weight3d(CUtensorMap* map, const void* ptr, long long E, long long R, long long C, int box_r) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || E <= 0 || R <= 0 || C <= 0) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(R), static_cast<cuuint64_t>(E)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(R) * static_cast<cuuint64_t>(C)};
  const cuuint32_t box[3] = {128u, static_cast<cuuint32_t>(box_r), 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

moe_status_t launch_grouped_gemm(int mode, const GemmMaps& maps, const GemmArgs& args,
                                 long long max_tiles, cudaStream_t stream) {
  if (args.E < 1 || args.E > MAX_E) return MOE_ERR_UNSUPPORTED_SHAPE;
  switch (mode) {
    case MODE_UP_SWIGLU: return launch_mode<MODE_UP_SWIGLU>(maps, args, max_tiles, stream);
    case MODE_PLAIN_BF16: return launch_mode<MODE_PLAIN_BF16>(maps, args, max_tiles, stream);
    case MODE_DGRAD_SWIGLU: return launch_mode<MODE_DGRAD_SWIGLU>(maps, args, max_tiles, stream);
    case MODE_WGRAD: return launch_mode<MODE_WGRAD>(maps, args, max_tiles, stream);
    case MODE_WGRAD_BF16: return launch_mode<MODE_WGRAD_BF16>(maps, args, max_tiles, stream);
    case MODE_UP_SWIGLU_MX: return launch_mode<MODE_UP_SWIGLU_MX>(maps, args, max_tiles, stream);
    case MODE_PLAIN_MX: return launch_mode<MODE_PLAIN_MX>(maps, args, max_tiles, stream);
    case MODE_DGRAD_SWIGLU_MX: return launch_mode<MODE_DGRAD_SWIGLU_MX>(maps, args, max_tiles, stream);
    default: return MOE_ERR_INVALID_ARG;
  }
}

}  // namespace moe
