// Host-side interface between the library's translation units (not part of the C ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/moe_gg.h"

namespace moe {

// ------------------------------------------------------------------ grouped GEMM (tcgen05)
enum GemmMode : int {
  // U = X W_ug^T per row segment, gate and up column blocks in one accumulator; the epilogue
  // writes bf16(P) for P = w * silu(gate) * up (w = 1 without routing weights), and optionally
  // U (24 bits) and P - bf16(P) (bf16).
  // A: rows [cap, d] K-major; B: W_ug [E, 2h, d].
  MODE_UP_SWIGLU = 0,
  // Y = P W per row segment with W [E, K, N] (N contiguous, MN-major B); bf16 store.
  MODE_PLAIN_BF16 = 1,
  // dA = dY W_down^T per row segment (W_down [E, h, d] K-major B); the epilogue applies the
  // SwiGLU backward with the saved U (24-bit) and writes dU = [dgate, dup] as a bf16 high/low pair
  // (out/out2, with their rows2d_store maps as the kernel's two output maps).
  MODE_DGRAD_SWIGLU = 2,
  // dW_e = (P_hi + P_lo)_e^T Q_e, contraction over the M_e rows of expert e (all operands
  // MN-major, two MMAs per K step into one accumulator); fp32 store, zeros for empty experts.
  MODE_WGRAD = 3,
  // as MODE_WGRAD with the high half of P only (plain bf16 activations, one MMA per K step)
  MODE_WGRAD_BF16 = 4,
  // MXFP8 versions of the row-grouped modes (mode - MODE_UP_SWIGLU_MX is the bf16 mode whose
  // epilogue they share): E4M3 operands, both K-major (A [cap, K] codes, B [E, N, K] codes), an
  // E8M0 scale per 32 elements of K in 512-byte atoms (sfa by the problem list's row tile,
  // sfb by expert and 128-row tile of N), block-scaled MMAs into one accumulator.
  MODE_UP_SWIGLU_MX = 5,   // B = W_ug codes along d; epilogue of MODE_UP_SWIGLU
  MODE_PLAIN_MX = 6,       // B = W^T codes [E, N, K]; epilogue of MODE_PLAIN_BF16
  MODE_DGRAD_SWIGLU_MX = 7 // B = W_down codes along d; epilogue of MODE_DGRAD_SWIGLU
};

// The tensor maps of one launch. They travel as one __grid_constant__ kernel parameter, so the
// kernel's TMA instructions read them from parameter space.
struct GemmMaps {
  CUtensorMap a, a_lo, b;     // operands; a_lo is the low half of A (MODE_WGRAD only)
  CUtensorMap out, out2;      // TMA store maps: DGRAD_SWIGLU dU high / low; WGRAD dW of the
                              // first / second problem
  CUtensorMap a2, a_lo2, b2;  // WGRAD modes: operands of the second problem
};

struct GemmArgs {
  const int32_t* offsets;  // inclusive offsets [E] on the device, or nullptr (uniform/single)
  int E;                   // experts in the problem list
  int uniform_rows;        // > 0: expert e owns rows [e*uniform_rows, (e+1)*uniform_rows)
  int single_expert;       // >= 0: one problem, expert `single_expert`, rows below
  int single_row0;
  int single_rows;
  int cap;                 // rows of the row-indexed buffers (device check of the offsets)
  int N;                   // output columns (UP_SWIGLU: h)
  int K;                   // contraction length of the row-grouped modes
  int Mdim;                // WGRAD: rows of each expert's gradient
  int h;                   // SwiGLU half width
  void* out;               // row-grouped bf16 output, or WGRAD fp32 [E, Mdim, N]
  long long ldo;           // elements per output row
  void* out2;              // UP_SWIGLU: optional U rounded to 24 bits, blocked by row tile (see u_block);
                           // DGRAD_SWIGLU: dU low half
  long long ldo2;
  void* out3;              // UP_SWIGLU: optional low half of P [cap, h] (P = w*A, or A)
  long long ldo3;
  // Optional routing weight of each row: w = row_weight[row_src[row]]. UP_SWIGLU writes
  // P = w*A (high half to `out`, low half to out3); DGRAD_SWIGLU scales dA by w before the
  // SwiGLU backward.
  const int32_t* row_src;
  const float* row_weight;
  const void* aux;         // DGRAD_SWIGLU: the saved U in the blocked layout of out2
  long long ld_aux;
  // First row tile of this problem list in the blocked U: 0 for a whole problem list, the row
  // tiles of the experts before it for one expert (single_expert)
  long long tile_base;
  // 1 when every bf16 row output is 32-byte aligned at each 16-column chunk (bases 32-byte
  // aligned; h % 16 == 0 for UP_SWIGLU and DGRAD_SWIGLU, N % 16 == 0 for PLAIN_BF16), so a chunk
  // row is one 32-byte store
  int vec32;
  // PLAIN_BF16, optional: row p of the output is written to row row_dst[p] of `out` instead of
  // row p (the down projection storing straight into token rows when top_k = 1)
  const int32_t* row_dst;
  // DGRAD_SWIGLU, optional: per row p, dw_np fp32 partial sums of <A_p, G_p> (A = SwiGLU(U)
  // unweighted, G = dy W_down^T before the routing weight), one per (column tile, warp half)
  float* dw_part;
  int dw_np;
  // WGRAD modes: number of independent problems in the launch (1 or 2). The second one has its
  // own operands (maps a2, a_lo2, b2), gradient shape (Mdim2 x N2), output (out_b / map out2)
  // and shares the experts and row segments of the first; its tiles follow the first's.
  int nprob;
  int N2;
  int Mdim2;
  void* out_b;
  long long ldo_b;
  // MXFP8 up/gate and dgrad modes, optional (mxq non-null): the next scaled GEMM's A operand
  // quantized in the epilogue from the bf16 values it stores (P = a_save; dU's high half):
  // codes [cap, mx_ldq] and scale atoms by the problem list's row tile, mx_kc 128-column chunks
  uint8_t* mxq;
  uint8_t* mxsf;
  int mx_ldq;
  int mx_kc;
  // MXFP8 modes: scale atoms of A (by row tile of the problem list) and of B (by expert and
  // 128-row tile of N, sfb_ntpad tiles per expert), sf_kc 128-element chunks of K per row
  const uint8_t* sfa;
  const uint8_t* sfb;
  int sf_kc;
  int sfb_ntpad;
  // Debug builds (MOE_GG_DEBUG) only: the extents the bounds checks compare against -- row
  // tiles of the blocked saved U (read or written), of the activation scale atoms read (sfa) and
  // of those the epilogue writes (mxsf), tiles of the weight scale atoms (sfb), and the rows of
  // the row_dst output
  long long dbg_u_tiles;
  long long dbg_sfa_tiles;
  long long dbg_mxsf_tiles;
  long long dbg_sfb_tiles;
  long long dbg_dst_rows;
  int32_t* status;         // optional device status word
  long long timeout_ns;    // bound of every wait of the main loops
  // bound of the teardown waits that let this CTA's in-flight copies and MMAs finish before it
  // frees tensor memory and exits (never below 2 s, whatever timeout_ns is)
  long long drain_ns;
};

// Launch one persistent grouped GEMM. `maps` holds the operand tensor maps described with each
// mode (unused entries are ignored). `max_tiles` bounds the grid (the exact tile count is only
// known on the device).
moe_status_t launch_grouped_gemm(int mode, const GemmMaps& maps, const GemmArgs& args,
                                 long long max_tiles, cudaStream_t stream);

// Tensor maps (bf16, 128-byte swizzle, zero fill outside the tensor).
//   rows2d: a [rows, cols] row-major matrix; box = 64 columns x box_rows rows.
//   weight3d: an [E, R, C] tensor; box = 64 x box_r x 1.
bool make_map_rows2d(CUtensorMap* map, const void* ptr, long long rows, long long cols,
                     int box_rows);
bool make_map_weight3d(CUtensorMap* map, const void* ptr, long long E, long long R, long long C,
                       int box_r);
//   grad3d_f32: an fp32 [E, R, C] gradient, stored through 16-column x 32-row boxes, 64B swizzle.
//   rows2d_store: a bf16 [rows, cols] row-major output, stored through 16-column x 32-row boxes,
//   32B swizzle (cols * 2 bytes a multiple of 16).
bool make_map_rows2d_store(CUtensorMap* map, const void* ptr, long long rows, long long cols);
bool make_map_grad3d_f32(CUtensorMap* map, const void* ptr, long long E, long long R, long long C);

//   u8 maps (MXFP8 codes, 128-byte swizzle): rows2d [rows, cols] with 128-byte x box_rows boxes;
//   weight3d [E, R, C] with 128-byte x box_r x 1 boxes.
bool make_map_u8_rows2d(CUtensorMap* map, const void* ptr, long long rows, long long cols, int box_rows);
bool make_map_u8_weight3d(CUtensorMap* map, const void* ptr, long long E, long long R, long long C, int box_r);

int gemm_tiles_n(int mode, int N);  // column tiles of one problem

// ------------------------------------------------------------------ debug build (debug.cuh)
// Check sites of the bounds checks; the names moe_debug_site_name() returns follow this order.
enum DbgSite : int {
  DBG_GG_ROW = 0,       // grouped kernel: an epilogue row against the row buffers' rows (cap)
  DBG_GG_TILE = 1,      // grouped kernel: a row tile of the blocked saved U
  DBG_GG_SLOT = 2,      // grouped kernel: a row's flat slot (row_src) against cap
  DBG_GG_DST = 3,       // grouped kernel: a destination row (row_dst) against the output's rows
  DBG_GG_SFA = 4,       // grouped kernel (MXFP8): a row tile of the activation scale atoms read
  DBG_GG_SFB = 5,       // grouped kernel (MXFP8): a tile of the weight scale atoms read
  DBG_GG_MXSF = 6,      // grouped kernel (MXFP8): a row tile of the scale atoms the epilogue writes
  DBG_COMBINE_ROW = 7,  // combine: an inverse-map row against T*top_k
  DBG_RWG_ROW = 8,      // routing-weight gradient: an inverse-map row against the slots
  DBG_ROUTE_POS = 9,    // route scatter: a slot's placed row against T*top_k
  DBG_MX_TILE = 10,     // MXFP8 quantization: a scale-atom tile against the atoms buffer
  DBG_SITES = 11
};

struct DbgRecord {
  int mask;         // bit s: check site s failed at least once
  int site;         // first failing site (-1: none)
  long long index;  // its index
  long long limit;  // and the bound the index had to stay below
};

// One per kernel translation unit: merge its record into *acc, clear it when `reset` (no-ops in
// release builds).
cudaError_t dbg_collect_grouped(DbgRecord* acc, bool reset);
cudaError_t dbg_collect_permute(DbgRecord* acc, bool reset);
cudaError_t dbg_collect_route(DbgRecord* acc, bool reset);
cudaError_t dbg_collect_mx(DbgRecord* acc, bool reset);

// ------------------------------------------------------------------ helpers
int device_sm_count();              // SMs of the current device (cached per device)
long long wait_timeout_ns();        // bound of device waits (default 2 s)
moe_status_t check_device();        // current device must be sm_103
moe_status_t cuda_fail(cudaError_t err);  // records the error text, returns MOE_ERR_CUDA
// Raise a kernel's dynamic shared-memory limit once per (kernel, device).
cudaError_t ensure_max_dynamic_smem(const void* kernel, int bytes);

// ------------------------------------------------------------------ routing / data movement
size_t route_workspace_bytes(long long n, int E);
moe_status_t launch_route(const int32_t* ids, int n, int E, int32_t* counts, int32_t* offsets,
                          int32_t* sorted_src, int32_t* inv_map, void* ws, cudaStream_t s);
moe_status_t launch_permute(const void* x, const int32_t* sorted_src, const int32_t* offsets,
                            const float* row_scale, int n, int k, int E, int d, void* xp,
                            cudaStream_t s);
// out[t] = 0 for the tokens with inv_map[t] < 0 (top_k = 1); d a multiple of 8
moe_status_t launch_zero_dropped_rows(const int32_t* inv_map, int T, int d, void* out, cudaStream_t s);
moe_status_t launch_combine(const void* y, const int32_t* inv_map, const float* weights, int T,
                            int k, int d, void* out, cudaStream_t s);
moe_status_t launch_pad_rows(const void* src, const int32_t* offsets, int E, int C, int cols,
                             void* dst, cudaStream_t s);
// Pitch change between a narrow row layout (rows in blocks of blk, sub-blocks of sub, `cols`
// columns) and a wide one (blocks of blk8, sub-blocks of sub8, cols8 columns, zero filled):
// to_wide packs (writes rows_out wide rows), else unpacks (writes rows_out narrow rows). With
// offsets, rows at or past M = offsets[E-1] are skipped. bf16 or fp32 elements.
moe_status_t launch_pitch_repack(const void* src, void* dst, bool fp32, long long rows_out,
                                int cols, int cols8, int blk, int sub, int blk8, int sub8,
                                bool to_wide, const int32_t* offsets, int E, cudaStream_t s);
// dw[s] = sum of the dw_np partials of row inv_map[s] in index order, 0 for a dropped slot.
moe_status_t launch_routing_weight_grad(const float* part, int np, const int32_t* inv_map,
                                        int n_slots, float* dw, cudaStream_t s);
// MXFP8 quantization (layouts in mx_quant.cu). Rows along K: with offsets, the rows p < M of a
// problem list (scale atoms by its 128-row tiles); else `rows` rows of weights with per_expert
// rows each (atoms by expert and 128-row tile, tiles padded to even). Columns: a weight
// [E, R, C] quantized along R into [E, C, R] codes.
int mx_ntpad(int N);
int mx_kc(int K);
moe_status_t launch_mx_quant_rows(const void* src, long long rows, int K, const int32_t* offsets, int E,
                                  int per_expert, void* q, void* sf, int32_t* status, cudaStream_t s);
size_t mx_workspace_bytes(int op, long long n, int E, int d, int h);  // the MOE_OP_MX_* sizes
// The permute's gather fused with the quantization of the gathered rows along d (xp nullable:
// the bf16 copy is written only when given).
moe_status_t launch_mx_permute_quant(const void* x, const int32_t* sorted_src, const int32_t* offsets, int E,
                                    int n, int k, int d, void* xp, void* q, void* sf, int32_t* status,
                                    cudaStream_t s);
moe_status_t launch_mx_quant_cols(const void* w, int E, int R, int C, void* q, void* sf, cudaStream_t s);
moe_status_t launch_unpad_rows(const void* src, const int32_t* offsets, int E, int C, int cap,
                               int cols, void* dst, cudaStream_t s);

}  // namespace moe
