/*
 * moe_gg.h -- C ABI of the device-scheduled ragged grouped GEMM for one SwiGLU
 * mixture-of-experts expert layer (GB300, sm_103a).
 *
 * The operation is the one of "Section 09: Grouped GEMM" (OLMo-core MoE report): routing turns
 * an expert layer into a ragged batch of products whose row counts M_e live on the device; the
 * counts are turned into cumulative int32 offsets on the device (Fig. 37), never copied to the
 * host, and one grouped kernel computes only the routed rows (§9.3, §9.4). Each expert is the
 * SwiGLU expert of Eq. 13:
 *     U_e = X_e W_ug,e^T        X_e [M_e, d],  W_ug,e [2h, d]  (gate rows [0,h), up rows [h,2h))
 *     Y_e = SwiGLU(U_e) W_down,e                W_down,e [h, d]
 * with SwiGLU(U) = silu(U[:, :h]) * U[:, h:]. Backward follows Eq. 15 / Table 15.
 *
 * Conventions shared by every entry point:
 *  - Every pointer is a DEVICE pointer owned by the caller, unless stated otherwise. The
 *    library allocates no device memory; scratch comes from the caller's workspace `ws`
 *    (size from moe_workspace_bytes()). Work is queued on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream) and the calls return without synchronising, except
 *    moe_loop_swiglu_fwd, which by design copies the offsets to the host.
 *  - bf16 tensors are passed as raw 16-bit patterns (moe_bf16), row-major and contiguous;
 *    fp32 and int32 tensors likewise.
 *  - Offsets are int32 inclusive segment ends of length E: expert e owns rows
 *    [offsets[e-1], offsets[e]) (offsets[-1] = 0), M = offsets[E-1] ("Section 09", Fig. 37:
 *    counts (1,4,3,2) give [1,5,8,10]). Rows p >= M of the row buffers are neither read for
 *    results nor written (§9.4: unused capacity stays outside the final offset).
 *  - Errors found on the host (null pointer, bad size, misalignment, small workspace) return a
 *    status before anything is launched. Conditions found on the device set bits in the
 *    optional `dev_status` word (atomic OR; the caller clears it and reads it when it chooses):
 *    MOE_DEV_TIMEOUT when a bounded wait inside a kernel gave up (the kernel then stops early
 *    instead of hanging), MOE_DEV_BAD_OFFSETS when offsets decrease or exceed the buffer rows
 *    (the affected kernel then computes nothing).
 *  - Accumulation: products of bf16 operands are summed in fp32 in tensor memory. A contraction
 *    longer than 8192 (K = d or h in the projections and dgrads, the rows of an expert in the
 *    wgrads) is summed in segments of 8192 whose partial sums are added in round-to-nearest
 *    fp32, which keeps its error at the level of an fp32 sum (the tensor core's own
 *    accumulator truncates). The MXFP8 calls do not segment.
 *  - Limits: 1 <= E <= 1024, 1 <= top_k <= 32, 1 <= d, h <= 2^20, T*top_k < 2^31. The
 *    grouped kernels read operands by TMA, which needs 16-byte row pitches (d and h multiples
 *    of 8). moe_permute, moe_unpermute_combine, moe_grouped_swiglu_fwd and moe_grouped_bwd also
 *    take other widths: the row kernels then move one element per lane step, and the two
 *    composite calls run the same kernels on zero-padded copies of width round_up(w, 8) held
 *    in their workspace (exact: the padding is zeros) and copy the results back. The single
 *    grouped-kernel entry points and the comparison variants need multiples of 8. Other
 *    shapes return MOE_ERR_UNSUPPORTED_SHAPE. Base pointers must be 16-byte aligned.
 */
#ifndef MOE_GG_H
#define MOE_GG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16;                 /* raw bfloat16 bits */
typedef struct CUstream_st* moe_stream_t;  /* identical to cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,          /* null pointer, negative size, misaligned pointer */
  MOE_ERR_UNSUPPORTED_SHAPE = 2,    /* shape outside the limits above */
  MOE_ERR_WORKSPACE_TOO_SMALL = 3,  /* ws_bytes < moe_workspace_bytes(...) */
  MOE_ERR_CUDA = 4,                 /* a CUDA runtime/driver call failed (see moe_last_cuda_error) */
  MOE_ERR_DEVICE_TIMEOUT = 5,       /* reserved for callers that map MOE_DEV_TIMEOUT to a status */
  MOE_ERR_UNSUPPORTED_DEVICE = 6    /* current device is not sm_103 */
} moe_status_t;

/* bits of the device status word */
#define MOE_DEV_TIMEOUT 0x1
#define MOE_DEV_BAD_OFFSETS 0x2

/* operations for moe_workspace_bytes */
typedef enum {
  MOE_OP_ROUTE = 0,       /* moe_route_offsets */
  MOE_OP_FWD = 1,         /* moe_grouped_swiglu_fwd */
  MOE_OP_BWD = 2,         /* moe_grouped_bwd (dU halves, routing-gradient partials) */
  MOE_OP_PADDED_BMM = 3,  /* moe_padded_bmm_swiglu_fwd (uses capacity_C) */
  MOE_OP_LOOP = 4,        /* moe_loop_swiglu_fwd */
  MOE_OP_SAVED = 5,       /* size of the `saved` buffer the forward fills for the backward */
  MOE_OP_MX_WEIGHTS = 6,  /* moe_mx_prepare_weights: the prepared MXFP8 weights */
  MOE_OP_MX_FWD = 7,      /* moe_grouped_swiglu_fwd_mxfp8 */
  MOE_OP_MX_BWD = 8,      /* moe_grouped_bwd_mxfp8 */
  MOE_OP_MX_ROW_SCALES = 9 /* moe_mx_quantize_rows: scale bytes for T*top_k rows of K = d */
} moe_op_t;

/* Bytes of caller workspace that `op` needs for these sizes (0 when none). Pure host
 * arithmetic; no CUDA call. Returns 0 for invalid sizes as well: validate with the call. */
size_t moe_workspace_bytes(int op, int T, int top_k, int E, int d, int h, int capacity_C);

/*
 * moe_route_offsets -- route histogram, cumulative offsets, placement and inverse map.
 * "Section 09: Grouped GEMM", Fig. 37 steps 1-2 and §9.3 (counts and inclusive int32 offsets
 * computed on the device); "grouped_mm" agent doc (sort rows by expert into contiguous blocks
 * after dropping ids outside [0, E); precomputed inverse map [N, top_k], sentinel-padded).
 *
 *  ids        [T*top_k] int32 expert id of each (token, slot), flat index t*top_k + j.
 *             Ids outside [0, E) are dropped: not counted, inv_map entry -1.
 *  counts     [E] out: rows routed to each expert.
 *  offsets    [E] out: inclusive prefix sum of counts.
 *  sorted_src [T*top_k] out: flat slot index placed at row p, for p < M; -1 for p >= M.
 *             Inside a segment rows keep increasing flat-index order (stable).
 *  inv_map    [T*top_k] out: row of each flat slot, -1 when dropped. inv_map[sorted_src[p]] = p.
 *  ws         workspace of moe_workspace_bytes(MOE_OP_ROUTE, T, top_k, E, 0, 0, 0) bytes.
 * Results are deterministic (no order-dependent atomics). T = 0 is allowed (counts = 0).
 */
moe_status_t moe_route_offsets(const int32_t* ids, int T, int top_k, int E, int32_t* counts,
                               int32_t* offsets, int32_t* sorted_src, int32_t* inv_map,
                               void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_permute -- gather token rows into expert-contiguous order (the forward gather x[idx] of
 * the "grouped_mm" agent doc); with row_scale it is also the combine's backward
 * (dY[p] = w[src] * dOut[src / top_k], Eq. 15 applied to the weighted sum).
 *
 *  x          [T, d] bf16 token rows.
 *  sorted_src [T*top_k], offsets [E] as written by moe_route_offsets.
 *  row_scale  nullable [T*top_k] fp32, indexed by flat slot; the product is rounded once.
 *  xp         [T*top_k, d] bf16 out: row p < M = x[sorted_src[p] / top_k] (* scale).
 */
moe_status_t moe_permute(const moe_bf16* x, const int32_t* sorted_src, const int32_t* offsets,
                         const float* row_scale, int T, int top_k, int E, int d, moe_bf16* xp,
                         moe_stream_t stream);

/*
 * moe_grouped_swiglu_fwd -- the device-scheduled grouped SwiGLU expert forward, Eq. 13.
 * Two persistent tcgen05 kernels walk the device problem list built from `offsets`
 * ("Section 09", Fig. 37 steps 3-4): (1) U = xp_e W_ug,e^T with SwiGLU fused into the
 * epilogue, writing A = SwiGLU(U); (2) y_e = A_e W_down,e. bf16 operands, fp32 accumulation in
 * tensor memory, bf16 results (one rounding each).
 *
 *  xp         [cap, d] bf16 rows in expert order (rows >= M ignored).
 *  offsets    [E] int32 inclusive; M = offsets[E-1] must be <= cap (else MOE_DEV_BAD_OFFSETS).
 *  sorted_src, weights  nullable pair: when weights ([T*top_k] fp32, by flat slot) is given,
 *             row p of the SwiGLU output is multiplied by w = weights[sorted_src[p]] in the
 *             up/gate epilogue (fp32, before the bf16 rounding), so y_p = (w A_p) W_down: the
 *             routing weight is applied before the combine (which is then called with
 *             weights = NULL) instead of inside it. The combine is linear, so the layer output
 *             is the same; the backward then gathers dOut without a rounding product.
 *  w_ug       [E, 2h, d] bf16;  w_down [E, h, d] bf16.
 *  y          [cap, d] bf16 out (rows < M written).
 *  a_save     [cap, h] bf16 out: bf16(P) with P = w*A (P = A without weights), the down
 *             projection's input.
 *  saved      nullable, moe_workspace_bytes(MOE_OP_SAVED, T, top_k, E, d, h) bytes for
 *             cap = T*top_k: what the backward needs beyond a_save, written when non-NULL
 *             (training). Byte 0: P - bf16(P), bf16 [cap, h] row-major. Byte
 *             round_up(cap*h*2, 256): U rounded to nearest even at 24 bits (the upper 24 bits
 *             of its fp32 pattern: 16 significant bits), blocked as the kernels' epilogues hold
 *             it -- for the G-th 128-row tile of the problem list (experts in order,
 *             ceil(M_e/128) tiles each, at most (cap + 127 E)/128), lane quadrant q (tile rows
 *             32q..32q+31) and 16-column chunk ci (ci < H = ceil(h/16): gate columns 16ci..;
 *             else up columns 16(ci-H)..), a 1536-byte block at byte ((G*4 + q)*2H + ci)*1536
 *             of three 512-byte planes: for tile row 32q+l and column j of the chunk, the upper
 *             16 of the 24 bits are the little-endian 16-bit word at byte (j/8)*512 + l*16 +
 *             (j%8)*2 and the lower 8 bits the byte at 1024 + l*16 + j. The slots of tile rows
 *             past the expert's segment are left unwritten. Keeping U to 16 significant bits and
 *             P as a bf16 high+low pair (a_save + the low half) lets the wgrads contract over
 *             long expert segments without the bf16 rounding of saved activations dominating
 *             the result; the blocked U makes each warp's store (and the dgrad's load) of one
 *             plane one contiguous 512-byte access.
 *  ws         moe_workspace_bytes(MOE_OP_FWD, ...) bytes: 0 (ws may be NULL) when d and h are
 *             multiples of 8, else the zero-padded copies of xp, y, a, W_ug, W_down. With h not
 *             a multiple of 8, `saved` holds the padded width round_up(h, 8) in place of h.
 */
moe_status_t moe_grouped_swiglu_fwd(const moe_bf16* xp, const int32_t* offsets,
                                    const int32_t* sorted_src, const float* weights, int E,
                                    int cap, int d, int h, const moe_bf16* w_ug,
                                    const moe_bf16* w_down, moe_bf16* y, moe_bf16* a_save,
                                    void* saved, void* ws, size_t ws_bytes, int32_t* dev_status,
                                    moe_stream_t stream);

/*
 * moe_grouped_bwd -- dgrad and wgrad of the SwiGLU expert, Eq. 15 and Table 15 ("Section 09"
 * §9.5): M_e is the output-row count of the dgrads and the contraction length of the wgrads.
 *   dA = w * (dy_e W_down,e^T);  dU = [dA*v*s*(1+g(1-s)), dA*silu(g)] with g,v = U[:, :h],
 *   U[:, h:], s = sigmoid(g);  dxp_e = dU W_ug,e;  dW_ug,e = dU^T xp_e;  dW_down,e = P_e^T dy_e
 * with w = weights[sorted_src[p]] and P = w*A (a_save + its saved low half) when weights are
 * given, else w = 1 and P = A.
 * dU is computed in fp32 in the dgrad epilogue and kept as a bf16 high+low pair; dxp uses the
 * high half, the wgrads contract both halves (two MMAs per K step) so that dW carries about
 * 16 significant bits of the activations instead of 8.
 *
 *  dy      [cap, d] bf16 upstream gradient at the grouped-GEMM boundary: the gradient of y, or,
 *          with weights, the plain gather of dOut (moe_permute with row_scale = NULL).
 *  xp, a_save, saved, sorted_src, weights as given to the forward (saved required here).
 *  dxp     [cap, d] bf16 out (rows < M).
 *  dw_ug   [E, 2h, d] fp32 out;  dw_down [E, h, d] fp32 out. Experts with M_e = 0 get zeros.
 *  inv_map, dw_route  nullable pair: when dw_route ([cap] fp32, by flat slot t*top_k + j,
 *          cap = T*top_k) is given, it receives the routing-weight gradient of the combine,
 *          dw_route[t*top_k+j] = <dOut[t], y~_p> with p = inv_map[t*top_k+j] and y~_p = A_p
 *          W_down,e the unweighted expert output (0 for a dropped slot). It is computed as
 *          <A_p, dy_p W_down,e^T> in the dgrad epilogue (dy = the gather of dOut), from the
 *          saved U and the fp32 accumulator, and summed over fixed partial slots in index order:
 *          deterministic.
 *  ws      moe_workspace_bytes(MOE_OP_BWD, ...) bytes: dU high and low (2 x [cap, 2h] bf16),
 *          then the routing-gradient partials ([cap, 2 ceil(h/256)] fp32, used with dw_route);
 *          for d or h not multiples of 8, first the zero-padded copies of dy, xp, dxp, a, the
 *          weights and the two gradients, then the above at the padded widths.
 */
moe_status_t moe_grouped_bwd(const moe_bf16* dy, const moe_bf16* xp, const moe_bf16* a_save,
                             const void* saved, const int32_t* offsets, const int32_t* sorted_src,
                             const float* weights, int E, int cap, int d, int h,
                             const moe_bf16* w_ug, const moe_bf16* w_down, moe_bf16* dxp,
                             float* dw_ug, float* dw_down, const int32_t* inv_map,
                             float* dw_route, void* ws, size_t ws_bytes, int32_t* dev_status,
                             moe_stream_t stream);

/*
 * The single kernels the two calls above are made of, one per step of the path, for callers
 * that schedule (or time) the steps themselves. Same conventions and the same `saved` layout;
 * sorted_src/weights as in moe_grouped_swiglu_fwd (nullable pair).
 *
 * moe_grouped_up_swiglu  -- U = xp_e W_ug,e^T and P = (w *) SwiGLU(U) (Eq. 13, first line);
 *                           writes a_save = bf16(P) and, when saved is non-NULL, U and P's low
 *                           half.
 * moe_grouped_down       -- y_e = a_e W_down,e (Eq. 13, second line); a [cap, h] bf16.
 * moe_grouped_down_dgrad_swiglu -- dA = (w *) dy_e W_down,e^T (Eq. 15 dgrad of the down
 *                           projection) with the SwiGLU backward fused: writes dU = [dgate, dup]
 *                           as bf16 high (du_hi) and low (du_lo) halves, each [cap, 2h]. With
 *                           dw_part (nullable, [cap, 2 ceil(h/256)] fp32) it also writes, for
 *                           every row p < M, the partial sums of <A_p, dy_p W_down,e^T> over
 *                           the row's 128-column pieces (see moe_routing_weight_grad).
 * moe_routing_weight_grad -- dw_route[s] = sum of the partials of row inv_map[s] in index order
 *                           (0 for a dropped slot), s < T*top_k: the routing-weight gradient of
 *                           the combine, as in moe_grouped_bwd.
 * moe_grouped_up_dgrad   -- dxp_e = dU_e W_ug,e (Eq. 15 dgrad of the up/gate projection).
 * moe_grouped_wgrad      -- dW_e = P_e^T Q_e over each expert's M_e rows (Eq. 15 wgrad;
 *                           Table 15: M_e is the contraction length). P = p_hi (+ p_lo when
 *                           non-NULL: both halves are contracted, ~16-bit activations) is
 *                           [cap, p_cols] bf16, Q [cap, q_cols] bf16, dW [E, p_cols, q_cols]
 *                           fp32; experts with M_e = 0 get zeros. For dW_down: P = a_save and
 *                           the saved low half, Q = dy; for dW_ug: P = dU halves, Q = xp.
 *                           p_cols and q_cols multiples of 8.
 */
moe_status_t moe_grouped_up_swiglu(const moe_bf16* xp, const int32_t* offsets,
                                   const int32_t* sorted_src, const float* weights, int E, int cap,
                                   int d, int h, const moe_bf16* w_ug, moe_bf16* a_save,
                                   void* saved, int32_t* dev_status, moe_stream_t stream);
moe_status_t moe_grouped_down(const moe_bf16* a, const int32_t* offsets, int E, int cap, int d,
                              int h, const moe_bf16* w_down, moe_bf16* y, int32_t* dev_status,
                              moe_stream_t stream);
moe_status_t moe_grouped_down_dgrad_swiglu(const moe_bf16* dy, const void* saved,
                                           const int32_t* offsets, const int32_t* sorted_src,
                                           const float* weights, int E, int cap, int d, int h,
                                           const moe_bf16* w_down, moe_bf16* du_hi,
                                           moe_bf16* du_lo, float* dw_part, int32_t* dev_status,
                                           moe_stream_t stream);
moe_status_t moe_routing_weight_grad(const float* dw_part, const int32_t* inv_map, int T,
                                     int top_k, int h, float* dw_route, moe_stream_t stream);
moe_status_t moe_grouped_up_dgrad(const moe_bf16* du_hi, const int32_t* offsets, int E, int cap,
                                  int d, int h, const moe_bf16* w_ug, moe_bf16* dxp,
                                  int32_t* dev_status, moe_stream_t stream);
moe_status_t moe_grouped_wgrad(const moe_bf16* p_hi, const moe_bf16* p_lo, int p_cols,
                               const moe_bf16* q, int q_cols, const int32_t* offsets, int E,
                               int cap, float* dw, int32_t* dev_status, moe_stream_t stream);

/*
 * moe_grouped_wgrad_dual -- two independent moe_grouped_wgrad problems over the same experts and
 * rows (the down projection's dW_down = P^T dy and the up/gate projection's dW_ug = dU^T xp of one
 * backward, Eq. 15 wgrad / Table 15) computed by one persistent launch: the second problem's
 * tiles follow the first's, so the two gradients share one pipeline fill and one tail. Each
 * problem's arguments mean what they mean for moe_grouped_wgrad; results are bit-identical to
 * two moe_grouped_wgrad calls. p1_lo and p2_lo must both be given or both be NULL.
 */
moe_status_t moe_grouped_wgrad_dual(const moe_bf16* p1_hi, const moe_bf16* p1_lo, int p1_cols,
                                    const moe_bf16* q1, int q1_cols, float* dw1,
                                    const moe_bf16* p2_hi, const moe_bf16* p2_lo, int p2_cols,
                                    const moe_bf16* q2, int q2_cols, float* dw2,
                                    const int32_t* offsets, int E, int cap, int32_t* dev_status,
                                    moe_stream_t stream);

/*
 * moe_unpermute_combine -- atomic-free weighted combine through the inverse map ("grouped_mm"
 * agent doc: the scatter-back becomes a gather plus a reduction):
 *     out[t] = sum_{j : inv_map[t*top_k+j] >= 0} w[t,j] * y[inv_map[t*top_k+j]]
 * accumulated in fp32 in slot order j, rounded once to bf16. weights NULL means all ones (then
 * it is the permute's backward, dx[t] = sum_j dxp[inv[t,j]]).
 *
 *  y [rows, d] bf16 (rows read: those inv_map names);  inv_map [T*top_k];  weights [T*top_k]
 *  fp32 or NULL;  out [T, d] bf16. Tokens whose slots are all dropped get zeros.
 */
moe_status_t moe_unpermute_combine(const moe_bf16* y, const int32_t* inv_map, const float* weights,
                                   int T, int top_k, int d, moe_bf16* out, moe_stream_t stream);

/*
 * moe_grouped_swiglu_fwd_top1_combine -- for top_k = 1, the forward and the combine in one pass:
 * the down projection stores row p straight into token row sorted_src[p] of `out`, the
 * direct-access write into the combine buffer of "Section 09: Grouped GEMM", §9.4. With one slot
 * per token the combine has no reduction to do (out[t] = y[inv[t]], the routing weight being
 * folded into the SwiGLU output as in moe_grouped_swiglu_fwd), so no scatter-add and no atomics
 * are needed; tokens whose slot was dropped (inv_map[t] = -1) get zero rows. Results are
 * bit-identical to moe_grouped_swiglu_fwd followed by moe_unpermute_combine with weights = NULL.
 *
 *  xp [T, d], offsets [E], sorted_src and inv_map [T] as moe_route_offsets wrote them for
 *  top_k = 1; weights nullable [T] fp32; out [T, d] bf16 (every row written); a_save [T, h] and
 *  saved (nullable) as moe_grouped_swiglu_fwd. d and h multiples of 8 (no zero-padded copies).
 */
moe_status_t moe_grouped_swiglu_fwd_top1_combine(const moe_bf16* xp, const int32_t* offsets,
                                                 const int32_t* sorted_src, const int32_t* inv_map,
                                                 const float* weights, int E, int T, int d, int h,
                                                 const moe_bf16* w_ug, const moe_bf16* w_down, moe_bf16* out,
                                                 moe_bf16* a_save, void* saved, int32_t* dev_status,
                                                 moe_stream_t stream);

/*
 * moe_padded_bmm_swiglu_fwd -- comparison variant: capacity-padded batched GEMM ("Section 09",
 * Eq. 14 and Fig. 35). Every expert is padded to capacity_C rows ([E, C, d], zero rows added),
 * the same tcgen05 kernels run the E uniform problems (all E*C rows are multiplied), and the
 * first min(M_e, C) rows of each expert are copied back; rows beyond C are dropped and get a
 * zero output row. Arguments as moe_grouped_swiglu_fwd; ws holds the padded buffers
 * (moe_workspace_bytes(MOE_OP_PADDED_BMM, ..., capacity_C)).
 */
moe_status_t moe_padded_bmm_swiglu_fwd(const moe_bf16* xp, const int32_t* offsets, int E, int cap,
                                       int d, int h, int capacity_C, const moe_bf16* w_ug,
                                       const moe_bf16* w_down, moe_bf16* y, void* ws,
                                       size_t ws_bytes, int32_t* dev_status, moe_stream_t stream);

/*
 * moe_loop_swiglu_fwd -- comparison variant: host-scheduled per-expert loop ("Section 09",
 * Fig. 36: the counts are copied to the host, the CPU waits, then one GEMM launch per expert
 * and projection). Copies `offsets` to the host and synchronises `stream` BY DESIGN; then
 * launches the same tcgen05 kernels once per non-empty expert. Arguments and results as
 * moe_grouped_swiglu_fwd (saved nullable, a_save required). Offsets that decrease or exceed
 * cap return MOE_ERR_INVALID_ARG (they are host-visible here).
 */
moe_status_t moe_loop_swiglu_fwd(const moe_bf16* xp, const int32_t* offsets, int E, int cap,
                                 int d, int h, const moe_bf16* w_ug, const moe_bf16* w_down,
                                 moe_bf16* y, moe_bf16* a_save, void* saved,
                                 int32_t* dev_status, moe_stream_t stream);

/*
 * MXFP8 variant -- "Section 09: Grouped GEMM", §9.5 (last paragraph): the routed MXFP8 path
 * runs the forward and the Dgrad as scaled grouped GEMMs and the Wgrad as BF16 grouped GEMM.
 * Format: OCP Microscaling MXFP8 -- blocks of 32 consecutive elements along the contraction
 * dimension share one power-of-two scale 2^s stored as E8M0 (s + 127), each element is FP8
 * E4M3; s = floor(log2(max |v|)) - 8 clamped to [-127, 127] (-127 for an all-zero block);
 * elements are v / 2^s rounded to nearest, ties to even, saturated to +-448. Every operand is
 * quantized along its own contraction dimension from its bf16 value: x and dy along d, the
 * SwiGLU output (a_save, bf16 P = w*A) along h, dU (its bf16 high half) along 2h, W_ug along d
 * (forward) and along 2h (dgrad), W_down along h (forward) and along d (dgrad). Products of
 * the block-scaled operands accumulate in fp32 in tensor memory (tcgen05.mma
 * kind::mxf8f6f4.block_scale). Shapes: d a multiple of 32, h a multiple of 128 (the gate and
 * up halves of W_ug then start on a 128-row scale tile), 1 <= E <= 1024; others return
 * MOE_ERR_UNSUPPORTED_SHAPE.
 *
 * Layouts. Codes of an operand [rows, K] are bytes, row-major. Scales come in 512-byte atoms,
 * one per (128-row tile, 128-element chunk of K): the scale of row r of the tile (0..127) and
 * 32-block kb of the chunk (0..3) is byte (r % 32) * 16 + (r / 32) * 4 + kb of atom
 * tile * ceil(K / 128) + chunk. For an activation the tiles are the problem list's 128-row
 * tiles (each expert's segment cut from its start; tile index = row tiles of the experts
 * before it + (p - start) / 128, at most (rows + 127 E) / 128 tiles); for a weight [E, N, K]
 * the tile of row n of expert e is e * NTp + n / 128 with NTp = ceil(N / 128) rounded up to even.
 *
 * moe_mx_prepare_weights -- quantize W_ug [E, 2h, d] and W_down [E, h, d] (bf16) into `mxw`
 *   (moe_workspace_bytes(MOE_OP_MX_WEIGHTS, 0, 1, E, d, h, 0) bytes, 256-byte aligned): four
 *   (codes, scales) pairs, each piece starting on a 256-byte boundary, in this order: W_ug
 *   along d (codes [E, 2h, d]); W_down along h (codes [E, d, h], the transpose); W_down along d
 *   (codes [E, h, d]); W_ug along 2h (codes [E, d, 2h], the transpose). Run once per weight
 *   update; the forward and the backward read it.
 * moe_permute_mxfp8 -- the permute's gather and the quantization of the gathered rows along d in
 *   one pass: for p < M, codes q[p] [d] and the scale atoms sf (by the problem list's tiles;
 *   moe_workspace_bytes(MOE_OP_MX_ROW_SCALES, T, top_k, E, d, h, 0) bytes) of x[sorted_src[p] /
 *   top_k], and, when xp is non-NULL, the bf16 row itself (what moe_permute writes). Gives the
 *   scaled forward its xp operand (and the scaled dgrad its dy: the gather of dOut) without a
 *   separate pass over the rows. d a multiple of 32.
 * moe_mx_quantize_rows -- quantize rows p < M = offsets[E-1] of x [cap, K] (bf16) into codes
 *   q [cap, K] and scale atoms sf (moe_workspace_bytes(MOE_OP_MX_ROW_SCALES, T, top_k, E, K, h,
 *   0) bytes for cap = T*top_k; h is ignored beyond its own check) by the problem list's tiles.
 *   Offsets that decrease or exceed cap set MOE_DEV_BAD_OFFSETS and nothing is written.
 * moe_grouped_swiglu_fwd_mxfp8 -- Eq. 13 with scaled GEMMs: U = q(xp) q(W_ug)^T, P = w*SwiGLU(U)
 *   in the up/gate epilogue (a_save = bf16(P), saved as in moe_grouped_swiglu_fwd; the same
 *   epilogue quantizes bf16(P) along h), then y = q(a_save) q(W_down). Arguments as
 *   moe_grouped_swiglu_fwd plus mxw and the nullable pair xq, xsf: the codes and scales of xp
 *   (from moe_permute_mxfp8 or moe_mx_quantize_rows); when they are NULL, xp is quantized here
 *   (xp may be NULL when they are given). ws holds the codes and scales of xp (unused when
 *   given) and of P (moe_workspace_bytes(MOE_OP_MX_FWD, ...), 256-byte aligned).
 * moe_grouped_bwd_mxfp8 -- Eq. 15: dA = w * q(dy) q(W_down)^T with the SwiGLU backward (dU high
 *   and low halves, routing-weight partials; the same epilogue quantizes dU's high half along
 *   2h), dxp = q(dU_hi) q(W_ug) (scaled GEMMs); dW_down = P^T dy and dW_ug = dU^T xp as BF16
 *   grouped GEMMs on both halves (one launch). Arguments as moe_grouped_bwd plus mxw and the
 *   nullable pair dyq, dysf: the codes and scales of dy (moe_permute_mxfp8 of dOut); when NULL,
 *   dy is quantized here (dy itself is always required: the BF16 wgrad reads it).
 *   ws = moe_workspace_bytes(MOE_OP_MX_BWD, ...) bytes (256-byte aligned): dU high, dU low,
 *   routing partials, then the codes and scales of dy (unused when given) and of dU.
 */
moe_status_t moe_mx_prepare_weights(const moe_bf16* w_ug, const moe_bf16* w_down, int E, int d, int h, void* mxw,
                                    size_t mxw_bytes, moe_stream_t stream);
moe_status_t moe_permute_mxfp8(const moe_bf16* x, const int32_t* sorted_src, const int32_t* offsets, int T,
                               int top_k, int E, int d, moe_bf16* xp, uint8_t* q, uint8_t* sf, int32_t* dev_status,
                               moe_stream_t stream);
moe_status_t moe_mx_quantize_rows(const moe_bf16* x, const int32_t* offsets, int E, int cap, int K, uint8_t* q,
                                  uint8_t* sf, int32_t* dev_status, moe_stream_t stream);
moe_status_t moe_grouped_swiglu_fwd_mxfp8(const moe_bf16* xp, const uint8_t* xq, const uint8_t* xsf,
                                          const int32_t* offsets, const int32_t* sorted_src, const float* weights,
                                          int E, int cap, int d, int h, const void* mxw, moe_bf16* y,
                                          moe_bf16* a_save, void* saved, void* ws, size_t ws_bytes,
                                          int32_t* dev_status, moe_stream_t stream);
moe_status_t moe_grouped_bwd_mxfp8(const moe_bf16* dy, const uint8_t* dyq, const uint8_t* dysf, const moe_bf16* xp,
                                   const moe_bf16* a_save, const void* saved, const int32_t* offsets,
                                   const int32_t* sorted_src,
                                   const float* weights, int E, int cap, int d, int h, const void* mxw,
                                   moe_bf16* dxp, float* dw_ug, float* dw_down, const int32_t* inv_map,
                                   float* dw_route, void* ws, size_t ws_bytes, int32_t* dev_status,
                                   moe_stream_t stream);

/*
 * moe_route_offsets_noalloc -- moe_route_offsets for callers that cannot allocate device memory.
 * The pages have no counterpart: this is a library convenience. Some callers have no way to
 * hand over a workspace: code that runs where cudaMalloc is not allowed or not safe (inside a
 * framework's allocator or stream callbacks, under a fixed memory budget, or from a language
 * binding with no device allocator of its own). This entry point takes no `ws`: the per-warp
 * histogram scratch lives in one array inside the library, MOE_NOALLOC_ROUTE_SCRATCH_BYTES
 * (1 MiB) in size, which every GPU that loads the library keeps until the process exits.
 *
 *  Arguments, results and status codes as moe_route_offsets (minus ws / ws_bytes); results are
 *  bit-identical to it. Returns MOE_ERR_WORKSPACE_TOO_SMALL when the scratch it would need,
 *  moe_workspace_bytes(MOE_OP_ROUTE, T, top_k, E, 0, 0, 0) = ceil(T*top_k/256) * E * 4 bytes,
 *  exceeds MOE_NOALLOC_ROUTE_SCRATCH_BYTES.
 *  Calls no cudaMalloc or cudaFree. The first call on each device looks up the array's device
 *  address (cudaGetSymbolAddress) with that device current; make that first call before any
 *  stream capture. The address is kept per device together with the device's current context
 *  and looked up again when that context changes (after cudaDeviceReset the array may move),
 *  so the first call after such a change is a set-up call too. Every call shares the one array and every call rewrites each entry before it
 *  reads it, so nothing has to start at zero; but two calls that overlap on the GPU (different
 *  streams, or different host threads) race on it and give wrong results.
 */
#define MOE_NOALLOC_ROUTE_SCRATCH_BYTES (1u << 20)
moe_status_t moe_route_offsets_noalloc(const int32_t* ids, int T, int top_k, int E,
                                       int32_t* counts, int32_t* offsets, int32_t* sorted_src,
                                       int32_t* inv_map, moe_stream_t stream);

/* Human-readable text of a status (static storage). */
const char* moe_status_string(moe_status_t status);

/* Text of the last CUDA error seen by this thread inside the library (static per thread). */
const char* moe_last_cuda_error(void);

/* Version of this ABI (incremented on incompatible change). */
int moe_abi_version(void);

/*
 * Debug build. The same sources compiled with -DMOE_GG_DEBUG (build.build(debug=True) ->
 * libmoe_gg_debug.so, the same ABI) stand in for a memory checker: each kernel checks the
 * global accesses whose index comes from device data (offsets, slot and inverse maps, tile
 * decoding) against the extent of the buffer it addresses, skips an access that fails (or
 * redirects a copy a barrier waits for to the buffer's first element) and records it; and each
 * entry point waits for its stream when it returns (not while the stream is being captured),
 * so that an asynchronous CUDA error is reported by the call that queued the faulting work.
 * Release builds compile the checks away.
 *
 * moe_debug_build -- 1 for a debug build, else 0.
 * moe_debug_report -- waits for the device (cudaDeviceSynchronize), then writes
 *   *site_mask   bit s set when check site s failed since the last reset; bit
 *                MOE_DEBUG_CALL_ERROR_BIT when an entry point found a CUDA error on its
 *                stream as it returned (moe_last_cuda_error() then names the call);
 *   *first_site  the first failing site (-1: none), *index its index, *limit the bound the
 *                index had to stay below (each pointer nullable),
 *   and clears the record when reset != 0. A release build writes 0 and -1 and returns MOE_OK.
 *   Returns MOE_ERR_CUDA when the device cannot be read.
 * moe_debug_site_name -- name of check site s ("?" when out of range; static storage).
 */
#define MOE_DEBUG_CALL_ERROR_BIT 30
int moe_debug_build(void);
moe_status_t moe_debug_report(int32_t* site_mask, int32_t* first_site, long long* index,
                              long long* limit, int reset);
const char* moe_debug_site_name(int site);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GG_H */
