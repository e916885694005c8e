/*
 * moe.h -- C ABI of libmoe.so: a single-GPU MoE layer for GB300 (sm_103a).
 *
 * The layer is the compute chain of the token-level dispatcher described in
 * "MoE Parallel Folding: Heterogeneous Parallelism Mappings for Efficient
 * Large-Scale MoE Model Training with Megatron Core" (arXiv 2504.14960),
 * study notes, "method overview": the router gives each token its Top-K
 * experts, a permutation makes each expert's tokens contiguous, the experts'
 * FFN runs, an un-permutation restores the token order; the backward runs the
 * same chain in reverse. The exchanges between ranks in that chain
 * (All-to-All-V, AllGather-V, ReduceScatter-V) are absent: one GPU holds every
 * expert, so each exchange is the identity.
 *
 * Conventions for every call below
 *  - Ownership: the caller allocates and owns every buffer. All tensor
 *    pointers are DEVICE pointers, 16-byte aligned, dense row-major with the
 *    layout stated. The library allocates nothing on the calls below.
 *  - Streams: every call is asynchronous on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream). No call synchronises the host or copies data
 *    to the host, except moe_get_status.
 *  - Data-dependent sizes stay on the device: the number of kept assignments
 *    and the per-expert row counts are read by later kernels from `offsets`.
 *    Buffers indexed by permuted row are sized for the worst case T*K rows.
 *  - Errors: argument checks that fail return MOE_ERR_INVALID_ARG or
 *    MOE_ERR_UNSUPPORTED before anything is launched; a failed launch returns
 *    MOE_ERR_CUDA. Device-side failures (a bounded wait that gave up, an index
 *    out of range) are recorded in the status word inside `ws` and read with
 *    moe_get_status; the kernel that saw one skips the bad access and returns.
 *  - Determinism: every output is bitwise reproducible from run to run.
 *  - dtype: MOE_BF16 means x, weights and activations are bf16 (accumulation
 *    in fp32); MOE_F32 means all of them are fp32. Logits, probabilities,
 *    combine weights, dXp, dx and every weight gradient are fp32 in both.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* bad pointer, size or alignment                    */
  MOE_ERR_UNSUPPORTED = 2, /* valid, but a shape the library has no kernel for */
  MOE_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed               */
  MOE_ERR_TIMEOUT = 4,     /* device: a bounded wait gave up (status word only)  */
  MOE_ERR_DEVICE = 5       /* device: an index check failed (status word only)   */
} moe_status_t;

enum { MOE_F32 = 0, MOE_BF16 = 1 };

typedef void *moe_stream_t; /* a cudaStream_t */

/* The problem statement of one MoE layer (study notes, "prerequisites":
 * Top-K gating and the capacity factor; "method overview" and "key modules":
 * drop and dropless routing, sub-sequence dropping).                          */
typedef struct {
  int64_t T;               /* tokens (micro-batch x sequence, flattened),
                              >= 1 and T * K < 2^31 (an empty batch is an
                              invalid shape: the caller skips the layer)     */
  int32_t d;               /* hidden size, a multiple of 8 (bf16) or 4 (fp32) */
  int32_t E;               /* routed experts, 1..64                          */
  int32_t K;               /* Top-K, 1..min(E, 8)                            */
  int32_t F;               /* routed expert SwiGLU intermediate size         */
  int32_t dtype;           /* MOE_BF16 or MOE_F32                            */
  int32_t drop;            /* 0 dropless, 1 capacity-factor dropping         */
  float capacity_factor;   /* CF, > 0 (used when drop = 1)                   */
  int64_t subseq_len;      /* S: drops are decided per block of S tokens of
                              the flat order; 0 means S = T (full sequence);
                              with drop = 1 the router needs S < 2^29
                              (else MOE_ERR_UNSUPPORTED)                     */
  int32_t renorm;          /* 1: combine weights renormalised over the K     */
  int32_t Fs;              /* shared expert SwiGLU size, 0 = none            */
} moe_shape_t;

/* Library version, "major.minor.patch". */
const char *moe_version(void);

/* Human-readable name of a status code. */
const char *moe_status_string(moe_status_t s);

/* Bytes of device workspace `ws` that the calls taking a `ws` need for this
 * shape (a multiple of 256; the caller allocates it 256-byte aligned and may
 * reuse it across calls on one stream). Returns 0 for an invalid shape. */
size_t moe_workspace_size(const moe_shape_t *shape);

/* Clears the device status word in `ws` (asynchronous). */
moe_status_t moe_clear_status(void *ws, moe_stream_t stream);

/* Synchronises `stream`, then returns the first device-side error recorded
 * in `ws` since the last moe_clear_status (MOE_OK if none). *info, if not
 * NULL, receives a kernel-specific detail word. */
moe_status_t moe_get_status(void *ws, moe_stream_t stream, uint32_t *info);

/* ---- forward ------------------------------------------------------------ */

/* Router: logits, softmax, Top-K, combine weights, capacity dropping.
 * Study notes, "method overview" (router Top-K), "prerequisites" (Top-K
 * gating, capacity factor), "key modules" and the quote of the paper's
 * section 3.3 (sub-sequence dropping is the default drop rule).
 *   x [T,d] dtype; W_r [E,d] dtype; b_r [E] fp32 or NULL (added to logits);
 *   w_sg [d] dtype or NULL: shared-expert gate vector;
 *   out: logits [T,E] fp32 = x W_r^T (+ b_r), accumulated in fp32 (bf16
 *        with d % 64 == 0: on the tensor cores, the K loop split in up to
 *        four fixed parts when the token count leaves SMs idle; the parts'
 *        fp32 sums are added in order, so the result is the same on every
 *        run on one GPU model);
 *        gate_logit [T] fp32 = x . w_sg (NULL iff w_sg is NULL);
 *        topk_idx [T,K] int32, topk_prob [T,K] fp32, topk_w [T,K] fp32,
 *        keep [T,K] uint8: as moe_route_topk.
 *   ws: workspace of moe_workspace_size(shape) bytes.                        */
moe_status_t moe_route(const moe_shape_t *shape, const void *x, const void *W_r,
                       const float *b_r, const void *w_sg, float *logits,
                       float *gate_logit, int32_t *topk_idx, float *topk_prob,
                       float *topk_w, uint8_t *keep, void *ws, moe_stream_t stream);

/* Top-K gating and capacity dropping from caller-supplied fp32 logits [T,E].
 * p = softmax(logits) computed in fp32 with a fixed operation order (own exp:
 * Cody-Waite reduction and degree-7 Taylor; pairwise sum; IEEE division).
 * topk_idx: K arg-max rounds over p, ties to the lower expert index, in
 * selection order; topk_prob = p at those experts; topk_w = topk_prob / Z with
 * Z = sum over the K slots in slot order (renorm = 1) or topk_prob (renorm 0).
 * keep[t,k] = 1 unless drop = 1 and the assignment is not among the
 * ceil(CF*S_j*K/E) highest-probability assignments of its (sub-sequence,
 * expert), ties to the lower token index. Kept weights are not renormalised
 * again after a drop.                                                        */
moe_status_t moe_route_topk(const moe_shape_t *shape, const float *logits,
                            int32_t *topk_idx, float *topk_prob, float *topk_w,
                            uint8_t *keep, void *ws, moe_stream_t stream);

/* Permutation map and row copy (study notes, "method overview": the
 * permutation makes each expert's tokens contiguous).
 *   in:  x [T,d] dtype; topk_idx, keep [T,K].
 *   out: counts [E] int32 (kept assignments per expert); offsets [E+1] int32
 *        (exclusive prefix of counts; offsets[E] = n_kept);
 *        row_of [T,K] int32: permuted row of each assignment, -1 if dropped;
 *        src_of [T*K] int32: t*K+k of each permuted row (first n_kept valid);
 *        Xp [T*K, d] dtype: Xp[row_of[t,k]] = x[t]; rows are expert-major and
 *        token-ascending inside an expert; rows >= n_kept are not written.
 *        Xp may be NULL: then only the map is built and no row is copied
 *        (for moe_expert_ffn_gather, which reads the rows from x itself). */
moe_status_t moe_permute(const moe_shape_t *shape, const void *x,
                         const int32_t *topk_idx, const uint8_t *keep, void *Xp,
                         int32_t *row_of, int32_t *src_of, int32_t *counts,
                         int32_t *offsets, void *ws, moe_stream_t stream);

/* GShard-style fixed layout (the alternative to the compact one; token
 * dropping only): expert e owns rows [e*C, (e+1)*C) of Xp, its kept rows
 * first (token-ascending, as moe_permute orders them) and zero rows after.
 * C = moe_padded_capacity(shape) = sum over sub-sequences of min(ceil(CF *
 * S_j * K / E), S_j), the most rows the capacity rule can keep for one
 * expert. MoE Parallel Folding study notes, "key modules" and "Q&A":
 * capacity-factor dropping bounds every expert's tokens, which is what lets a
 * dispatcher use fixed-size buffers.
 * moe_padded_capacity returns 0 when shape->drop is 0, the shape is invalid,
 * or E*C does not fit in int32.
 *   out: Xp [E*C, d]; row_of [T,K] (-1 when dropped); src_of [E*C] (t*K+k of
 *        each kept row, -1 on padding rows); counts [E]; offsets [E+1] =
 *        {0, C, 2C, ..., E*C}, so moe_expert_ffn(max_rows = E*C, n_groups = E)
 *        runs every padded row (zero rows give zero outputs) and
 *        moe_unpermute / moe_unpermute_bwd / moe_permute_bwd read row_of as
 *        for the compact layout.
 * Errors: as moe_permute; MOE_ERR_UNSUPPORTED when shape->drop is 0; a kept
 * count above C (keep not produced by the capacity rule) records
 * MOE_ERR_DEVICE in the status word and leaves that slot dropped.           */
int64_t moe_padded_capacity(const moe_shape_t *shape);
moe_status_t moe_permute_padded(const moe_shape_t *shape, const void *x,
                                const int32_t *topk_idx, const uint8_t *keep, void *Xp,
                                int32_t *row_of, int32_t *src_of, int32_t *counts,
                                int32_t *offsets, void *ws, moe_stream_t stream);

/* Largest token count T that moe_permute_noalloc accepts. */
#define MOE_PERMUTE_NOALLOC_MAX_TOKENS 131072

/* moe_permute for callers that cannot allocate device memory: the same
 * outputs as moe_permute (bit for bit), with no workspace argument. The paper
 * has no counterpart; this is a convenience of this library.
 * Who needs it: code that runs where cudaMalloc is not allowed or not safe --
 * inside a custom allocator's callbacks, under a fixed device-memory budget
 * reserved at start-up (serving processes that pin all memory up front), or
 * on a latency path that must not risk the implicit device synchronisation a
 * cudaMalloc/cudaFree can cause.
 * How: the map build's scratch (per-block expert counts, 128 KB) is a fixed
 * array inside libmoe.so, resident on every GPU that loads the library until
 * the process exits. The first call in each CUDA context (on each device, or
 * again after cudaDeviceReset) looks the array's device address up
 * (cudaGetSymbolAddress, with that device current) and caches it under the
 * context's ID; make that first call before any stream capture. No call
 * allocates.
 * Limits: T <= MOE_PERMUTE_NOALLOC_MAX_TOKENS, else MOE_ERR_UNSUPPORTED; E <= 64
 * as everywhere. Every call uses the same array: two calls that can run at the
 * same time on one GPU (different streams or host threads without ordering
 * between them) race and corrupt each other's maps; order them. Each call
 * rewrites all the scratch it reads, so the previous call's contents never
 * leak into a result. There is no workspace, so no device status word is
 * recorded: an out-of-range expert index is skipped (its row_of is -1), and
 * a row copy whose bounded wait gave up (which would mean a stalled copy
 * engine) leaves its token's rows of Xp unwritten without any report.      */
moe_status_t moe_permute_noalloc(const moe_shape_t *shape, const void *x,
                                 const int32_t *topk_idx, const uint8_t *keep, void *Xp,
                                 int32_t *row_of, int32_t *src_of, int32_t *counts,
                                 int32_t *offsets, moe_stream_t stream);

/* Grouped SwiGLU FFN (study notes, "method overview": expert FFN
 * computation). Group g owns rows [offsets[g], offsets[g+1]) of Xp.
 *   dtype: MOE_BF16 (tcgen05 tensor-core path) or MOE_F32;
 *   max_rows: rows allocated in Xp/A_save/H_save/Yp (offsets[n_groups] must
 *   not exceed it); d, F as in moe_shape_t; n_groups: experts (1 for a shared
 *   expert with offsets = {0, T}).
 *   W_gu [n_groups, 2F, d] (rows [0,F) gate, [F,2F) up); W_down [n_groups,d,F].
 *   out: A_save [max_rows, 2F] = [G|U] (NULL: not stored; the backward needs
 *        it); H_save [max_rows, F] = silu(G)*U (required: it is also the
 *        input of the down projection); Yp [max_rows, d] = H W_down^T.
 *        Only rows < offsets[n_groups] are written.
 *   ws: any workspace of this library (only its status word is used).
 *   bf16 requires d % 128 == 0 and F % 128 == 0 (else MOE_ERR_UNSUPPORTED);
 *   fp32 requires d % 4 == 0.                                                */
moe_status_t moe_expert_ffn(int32_t dtype, int64_t max_rows, int32_t d, int32_t F,
                            int32_t n_groups, const int32_t *offsets, const void *Xp,
                            const void *W_gu, const void *W_down, void *A_save,
                            void *H_save, void *Yp, void *ws, moe_stream_t stream);

/* The grouped SwiGLU FFN of moe_expert_ffn with the permutation fused into
 * its gate/up GEMM (study notes, "method overview": the permutation feeds the
 * experts' FFN directly): instead of reading Xp, the GEMM gathers permuted
 * row R from x as x[src_of[R] / K], so the permuted copy of the tokens is
 * neither written nor read back. Outputs equal moe_expert_ffn's on
 * Xp = permute(x) bit for bit.
 *   x [T, d] bf16 (the layer's tokens); src_of [>= offsets[n_groups]] int32
 *   as written by moe_permute / moe_permute_padded (t*K + k of each permuted
 *   row; a negative entry, the padded layout's padding rows, gives a zero
 *   row); T, K as in moe_shape_t. Other arguments as moe_expert_ffn
 *   (bf16 only; d % 128 == 0, F % 128 == 0).
 * Errors: as moe_expert_ffn; an src_of entry >= T*K records MOE_ERR_DEVICE
 *   in the status word and gives a zero row; MOE_ERR_UNSUPPORTED when the
 *   CTA-pair GEMM kernels are disabled.                                      */
moe_status_t moe_expert_ffn_gather(int64_t max_rows, int32_t d, int32_t F, int32_t n_groups,
                                   const int32_t *offsets, const void *x, int64_t T, int32_t K,
                                   const int32_t *src_of, const void *W_gu, const void *W_down,
                                   void *A_save, void *H_save, void *Yp, void *ws,
                                   moe_stream_t stream);

/* Un-permutation with the weighted Top-K combine (study notes, "method
 * overview": the un-permutation restores the original token order).
 *   out[t] = sum over kept slots k, in slot order, of topk_w[t,k] *
 *   Yp[row_of[t,k]] (+ sigmoid(gate_logit[t]) * Ys[t]), summed in fp32 and
 *   stored once in dtype. Ys [T,d] and gate_logit [T] are both NULL or both
 *   set. A token with every slot dropped and no shared expert outputs 0.     */
moe_status_t moe_unpermute(const moe_shape_t *shape, const void *Yp,
                           const int32_t *row_of, const float *topk_w, const void *Ys,
                           const float *gate_logit, void *out, moe_stream_t stream);

/* ---- backward (study notes, "method overview": the backward runs the
 *      chain in reverse) -------------------------------------------------- */

/* dYp[row_of[t,k]] = dtype(topk_w[t,k] * dout[t]) for kept slots;
 * dw[t,k] = <dout[t], Yp[row_of[t,k]]> fp32 (0 when dropped);
 * with a shared expert: dYs[t] = dtype(s_t * dout[t]), dz[t] = s_t (1 - s_t)
 * <dout[t], Ys[t]> with s_t = sigmoid(gate_logit[t]). Ys, gate_logit, dYs, dz
 * are all NULL or all set.                                                  */
moe_status_t moe_unpermute_bwd(const moe_shape_t *shape, const void *dout,
                               const void *Yp, const int32_t *row_of,
                               const float *topk_w, const void *Ys,
                               const float *gate_logit, void *dYp, float *dw,
                               void *dYs, float *dz, moe_stream_t stream);

/* Workspace bytes moe_expert_ffn_bwd needs: the status word and, for bf16,
 * the weight-gradient GEMMs' per-group tensor maps. moe_workspace_size()
 * never returns less than this for a valid shape.                           */
#define MOE_FFN_BWD_WORKSPACE_BYTES 33280u

/* Backward of moe_expert_ffn (same argument meanings).
 *   in:  dYp [max_rows,d] dtype; Xp; A_save; H_save; W_gu; W_down.
 *   out: dXp [max_rows, d] fp32 = dA W_gu; dW_gu [n_groups,2F,d] fp32 =
 *        dA^T Xp; dW_down [n_groups,d,F] fp32 = dYp^T H (zero for a group
 *        with no rows);
 *   dA [max_rows, 2F] dtype: caller-owned buffer that receives
 *   [dG | dU] = [dH*U*sg*(1+G(1-sg)) | dH*G*sg], dH = dYp W_down,
 *   sg = sigmoid(G), G|U from A_save.
 *   ws: ws_bytes bytes, 16-byte aligned; ws_bytes below
 *   MOE_FFN_BWD_WORKSPACE_BYTES returns MOE_ERR_INVALID_ARG.                 */
moe_status_t moe_expert_ffn_bwd(int32_t dtype, int64_t max_rows, int32_t d, int32_t F,
                                int32_t n_groups, const int32_t *offsets,
                                const void *dYp, const void *Xp, const void *A_save,
                                const void *H_save, const void *W_gu,
                                const void *W_down, void *dA, float *dXp,
                                float *dW_gu, float *dW_down, void *ws, size_t ws_bytes,
                                moe_stream_t stream);

/* dx[t] = sum over kept slots of dXp[row_of[t,k]] (+ dx_add[t]), fp32.
 * dXp [T*K,d] fp32; dx_add [T,d] fp32 or NULL; dx [T,d] fp32.               */
moe_status_t moe_permute_bwd(const moe_shape_t *shape, const float *dXp,
                             const int32_t *row_of, const float *dx_add, float *dx,
                             moe_stream_t stream);

/* Sum of partial results in part order (the arithmetic of a ReduceScatter-V
 * over an expert-tensor-parallel group, done on one GPU): out[i] =
 * dtype(((partials[0][i] + partials[1][i]) + ...) + partials[n_parts-1][i]),
 * fp32 additions, one rounding. MoE Parallel Folding study notes, "method
 * overview": ETP splits an expert's FFN dimension over ranks and sums the
 * partial outputs (ReduceScatter-V); here the F-shards of one expert run as
 * separate moe_expert_ffn calls and this call adds their outputs.
 *   partials [n_parts, rows, d] dtype, contiguous; out [rows, d] dtype (may
 *   not alias partials). dtype MOE_BF16 or MOE_F32; 1 <= n_parts <= 16;
 *   d a multiple of 8 (bf16) or 4 (fp32); pointers 16-byte aligned.
 * Errors: MOE_ERR_INVALID_ARG for NULL/misaligned pointers or bad sizes.    */
moe_status_t moe_sum_partials(int32_t dtype, int32_t n_parts, int64_t rows, int32_t d,
                              const void *partials, void *out, moe_stream_t stream);

/* Router backward. g = dw [T,K]; renorm: dp_j = (g_j - sum_k g_k w_k) / Z on
 * the Top-K (Z = sum of topk_prob), else dp = g there; dp = 0 elsewhere;
 * p = softmax(logits) as in moe_route_topk; dl_i = p_i (dp_i - sum_j p_j dp_j).
 *   out: dW_r [E,d] fp32 = dl^T x; db_r [E] fp32 = sum_t dl (NULL: skipped);
 *        dx_router [T,d] fp32 = (dx_in or 0) + dl W_r (+ dz w_sg);
 *        dw_sg [d] fp32 = dz^T x (NULL iff dz is NULL).
 *   w_sg, dz, dw_sg: all NULL or all set. dx_in [T,d] fp32 or NULL.        */
moe_status_t moe_route_bwd(const moe_shape_t *shape, const void *x, const void *W_r,
                           const void *w_sg, const float *logits,
                           const int32_t *topk_idx, const float *topk_prob,
                           const float *topk_w, const float *dw, const float *dz,
                           const float *dx_in, float *dW_r, float *db_r,
                           float *dw_sg, float *dx_router, void *ws,
                           moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
