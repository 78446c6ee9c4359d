/*
 * attn_bwd.h -- C ABI of the GB300 (sm_103a) fused softmax-attention backward.
 *
 * Given Q, K, V, O, dO and the per-row natural-log log-sum-exp of a softmax
 * attention forward, the library computes dQ, dK and dV without materialising
 * any S x S matrix.  The operation is the unsplit backward of the TileOPs pull
 * request "Serve MHA backward on a warp-specialized SM90 kernel and time FA3's
 * backward alone" (section "TileFoundry Description", program "Reference"):
 *
 *   delta_i = sum_d O_id dO_id
 *   P_ij    = exp(scale * q_i.k_j - LSE_i)   where key j is visible to query i, else 0
 *   dV_j    = sum_i P_ij dO_i
 *   dP_ij   = dO_i . v_j
 *   dS_ij   = P_ij (dP_ij - delta_i) scale
 *   dQ_i    = sum_j dS_ij k_j                 dK_j = sum_i dS_ij q_i
 *
 * split, as on that page's "Tiled" program and its three-launch summary, into
 * a preprocess (delta), a main kernel that owns key blocks (dK, dV written
 * once; dQ accumulated in f32) and a dQ landing pass (scale and cast).
 * Grouped-query attention follows the flash-linear-attention issue "Evaluate
 * KV-head-owned GQA dKV backward" (section "Bounded scope", items 1-2): one
 * CTA owns a key tile of one KV head and loops over the G query heads of the
 * group.  Top-k sparse attention over a shared latent K/V row follows the
 * tilelang pull request "Adaptive threads for sparse MLA backward".
 *
 * Conventions for every entry point:
 *   - Tensors are BSHD (batch, sequence, head, head-dim) in device memory,
 *     addressed as base + b*st.b + s*st.s + h*st.h + d (element strides; the
 *     head-dim stride is 1).  Base pointers and the strides b, s, h (in bytes)
 *     must be 16-byte aligned.  16-bit tensors hold ATTN_DT_F16 or
 *     ATTN_DT_BF16 values as given by ``dtype``.
 *   - The caller owns every buffer, including the workspace; the library
 *     allocates nothing and keeps no state between calls.  Calls on different
 *     streams are independent as long as each uses its own workspace.
 *   - ``stream`` is a cudaStream_t (NULL: the legacy default stream).  All
 *     work is asynchronous; a call returns after queueing its launches.
 *   - A call either queues all of its launches or returns an error before
 *     queueing any: argument errors come back as ATTN_ERR_INVALID_ARG or
 *     ATTN_ERR_UNSUPPORTED, never as a silent fallback.  Faults found by the
 *     kernels themselves (a bounded wait that ran out) are recorded in the
 *     workspace and reported by attn_bwd_check_error.
 *   - One call per backward: attn_bwd / attn_bwd_gqa (dense) and
 *     attn_bwd_sparse (top-k) take Q, K, V, O, dO and the LSE, validate every
 *     argument, then queue the three launches on ``stream`` and deliver dQ,
 *     dK and dV (or dQ and dKV).  The launches are also exported one by one
 *     (the split form): attn_bwd_preprocess, then attn_bwd_gqa_main (or
 *     attn_bwd_sparse_main), then attn_bwd_dq_land (or attn_bwd_sparse_land),
 *     on one stream with the same workspace.
 */
#ifndef ATTN_BWD_H_
#define ATTN_BWD_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_BWD_API __attribute__((visibility("default")))
#else
#define ATTN_BWD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { ATTN_DT_F16 = 0, ATTN_DT_BF16 = 1 } attn_dtype_t;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer or stride */
  ATTN_ERR_UNSUPPORTED = 2, /* well-formed but outside what the kernels serve (head dim, group size, ...) */
  ATTN_ERR_WORKSPACE = 3,   /* workspace missing or smaller than attn_bwd_workspace_size() */
  ATTN_ERR_LAUNCH = 4,      /* the CUDA runtime refused a launch */
  ATTN_ERR_TIMEOUT = 5,     /* a kernel's bounded wait ran out (reported by attn_bwd_check_error) */
  ATTN_ERR_DEVICE = 6       /* a CUDA error surfaced while synchronising */
} attn_status_t;

/* Element strides of a BSHD tensor (or b, h, s strides of an LSE [B,H,S]). */
typedef struct {
  int64_t b, s, h;
} attn_strides_t;

/* Which keys a query sees, within one sequence.  Sequences: each batch row,
 * or, when cu_seqlens is given (B must be 1), the packed ranges
 * [cu_seqlens[n], cu_seqlens[n+1]) along S.  Positions are local to a
 * sequence.  Query i stands at key position i + off, where off = Sk - S for
 * a dense row of S queries and Sk keys and off = 0 otherwise (the masks are
 * aligned at the end of the row, so the last query sees the last key; the
 * pages define the masks for square problems only, and this is the reading
 * taken for rows whose lengths differ).  Query i sees key j iff
 *   causal == 0 and window_left < 0 : always,
 *   causal != 0                     : j <= i + off  (the page's "cols <= rows"),
 *   window_left = W > 0             : i + off - W < j <= i + off  (implies causal).
 * A query that sees no key (i + off < 0) gets dQ = 0 and adds nothing to dK,
 * dV; its LSE row is expected to be -inf (any value is accepted: it is never
 * used as an operand).
 * cu_seqlens: device int32 [num_seqs + 1], non-decreasing from 0 and ending
 * at most at S (the kernels clamp to S); NULL for dense batches.  Rows past
 * cu_seqlens[num_seqs] belong to no sequence: the kernels never use their Q,
 * K, V, dO, O or LSE values as operands (tiles that overhang them are zeroed
 * in shared memory after the load), so they may hold anything, NaN included;
 * dQ rows there are written as zero and dK/dV rows there are not written.
 * No longest-sequence length is needed: the persistent kernels compute the
 * tile count of every sequence on the device.
 * kv_len: keys per batch row of a dense batch, Sk (k, v, dk, dv are then
 * [B,Sk,HKV,D]); 0 means Sk = S.  Must be 0 or S when cu_seqlens is given. */
typedef struct {
  int32_t causal;
  int32_t window_left;
  const int32_t* cu_seqlens;
  int32_t num_seqs;
  int32_t kv_len;
} attn_mask_t;

/* Bytes of workspace one backward call needs: a 256-byte header (device error
 * word, tile counter), LSE*log2(e) and delta as f32 [B,H,S], the f32 dQ
 * accumulator [B,S,H,Dq], and ``dkv_elems`` f32 for a sparse dKV accumulator
 * (0 for dense).  Every region is 256-byte aligned. */
ATTN_BWD_API size_t attn_bwd_workspace_size(int64_t B, int64_t S, int64_t H, int64_t Dq, int64_t dkv_elems);

/* Workspace bytes with which the one-call dense backward (attn_bwd_gqa,
 * attn_bwd) may split the last round of key tiles: at head dim 128, on an
 * unmasked dense batch with G >= 2, when the tiles do not divide evenly over
 * the persistent CTAs, the last round's tiles are drawn as units of fewer query
 * heads whose dK/dV partials are added in f32 behind the dQ accumulator (at
 * most 256 tiles, 2*D*128 + 4 values each).  Any workspace of at least
 * attn_bwd_workspace_size(B, S, HQ, D, 0) bytes stays valid: without room for
 * the partials the tiles are drawn whole.  0 for negative sizes. */
ATTN_BWD_API size_t attn_bwd_gqa_workspace_size(int64_t B, int64_t S, int64_t HQ, int64_t D);

/* Split form, launch 1: delta_i = sum_d O_id dO_id (f32), LSE*log2(e), zeroed dQ (and
 * dKV) accumulators, cleared error word and tile counter.  The delta row
 * preprocess of the TileOPs page ("delta_rows" in its Base and Tiled
 * programs).
 *   o, dO : [B,S,H,Dv] 16-bit;  lse : f32, lse[b*slse.b + h*slse.h + s*slse.s]
 *   Dq    : head dim of Q (sizes the dQ accumulator; 0 for the sparse path,
 *           which needs none); dkv_elems as above.
 * Dv must be a multiple of 8 and at most 1024. */
ATTN_BWD_API attn_status_t attn_bwd_preprocess(const void* o, attn_strides_t so, const void* dO, attn_strides_t sdo,
                                  const float* lse, attn_strides_t slse, int64_t B, int64_t S, int64_t H,
                                  int64_t Dv, int64_t Dq, int64_t dkv_elems, attn_dtype_t dtype, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* Group sizes G = HQ / HKV the dense path accepts: at most 16 query heads per
 * KV head in either dtype (larger groups return ATTN_ERR_UNSUPPORTED).  P and
 * dS are rounded to the input dtype before the dV and dK products, as the
 * TileOPs page's "Tiled" program does.  With bf16's 8-bit significand the
 * rounding errors of large P (short causal rows), summed over the group's
 * heads, would exceed the bf16 tolerance from G = 8 on; so for bf16 groups of
 * more than 4 heads a step whose largest P exceeds 1/8 also adds the 16-bit
 * rounding residuals of P and dS through a second pair of dV / dK products.
 * Steps of long rows, whose P stay small, run without them. */
#define ATTN_BWD_MAX_GROUP_F16 16
#define ATTN_BWD_MAX_GROUP_BF16 16

/* The whole dense backward of grouped-query attention in one call: the
 * TileOPs page's three launches behind one op call ("Summary": preprocess,
 * main kernel, dQ landing), queued on ``stream`` after every argument has
 * been checked, so a call either queues all three or nothing.
 *   q, o, dO, dq : [B,S,HQ,D] 16-bit;  k, v, dk, dv : [B,Sk,HKV,D] 16-bit
 *   (Sk = mask->kv_len if mask and kv_len > 0, else S);
 *   lse : f32 natural-log LSE [B,HQ,S] of the forward with strides slse
 *   (b, s, h);  dq, dk, dv are written (dK and dV once per key row by their
 *   owning CTA, dQ = sm_scale * the f32 sum of its partials).
 *   D in {64, 128};  G = HQ / HKV within the limits above;  S >= 1;  B == 1
 *   when varlen;  sm_scale finite.  Query head h reads KV head h / G.
 *   workspace : at least attn_bwd_workspace_size(B, S, HQ, D, 0) bytes,
 *   16-byte aligned, owned by the caller; its contents on entry do not matter;
 *   attn_bwd_gqa_workspace_size(B, S, HQ, D) bytes allow the last-round split.
 * Errors: ATTN_ERR_INVALID_ARG (null or misaligned pointer, bad stride, size
 * or mask), ATTN_ERR_UNSUPPORTED (head dim, group size, dtype, sizes past
 * 2^31 rows), ATTN_ERR_WORKSPACE, all before anything is queued;
 * ATTN_ERR_LAUNCH if the runtime refuses a launch. */
ATTN_BWD_API attn_status_t attn_bwd_gqa(const void* q, attn_strides_t sq, const void* k, attn_strides_t sk,
                                        const void* v, attn_strides_t sv, const void* o, attn_strides_t so,
                                        const void* dO, attn_strides_t sdo, const float* lse, attn_strides_t slse,
                                        int64_t B, int64_t S, int64_t HQ, int64_t HKV, int64_t D, attn_dtype_t dtype,
                                        float sm_scale, const attn_mask_t* mask, void* dq, attn_strides_t sdq,
                                        void* dk, attn_strides_t sdk, void* dv, attn_strides_t sdv, void* workspace,
                                        size_t workspace_bytes, void* stream);

/* The forward whose outputs the backward takes: O = softmax(scale Q K^T) V
 * under the mask, and the natural-log LSE of every query row (the TileOPs
 * page's backward op takes q, k, v, o, do, lse, "Summary"; the rows computed
 * are the first half of its "Reference" program: masked scores, their softmax
 * and log-sum-exp).  Persistent CTAs, one per SM, walk units of two 128-row
 * query tiles of one query head;
 * tcgen05 MMAs with the scores and O in tensor memory, the row max updated
 * lazily (O rescaled only when a row max grows by more than 2^8).
 *   q, o : [B,S,HQ,D] 16-bit;  k, v : [B,Sk,HKV,D] 16-bit (Sk as for
 *   attn_bwd_gqa);  lse : f32, lse[b*slse.b + h*slse.h + s*slse.s] (written);
 *   o is written in the input dtype.  A query that sees no key gets O = 0 and
 *   LSE = -inf.  Rows past cu_seqlens[num_seqs] are not written; their K/V
 *   rows may hold anything (they are zeroed in shared memory before use).
 *   D in {64, 128};  any G = HQ / HKV;  sm_scale finite and > 0.
 *   workspace : at least 256 bytes, 16-byte aligned (the header of a backward
 *   workspace serves); its error word is cleared by the call and
 *   attn_bwd_check_error reports a kernel whose bounded wait ran out.
 * Errors: ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_WORKSPACE
 * before anything is queued; ATTN_ERR_LAUNCH if the runtime refuses. */
ATTN_BWD_API attn_status_t attn_fwd_gqa(const void* q, attn_strides_t sq, const void* k, attn_strides_t sk,
                                        const void* v, attn_strides_t sv, int64_t B, int64_t S, int64_t HQ,
                                        int64_t HKV, int64_t D, attn_dtype_t dtype, float sm_scale,
                                        const attn_mask_t* mask, void* o, attn_strides_t so, float* lse,
                                        attn_strides_t slse, void* workspace, size_t workspace_bytes, void* stream);

/* Multi-head attention: attn_bwd_gqa with HQ == HKV == H (the page's MHA op is
 * GQA with H_kv = H). */
ATTN_BWD_API attn_status_t attn_bwd(const void* q, attn_strides_t sq, const void* k, attn_strides_t sk, const void* v,
                                    attn_strides_t sv, const void* o, attn_strides_t so, const void* dO,
                                    attn_strides_t sdo, const float* lse, attn_strides_t slse, int64_t B, int64_t S,
                                    int64_t H, int64_t D, attn_dtype_t dtype, float sm_scale, const attn_mask_t* mask,
                                    void* dq, attn_strides_t sdq, void* dk, attn_strides_t sdk, void* dv,
                                    attn_strides_t sdv, void* workspace, size_t workspace_bytes, void* stream);

/* Split form, launch 2 of the dense path: one CTA per (key tile of 128 rows,
 * KV head, batch) keeps K and V in shared memory and dK, dV in tensor memory,
 * loops over the G query heads of its group and their query blocks, writes dK
 * (times sm_scale) and dV once in the input dtype and adds its dQ partials
 * into the workspace accumulator (the "Tiled" program's placement; KV-head
 * ownership as in the flash-linear-attention issue, "Bounded scope" items
 * 1-2).  Arguments as for attn_bwd_gqa; needs attn_bwd_preprocess first and
 * attn_bwd_dq_land after it, on the same stream and workspace. */
ATTN_BWD_API attn_status_t attn_bwd_gqa_main(const void* q, attn_strides_t sq, const void* k, attn_strides_t sk,
                                             const void* v, attn_strides_t sv, const void* dO, attn_strides_t sdo,
                                             int64_t B, int64_t S, int64_t HQ, int64_t HKV, int64_t D,
                                             attn_dtype_t dtype, float sm_scale, const attn_mask_t* mask, void* dk,
                                             attn_strides_t sdk, void* dv, attn_strides_t sdv, void* workspace,
                                             size_t workspace_bytes, void* stream);

/* Split form, launch 3 of the dense path: dQ = cast(sm_scale * dQacc), the
 * TileOPs page's "dq_land".
 *   dq : [B,S,H,D] 16-bit (written).  B*S*H below 2^31, else
 *   ATTN_ERR_UNSUPPORTED. */
ATTN_BWD_API attn_status_t attn_bwd_dq_land(void* dq, attn_strides_t sdq, int64_t B, int64_t S, int64_t H, int64_t D,
                               attn_dtype_t dtype, float sm_scale, const void* workspace, size_t workspace_bytes,
                               void* stream);

/* The whole top-k sparse backward over shared latent rows (the tilelang
 * sparse MLA backward) in one call: the preprocess (delta, LSE*log2(e), a
 * zeroed f32 dKV accumulator; no dQ accumulator), the sparse kernel and the
 * dKV cast, queued on ``stream`` after every argument has been checked.
 * Query t of batch b, head h (KV head g = h / (H/HKV)) attends the latent rows
 * kv[b, idx[b,t,g,s], g, :] for every slot s whose index lies in [0, SKV);
 * other entries (-1 pads) are not visible.  K is the whole DQK-wide row, V its
 * first DV columns, and dKV = dK + [dV, 0].
 *   q, dq : [B,S,H,DQK];  kv, dkv : [B,SKV,HKV,DQK], kv stored densely (row
 *   stride DQK);  o, dO : [B,S,H,DV] 16-bit;  lse : f32 [B,H,S] with strides
 *   slse (b, s, h);  idx : int32 [B,S,HKV,topk] with strides sidx (slot
 *   stride 1);  DQK = 576, DV = 512;  G = H / HKV <= 64;  topk >= 1.
 *   workspace : attn_bwd_workspace_size(B, S, H, 0, B*SKV*HKV*DQK) bytes.
 * A group of G < 64 heads (a tensor-parallel split of the heads) is computed
 * padded to 64 heads whose extra rows contribute exactly zero, so it takes
 * 64/G times the work of its own heads.  Errors as for attn_bwd_gqa. */
ATTN_BWD_API attn_status_t attn_bwd_sparse(const void* q, attn_strides_t sq, const void* kv, attn_strides_t skv,
                                           const void* o, attn_strides_t so, const void* dO, attn_strides_t sdo,
                                           const float* lse, attn_strides_t slse, const int32_t* idx,
                                           attn_strides_t sidx, int64_t B, int64_t S, int64_t SKV, int64_t H,
                                           int64_t HKV, int64_t DQK, int64_t DV, int64_t topk, attn_dtype_t dtype,
                                           float sm_scale, void* dq, attn_strides_t sdq, void* dkv,
                                           attn_strides_t sdkv, void* workspace, size_t workspace_bytes,
                                           void* stream);

/* Split form, launch 2 of the sparse path: one CTA owns a (token, KV head)
 * pair with all of its query heads, so dQ (which already includes sm_scale)
 * is written here, once; dKV partials are added into the workspace's f32 dKV
 * accumulator, which attn_bwd_sparse_land casts.  The preprocess before it
 * runs with Dq = 0 (no dQ accumulator) and dkv_elems = B*SKV*HKV*DQK.
 * Arguments as for attn_bwd_sparse. */
ATTN_BWD_API attn_status_t attn_bwd_sparse_main(const void* q, attn_strides_t sq, const void* kv, attn_strides_t skv,
                                                const void* dO, attn_strides_t sdo, const int32_t* idx,
                                                attn_strides_t sidx, int64_t B, int64_t S, int64_t SKV, int64_t H,
                                                int64_t HKV, int64_t DQK, int64_t DV, int64_t topk,
                                                attn_dtype_t dtype, float sm_scale, void* dq, attn_strides_t sdq,
                                                void* workspace, size_t workspace_bytes, void* stream);

/* Split form, launch 3 of the sparse path: dKV = cast(dKVacc) (the sparse
 * kernel applies sm_scale to dS itself: dKV mixes the scaled dK term with the
 * unscaled dV term, so the scale cannot be folded into a landing pass as on
 * the dense path).  B, S, H locate the workspace regions as at preprocess
 * time.
 *   dkv : [B,SKV,HKV,DQK] 16-bit (written).  B*SKV*HKV below 2^31, else
 *   ATTN_ERR_UNSUPPORTED. */
ATTN_BWD_API attn_status_t attn_bwd_sparse_land(void* dkv, attn_strides_t sdkv, int64_t B, int64_t S, int64_t SKV,
                                                int64_t H, int64_t HKV, int64_t DQK, attn_dtype_t dtype,
                                                const void* workspace, size_t workspace_bytes, void* stream);

/* Synchronises ``stream`` and reports the device error word of ``workspace``:
 * ATTN_OK, ATTN_ERR_TIMEOUT (a bounded wait ran out; *device_code, if not
 * NULL, receives the site code) or ATTN_ERR_DEVICE (a CUDA error). */
ATTN_BWD_API attn_status_t attn_bwd_check_error(const void* workspace, void* stream, int32_t* device_code);

/* Static description of a status code. */
ATTN_BWD_API const char* attn_bwd_status_string(attn_status_t status);

/* Host-side schedule helper, exported so that the tile/mask derivation can be
 * checked against a brute-force mask: the half-open range [*lo, *hi) of query
 * blocks of ``block_q`` rows that a key tile [k0, k0 + block_k) of a sequence
 * of ``len`` positions must visit so that no visible (query, key) pair is
 * missed and no block without one is visited. */
ATTN_BWD_API void attn_bwd_query_block_range(int32_t k0, int32_t block_k, int32_t len, int32_t causal, int32_t window_left,
                                int32_t block_q, int32_t* lo, int32_t* hi);

/* The same for a dense row of ``q_len`` queries and ``kv_len`` keys whose
 * masks are aligned at the end of the row (query i at key position
 * i + kv_len - q_len, as attn_mask_t describes); with q_len == kv_len it
 * equals attn_bwd_query_block_range. */
ATTN_BWD_API void attn_bwd_query_block_range_qk(int32_t k0, int32_t block_k, int32_t kv_len, int32_t q_len,
                                                int32_t causal, int32_t window_left, int32_t block_q, int32_t* lo,
                                                int32_t* hi);

/* Host-side schedule helper, exported so that the persistent tile order of the
 * dense kernels can be checked on the host.  Tile ``t`` is the t-th draw from
 * the tile counter of a launch over B batch rows, S positions and HKV KV heads
 * with the mask (causal, window_left) and, for packed sequences, cu_seqlens
 * (HOST memory here, [num_seqs + 1]; NULL for dense batches).  Tiles are 128
 * keys, query blocks 128 rows; dense batches go through the (batch, KV head)
 * pairs in groups of 8, key block major inside a group (the longest tiles of a
 * group first under a causal mask), packed sequences key block major over all
 * pairs.  (A launch sizes its groups by the CTAs in flight: rows with more key
 * tiles per pair than CTAs take groups of one pair; this helper shows the
 * groups of 8.)  Writes out[0..6] = {valid, b, kv head, sequence start, first key
 * (sequence-local), first query block, number of query blocks}; valid = 0 for
 * a draw past the last tile or invalid sizes (B, S, HKV < 1). */
ATTN_BWD_API void attn_bwd_tile_schedule(int32_t t, int32_t B, int32_t S, int32_t HKV, int32_t causal,
                                         int32_t window_left, const int32_t* cu_seqlens, int32_t num_seqs,
                                         int32_t* out);

/* Host-side plan of the last-round split for ``tiles`` equal key tiles on
 * ``ctas`` persistent CTAs with G query heads per KV head: out[0..2] =
 * {first split draw, split tiles, query heads per unit}, all 0 when the tiles
 * are drawn whole (the split shortens the last round by less than a quarter
 * tile, half a tile at G = 2, or G < 2, or the tiles divide evenly). */
ATTN_BWD_API void attn_bwd_tail_plan(int64_t tiles, int32_t ctas, int32_t G, int32_t* out);

/* attn_bwd_tile_schedule for an unmasked dense batch with G query heads per KV
 * head and a last-round split (tail_tiles = 0: none): out[0..9] = the seven
 * values above, then {first query head of the unit within the group, query
 * heads, partials slot (-1 for a whole tile)}. */
ATTN_BWD_API void attn_bwd_tile_schedule_split(int32_t t, int32_t B, int32_t S, int32_t HKV, int32_t G,
                                               int32_t tail_start, int32_t tail_tiles, int32_t tail_hpu,
                                               int32_t* out);

/* Self-test of the bounded-wait machinery: launches one CTA that waits on a
 * barrier nothing signals, with a ``timeout_us`` limit, and returns what
 * attn_bwd_check_error then reports (ATTN_ERR_TIMEOUT when the machinery
 * works).  Needs a workspace of at least 256 bytes. */
ATTN_BWD_API attn_status_t attn_bwd_selftest_timeout(void* workspace, size_t workspace_bytes, int32_t timeout_us, void* stream);

/* Size of the library-held workspace of attn_bwd_gqa_noalloc (32 MiB). */
#define ATTN_BWD_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/* The whole dense backward (attn_bwd_gqa's three launches on ``stream``) for
 * callers that cannot allocate device memory: plugins running inside a
 * framework that owns all device memory through its own pool, and
 * latency-critical loops that cannot afford the device-wide synchronisation
 * of cudaMalloc/cudaFree.  This entry point is a convenience of this library;
 * the pages it follows have no counterpart.
 *
 * Instead of a workspace argument it uses one device array of
 * ATTN_BWD_NOALLOC_SCRATCH_BYTES that the library holds, on every GPU that
 * loads it, until the process exits; it allocates nothing.  Problems whose
 * attn_bwd_workspace_size(B, S, HQ, D, 0) exceeds that size are rejected with
 * ATTN_ERR_WORKSPACE, and every other argument is checked as attn_bwd_gqa
 * checks it, before anything is queued.  The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress) with that device current
 * and keeps it for the life of the process; make that first call before any
 * stream capture, and do not use this entry point across a device reset
 * (cudaDeviceReset), after which the kept address is stale.  All calls on a
 * device share the array: calls whose work overlaps on the GPU (different
 * streams, or several host threads) race and corrupt each other's results, so
 * serialise them.  The preprocess clears what must start at zero, so earlier
 * calls' leftovers do not matter.  Errors found by the kernels themselves (a
 * bounded wait that ran out) are recorded in the array; read them with
 * attn_bwd_noalloc_check_error.
 *   Arguments as for attn_bwd_gqa, without the workspace. */
ATTN_BWD_API attn_status_t attn_bwd_gqa_noalloc(const void* q, attn_strides_t sq, const void* k, attn_strides_t sk,
                                                const void* v, attn_strides_t sv, const void* o, attn_strides_t so,
                                                const void* dO, attn_strides_t sdo, const float* lse,
                                                attn_strides_t slse, int64_t B, int64_t S, int64_t HQ, int64_t HKV,
                                                int64_t D, attn_dtype_t dtype, float sm_scale,
                                                const attn_mask_t* mask, void* dq, attn_strides_t sdq, void* dk,
                                                attn_strides_t sdk, void* dv, attn_strides_t sdv, void* stream);

/* attn_bwd_check_error for the array of attn_bwd_gqa_noalloc on the current
 * device: synchronises ``stream`` and reports ATTN_OK, ATTN_ERR_TIMEOUT (with
 * the site code in *device_code, if not NULL) or ATTN_ERR_DEVICE.  The next
 * attn_bwd_gqa_noalloc call on the device clears the recorded error. */
ATTN_BWD_API attn_status_t attn_bwd_noalloc_check_error(void* stream, int32_t* device_code);

/* Device scratch bytes that attn_bwd_gqa_host needs to process the problem
 * in about ``chunks`` chunks (0 for an invalid shape). */
ATTN_BWD_API size_t attn_bwd_host_scratch_size(int64_t B, int64_t S, int64_t HQ, int64_t HKV, int64_t D,
                                               int64_t chunks);

/* The dense backward from host buffers to host buffers, with the
 * host<->device copies overlapped with the kernels.  This entry point is a
 * convenience of this library; the pages it follows have no counterpart.
 *
 * The problem is split into chunks of batch rows and KV heads; a chunk (its
 * KV heads and their query heads) is independent of the others.  With
 * chunks >= B each batch row is split into ceil(HKV / ceil(HKV / (chunks / B)))
 * ranges of KV heads; with chunks < B a chunk is ceil(B / chunks) whole batch
 * rows.  Each chunk is copied in (strided slices of the host tensors into
 * contiguous device buffers, on ``copy_in_stream``), run through attn_bwd_gqa (its three
 * launches, on ``stream``) and copied out (on
 * ``copy_out_stream``), with two buffer slots so that copies of neighbouring
 * chunks overlap the kernels.  The copies start after the work queued on
 * ``stream`` before the call, and ``stream`` waits for the last copy-out, so
 * synchronising ``stream`` covers the whole call.  The three streams must be
 * distinct for the work to overlap.
 *   q, o, dO, dq : host [B,S,HQ,D] 16-bit, contiguous;  k, v, dk, dv : host
 *   [B,S,HKV,D] 16-bit, contiguous;  lse : host f32 [B,HQ,S] (natural log),
 *   contiguous.  Host buffers should be page-locked (with pageable memory the
 *   copies are correct but do not overlap); dq, dk, dv are written.
 *   mask : as for attn_bwd_gqa (cu_seqlens in device memory); kv_len must be
 *   0 or S here (ATTN_ERR_INVALID_ARG otherwise).
 *   scratch : device memory of attn_bwd_host_scratch_size(...) bytes, 256-byte
 *   aligned, owned by the caller; it starts with the workspace of one chunk,
 *   so attn_bwd_check_error(scratch, stream, ...) reports device errors.
 * The call creates CUDA events and releases them before it returns (each is
 * freed once the work that uses it completes); it allocates no memory.
 * Returns an error before queueing anything for invalid arguments; an error
 * from a later step leaves the chunks queued so far in flight. */
ATTN_BWD_API attn_status_t attn_bwd_gqa_host(const void* q, const void* k, const void* v, const void* o,
                                             const void* dO, const float* lse, int64_t B, int64_t S, int64_t HQ,
                                             int64_t HKV, int64_t D, attn_dtype_t dtype, float sm_scale,
                                             const attn_mask_t* mask, void* dq, void* dk, void* dv, void* scratch,
                                             size_t scratch_bytes, int64_t chunks, void* stream,
                                             void* copy_in_stream, void* copy_out_stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_BWD_H_ */
