/* Attention-sink gradient of the fused softmax-attention backward (C ABI).
 *
 * Companion of attn_bwd.h: the same types, status codes and workspace.  A
 * sink is one extra logit per query head in every row's softmax
 * normalisation, with no value; its gradient is a per-head sum over the rows
 * that the dense backward's preprocess has prepared in the workspace. */
#ifndef ATTN_BWD_SINK_H
#define ATTN_BWD_SINK_H

#include "attn_bwd.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Gradient of per-query-head attention-sink logits: dsink[h] = -sum over the
 * rows i of every sequence (all batch rows; with cu_seqlens, rows
 * cu_seqlens[0] .. cu_seqlens[num_seqs] - 1) of exp(sink[h] - LSE_hi) delta_hi.
 * A sink is read as one extra logit per query head that joins every row's
 * softmax normalisation and carries no value: the forward's LSE includes
 * exp(sink[h]) and O is normalised by it, and dQ, dK, dV of the real keys are
 * then those of attn_bwd_gqa with that O and LSE.  The sink's own column has
 * dP = 0, so its dS is -P_sink delta_i, summed over the rows (the
 * flash-linear-attention issue "Evaluate KV-head-owned GQA dKV backward"
 * names dsink among the gradients of its frozen correctness contract without
 * a formula; this is the plain reading of an attention sink).
 *   sink   : f32 [HQ] on the device;  dsink : f32 [HQ] on the device, written
 *   workspace : the workspace of an attn_bwd_gqa / attn_bwd call (or of
 *   attn_bwd_preprocess) on the same stream, with the same B, S, HQ and mask:
 *   its LSE2 and delta rows are read.  Rows whose LSE is not finite add nothing.
 * One launch, one block per head, additions in a fixed order (the same result
 * from run to run).  Errors: ATTN_ERR_INVALID_ARG (null or misaligned pointer,
 * bad size or mask), ATTN_ERR_UNSUPPORTED (sizes past 2^31 rows),
 * ATTN_ERR_WORKSPACE, ATTN_ERR_LAUNCH. */
ATTN_BWD_API attn_status_t attn_bwd_sink_grad(const float* sink, int64_t B, int64_t S, int64_t HQ,
                                              const attn_mask_t* mask, const void* workspace,
                                              size_t workspace_bytes, float* dsink, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_BWD_SINK_H */
