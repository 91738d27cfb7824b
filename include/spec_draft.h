/*
 * spec_draft.h -- one draft step of a drafter that reuses the target's LM
 * head (sm_103a).
 *
 * Page: quochung.cyou A.I article on speculative decoding, the EAGLE part (a
 * small draft decoder layer estimates the hidden state h-hat the target
 * would produce; the target's own LM head turns h-hat into probabilities
 * over the vocabulary, from which the candidate token is taken).  One step:
 *
 *   z_q[b,:] = h_hat[b,:] . W_lm          (the target's LM head)
 *   T > 0:  x_b ~ softmax(z_q[b] / T), drawn by inverse CDF over ascending
 *           token ids on uniforms[b] (the rule of the verify step's
 *           correction and bonus draws): x_b = smallest v with
 *           C_v > u_b * S, so that x_b ~ q exactly;
 *   T == 0: x_b = argmax_v z_q[b,v], ties to the lowest id.
 *
 * Step j of a round drafts slot j: its logits are the verify step's draft
 * logits row b*K+j, so `out_logits` may point into a [B][K][V] draft-logits
 * buffer at slot j with row stride ld = K*V.
 *
 * Arguments (device pointers, caller-owned, as in spec_verify.h):
 *   hidden      bf16 [B][d]   the draft model's h-hat, one row per sequence
 *   W_lm        bf16 [V][d]   the target's LM-head weight
 *   uniforms    f32  [B]      in [0, 1); ignored (may be NULL) when T == 0
 *   out_tokens  int32 [B]     x_b, or -1 when the row's logits were not
 *                             finite (error word bit SPEC_DEVERR_NONFINITE)
 *   out_logits  f32, row b at out_logits + b*ld (ld >= V); may be NULL (the
 *               logits then live in the workspace); must be NULL when T == 0
 *               (the greedy step never materialises logits)
 *   dims        B, d, V as in spec_verify (K is ignored)
 * Workspace: spec_draft_step_workspace_bytes(dims, T) bytes, 16-byte
 * aligned, no initialisation; its error word is read with
 * spec_verify_read_error.  Alignment: 16 bytes for hidden, W_lm and
 * workspace, 4 for out_logits (any slot of a draft-logits buffer); d % 8 ==
 * 0.
 */
#ifndef SPEC_DRAFT_H_
#define SPEC_DRAFT_H_

#include "spec_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Workspace bytes of one draft step (0 if the sizes or T are invalid). */
SPEC_API size_t spec_draft_step_workspace_bytes(spec_dims dims, float temperature);

/* One draft step (see above).  Errors as spec_verify, plus SPEC_ERR_ARG for
 * out_logits given with T == 0 or ld < V. */
SPEC_API spec_status spec_draft_step(const void *hidden, const void *W_lm, const float *uniforms, float temperature,
                                     int32_t *out_tokens, float *out_logits, int64_t ld, spec_dims dims,
                                     void *workspace, size_t workspace_bytes, spec_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_DRAFT_H_ */
