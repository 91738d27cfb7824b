/*
 * spec_tree.h -- C ABI of tree-shaped candidate verification (sm_103a).
 *
 * Pages: "Speculative Decoding: Memverifikasi Token Draft secara Paralel",
 * section "Sampling eksak memerlukan aturan koreksi" (tree-shaped candidates
 * are a variant that needs its own distribution claim; the acceptance ratio
 * min(1, p/q) and the positive residual max(0, p - q)), with the prefix
 * rule of "Penolakan memotong prefix yang diterima".
 *
 * Tree: N nodes per sequence.  Node 0 is the root (the last committed
 * token's position); node i >= 1 carries draft token tokens[b][i] and a
 * parent parents[b][i] < i (parents[b][0] = -1).  Target row i (one row per
 * node, from one tree-attention pass) is the target's next-token
 * distribution after the path to node i; draft row i is the distribution
 * node i's children were drawn from.  The children of a node must be
 * independent draws from that node's draft distribution (repeats allowed):
 * that is the condition under which the rule below reproduces the target
 * distribution exactly.
 *
 * Rule (T > 0), p = softmax(z_p / T), q = softmax(z_q / T):
 *   walk from the root; at node c the working distribution is r = p_c; the
 *   children of c are tried in ascending node index: child k with token x is
 *   accepted iff uniforms[b][k] < min(1, r(x) / q_c(x)); a rejection
 *   replaces r by max(0, r - q_c) normalised (unchanged if that has no
 *   mass); an acceptance moves to the child.  When every child was rejected
 *   the emitted token y ~ r; when the accepted node has no children,
 *   y ~ p of that node (the bonus).  y is the inverse-CDF draw of the chain
 *   rule (ascending ids, smallest v with C_v > u*S) on uniforms[b][0].
 * T == 0: a child is accepted iff its token is the argmax of the current
 *   node's target row (ties to the lowest id); y = argmax of the last row.
 *
 * Outputs: out_tokens int32 [B][N]: the accepted nodes' tokens in walk
 * order, then y, then -1; out_path int32 [B][N]: the accepted node indices
 * (the cache entries to keep), then -1; out_num_accepted int32 [B]: their
 * count n, or -1 for a sequence with invalid input (a parent outside
 * [0, i), a token outside [0, V), a non-finite logit in a visited row), whose
 * outputs are then all -1 (error-word bits as in spec_verify.h).
 *
 * Layout: hidden bf16 [B*N][d] (row b*N+i = node i of sequence b), W_lm bf16
 * [V][d], draft_logits and target_logits f32 [B*N][V], tokens / parents /
 * uniforms [B][N].  Sizes: 1 <= N <= 256, V <= 196608, B*N <= 2^24, d % 8
 * == 0.  Ownership, asynchrony, alignment (16 bytes) and the error word
 * (spec_verify_read_error on the workspace) as in spec_verify.h; the
 * workspace needs no initialisation.
 *
 * Execution (T > 0): one thread-block cluster per tree walks it; the
 * library takes clusters of 16, 12 or 8 CTAs, the largest of which all B
 * trees are resident at once.  The environment variable
 * SPEC_TREE_CLUSTER_CTAS = 8, 12 or 16 forces one of these sizes where such
 * a cluster fits (read at every call; the tokens drawn are the same up to
 * the draw band of the summation order).
 */
#ifndef SPEC_TREE_H_
#define SPEC_TREE_H_

#include "spec_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t B; /* sequences */
  int32_t N; /* nodes per tree, root included */
  int32_t d; /* hidden size (ignored by spec_tree_verify_from_logits) */
  int32_t V; /* vocabulary size */
} spec_tree_dims;

/* Workspace bytes (0 if the sizes or T are invalid).  `logits_in_workspace`
 * reserves room for the target logits when the caller keeps none. */
SPEC_API size_t spec_tree_workspace_bytes(spec_tree_dims dims, float temperature, int32_t logits_in_workspace);

/* LM head over every node's hidden state, then the tree walk.
 * out_target_logits (optional, T > 0 only) receives the target logits. */
SPEC_API spec_status spec_tree_verify(const void *hidden, const void *W_lm, const float *draft_logits,
                                      const int32_t *tokens, const int32_t *parents, const float *uniforms,
                                      float temperature, int32_t *out_tokens, int32_t *out_path,
                                      int32_t *out_num_accepted, spec_tree_dims dims, void *workspace,
                                      size_t workspace_bytes, float *out_target_logits, spec_stream_t stream);

/* The tree walk on given target logits. */
SPEC_API spec_status spec_tree_verify_from_logits(const float *target_logits, const float *draft_logits,
                                                  const int32_t *tokens, const int32_t *parents,
                                                  const float *uniforms, float temperature, int32_t *out_tokens,
                                                  int32_t *out_path, int32_t *out_num_accepted, spec_tree_dims dims,
                                                  void *workspace, size_t workspace_bytes, spec_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_TREE_H_ */
