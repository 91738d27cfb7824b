/*
 * spec_ngram.h -- C ABI of the prompt-lookup (n-gram) drafter (sm_103a).
 *
 * Page: quochung.cyou A.I article on speculative decoding, section "Vấn đề
 * 3: Làm sao khi không muốn train drafter?" (Prompt Lookup Decoding: match
 * the tail of the output being generated against the prompt and earlier
 * output, propose what followed, verify with the target; no drafter
 * weights).  It pairs with the greedy verify step (spec_verify with
 * temperature 0), which accepts a draft only where it equals the target's
 * argmax.
 *
 * Rule, per sequence with history h[0..L) (prompt then output so far):
 *   for n = n_max down to n_min: the key is h[L-n..L); an occurrence is a
 *   start s < L-n with h[s..s+n) equal to the key; the first n with an
 *   occurrence wins and, for it, the smallest s;
 *   drafts[0..count) = h[s+n .. s+n+count), count = min(K, L-s-n);
 *   no occurrence for any n: count = 0;
 *   drafts[count..K) = the last proposed token (h[L-1] when count = 0,
 *   0 when L = 0).
 *
 * Layout: history int32 [B][max_len] (row b holds its lengths[b] tokens,
 * the rest of the row is ignored), lengths int32 [B], out_drafts int32
 * [B][K], out_count int32 [B].  A sequence whose length lies outside
 * [0, max_len] gets out_count = -1 and out_drafts = -1 (which the verify
 * step reports as an invalid sequence) and sets SPEC_NGRAM_DEVERR_LENGTH in
 * the error word.
 *
 * Ownership and asynchrony as in spec_verify.h.  `workspace` holds
 * spec_ngram_workspace_bytes(dims) bytes of device memory; zero it once
 * before its first use (every call leaves it ready for the next).  Calls
 * that share a workspace must not run concurrently (same stream is fine).
 * Sizes: 1 <= B <= 65535, 4 <= max_len <= 2^30 with max_len % 4 == 0 (rows
 * of whole 16-byte words), 1 <= K <= 32, 1 <= n_min <= n_max <= 16.
 * Alignment: history and workspace 16 bytes, the other pointers 4.
 */
#ifndef SPEC_NGRAM_H_
#define SPEC_NGRAM_H_

#include "spec_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

#define SPEC_NGRAM_DEVERR_LENGTH 1
#define SPEC_NGRAM_DEVERR_TIMEOUT 2 /* a staging copy did not complete in time */

typedef struct {
  int32_t B;       /* sequences */
  int32_t max_len; /* history row stride (tokens) */
  int32_t K;       /* drafts per sequence */
  int32_t n_min;   /* shortest key tried */
  int32_t n_max;   /* longest key tried */
} spec_ngram_dims;

/* Workspace bytes for `dims` (0 if the sizes are invalid). */
SPEC_API size_t spec_ngram_workspace_bytes(spec_ngram_dims dims);

/* Propose K drafts per sequence (see above).  Returns SPEC_ERR_ARG for a null
 * pointer, SPEC_ERR_DIMS for sizes outside the ranges above, SPEC_ERR_ALIGN,
 * SPEC_ERR_WORKSPACE for a short workspace, SPEC_ERR_CUDA for a launch
 * failure. */
SPEC_API spec_status spec_ngram_propose(const int32_t *history, const int32_t *lengths, int32_t *out_drafts,
                                        int32_t *out_count, spec_ngram_dims dims, void *workspace,
                                        size_t workspace_bytes, spec_stream_t stream);

/* Synchronises `stream` and copies the error word of the latest call on
 * this workspace (SPEC_NGRAM_DEVERR_* bits) to *error_word. */
SPEC_API spec_status spec_ngram_read_error(void *workspace, int32_t *error_word, spec_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_NGRAM_H_ */
