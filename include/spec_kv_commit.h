/*
 * spec_kv_commit.h -- C ABI of the KV-cache commit that follows the verify
 * step (sm_103a).
 *
 * Pages: "Speculative Decoding: Memverifikasi Token Draft secara Paralel",
 * section "Verifikasi mengubah jalur cache" (the target pass computes cache
 * state for every candidate position before the survivors are known; the
 * entries of the discarded suffix must not become committed state; a
 * separate draft model's cache must be advanced consistently with the
 * accepted prefix and the correction; truncation, staged writes or index
 * management are all acceptable), with the prefix rule of "Penolakan
 * memotong prefix yang diterima".
 *
 * Reading.  One round's pass consumed, per sequence, the pending token and
 * then the drafts, at positions L .. L+S-1 (L = committed length before the
 * round): S = K+1 entries for the target model, S = K for a separate draft
 * model (its last draft was never fed back).  With n drafts accepted
 * (out_num_accepted of spec_verify) the first
 *
 *     keep = min(n + 1, S)      (0 when n < 0, a sequence the verify step
 *                                flagged as invalid)
 *
 * entries are the committed ones; the rest are dropped.  The correction or
 * bonus token has no entry: it is the next round's pending token.
 *
 * Layout (all dense, row-major, entries of entry_bytes bytes):
 *   pool        [layers][num_pages][page_size][entry_bytes]   device, in/out
 *   staged      [layers][B][S][entry_bytes]                   device, or NULL
 *   block_table int32 [B][max_pages]: page of positions
 *               p*page_size .. (p+1)*page_size-1 of sequence b  device
 *   seq_len     int32 [B]: committed length, advanced by keep     device, in/out
 *   num_accepted int32 [B]                                       device
 *
 * Staged mode (staged != NULL): entry i of sequence b, every layer, is
 * copied to position L_b + i (page block_table[b][(L_b+i)/page_size], slot
 * (L_b+i) % page_size) for i < keep_b, and seq_len[b] becomes L_b + keep_b.
 * In-place mode (staged == NULL): the pass already wrote its entries at
 * their positions; only seq_len advances (index-based truncation of the
 * rejected suffix, nothing is copied).
 *
 * A sequence whose committed range needs a block-table column >= max_pages
 * or a page id outside [0, num_pages), or whose seq_len is negative, is left
 * untouched (no copy, no length change) and sets a bit of the error word.
 *
 * Ownership and asynchrony as in spec_verify.h: caller-owned device memory,
 * work enqueued on `stream`, nothing allocated.  `workspace` holds
 * spec_kv_commit_workspace_bytes(dims) bytes of device memory (the error
 * word, a completion ticket and the table of kept entries).  Zero it once
 * before its first use: every call leaves the ticket at zero again.  Calls
 * that share a workspace must not run concurrently (the same stream is
 * fine).  The error word is rewritten by every call.
 * Alignment: pool, staged and workspace 16-byte aligned, entry_bytes % 16 ==
 * 0.  Sizes: 1 <= B <= 65535, 1 <= S <= 256, 1 <= layers <= 65535,
 * page_size, num_pages, max_pages >= 1; max_pages * page_size < 2^31; pool
 * and staged byte sizes must fit in 63 bits.
 */
#ifndef SPEC_KV_COMMIT_H_
#define SPEC_KV_COMMIT_H_

#include "spec_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

/* error-word bits */
#define SPEC_KV_DEVERR_CAPACITY 1 /* committed range past the block table */
#define SPEC_KV_DEVERR_PAGE 2     /* block-table entry outside the pool */
#define SPEC_KV_DEVERR_LENGTH 4   /* negative seq_len */

typedef struct {
  int32_t B;           /* sequences */
  int32_t S;           /* staged entries per sequence (K+1 target, K draft) */
  int32_t layers;      /* layers (pool and staged planes) */
  int32_t page_size;   /* positions per page */
  int32_t num_pages;   /* pages per layer plane of the pool */
  int32_t max_pages;   /* block-table columns */
  int64_t entry_bytes; /* bytes of one (layer, position) entry */
} spec_kv_dims;

/* Workspace bytes for `dims` (0 if the sizes are invalid). */
SPEC_API size_t spec_kv_commit_workspace_bytes(spec_kv_dims dims);

/* Commit one round (see above).  Returns SPEC_ERR_ARG for a null required
 * pointer, SPEC_ERR_DIMS for sizes outside the ranges above,
 * SPEC_ERR_ALIGN for misalignment, SPEC_ERR_WORKSPACE for a workspace
 * smaller than spec_kv_commit_workspace_bytes(dims), SPEC_ERR_CUDA for a
 * launch failure. */
SPEC_API spec_status spec_kv_commit(const int32_t *num_accepted, int32_t *seq_len, const int32_t *block_table,
                                    const void *staged, void *pool, spec_kv_dims dims, void *workspace,
                                    size_t workspace_bytes, spec_stream_t stream);

/* Synchronises `stream` and copies the error word of the latest call on
 * this workspace (SPEC_KV_DEVERR_* bits, 0 = every sequence committed) to
 * *error_word. */
SPEC_API spec_status spec_kv_commit_read_error(void *workspace, int32_t *error_word, spec_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_KV_COMMIT_H_ */
