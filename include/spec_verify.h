/*
 * spec_verify.h -- C ABI of the target-side verify-and-accept step of
 * speculative decoding on one GB300 GPU (sm_103a).
 *
 * The step (pages: quochung.cyou A.I article on speculative decoding,
 * sections "Một vòng speculative decoding", "Modified rejection sampling"
 * and its sub-sections "Giải pháp", "Khi reject thì lấy token từ đâu?",
 * "Toàn bộ thuật toán cho một token", "Áp dụng thuật toán";
 * "Speculative Decoding: Memverifikasi Token Draft secara Paralel",
 * sections "Sampling eksak memerlukan aturan koreksi" and "Penolakan
 * memotong prefix yang diterima"; "57 Speculative Decoding", section
 * "Идея и механизм" with its acceptance, residual and exactness equations):
 *
 *   z_p[b,j,:] = h[b,j,:] . W_lm                      (LM head, j = 0..K)
 *   p_j = softmax(z_p[b,j] / T),  q_j = softmax(z_q[b,j] / T)
 *   draft x_j accepted iff u[b][j] < min(1, p_j(x_j) / q_j(x_j)), left to
 *   right; n_b = number of leading accepts
 *   n_b < K: y ~ max(0, p_{n_b} - q_{n_b}) normalised (the correction)
 *   n_b = K: y ~ p_K (the bonus token)
 *   y is drawn by inverse CDF over ascending token ids on u[b][K]:
 *   y = smallest v with C_v > u*S, C_v = sum_{t<=v} r_t, S = sum_t r_t.
 *   T == 0 is greedy: x_j accepted iff it is the argmax of row j (ties to
 *   the lowest id), y = argmax of row n_b.
 *
 * Conventions for every entry point below
 *   - Pointers named "device" are device memory of the current CUDA device,
 *     owned by the caller, and must stay valid until the work enqueued on
 *     `stream` has finished.  Nothing is allocated by the library; scratch
 *     space is the caller's `workspace`.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) with no host synchronisation, except where stated.
 *   - Layouts are dense row-major with no padding:
 *       hidden        bf16  [B*(K+1)][d]   row b*(K+1)+j = position j of seq b
 *       W_lm          bf16  [V][d]         (d x V column-major, the nn.Linear
 *                                           weight layout)
 *       target_logits f32   [B*(K+1)][V]
 *       draft_logits  f32   [B*K][V]       row b*K+j = draft slot j of seq b
 *       draft_tokens  int32 [B][K]
 *       uniforms      f32   [B][K+1]       u[b][0..K-1] accept tests,
 *                                           u[b][K] the correction/bonus draw
 *       out_tokens    int32 [B][K+1]       accepted drafts, then y, then -1
 *       out_num_accepted int32 [B]         n_b, or -1 if the sequence's
 *                                           inputs were invalid on the device
 *   - Alignment: every device pointer 16-byte aligned; d % 8 == 0 for the
 *     LM head (rows of hidden and W_lm must start on 16-byte boundaries).
 *   - Sizes: B >= 1, 0 <= K <= 32, V >= 1, 8 <= d (LM head); B*(K+1) and
 *     B*K*V etc. must fit the index types (checked).
 *   - Errors detectable on the host are returned synchronously and nothing
 *     is enqueued.  Invalid data found on the device (a draft token outside
 *     [0, V), a non-finite logit) marks the affected sequence
 *     (out_num_accepted[b] = -1, out_tokens[b][:] = -1) and sets a bit of the
 *     workspace's error word; read it with spec_verify_read_error.
 */
#ifndef SPEC_VERIFY_H_
#define SPEC_VERIFY_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SPEC_API __attribute__((visibility("default")))
#else
#define SPEC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle as cudaStream_t (the runtime's stream type is this pointer). */
typedef struct CUstream_st *spec_stream_t;

typedef struct {
  int32_t B; /* sequences */
  int32_t K; /* drafted tokens per sequence (0 = bonus token only) */
  int32_t d; /* hidden size (ignored by the *_from_logits entry points) */
  int32_t V; /* vocabulary size */
} spec_dims;

typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_ARG = 1,          /* null pointer where one is required, bad temperature */
  SPEC_ERR_DIMS = 2,         /* a size out of range */
  SPEC_ERR_ALIGN = 3,        /* pointer or leading dimension misaligned */
  SPEC_ERR_WORKSPACE = 4,    /* workspace NULL or smaller than required */
  SPEC_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed */
  SPEC_ERR_ARCH = 6,         /* current device is not sm_103 (GB300) */
  SPEC_ERR_DEVICE_INPUT = 7, /* returned by spec_verify_read_error only */
  SPEC_ERR_SCRATCH_LIMIT = 8 /* request larger than the fixed scratch of the no-allocation entry point */
} spec_status;

/* Bits of the device error word (spec_verify_read_error). */
#define SPEC_DEVERR_TOKEN_RANGE 0x1 /* a draft token outside [0, V) */
#define SPEC_DEVERR_NONFINITE 0x2   /* a NaN/Inf target or draft logit */
#define SPEC_DEVERR_TIMEOUT 0x4     /* a bounded on-chip wait gave up */

/* Fields of out_debug, float [B][K+1][SPEC_DEBUG_FIELDS], sampling path:
 *   [0] p_j(x_j)   [1] q_j(x_j)   [2] a_j = min(1, p_j(x_j)/q_j(x_j))      (j < K)
 *   [3] log sum_v exp(z_p[b,j,v]/T)                                        (j <= K)
 *   [4] log sum_v exp(z_q[b,j,v]/T)                                        (j < K)
 *   [5] at j = n_b: mass of the row the draw used, sum max(0, p-q) for a
 *       correction, 1 for the bonus; 0 elsewhere
 * greedy path (T == 0): [0] max_v z_p[b,j,v]  [1] its lowest argmax id; rest 0.
 * Entries that do not apply are 0. */
#define SPEC_DEBUG_FIELDS 6

/* Version of this ABI (bumped on any signature or layout change). */
SPEC_API int32_t spec_abi_version(void);

/* Human-readable name of a status. Never NULL. */
SPEC_API const char *spec_status_string(spec_status status);

/*
 * Bytes of device workspace that spec_verify needs for `dims` at
 * `temperature` (T == 0 selects the greedy layout).  When
 * `logits_in_workspace` is non-zero the target logits (f32 [B*(K+1)][V]) are
 * kept in the workspace; pass 0 when the caller supplies out_target_logits.
 * Returns 0 for invalid dims.
 */
SPEC_API size_t spec_verify_workspace_bytes(spec_dims dims, float temperature, int32_t logits_in_workspace);

/*
 * The whole step from hidden states (LM head, then verify-and-accept).
 *
 * hidden, W_lm          device bf16, layouts above.
 * draft_logits          device f32 [B*K][V]; may be NULL iff temperature == 0.
 * draft_tokens          device int32 [B][K] (may be NULL iff K == 0).
 * uniforms              device f32 [B][K+1] in [0,1); ignored (may be NULL)
 *                       iff temperature == 0.
 * temperature           T >= 0 and finite; 0 selects greedy.
 * out_tokens, out_num_accepted   device int32 outputs.
 * workspace             device scratch of at least
 *                       spec_verify_workspace_bytes(dims, T, out_target_logits == NULL);
 *                       its contents need no initialisation and are
 *                       overwritten.  Two calls must not share a workspace
 *                       while both are in flight.
 * out_target_logits     optional device f32 [B*(K+1)][V]: receives z_p
 *                       (T > 0 only; must be NULL when T == 0, where the
 *                       greedy path never materialises the logits).
 * out_debug             optional device f32 [B][K+1][SPEC_DEBUG_FIELDS].
 *
 * Dense part: the LM head is a bf16 x bf16 -> f32 contraction on the
 * tensor cores (tcgen05, TMEM accumulators, TMA-fed), streaming W_lm once.
 * Decision arithmetic (no f64 anywhere): exp(z/T) is evaluated as 2^(z*c)
 * with c = log2(e)/T held as a pair of f32 values; every row normaliser and
 * every residual mass or prefix sum is a float-float (paired f32, TwoSum)
 * sum of terms scaled against an integer power-of-two reference, so the
 * scaling is exact and the sums carry no systematic error above ~1e-12
 * (each token's own term keeps the f32 rounding of one exponent and one
 * exp2f); the ratio S_p/S_q used by the residual is a float-float quotient.
 */
SPEC_API spec_status spec_verify(const void *hidden, const void *W_lm, const float *draft_logits,
                        const int32_t *draft_tokens, const float *uniforms, float temperature,
                        int32_t *out_tokens, int32_t *out_num_accepted, spec_dims dims,
                        void *workspace, size_t workspace_bytes, float *out_target_logits,
                        float *out_debug, spec_stream_t stream);

/*
 * spec_verify with per-stage timing: identical arguments and work, plus
 * `stage_events`, an array of 3 cudaEvent_t handles (created by the caller)
 * recorded on `stream` before the LM-head kernel, between the LM head (with
 * its fused softmax statistics) and the finishing kernel, and after it.  The events sit
 * between the launches, so the finishing kernel no longer overlaps the
 * head's tail; use it to attribute time, not to measure the step.
 */
SPEC_API spec_status spec_verify_timed(const void *hidden, const void *W_lm, const float *draft_logits,
                                       const int32_t *draft_tokens, const float *uniforms, float temperature,
                                       int32_t *out_tokens, int32_t *out_num_accepted, spec_dims dims,
                                       void *workspace, size_t workspace_bytes, float *out_target_logits,
                                       float *out_debug, spec_stream_t stream, void *const *stage_events);

/*
 * The verify-and-accept part alone, on given target logits
 * (device f32 [B*(K+1)][V]); same arguments and rules as spec_verify
 * otherwise.  dims.d is ignored.  Workspace: at least
 * spec_verify_from_logits_workspace_bytes(dims, T) bytes (with no LM head
 * there is no stream-K area and one partial per 4096-token chunk, so this is
 * at most spec_verify_workspace_bytes(dims, T, 0), which also suffices).
 */
SPEC_API size_t spec_verify_from_logits_workspace_bytes(spec_dims dims, float temperature);

SPEC_API spec_status spec_verify_from_logits(const float *target_logits, const float *draft_logits,
                                    const int32_t *draft_tokens, const float *uniforms,
                                    float temperature, int32_t *out_tokens,
                                    int32_t *out_num_accepted, spec_dims dims, void *workspace,
                                    size_t workspace_bytes, float *out_debug,
                                    spec_stream_t stream);

/*
 * spec_verify_from_logits for callers that cannot allocate device memory.
 * (No counterpart on the pages: this is a deployment variant of the same step.)
 *
 * Some callers have no room to allocate at all while they decode: a serving
 * process that reserved the whole GPU at start-up for its weights and its
 * key-value cache has nothing left for a cudaMalloc, and one that does find
 * memory would stall every stream of the device on the call's implicit
 * synchronisation in the middle of a decoding step.  This entry point takes
 * the same inputs and outputs as spec_verify_from_logits but no workspace:
 * its scratch is a fixed array of SPEC_NOALLOC_SCRATCH_BYTES bytes of device
 * memory inside the library, which every GPU that loads the library holds
 * until the process exits.
 *
 *  - Requests whose workspace, spec_verify_from_logits_workspace_bytes(dims, T),
 *    would exceed SPEC_NOALLOC_SCRATCH_BYTES are refused with
 *    SPEC_ERR_SCRATCH_LIMIT before anything is enqueued (and before any
 *    pointer is looked at); a request of exactly that size is served.
 *  - The first call on a device looks up the array's device address (a
 *    runtime query, once per device, with that device current); make that
 *    first call before capturing any stream on the device.
 *  - Every call on a device shares the one array.  Calls whose work overlaps
 *    on the GPU (different streams, different host threads without ordering)
 *    race on it and corrupt each other's results; order them.  Each call
 *    clears what it needs cleared itself, so stale contents of the last call
 *    do no harm.
 *  - Nothing is allocated: no cudaMalloc, no cudaFree, no allocating library
 *    routine.  Error reporting as in spec_verify_from_logits; the device
 *    error word lives in the shared array and is read with
 *    spec_verify_noalloc_read_error.
 */
#define SPEC_NOALLOC_SCRATCH_BYTES (1u << 20)
SPEC_API spec_status spec_verify_from_logits_noalloc(const float *target_logits, const float *draft_logits,
                                                     const int32_t *draft_tokens, const float *uniforms,
                                                     float temperature, int32_t *out_tokens,
                                                     int32_t *out_num_accepted, spec_dims dims, float *out_debug,
                                                     spec_stream_t stream);

/* Device error word of the no-allocation entry point's last call on the
 * current device (synchronises `stream` first); as spec_verify_read_error. */
SPEC_API spec_status spec_verify_noalloc_read_error(int32_t *error_word, spec_stream_t stream);

/*
 * LM head alone (page "quochung.cyou" section "Hidden state": the final hidden
 * state goes through the LM head to a score for every token):
 * logits[m][v] = sum_k hidden[m][k] * W_lm[v][k], bf16 inputs, f32 accumulate
 * and output.  hidden device bf16 [M][d], W_lm device bf16 [V][d], logits
 * device f32 [M][V].  1 <= M <= 2^24, 8 <= d <= 2^20 with d % 8 == 0.
 * No workspace.
 */
SPEC_API spec_status spec_lm_head(const void *hidden, const void *W_lm, float *logits, int32_t M,
                         int32_t d, int32_t V, spec_stream_t stream);

/*
 * spec_verify with the per-step tensors in HOST memory (pinned host memory
 * lets the copies run asynchronously; pageable memory also works, with
 * synchronous copies).  W_lm stays in device memory (the model's weight).
 * The call copies hidden, draft_logits, draft_tokens and uniforms to the
 * device, runs spec_verify, copies out_tokens and out_num_accepted back and
 * synchronises `stream` before returning, so the host outputs are ready.
 * device_workspace must hold spec_verify_host_workspace_bytes(dims, T) bytes.
 */
SPEC_API size_t spec_verify_host_workspace_bytes(spec_dims dims, float temperature);
SPEC_API spec_status spec_verify_host(const void *hidden_host, const void *W_lm_device,
                             const float *draft_logits_host, const int32_t *draft_tokens_host,
                             const float *uniforms_host, float temperature,
                             int32_t *out_tokens_host, int32_t *out_num_accepted_host,
                             spec_dims dims, void *device_workspace, size_t workspace_bytes,
                             spec_stream_t stream);

/* spec_verify_host without the final synchronisation: the copies and the
 * step are enqueued on `stream` and the call returns.  The host buffers must
 * stay valid and unmodified, and the outputs must not be read, until the
 * work on `stream` has completed (e.g. cudaStreamSynchronize or an event);
 * with pinned host buffers the copies are asynchronous, so a caller can keep
 * several steps in flight on several streams, each with its own workspace
 * and buffers. */
SPEC_API spec_status spec_verify_host_async(const void *hidden_host, const void *W_lm_device,
                                            const float *draft_logits_host, const int32_t *draft_tokens_host,
                                            const float *uniforms_host, float temperature,
                                            int32_t *out_tokens_host, int32_t *out_num_accepted_host,
                                            spec_dims dims, void *device_workspace, size_t workspace_bytes,
                                            spec_stream_t stream);

/*
 * Synchronises `stream`, then reads the device error word of `workspace`
 * (the one used by the last spec_verify / spec_verify_from_logits call) into
 * *error_word (SPEC_DEVERR_* bits).  Returns SPEC_OK when it is 0,
 * SPEC_ERR_DEVICE_INPUT when a bit is set, SPEC_ERR_CUDA on a CUDA failure.
 */
SPEC_API spec_status spec_verify_read_error(const void *workspace, int32_t *error_word,
                                   spec_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H_ */
