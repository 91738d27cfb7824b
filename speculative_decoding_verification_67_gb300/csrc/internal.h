// Internal interfaces between the C-ABI layer (capi.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace sv {

// Per-device facts the launches depend on.
struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  int max_smem_optin = 0;
};

// Device error word bits (mirror SPEC_DEVERR_* of the public header).
constexpr int kErrTokenRange = 0x1;
constexpr int kErrNonFinite = 0x2;
constexpr int kErrTimeout = 0x4;

// ------------------------------------------------------------------ LM head
// Output modes of the LM-head epilogue.
enum class HeadOut : int {
  kLogits = 0,   // f32 logits [M][V]
  kArgmax = 1,   // per (vocab tile, row) max and lowest argmax: [num_vt][M]
};

constexpr int kHeadTileV = 128;   // vocabulary rows per tile (MMA M)
constexpr int kHeadTileK = 64;    // hidden elements per pipeline stage (128-byte rows)

struct HeadPlan {
  int N = 0;            // positions per tile (MMA N), multiple of 16, <= 256
  int num_chunks = 0;   // position chunks, ceil(M / N)
  int num_vt = 0;       // vocabulary tiles, ceil(V / 128)
  int num_tiles = 0;    // num_vt * num_chunks
  int num_kb = 0;       // ceil(d / 64)
  int stages = 0;       // shared-memory pipeline depth
  uint32_t tmem_cols = 0;
  size_t smem_bytes = 0;
  int grid = 0;
};

HeadPlan plan_head(int M, int d, int V, const DeviceInfo& dev);

// Enqueues the LM head.  Returns cudaSuccess or the first CUDA error;
// *encode_failed is set when building a TMA descriptor failed.
cudaError_t launch_head(const void* hidden, const void* W, int M, int d, int V, HeadOut mode,
                        float* logits, float* part_max, int* part_idx, int* err,
                        const DeviceInfo& dev, cudaStream_t stream, bool* encode_failed);

// ------------------------------------------------------------------ verify
constexpr int kRowChunk = 8192;   // vocab elements per CTA of the row-statistics pass
constexpr int kResChunk = 4096;   // vocab elements per CTA of the residual pass
constexpr int kMaxK = 32;

// Per (row, chunk) partial of the softmax normaliser of z/T.
struct RowPart {
  float m;      // max of z/T over the chunk
  int bad;      // a non-finite logit was seen
  double s;     // sum exp(z/T - m) over the chunk
};

// Per-sequence state handed from the decision to the residual pass.
struct SeqState {
  int n;          // accepted drafts
  int bad;        // invalid input: skip
  float m_p;      // max of z_p/T on row n
  float m_q;      // max of z_q/T on row n (n < K)
  double S_p;     // sum exp(z_p/T - m_p) on row n
  double S_q;     // same for the draft row (n < K)
  double kappa;   // S_p / S_q
};

struct VerifyArgs {
  int B, K, V;
  float T;
  const float* zp;          // [B*(K+1)][V]
  const float* zq;          // [B*K][V]
  const int32_t* x;         // [B][K]
  const float* u;           // [B][K+1]
  int32_t* out_tokens;      // [B][K+1]
  int32_t* out_n;           // [B]
  float* out_debug;         // [B][K+1][6] or null
  // workspace
  int* err;
  unsigned* tickets_a;      // [B]
  unsigned* tickets_b;      // [B]
  RowPart* parts;           // [R][CA], R = B*(K+1) + B*K
  SeqState* seq;            // [B]
  double* res_sums;         // [B][CB]
  int CA, CB;
};

cudaError_t launch_verify_sampling(const VerifyArgs& a, cudaStream_t stream);

struct GreedyArgs {
  int B, K, V;
  int P;                    // partitions of the vocabulary (partials per row)
  const float* part_max;    // [P][M]
  const int* part_idx;      // [P][M]  (-2 marks a non-finite logit)
  const int32_t* x;         // [B][K]
  int32_t* out_tokens;
  int32_t* out_n;
  float* out_debug;
  int* err;
};

// Scratch the greedy finish needs after the partition partials (bytes, for M rows),
// and its launch; `ticket` must be zero before the launch.
size_t greedy_scratch_bytes(int M);
cudaError_t launch_greedy_finish_ws(const GreedyArgs& a, void* scratch, unsigned* ticket, cudaStream_t stream);

// Row argmax partials from given logits ([M][V] -> [P][M], P = ceil(V / kRowChunk)).
cudaError_t launch_row_argmax(const float* logits, int M, int V, float* part_max, int* part_idx,
                              cudaStream_t stream);

}  // namespace sv
