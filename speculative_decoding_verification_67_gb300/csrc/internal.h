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
  kArgmax = 1,   // per (row, vocab tile) max and lowest argmax: [M][num_vt]
};

constexpr int kHeadTileV = 128;   // vocabulary rows per tile (MMA M)
constexpr int kHeadTileK = 64;    // hidden elements per pipeline stage (128-byte rows)

struct HeadPlan {
  bool precise = false; // per-hidden-block TMEM slots summed in registers (N = 32 or 64)
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
constexpr int kChunk = 4096;      // vocabulary tokens per CTA of the per-row passes
constexpr int kMaxK = 32;

// Per (row, chunk) softmax normaliser of z/T: sum over the chunk of
// 2^(z*log2(e)/T - k), k the chunk's integer reference, as a float pair.
struct ChunkStat {
  float k;      // integer-valued reference exponent (base 2)
  int bad;      // a non-finite logit was seen
  float s_hi, s_lo;
};

// Per-sequence state handed from the decision to the residual pass.
struct SeqState {
  int n;          // accepted drafts
  int bad;        // invalid input: skip
  float k_p;      // reference exponent of target row n
  float k_q;      // reference exponent of draft row n (n < K)
  float2 S_p;     // normaliser of target row n against k_p (float pair)
  float2 S_q;     // same for the draft row (n < K)
  float2 kappa;   // S_p / S_q (float pair)
};

struct VerifyArgs {
  int B, K, V;
  float c_hi, c_lo;         // log2(e) / T as a float pair
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
  ChunkStat* stats;         // [R][CA], R = B*(K+1) + B*K
  SeqState* seq;            // [B]
  float2* res_sums;         // [B][CB]
  int CA, CB;
};

// log2(e) / T split into a float pair.
void exponent_constant(float temperature, float* c_hi, float* c_lo);

cudaError_t launch_verify_sampling(const VerifyArgs& a, cudaStream_t stream);

struct GreedyArgs {
  int B, K, V;
  int P;                    // partitions of the vocabulary (partials per row)
  const float* part_max;    // [M][P]
  const int* part_idx;      // [M][P]  (-2 marks a non-finite logit)
  const int32_t* x;         // [B][K]
  int32_t* out_tokens;
  int32_t* out_n;
  float* out_debug;
  int* err;
};

cudaError_t launch_greedy_finish(const GreedyArgs& a, cudaStream_t stream);

// Row argmax partials from given logits ([M][V] -> [M][P], P = ceil(V / kChunk)).
cudaError_t launch_row_argmax(const float* logits, int M, int V, float* part_max, int* part_idx,
                              cudaStream_t stream);

}  // namespace sv
