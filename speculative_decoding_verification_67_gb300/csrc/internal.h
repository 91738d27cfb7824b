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

// The current device's facts (cached per device); SPEC_ERR_ARCH unless it
// is compute capability 10.3.  Returns a spec_status value.
int current_device(DeviceInfo& out);

// Device error word bits (mirror SPEC_DEVERR_* of the public header).
constexpr int kErrTokenRange = 0x1;
constexpr int kErrNonFinite = 0x2;
constexpr int kErrTimeout = 0x4;

// ------------------------------------------------------------------ partials
constexpr int kChunk = 4096;      // vocabulary tokens per unit of the per-row passes
constexpr int kMaxK = 32;

// Stored softmax-normaliser partial of one row over some of its tokens:
// sum of 2^(z*log2(e)/T - k) as a float pair against the integer-valued
// reference k (-inf when no token contributed).
struct StatPart {
  float k;
  float s_hi, s_lo;
  int bad;       // a non-finite logit was seen
};

// ------------------------------------------------------------------ LM head
// Output modes of the LM-head epilogue.
enum class HeadOut : int {
  kLogits = 0,   // f32 logits [M][V]
  kArgmax = 1,   // per (row, vocab tile) max and lowest argmax: [M][num_vt]
  kStats = 2,    // logits, plus softmax partials of every target row and of
                 // the draft rows (the sampling step's statistics)
};

constexpr int kHeadTileV = 128;   // vocabulary rows per tile (MMA M)
constexpr int kHeadTileK = 64;    // hidden elements per pipeline stage (128-byte rows)

struct HeadPlan {
  bool precise = false; // groups of hidden blocks in rotating TMEM slots, summed in registers
  int N = 0;            // positions per tile (MMA N), multiple of 16, <= 256
  int num_chunks = 0;   // position chunks, ceil(M / N)
  int num_vt = 0;       // vocabulary tiles, ceil(V / 128)
  int num_tiles = 0;    // num_vt * num_chunks
  int num_kb = 0;       // ceil(d / 64)
  int kbs = 1;          // hidden blocks per pipeline stage (large-batch kernel: 2 when num_kb is even)
  int stages = 0;       // shared-memory pipeline depth
  uint32_t tmem_cols = 0;
  size_t smem_bytes = 0;
  int grid = 0;
  int target_parts = 0;  // target-row partials per row (one per CTA, small-batch statistics)
  // stream-K schedule (precise scheme with a fixup buffer): every CTA takes an
  // equal contiguous range of the num_tiles * groups (tile, 4-block group) units
  bool streamk = false;
  int groups = 1;        // units per tile
  // the large-batch kernel (above 64 positions, logits or greedy partials):
  // chunks of N <= 256 positions, two N-column TMEM slots of gkb hidden
  // blocks each, summed in registers by eight epilogue warps
  bool large = false;
  // ... on CTA pairs (tcgen05 cta_group::2, 256-row vocabulary tiles)
  bool pair = false;
  int gkb = 4;           // hidden blocks accumulated per TMEM slot (precise schemes)
};

// Upper bound of the LM head's grid (sizes the per-CTA workspace areas).
constexpr int kMaxHeadGrid = 256;
// Fixup area of the stream-K schedule: 128 x 64 floats per CTA, then 4
// 64-bit flags per CTA.
constexpr size_t kFixupFloatsPerCta = 128 * 64;
constexpr size_t kFixupBytes = kMaxHeadGrid * (kFixupFloatsPerCta * 4 + 4 * 8);

HeadPlan plan_head(int M, int d, int V, HeadOut mode, const DeviceInfo& dev, bool streamk = false);

// Sampling-step statistics the LM head produces alongside the logits.
struct HeadStats {
  float c_hi = 0.f, c_lo = 0.f;   // log2(e) / T as a float pair
  StatPart* tpart = nullptr;      // [M][plan.target_parts]
  const float* zq = nullptr;      // draft logits [draft_rows][V]
  int draft_rows = 0;
  StatPart* dpart = nullptr;      // [draft_rows][ceil(V / kChunk)]
  unsigned* tickets = nullptr;    // [n_tickets] zeroed by the kernel
  int n_tickets = 0;
};

// Enqueues the LM head.  Returns cudaSuccess or the first CUDA error;
// *encode_failed is set when building a TMA descriptor failed.  When
// zero_err is set, the kernel clears *err before anything can report.
// `ldz` is the row stride of `logits` in floats (0: V).  `fixup` (kFixupBytes,
// no initialisation needed) enables the stream-K schedule of the precise scheme.
cudaError_t launch_head(const void* hidden, const void* W, int M, int d, int V, HeadOut mode,
                        float* logits, float* part_max, int* part_idx, const HeadStats* stats, int* err,
                        bool zero_err, const DeviceInfo& dev, cudaStream_t stream, bool* encode_failed,
                        long long ldz = 0, void* fixup = nullptr);

// ------------------------------------------------------------------ verify
struct VerifyArgs {
  int B, K, V;
  float c_hi, c_lo;         // log2(e) / T as a float pair
  const float* zp;          // [B*(K+1)] rows of V, row stride ldp
  long long ldp;            // row stride of zp in floats (>= V)
  const float* zq;          // [B*K][V]
  const int32_t* x;         // [B][K]
  const float* u;           // [B][K+1]
  int32_t* out_tokens;      // [B][K+1]
  int32_t* out_n;           // [B]
  float* out_debug;         // [B][K+1][6] or null
  // workspace
  int* err;
  unsigned* tickets;        // [B] (zeroed by the kernel producing the statistics)
  const StatPart* tpart;    // [B*(K+1)][Pt]
  const StatPart* dpart;    // [B*K][Pd]
  int Pt, Pd;
  float2* res_sums;         // [B][CB]
  int CB;
  int G;                    // chunks per CTA of the grid finishing kernel (set at launch)
};

// log2(e) / T split into a float pair.
void exponent_constant(float temperature, float* c_hi, float* c_lo);

// Softmax partials of given target and draft logits (per row and 4096-token
// chunk); clears *err first when err is given and zero_err is set, and the
// n_tickets tickets.  Target row r starts at zp + r * ldp (ldp 0: V).
cudaError_t launch_row_stats(const float* zp, const float* zq, int M, int draft_rows, int V, float c_hi, float c_lo,
                             StatPart* tpart, StatPart* dpart, int* err, unsigned* tickets, int n_tickets,
                             cudaStream_t stream, long long ldp = 0, bool zero_err = true);

// Decision and residual draw (one launch, chained with programmatic
// dependent launch after the statistics).
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

// Row argmax partials from given logits ([M][V] -> [M][P], P = ceil(V / kChunk));
// clears *err first.
cudaError_t launch_row_argmax(const float* logits, int M, int V, float* part_max, int* part_idx, int* err,
                              cudaStream_t stream);

// Launch with programmatic stream serialization: the kernel may start
// while its predecessor on the stream finishes and must begin with
// griddep_wait() before touching the predecessor's outputs.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t stream,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace sv
