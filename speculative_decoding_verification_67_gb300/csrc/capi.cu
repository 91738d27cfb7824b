// C ABI of the verify-and-accept step: argument checks, workspace layout and
// the launch sequence.  Declared in include/spec_verify.h.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "spec_draft.h"
#include "spec_verify.h"

namespace sv {

namespace {
std::mutex g_dev_mu;
DeviceInfo g_dev[64];
}  // namespace

int current_device(DeviceInfo& out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
  if (dev < 0 || dev >= 64) return SPEC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& di = g_dev[dev];
  if (di.device < 0) {
    DeviceInfo t;
    t.device = dev;
    if (cudaDeviceGetAttribute(&t.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&t.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&t.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&t.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return SPEC_ERR_CUDA;
    di = t;
  }
  out = di;
  if (out.cc_major != 10 || out.cc_minor != 3) return SPEC_ERR_ARCH;
  return SPEC_OK;
}

}  // namespace sv

namespace {

using sv::DeviceInfo;

constexpr size_t kAlign = 256;
constexpr int kAbiVersion = 1;
constexpr long long kMaxRows = 1ll << 24;  // rows of the per-row passes (grid.x)

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Workspace layout.  Nothing needs initialising by the caller: the first
// kernel of a call clears the error word, and the kernel producing the
// softmax statistics clears the tickets the finishing kernel counts on.
struct Layout {
  size_t ctrl_bytes = 0;
  size_t fix = 0;                                     // stream-K fixup of the precise LM head (M <= 64)
  size_t tpart = 0, dpart = 0, res = 0, logits = 0;  // sampling
  size_t pmax = 0, pidx = 0;                                   // greedy
  int CA = 0, P = 0;
  size_t total = 0;
};

// int[0] error word, int[1 .. 1+B) tickets of the residual pass.
constexpr int kCtrlErr = 0, kCtrlTickets = 1;

Layout make_layout(int B, int K, int V, bool greedy, bool logits_in_ws, bool from_logits) {
  Layout L;
  const size_t M = static_cast<size_t>(B) * (K + 1);
  const size_t num_vt = (static_cast<size_t>(V) + sv::kHeadTileV - 1) / sv::kHeadTileV;
  size_t off = round_up(sizeof(int) * (kCtrlTickets + static_cast<size_t>(B)));
  L.ctrl_bytes = off;
  L.CA = (V + sv::kChunk - 1) / sv::kChunk;
  const bool precise_head = !from_logits && M <= 64;
  if (precise_head) {
    L.fix = off;
    off += round_up(sv::kFixupBytes);
  }
  if (!greedy) {
    // the LM head writes one partial per CTA (at most kMaxHeadGrid CTAs), the
    // streaming pass over given logits one per 4096-token chunk
    L.tpart = off;
    const size_t parts = from_logits ? static_cast<size_t>(L.CA)
                                     : std::max(static_cast<size_t>(L.CA), static_cast<size_t>(sv::kMaxHeadGrid));
    off += round_up(sizeof(sv::StatPart) * M * parts);
    L.dpart = off;
    off += round_up(sizeof(sv::StatPart) * static_cast<size_t>(B) * K * L.CA);
    L.res = off;
    off += round_up(sizeof(float2) * static_cast<size_t>(B) * L.CA);
    if (logits_in_ws) {
      L.logits = off;
      off += round_up(sizeof(float) * M * static_cast<size_t>(V));
    }
  } else {
    L.P = from_logits ? L.CA : static_cast<int>(num_vt);
    L.pmax = off;
    off += round_up(sizeof(float) * static_cast<size_t>(L.P) * M);
    L.pidx = off;
    off += round_up(sizeof(int) * static_cast<size_t>(L.P) * M);
  }
  L.total = off;
  return L;
}

// Whether the large-batch LM head's two side warps can reduce the draft rows
// within the head's own run.  Measured on GB300 they stream ~0.25 TB/s in all
// (two warps per SM beside the epilogue), and the head lasts about the longer
// of its weight stream (~6.5 TB/s) and its products (~1.3 PFLOP/s): at
// B = 16, K = 4, V = 128256 (33 MB of draft logits) they fit and save the
// pass; at B = 64, K = 8, d = 8192, V = 152064 (311 MB) they outlasted the
// head by ~70 us, against ~55 us for the streaming pass after it.
bool draft_fits_side_warps(int M, int draft_rows, int d, int V) {
  const double draft_bytes = 4.0 * draft_rows * V;
  const double head_ns = std::max(2.0 * V * d / 6500.0, 2.0 * M * static_cast<double>(d) * V / 1.3e6);
  return draft_bytes <= 250.0 * head_ns;
}

bool dims_ok(const spec_dims& d, bool need_head) {
  if (d.B < 1 || d.K < 0 || d.K > sv::kMaxK || d.V < 1) return false;
  const long long M = static_cast<long long>(d.B) * (d.K + 1);
  const long long R = M + static_cast<long long>(d.B) * d.K;
  if (R > kMaxRows) return false;
  if (static_cast<long long>(d.V) * M > (1ll << 40)) return false;
  if (need_head && (d.d < 8 || d.d % 8 != 0 || d.d > (1 << 20))) return false;
  return true;
}

spec_status device_status(DeviceInfo& out) { return static_cast<spec_status>(sv::current_device(out)); }

spec_status check_sampling_inputs(const spec_dims& d, float T, const float* draft_logits,
                                  const int32_t* draft_tokens, const float* uniforms, const int32_t* out_tokens,
                                  const int32_t* out_n, const float* out_debug) {
  if (!(T >= 0.f) || !std::isfinite(T)) return SPEC_ERR_ARG;
  if (!out_tokens || !out_n) return SPEC_ERR_ARG;
  if (d.K > 0 && !draft_tokens) return SPEC_ERR_ARG;
  if (T > 0.f) {
    if (!uniforms) return SPEC_ERR_ARG;
    if (d.K > 0 && !draft_logits) return SPEC_ERR_ARG;
    if (draft_logits && !aligned(draft_logits, 16)) return SPEC_ERR_ALIGN;
    if (!aligned(uniforms, 4)) return SPEC_ERR_ALIGN;
  }
  if ((draft_tokens && !aligned(draft_tokens, 4)) || !aligned(out_tokens, 4) || !aligned(out_n, 4) ||
      (out_debug && !aligned(out_debug, 4)))
    return SPEC_ERR_ALIGN;
  return SPEC_OK;
}

sv::VerifyArgs sampling_args(const Layout& L, const spec_dims& d, float T, const float* zp, const float* zq,
                             const int32_t* x, const float* u, int32_t* out_tokens, int32_t* out_n,
                             float* out_debug, char* ws, int Pt) {
  sv::VerifyArgs a;
  a.B = d.B;
  a.K = d.K;
  a.V = d.V;
  sv::exponent_constant(T, &a.c_hi, &a.c_lo);
  a.zp = zp;
  a.ldp = d.V;
  a.zq = zq;
  a.x = x;
  a.u = u;
  a.out_tokens = out_tokens;
  a.out_n = out_n;
  a.out_debug = out_debug;
  int* ctrl = reinterpret_cast<int*>(ws);
  a.err = ctrl + kCtrlErr;
  a.tickets = reinterpret_cast<unsigned*>(ctrl + kCtrlTickets);
  a.tpart = reinterpret_cast<const sv::StatPart*>(ws + L.tpart);
  a.dpart = reinterpret_cast<const sv::StatPart*>(ws + L.dpart);
  a.Pt = Pt;
  a.Pd = L.CA;
  a.res_sums = reinterpret_cast<float2*>(ws + L.res);
  a.G = 1;
  a.CB = L.CA;
  return a;
}

sv::GreedyArgs greedy_args(const Layout& L, const spec_dims& d, const int32_t* x, int32_t* out_tokens,
                           int32_t* out_n, float* out_debug, char* ws) {
  sv::GreedyArgs g;
  g.B = d.B;
  g.K = d.K;
  g.V = d.V;
  g.P = L.P;
  g.part_max = reinterpret_cast<const float*>(ws + L.pmax);
  g.part_idx = reinterpret_cast<const int*>(ws + L.pidx);
  g.x = x;
  g.out_tokens = out_tokens;
  g.out_n = out_n;
  g.out_debug = out_debug;
  g.err = reinterpret_cast<int*>(ws) + kCtrlErr;
  return g;
}

}  // namespace

extern "C" {

int32_t spec_abi_version(void) { return kAbiVersion; }

const char* spec_status_string(spec_status s) {
  switch (s) {
    case SPEC_OK: return "SPEC_OK";
    case SPEC_ERR_ARG: return "SPEC_ERR_ARG: invalid argument (null pointer or temperature)";
    case SPEC_ERR_DIMS: return "SPEC_ERR_DIMS: size out of range";
    case SPEC_ERR_ALIGN: return "SPEC_ERR_ALIGN: misaligned pointer or hidden size";
    case SPEC_ERR_WORKSPACE: return "SPEC_ERR_WORKSPACE: workspace missing or too small";
    case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA: CUDA call failed";
    case SPEC_ERR_ARCH: return "SPEC_ERR_ARCH: current device is not sm_103 (GB300)";
    case SPEC_ERR_DEVICE_INPUT: return "SPEC_ERR_DEVICE_INPUT: invalid input found on the device";
    case SPEC_ERR_SCRATCH_LIMIT:
      return "SPEC_ERR_SCRATCH_LIMIT: request larger than the no-allocation entry point's fixed scratch";
  }
  return "SPEC_ERR_UNKNOWN";
}

size_t spec_verify_workspace_bytes(spec_dims dims, float temperature, int32_t logits_in_workspace) {
  if (!dims_ok(dims, false) || !(temperature >= 0.f)) return 0;
  return make_layout(dims.B, dims.K, dims.V, temperature == 0.f, logits_in_workspace != 0, false).total;
}

size_t spec_verify_from_logits_workspace_bytes(spec_dims dims, float temperature) {
  if (!dims_ok(dims, false) || !(temperature >= 0.f) || !std::isfinite(temperature)) return 0;
  return make_layout(dims.B, dims.K, dims.V, temperature == 0.f, false, true).total;
}

}  // extern "C"

namespace {

spec_status verify_impl(const void* hidden, const void* W_lm, const float* draft_logits,
                        const int32_t* draft_tokens, const float* uniforms, float temperature,
                        int32_t* out_tokens, int32_t* out_num_accepted, spec_dims dims, void* workspace,
                        size_t workspace_bytes, float* out_target_logits, float* out_debug,
                        spec_stream_t stream, void* const* ev, long long ldz = 0) {
  if (!dims_ok(dims, true)) return SPEC_ERR_DIMS;
  if (!hidden || !W_lm) return SPEC_ERR_ARG;
  if (!aligned(hidden, 16) || !aligned(W_lm, 16)) return SPEC_ERR_ALIGN;
  spec_status st = check_sampling_inputs(dims, temperature, draft_logits, draft_tokens, uniforms, out_tokens,
                                         out_num_accepted, out_debug);
  if (st != SPEC_OK) return st;
  const bool greedy = temperature == 0.f;
  if (greedy && out_target_logits) return SPEC_ERR_ARG;
  if (out_target_logits && !aligned(out_target_logits, 4)) return SPEC_ERR_ALIGN;
  const Layout L = make_layout(dims.B, dims.K, dims.V, greedy, !greedy && !out_target_logits, false);
  if (!workspace || workspace_bytes < L.total) return SPEC_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return SPEC_ERR_ALIGN;
  DeviceInfo dev;
  st = device_status(dev);
  if (st != SPEC_OK) return st;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const int M = dims.B * (dims.K + 1);
  int* err = reinterpret_cast<int*>(ws) + kCtrlErr;
  bool enc_fail = false;
  cudaError_t e;
  auto mark = [&](int i) -> bool {
    return !ev || cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev[i]), s) == cudaSuccess;
  };
  if (!mark(0)) return SPEC_ERR_CUDA;
  if (greedy) {
    e = sv::launch_head(hidden, W_lm, M, dims.d, dims.V, sv::HeadOut::kArgmax, nullptr,
                        reinterpret_cast<float*>(ws + L.pmax), reinterpret_cast<int*>(ws + L.pidx), nullptr, err,
                        true, dev, s, &enc_fail, 0, L.fix ? ws + L.fix : nullptr);
    if (enc_fail || e != cudaSuccess || !mark(1)) return SPEC_ERR_CUDA;
    const sv::GreedyArgs g = greedy_args(L, dims, draft_tokens, out_tokens, out_num_accepted, out_debug, ws);
    e = sv::launch_greedy_finish(g, s);
    return (e == cudaSuccess && mark(2)) ? SPEC_OK : SPEC_ERR_CUDA;
  }
  float* logits = out_target_logits ? out_target_logits : reinterpret_cast<float*>(ws + L.logits);
  if (!out_target_logits || ldz <= 0) ldz = dims.V;
  const sv::HeadPlan plan = sv::plan_head(M, dims.d, dims.V, sv::HeadOut::kStats, dev, L.fix != 0);
  sv::HeadStats hs;
  sv::exponent_constant(temperature, &hs.c_hi, &hs.c_lo);
  hs.tpart = reinterpret_cast<sv::StatPart*>(ws + L.tpart);
  hs.zq = draft_logits;
  const bool draft_in_head = !plan.large || draft_fits_side_warps(M, dims.B * dims.K, dims.d, dims.V);
  hs.draft_rows = draft_in_head ? dims.B * dims.K : 0;
  hs.dpart = reinterpret_cast<sv::StatPart*>(ws + L.dpart);
  hs.tickets = reinterpret_cast<unsigned*>(reinterpret_cast<int*>(ws) + kCtrlTickets);
  hs.n_tickets = dims.B;
  // The LM head's epilogue produces the target statistics as it writes the
  // logits (one partial per CTA and row), and its side warps reduce the draft
  // rows meanwhile, unless they would outlast the head: then a streaming pass
  // after it reduces them (keeping the head's error word).
  e = sv::launch_head(hidden, W_lm, M, dims.d, dims.V, sv::HeadOut::kStats, logits, nullptr, nullptr, &hs, err,
                      true, dev, s, &enc_fail, ldz, L.fix ? ws + L.fix : nullptr);
  if (enc_fail || e != cudaSuccess) return SPEC_ERR_CUDA;
  if (!draft_in_head && dims.K > 0) {
    e = sv::launch_row_stats(draft_logits, draft_logits, 0, dims.B * dims.K, dims.V, hs.c_hi, hs.c_lo, nullptr,
                             hs.dpart, err, nullptr, 0, s, 0, false);
    if (e != cudaSuccess) return SPEC_ERR_CUDA;
  }
  if (!mark(1)) return SPEC_ERR_CUDA;
  sv::VerifyArgs a = sampling_args(L, dims, temperature, logits, draft_logits, draft_tokens, uniforms,
                                   out_tokens, out_num_accepted, out_debug, ws, plan.target_parts);
  a.ldp = ldz;
  e = sv::launch_verify_sampling(a, s);
  return (e == cudaSuccess && mark(2)) ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace

extern "C" {

spec_status spec_verify(const void* hidden, const void* W_lm, const float* draft_logits,
                        const int32_t* draft_tokens, const float* uniforms, float temperature,
                        int32_t* out_tokens, int32_t* out_num_accepted, spec_dims dims, void* workspace,
                        size_t workspace_bytes, float* out_target_logits, float* out_debug,
                        spec_stream_t stream) {
  return verify_impl(hidden, W_lm, draft_logits, draft_tokens, uniforms, temperature, out_tokens,
                     out_num_accepted, dims, workspace, workspace_bytes, out_target_logits, out_debug, stream,
                     nullptr);
}

spec_status spec_verify_timed(const void* hidden, const void* W_lm, const float* draft_logits,
                              const int32_t* draft_tokens, const float* uniforms, float temperature,
                              int32_t* out_tokens, int32_t* out_num_accepted, spec_dims dims, void* workspace,
                              size_t workspace_bytes, float* out_target_logits, float* out_debug,
                              spec_stream_t stream, void* const* stage_events) {
  if (!stage_events || !stage_events[0] || !stage_events[1] || !stage_events[2]) return SPEC_ERR_ARG;
  return verify_impl(hidden, W_lm, draft_logits, draft_tokens, uniforms, temperature, out_tokens,
                     out_num_accepted, dims, workspace, workspace_bytes, out_target_logits, out_debug, stream,
                     stage_events);
}

spec_status spec_verify_from_logits(const float* target_logits, const float* draft_logits,
                                    const int32_t* draft_tokens, const float* uniforms, float temperature,
                                    int32_t* out_tokens, int32_t* out_num_accepted, spec_dims dims,
                                    void* workspace, size_t workspace_bytes, float* out_debug,
                                    spec_stream_t stream) {
  if (!dims_ok(dims, false)) return SPEC_ERR_DIMS;
  if (!target_logits) return SPEC_ERR_ARG;
  if (!aligned(target_logits, 16)) return SPEC_ERR_ALIGN;
  spec_status st = check_sampling_inputs(dims, temperature, draft_logits, draft_tokens, uniforms, out_tokens,
                                         out_num_accepted, out_debug);
  if (st != SPEC_OK) return st;
  const bool greedy = temperature == 0.f;
  const Layout L = make_layout(dims.B, dims.K, dims.V, greedy, false, true);
  if (!workspace || workspace_bytes < L.total) return SPEC_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return SPEC_ERR_ALIGN;
  DeviceInfo dev;
  st = device_status(dev);
  if (st != SPEC_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int* err = reinterpret_cast<int*>(ws) + kCtrlErr;
  const int M = dims.B * (dims.K + 1);
  cudaError_t e;
  if (greedy) {
    e = sv::launch_row_argmax(target_logits, M, dims.V, reinterpret_cast<float*>(ws + L.pmax),
                              reinterpret_cast<int*>(ws + L.pidx), err, s);
    if (e != cudaSuccess) return SPEC_ERR_CUDA;
    const sv::GreedyArgs g = greedy_args(L, dims, draft_tokens, out_tokens, out_num_accepted, out_debug, ws);
    e = sv::launch_greedy_finish(g, s);
    return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
  }
  float c_hi, c_lo;
  sv::exponent_constant(temperature, &c_hi, &c_lo);
  e = sv::launch_row_stats(target_logits, draft_logits, M, dims.B * dims.K, dims.V, c_hi, c_lo,
                           reinterpret_cast<sv::StatPart*>(ws + L.tpart), reinterpret_cast<sv::StatPart*>(ws + L.dpart),
                           err, reinterpret_cast<unsigned*>(reinterpret_cast<int*>(ws) + kCtrlTickets), dims.B, s);
  if (e != cudaSuccess) return SPEC_ERR_CUDA;
  const sv::VerifyArgs a = sampling_args(L, dims, temperature, target_logits, draft_logits, draft_tokens, uniforms,
                                         out_tokens, out_num_accepted, out_debug, ws, L.CA);
  e = sv::launch_verify_sampling(a, s);
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------- no allocation
// Scratch of spec_verify_from_logits_noalloc: one fixed array per device,
// shared by every call on that device (see the header).
static __device__ __align__(256) unsigned char g_noalloc_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {nullptr};

// Device address of the scratch array on the current device; looked up once
// per device (host code cannot use the symbol's name as an address).
spec_status noalloc_scratch(const DeviceInfo& dev, char** out) {
  if (dev.device < 0 || dev.device >= static_cast<int>(sizeof(g_noalloc_ptr) / sizeof(g_noalloc_ptr[0])))
    return SPEC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev.device]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return SPEC_ERR_CUDA;
    g_noalloc_ptr[dev.device] = ptr;
  }
  *out = static_cast<char*>(g_noalloc_ptr[dev.device]);
  return SPEC_OK;
}

}  // namespace

extern "C" {

spec_status spec_verify_from_logits_noalloc(const float* target_logits, const float* draft_logits,
                                            const int32_t* draft_tokens, const float* uniforms, float temperature,
                                            int32_t* out_tokens, int32_t* out_num_accepted, spec_dims dims,
                                            float* out_debug, spec_stream_t stream) {
  if (!dims_ok(dims, false)) return SPEC_ERR_DIMS;
  if (!(temperature >= 0.f) || !std::isfinite(temperature)) return SPEC_ERR_ARG;
  // the same rule the header states: the exact from-logits workspace size
  if (spec_verify_from_logits_workspace_bytes(dims, temperature) > SPEC_NOALLOC_SCRATCH_BYTES)
    return SPEC_ERR_SCRATCH_LIMIT;
  DeviceInfo dev;
  spec_status st = device_status(dev);
  if (st != SPEC_OK) return st;
  char* scratch = nullptr;
  st = noalloc_scratch(dev, &scratch);
  if (st != SPEC_OK) return st;
  return spec_verify_from_logits(target_logits, draft_logits, draft_tokens, uniforms, temperature, out_tokens,
                                 out_num_accepted, dims, scratch, SPEC_NOALLOC_SCRATCH_BYTES, out_debug, stream);
}

spec_status spec_verify_noalloc_read_error(int32_t* error_word, spec_stream_t stream) {
  if (!error_word) return SPEC_ERR_ARG;
  DeviceInfo dev;
  spec_status st = device_status(dev);
  if (st != SPEC_OK) return st;
  char* scratch = nullptr;
  st = noalloc_scratch(dev, &scratch);
  if (st != SPEC_OK) return st;
  return spec_verify_read_error(scratch, error_word, stream);
}

// One draft step = the verify path with no drafts: the LM head on the B
// draft rows (fused softmax statistics), then the bonus draw from row 0 of
// each sequence (or the greedy argmax).  The accept counts it also produces
// (always 0, or -1 for a row with non-finite logits) go to the end of the
// workspace.
size_t spec_draft_step_workspace_bytes(spec_dims dims, float temperature) {
  dims.K = 0;
  if (!dims_ok(dims, true) || !(temperature >= 0.f) || !std::isfinite(temperature)) return 0;
  const Layout L = make_layout(dims.B, 0, dims.V, temperature == 0.f, temperature > 0.f, false);
  return L.total + round_up(sizeof(int32_t) * static_cast<size_t>(dims.B));
}

spec_status spec_draft_step(const void* hidden, const void* W_lm, const float* uniforms, float temperature,
                            int32_t* out_tokens, float* out_logits, int64_t ld, spec_dims dims, void* workspace,
                            size_t workspace_bytes, spec_stream_t stream) {
  dims.K = 0;
  if (!dims_ok(dims, true)) return SPEC_ERR_DIMS;
  if (!(temperature >= 0.f) || !std::isfinite(temperature)) return SPEC_ERR_ARG;
  const bool greedy = temperature == 0.f;
  if (greedy && out_logits) return SPEC_ERR_ARG;
  if (out_logits && ld < dims.V) return SPEC_ERR_ARG;
  const Layout L = make_layout(dims.B, 0, dims.V, greedy, !greedy && !out_logits, false);
  const size_t need = L.total + round_up(sizeof(int32_t) * static_cast<size_t>(dims.B));
  if (!workspace || workspace_bytes < need) return SPEC_ERR_WORKSPACE;
  int32_t* n_scratch = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + L.total);
  return verify_impl(hidden, W_lm, nullptr, nullptr, uniforms, temperature, out_tokens, n_scratch, dims, workspace,
                     L.total, out_logits, nullptr, stream, nullptr, out_logits ? ld : 0);
}

spec_status spec_lm_head(const void* hidden, const void* W_lm, float* logits, int32_t M, int32_t d, int32_t V,
                         spec_stream_t stream) {
  if (M < 1 || M > kMaxRows || V < 1 || d < 8 || d % 8 != 0 || d > (1 << 20)) return SPEC_ERR_DIMS;
  if (!hidden || !W_lm || !logits) return SPEC_ERR_ARG;
  if (!aligned(hidden, 16) || !aligned(W_lm, 16) || !aligned(logits, 16)) return SPEC_ERR_ALIGN;
  DeviceInfo dev;
  spec_status st = device_status(dev);
  if (st != SPEC_OK) return st;
  bool enc_fail = false;
  const cudaError_t e = sv::launch_head(hidden, W_lm, M, d, V, sv::HeadOut::kLogits, logits, nullptr, nullptr,
                                        nullptr, nullptr, false, dev, reinterpret_cast<cudaStream_t>(stream),
                                        &enc_fail);
  if (enc_fail || e != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

// Host-buffer variant: staging areas follow the regular workspace.
namespace {
struct HostStage {
  size_t base = 0, hidden = 0, dl = 0, tok = 0, u = 0, out_tok = 0, out_n = 0, total = 0;
};
HostStage host_stage(const spec_dims& d, float T) {
  HostStage h;
  const bool greedy = T == 0.f;
  const size_t M = static_cast<size_t>(d.B) * (d.K + 1);
  size_t off = make_layout(d.B, d.K, d.V, greedy, !greedy, false).total;
  h.base = off;
  h.hidden = off;
  off += round_up(M * static_cast<size_t>(d.d) * 2);
  h.dl = off;
  if (!greedy) off += round_up(static_cast<size_t>(d.B) * d.K * static_cast<size_t>(d.V) * 4);
  h.tok = off;
  off += round_up(static_cast<size_t>(d.B) * d.K * 4 + 4);
  h.u = off;
  if (!greedy) off += round_up(M * 4);
  h.out_tok = off;
  off += round_up(M * 4);
  h.out_n = off;
  off += round_up(static_cast<size_t>(d.B) * 4);
  h.total = off;
  return h;
}
}  // namespace

size_t spec_verify_host_workspace_bytes(spec_dims dims, float temperature) {
  if (!dims_ok(dims, true) || !(temperature >= 0.f)) return 0;
  return host_stage(dims, temperature).total;
}

spec_status spec_verify_host_async(const void* hidden_host, const void* W_lm_device, const float* draft_logits_host,
                                   const int32_t* draft_tokens_host, const float* uniforms_host, float temperature,
                                   int32_t* out_tokens_host, int32_t* out_num_accepted_host, spec_dims dims,
                                   void* device_workspace, size_t workspace_bytes, spec_stream_t stream) {
  if (!dims_ok(dims, true)) return SPEC_ERR_DIMS;
  if (!hidden_host || !W_lm_device || !out_tokens_host || !out_num_accepted_host) return SPEC_ERR_ARG;
  if (!(temperature >= 0.f) || !std::isfinite(temperature)) return SPEC_ERR_ARG;
  const bool greedy = temperature == 0.f;
  if (dims.K > 0 && !draft_tokens_host) return SPEC_ERR_ARG;
  if (!greedy && (!uniforms_host || (dims.K > 0 && !draft_logits_host))) return SPEC_ERR_ARG;
  const HostStage h = host_stage(dims, temperature);
  if (!device_workspace || workspace_bytes < h.total) return SPEC_ERR_WORKSPACE;
  if (!aligned(device_workspace, 16)) return SPEC_ERR_ALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(device_workspace);
  const size_t M = static_cast<size_t>(dims.B) * (dims.K + 1);
  const size_t nx = static_cast<size_t>(dims.B) * dims.K;
  if (cudaMemcpyAsync(ws + h.hidden, hidden_host, M * dims.d * 2, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return SPEC_ERR_CUDA;
  if (nx > 0 && cudaMemcpyAsync(ws + h.tok, draft_tokens_host, nx * 4, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return SPEC_ERR_CUDA;
  if (!greedy) {
    if (nx > 0 && cudaMemcpyAsync(ws + h.dl, draft_logits_host, nx * static_cast<size_t>(dims.V) * 4,
                                  cudaMemcpyHostToDevice, s) != cudaSuccess)
      return SPEC_ERR_CUDA;
    if (cudaMemcpyAsync(ws + h.u, uniforms_host, M * 4, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return SPEC_ERR_CUDA;
  }
  spec_status st = spec_verify(ws + h.hidden, W_lm_device, greedy ? nullptr : reinterpret_cast<float*>(ws + h.dl),
                               nx > 0 ? reinterpret_cast<int32_t*>(ws + h.tok) : nullptr,
                               greedy ? nullptr : reinterpret_cast<float*>(ws + h.u), temperature,
                               reinterpret_cast<int32_t*>(ws + h.out_tok), reinterpret_cast<int32_t*>(ws + h.out_n),
                               dims, ws, h.base, nullptr, nullptr, stream);
  if (st != SPEC_OK) return st;
  if (cudaMemcpyAsync(out_tokens_host, ws + h.out_tok, M * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemcpyAsync(out_num_accepted_host, ws + h.out_n, static_cast<size_t>(dims.B) * 4,
                      cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

spec_status spec_verify_host(const void* hidden_host, const void* W_lm_device, const float* draft_logits_host,
                             const int32_t* draft_tokens_host, const float* uniforms_host, float temperature,
                             int32_t* out_tokens_host, int32_t* out_num_accepted_host, spec_dims dims,
                             void* device_workspace, size_t workspace_bytes, spec_stream_t stream) {
  const spec_status st = spec_verify_host_async(hidden_host, W_lm_device, draft_logits_host, draft_tokens_host,
                                                uniforms_host, temperature, out_tokens_host, out_num_accepted_host,
                                                dims, device_workspace, workspace_bytes, stream);
  if (st != SPEC_OK) return st;
  return cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status spec_verify_read_error(const void* workspace, int32_t* error_word, spec_stream_t stream) {
  if (!workspace || !error_word) return SPEC_ERR_ARG;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return SPEC_ERR_CUDA;
  if (cudaMemcpy(error_word, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return *error_word == 0 ? SPEC_OK : SPEC_ERR_DEVICE_INPUT;
}

}  // extern "C"
