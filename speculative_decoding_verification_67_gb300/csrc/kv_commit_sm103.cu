// KV-cache commit after the verify step ("Speculative Decoding: Memverifikasi
// Token Draft secara Paralel", section "Verifikasi mengubah jalur cache").
// Declared in include/spec_kv_commit.h.
//
// The copy is a plain HBM stream: one warp per (kept entry, layer), every kept
// byte read once and written once in 16-byte vectors, eight loads in flight
// per lane before the stores.  What has to happen first is a plan: which
// entries are kept (an exclusive scan of keep over the sequences) and where
// each one goes (a block-table lookup).
//
// Up to kFusedMaxB sequences, one kernel does both: every CTA scans the
// accept counts into shared memory itself (a few hundred bytes read from L2),
// copies its share, and the last CTA to finish (a grid-wide ticket) advances
// the lengths, which every CTA has read by then.  Above that, a one-CTA plan
// kernel writes the table of kept entries to the workspace and advances the
// lengths, and the copy kernel, launched as its programmatic dependent, reads
// the table.  In-place mode runs the plan alone.
#include <cstdint>

#include "internal.h"
#include "sm103_ptx.cuh"
#include "spec_kv_commit.h"

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kCopyThreads = 256;
constexpr int kCopyWarps = kCopyThreads / 32;
constexpr int kCopyCtasPerSm = 8;
constexpr int kLoadsInFlight = 8;
constexpr int kMaxStaged = 256;
constexpr size_t kCtrlBytes = 256;  // int err, int kept-entry count, unsigned ticket
constexpr int kFusedMaxB = 4096;
constexpr int kFusedCtasPerSm = 4;

struct KvArgs {
  const int32_t* n;
  int32_t* seq_len;
  const int32_t* bt;
  const uint4* staged;  // null in in-place mode
  uint4* pool;
  int B, S, layers, page_size, num_pages, max_pages;
  long long entry_vecs;
  int* ctrl;      // [0] error word, [1] kept entries, [2] ticket of the fused kernel
  int2* table;    // [B*S] (staging row b*S+i, pool row page*page_size+slot)
};

__device__ __forceinline__ int kept(int n, int S) { return n < 0 ? 0 : min(n + 1, S); }

// Error bits of committing `keep` entries at L.. of sequence b (0 = valid).
__device__ int range_error(const KvArgs& a, int b, int L, int keep) {
  if (L < 0) return SPEC_KV_DEVERR_LENGTH;
  if (keep == 0) return 0;
  const long long last = static_cast<long long>(L) + keep - 1;
  if (last / a.page_size >= a.max_pages) return SPEC_KV_DEVERR_CAPACITY;
  for (long long col = L / a.page_size; col <= last / a.page_size; ++col) {
    const int page = a.bt[static_cast<long long>(b) * a.max_pages + col];
    if (page < 0 || page >= a.num_pages) return SPEC_KV_DEVERR_PAGE;
  }
  return 0;
}

// Exclusive block scan of one int per thread (kPlanThreads threads).
__device__ int block_excl_scan(int v, int* warp_tot, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = warp_tot[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, off);
      if (lane >= off) t += y;
    }
    warp_tot[lane] = t;  // inclusive
  }
  __syncthreads();
  total = warp_tot[31];
  const int before = warp == 0 ? 0 : warp_tot[warp - 1];
  __syncthreads();  // warp_tot is reused by the next call
  return before + x - v;
}

__global__ void __launch_bounds__(kPlanThreads) kv_plan_kernel(const KvArgs a) {
  __shared__ int warp_tot[32];
  __shared__ int s_err;
  sv::griddep_launch_dependents();  // the copy kernel may launch; it waits for this grid to finish
  if (threadIdx.x == 0) s_err = 0;
  __syncthreads();
  int base = 0;
  for (int b0 = 0; b0 < a.B; b0 += kPlanThreads) {
    const int b = b0 + threadIdx.x;
    int keep = 0, L = 0, e = 0;
    if (b < a.B) {
      L = a.seq_len[b];
      keep = kept(a.n[b], a.S);
      e = range_error(a, b, L, keep);
      if (e) {
        atomicOr(&s_err, e);
        keep = 0;
      }
    }
    int total;
    const int off = base + block_excl_scan(keep, warp_tot, total);
    if (a.table != nullptr) {
      for (int i = 0; i < keep; ++i) {
        const long long pos = static_cast<long long>(L) + i;
        const int page = a.bt[static_cast<long long>(b) * a.max_pages + pos / a.page_size];
        a.table[off + i] = make_int2(b * a.S + i, static_cast<int>(page * static_cast<long long>(a.page_size) +
                                                                   pos % a.page_size));
      }
    }
    if (b < a.B && !e) a.seq_len[b] = L + keep;
    base += total;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    a.ctrl[0] = s_err;
    a.ctrl[1] = base;
  }
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Copies the kept entry k (all of its entry_vecs vectors) of one layer with
// one warp.
__device__ __forceinline__ void copy_entry(const uint4* src, uint4* dst, long long entry_vecs, int lane) {
  for (long long v0 = 0; v0 < entry_vecs; v0 += 32 * kLoadsInFlight) {
    uint4 r[kLoadsInFlight];
#pragma unroll
    for (int j = 0; j < kLoadsInFlight; ++j) {
      const long long v = v0 + lane + 32 * j;
      if (v < entry_vecs) r[j] = ld_stream(src + v);
    }
#pragma unroll
    for (int j = 0; j < kLoadsInFlight; ++j) {
      const long long v = v0 + lane + 32 * j;
      if (v < entry_vecs) dst[v] = r[j];
    }
  }
}

__global__ void __launch_bounds__(kCopyThreads) kv_copy_kernel(const KvArgs a) {
  sv::griddep_wait();  // the plan kernel's table and count are complete and visible
  const int kt = a.ctrl[1];
  const long long units = static_cast<long long>(kt) * a.layers;
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * kCopyWarps;
  const long long plane_src = static_cast<long long>(a.B) * a.S;
  const long long plane_dst = static_cast<long long>(a.num_pages) * a.page_size;
  for (long long u = static_cast<long long>(blockIdx.x) * kCopyWarps + (threadIdx.x >> 5); u < units; u += warps) {
    const int k = static_cast<int>(u % kt);
    const long long layer = u / kt;
    const int2 t = a.table[k];
    copy_entry(a.staged + (layer * plane_src + t.x) * a.entry_vecs, a.pool + (layer * plane_dst + t.y) * a.entry_vecs,
               a.entry_vecs, lane);
  }
}

__global__ void __launch_bounds__(kCopyThreads) kv_commit_fused_kernel(const KvArgs a) {
  __shared__ int s_off[kFusedMaxB + 1];  // exclusive prefix of keep
  __shared__ int s_len[kFusedMaxB];
  __shared__ int warp_tot[kCopyWarps];
  __shared__ int s_err, s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) s_err = 0;
  __syncthreads();
  for (int b = threadIdx.x; b < a.B; b += kCopyThreads) {
    const int L = a.seq_len[b];
    int keep = kept(a.n[b], a.S);
    const int e = range_error(a, b, L, keep);
    if (e) {
      atomicOr(&s_err, e);
      keep = 0;
    }
    s_len[b] = L;
    s_off[b] = keep;
  }
  __syncthreads();
  // exclusive scan of s_off[0..B) in chunks of kCopyThreads
  int carry = 0;
  for (int b0 = 0; b0 < a.B; b0 += kCopyThreads) {
    const int b = b0 + threadIdx.x;
    const int v = b < a.B ? s_off[b] : 0;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    int before = carry, total = carry;
    for (int w = 0; w < kCopyWarps; ++w) {
      if (w < warp) before += warp_tot[w];
      total += warp_tot[w];
    }
    if (b < a.B) s_off[b] = before + x - v;
    carry = total;
    __syncthreads();
  }
  if (threadIdx.x == 0) s_off[a.B] = carry;
  __syncthreads();
  const int kt = carry;

  const long long units = static_cast<long long>(kt) * a.layers;
  const long long warps = static_cast<long long>(gridDim.x) * kCopyWarps;
  const long long plane_src = static_cast<long long>(a.B) * a.S;
  const long long plane_dst = static_cast<long long>(a.num_pages) * a.page_size;
  for (long long u = static_cast<long long>(blockIdx.x) * kCopyWarps + warp; u < units; u += warps) {
    const int k = static_cast<int>(u % kt);
    const long long layer = u / kt;
    int lo = 0, hi = a.B;  // the sequence b with s_off[b] <= k < s_off[b+1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_off[mid] <= k) lo = mid; else hi = mid;
    }
    const int b = lo, i = k - s_off[b];
    const long long pos = static_cast<long long>(s_len[b]) + i;
    const int page = a.bt[static_cast<long long>(b) * a.max_pages + pos / a.page_size];
    const uint4* src = a.staged + (layer * plane_src + static_cast<long long>(b) * a.S + i) * a.entry_vecs;
    uint4* dst = a.pool + (layer * plane_dst + static_cast<long long>(page) * a.page_size + pos % a.page_size) *
                              a.entry_vecs;
    copy_entry(src, dst, a.entry_vecs, lane);
  }

  // the last CTA to finish advances the lengths (every CTA has read them)
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(reinterpret_cast<unsigned*>(a.ctrl + 2), 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  for (int b = threadIdx.x; b < a.B; b += kCopyThreads) a.seq_len[b] = s_len[b] + (s_off[b + 1] - s_off[b]);
  if (threadIdx.x == 0) {
    a.ctrl[0] = s_err;
    a.ctrl[1] = kt;
    a.ctrl[2] = 0;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool dims_ok(const spec_kv_dims& d) {
  if (d.B < 1 || d.B > 65535 || d.S < 1 || d.S > kMaxStaged || d.layers < 1 || d.layers > 65535 ||
      d.page_size < 1 || d.num_pages < 1 || d.max_pages < 1 || d.entry_bytes < 16 || d.entry_bytes % 16 != 0)
    return false;
  const double pool_bytes = static_cast<double>(d.layers) * d.num_pages * d.page_size * d.entry_bytes;
  const double staged_bytes = static_cast<double>(d.layers) * d.B * d.S * d.entry_bytes;
  if (pool_bytes > 9.0e18 || staged_bytes > 9.0e18) return false;
  if (static_cast<double>(d.max_pages) * d.page_size >= 2147483647.0) return false;   // positions fit int32
  if (static_cast<double>(d.num_pages) * d.page_size >= 2147483647.0) return false;   // pool rows fit int32
  return true;
}

size_t workspace_bytes(const spec_kv_dims& d) {
  return kCtrlBytes + (sizeof(int2) * static_cast<size_t>(d.B) * d.S + 255) / 256 * 256;
}

}  // namespace

extern "C" {

size_t spec_kv_commit_workspace_bytes(spec_kv_dims dims) { return dims_ok(dims) ? workspace_bytes(dims) : 0; }

spec_status spec_kv_commit(const int32_t* num_accepted, int32_t* seq_len, const int32_t* block_table,
                           const void* staged, void* pool, spec_kv_dims dims, void* workspace,
                           size_t workspace_bytes_given, spec_stream_t stream) {
  if (!num_accepted || !seq_len || !block_table || !workspace) return SPEC_ERR_ARG;
  if (staged && !pool) return SPEC_ERR_ARG;
  if (!dims_ok(dims)) return SPEC_ERR_DIMS;
  if (!aligned16(workspace) || (staged && !aligned16(staged)) || (pool && !aligned16(pool)) ||
      (reinterpret_cast<uintptr_t>(num_accepted) & 3u) || (reinterpret_cast<uintptr_t>(seq_len) & 3u) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u))
    return SPEC_ERR_ALIGN;
  if (workspace_bytes_given < workspace_bytes(dims)) return SPEC_ERR_WORKSPACE;
  sv::DeviceInfo dev;
  const int st = sv::current_device(dev);
  if (st != SPEC_OK) return static_cast<spec_status>(st);

  KvArgs a;
  a.n = num_accepted;
  a.seq_len = seq_len;
  a.bt = block_table;
  a.staged = static_cast<const uint4*>(staged);
  a.pool = static_cast<uint4*>(pool);
  a.B = dims.B;
  a.S = dims.S;
  a.layers = dims.layers;
  a.page_size = dims.page_size;
  a.num_pages = dims.num_pages;
  a.max_pages = dims.max_pages;
  a.entry_vecs = dims.entry_bytes / 16;
  a.ctrl = static_cast<int*>(workspace);
  a.table = staged ? reinterpret_cast<int2*>(static_cast<char*>(workspace) + kCtrlBytes) : nullptr;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const long long max_units = static_cast<long long>(dims.B) * dims.S * dims.layers;
  const long long want = (max_units + kCopyWarps - 1) / kCopyWarps;
  const long long cap = static_cast<long long>(dev.sm_count) * kCopyCtasPerSm;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  if (staged && dims.B <= kFusedMaxB) {
    // one wave: the fused kernel keeps four CTAs per SM (64 registers a thread)
    const long long fcap = static_cast<long long>(dev.sm_count) * kFusedCtasPerSm;
    const unsigned fgrid = static_cast<unsigned>(want < fcap ? want : fcap);
    kv_commit_fused_kernel<<<fgrid, kCopyThreads, 0, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
  }
  kv_plan_kernel<<<1, kPlanThreads, 0, s>>>(a);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  if (staged && sv::launch_dependent(kv_copy_kernel, dim3(grid), dim3(kCopyThreads), s, a) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

spec_status spec_kv_commit_read_error(void* workspace, int32_t* error_word, spec_stream_t stream) {
  if (!workspace || !error_word) return SPEC_ERR_ARG;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemcpy(error_word, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

}  // extern "C"
