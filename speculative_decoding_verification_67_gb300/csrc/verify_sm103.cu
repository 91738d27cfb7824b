// Vocabulary-parallel verify-and-accept kernels (sm_103a, CUDA cores).
//
// Sampling path (T > 0).  The softmax(z/T) normaliser partials of every
// target row and draft row come from the LM-head kernel (its epilogue and
// two side warps) or, on given logits, from row_stats_kernel.  Then one
// launch, chained with programmatic dependent launch: finish_kernel, grid
// (sequences) x (groups of consecutive chunks of 4096 tokens, as few
// chunks per CTA as let the grid be resident at once).  Every CTA of a
// sequence
//
//  1. merges the partials of the sequence's 2K+1 rows into their
//     normalisers (page "quochung.cyou" A.I article, section "Forward pass":
//     the scores form a distribution summing to 100%), gathers p_j(x_j) and
//     q_j(x_j), runs the accept test u_j < min(1, p_j(x_j) / q_j(x_j))
//     (section "Modified rejection sampling / Giải pháp") and takes the
//     accepted prefix with one warp ballot (section "Áp dụng thuật toán":
//     left to right, stop at the first rejection) -- the same arithmetic in
//     every CTA, so the same decision, with no exchange between CTAs;
//  2. reduces its chunks of the row pair at the first rejection n_b to the
//     mass of max(0, p - q) (section "Khi reject thì lấy token từ đâu?"), or
//     of p_K for the bonus token when n_b = K.  The last CTA of the
//     sequence (atomic ticket; no CTA ever waits for another) finds the
//     chunk holding u*S and rescans it with a block-wide prefix scan for the
//     smallest token whose cumulative mass exceeds u*S (inverse CDF,
//     ascending token id).
//
// Rows of at most 32 chunks (V <= 131072) take finish_cluster_kernel
// instead whenever every sequence's cluster is resident at once: one
// cluster per sequence (one chunk per CTA up to 8 chunks, two
// above, so at most 16 CTAs), the chunk masses exchanged through
// distributed shared memory, and the warps owning the drawn chunk scanning
// it from the terms they still hold in registers; the same arithmetic, the
// same tokens.
//
// Arithmetic: see verify_math.cuh (exact power-of-two rescaling of
// partials, float-float sums, exponent map z * log2(e)/T as a float pair);
// nothing here uses f64 (slow on this part).
//
// Greedy path (T = 0): the LM head writes per-(row, vocabulary tile)
// (max, lowest argmax) partials; greedy_finish_kernel reduces them and
// compares the drafts with the argmax left to right (section "Một vòng
// speculative decoding", Bước 3).
#include <algorithm>
#include <atomic>
#include <cfloat>
#include <climits>

#include "internal.h"
#include "sm103_ptx.cuh"
#include "verify_math.cuh"

namespace sv {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPer = kChunk / kThreads;  // 16 tokens per thread
static_assert(kPer == 16, "load16 handles 16 tokens per thread");

// The kThreads threads that hold one chunk: the whole block of finish_kernel,
// one chunk's warps of a finish_cluster_kernel block (chunk h owns warps
// h*kWarps .. h*kWarps+kWarps-1).  Named barrier 1 over them alone, and a
// warp's index among them.
__device__ __forceinline__ void chunk_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }
__device__ __forceinline__ int chunk_warp() { return (threadIdx.x >> 5) % kWarps; }

// ------------------------------------------------------------ block helpers
__device__ __forceinline__ int warp_max_i(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__device__ __forceinline__ int warp_min_i(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

// Exclusive prefix sum (thread order) of a float-float value over one
// chunk's threads, and their total.  sm: kWarps pairs.
__device__ void block_excl_scan_ff(ff v, ff& excl, ff& total, ff* sm) {
  const int lane = threadIdx.x & 31, warp = chunk_warp();
  ff incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    ff o{__shfl_up_sync(0xffffffffu, incl.hi, off), __shfl_up_sync(0xffffffffu, incl.lo, off)};
    if (lane >= off) incl = ff_add(o, incl);
  }
  ff ex{__shfl_up_sync(0xffffffffu, incl.hi, 1), __shfl_up_sync(0xffffffffu, incl.lo, 1)};
  if (lane == 0) ex = {0.f, 0.f};
  if (lane == 31) sm[warp] = incl;
  chunk_sync();
  ff off{0.f, 0.f}, tot{0.f, 0.f};
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    if (w == warp) off = tot;
    tot = ff_add(tot, sm[w]);
  }
  chunk_sync();
  excl = ff_add(off, ex);
  total = tot;
}

// Ticket: true in every thread of the block that arrives last among
// `expected` blocks counted on *counter; earlier blocks' writes made before
// their ticket are visible to it afterwards.
__device__ bool last_block_ticket(unsigned* counter, unsigned expected, int* sm) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned t = atomicAdd(counter, 1u);
    sm[0] = (t == expected - 1u) ? 1 : 0;
  }
  __syncthreads();
  const bool last = sm[0] != 0;
  if (last) __threadfence();
  return last;
}

// 16 consecutive floats of a row (tokens e0 .. e0+15) with bounds; bit i of
// `valid` tells whether token e0+i exists.
template <bool kVec>
__device__ __forceinline__ void load16(const float* __restrict__ row, int e0, int V, float (&z)[kPer],
                                       unsigned& valid) {
  valid = 0;
  if (kVec && e0 + kPer <= V) {
#pragma unroll
    for (int i = 0; i < kPer / 4; ++i) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(row + e0) + i);
      z[4 * i] = f.x;
      z[4 * i + 1] = f.y;
      z[4 * i + 2] = f.z;
      z[4 * i + 3] = f.w;
    }
    valid = 0xffffu;
  } else {
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const bool in = e0 + i < V;
      z[i] = in ? row[e0 + i] : 0.f;
      valid |= in ? (1u << i) : 0u;
    }
  }
}

// ---------------------------------------------------------------- statistics
constexpr int kStatThreads = 128;  // the per-row statistics pass: 4 warps a block, several blocks an SM

// 32 consecutive values per lane of a 1024-token block [base, base + 1024) of
// a row, in eight 128-bit loads per lane (lane l holds tokens base + 4(32j + l)
// .. +3 for j = 0..7, so every load instruction covers 512 contiguous bytes);
// bit t of `valid` tells whether value t exists.
template <bool kVec>
__device__ __forceinline__ void load_block32(const float* __restrict__ z, int base, int V, int lane, float (&v)[32],
                                             unsigned& valid) {
  valid = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int e = base + (j * 32 + lane) * 4;
    if (kVec && e + 3 < V) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(z + e));
      v[4 * j] = f.x;
      v[4 * j + 1] = f.y;
      v[4 * j + 2] = f.z;
      v[4 * j + 3] = f.w;
      valid |= 0xfu << (4 * j);
    } else {
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const bool in = e + t < V;
        v[4 * j + t] = in ? z[e + t] : 0.f;
        valid |= in ? (1u << (4 * j + t)) : 0u;
      }
    }
  }
}

// Folds one lane's 32 values into its running partial: the block reference
// ceil(max z c) raises the partial's (exact power-of-two rescale), then the
// block's terms are added.  Missing and non-finite values
// add nothing; a non-finite one marks the partial.
__device__ __forceinline__ void fold_block32(const float (&v)[32], unsigned valid, Expo c, Partial& lp) {
  if (valid == 0xffffffffu) {
    // Full block: the largest exponent from the largest logit (z -> z c is
    // monotone, c > 0), the terms without per-value masks.  A non-finite
    // value makes the block sum non-finite; only then does the block take
    // the masked path below (same arithmetic otherwise, same result).
    float zm = v[0];
#pragma unroll
    for (int t = 1; t < 32; ++t) zm = fmaxf(zm, v[t]);
    const float hm = expo_hi(zm, c);
    if (isfinite(hm)) {
      const float kn = ceilf(hm);
      const float k = lp.k == -INFINITY ? kn : fmaxf(lp.k, kn);
      float t[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float h = expo_hi(v[i], c);
        t[i] = exp2f((h - k) + expo_lo(v[i], h, c));
      }
#pragma unroll
      for (int w = 16; w > 0; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) t[i] += t[i + w];
      if (isfinite(t[0])) {
        if (lp.k != -INFINITY && kn > lp.k) {
          const float sc = pow2_nonpos(lp.k - kn);
          lp.s = {lp.s.hi * sc, lp.s.lo * sc};
        }
        lp.k = k;
        lp.s = ff_add_f(lp.s, t[0]);
        return;
      }
    }
  }
  float hm = -INFINITY;
  unsigned use = 0;  // bit t: value t exists and z c is finite
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    const float h = expo_hi(v[t], c);
    const bool in = (valid >> t) & 1u;
    const bool fin = isfinite(h);
    lp.bad |= (in && !fin) ? 1 : 0;
    use |= (in && fin) ? (1u << t) : 0u;
    hm = fmaxf(hm, (in && fin) ? h : -INFINITY);
  }
  if (hm == -INFINITY) return;
  const float kn = ceilf(hm);
  if (lp.k == -INFINITY) {
    lp.k = kn;
  } else if (kn > lp.k) {
    const float sc = pow2_nonpos(lp.k - kn);
    lp.s = {lp.s.hi * sc, lp.s.lo * sc};
    lp.k = kn;
  }
  // the 32 terms (each <= 1) summed pairwise (rounding error <= 5 half-ulps
  // of the block sum, below the terms' own exp2f error), then added to the
  // running partial with a compensated add
  float t[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float h = expo_hi(v[i], c);
    const float e = exp2f((h - lp.k) + expo_lo(v[i], h, c));
    t[i] = ((use >> i) & 1u) ? e : 0.f;
  }
#pragma unroll
  for (int w = 16; w > 0; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) t[i] += t[i + w];
  lp.s = ff_add_f(lp.s, t[0]);
}

// Softmax partials of given logits, one per (row, 4096-token chunk) unit;
// rows [0, M) are target rows (stride ldp), the rest draft rows (stride V).
// Each warp takes whole units (warp-strided over the grid) and streams a
// unit in four 1024-token blocks, loading the next block before folding the
// current one, then merges its lanes: no block barrier and no serial merge
// per unit (one unit per block with a block merge reached ~1.7 TB/s).
template <bool kVec>
__global__ void __launch_bounds__(kStatThreads, 3) row_stats_kernel(const float* __restrict__ zp,
                                                             const float* __restrict__ zq, int M, int V,
                                                             long long ldp, Expo c, StatPart* tpart, StatPart* dpart,
                                                             int P, long long units, int* err, unsigned* tickets,
                                                             int n_tickets, int zero_err) {
  const int lane = threadIdx.x & 31;
  if (blockIdx.x == 0) {
    if (zero_err && err && threadIdx.x == 0) *err = 0;
    for (int i = threadIdx.x; i < n_tickets; i += kStatThreads) tickets[i] = 0u;
  }
  constexpr int kStatWarps = kStatThreads / 32;
  const long long nw = static_cast<long long>(gridDim.x) * kStatWarps;
  for (long long u = static_cast<long long>(blockIdx.x) * kStatWarps + (threadIdx.x >> 5); u < units; u += nw) {
    const int row = static_cast<int>(u / P), chunk = static_cast<int>(u % P);
    const float* z = row < M ? zp + static_cast<size_t>(row) * ldp : zq + static_cast<size_t>(row - M) * V;
    const int base = chunk * kChunk;
    Partial lp = partial_empty();
    float cur[32];
    unsigned cv;
    load_block32<kVec>(z, base, V, lane, cur, cv);
#pragma unroll 1
    for (int blk = 0; blk < kChunk / 1024; ++blk) {
      float nxt[32];
      unsigned nv = 0;
      if (blk + 1 < kChunk / 1024) load_block32<kVec>(z, base + (blk + 1) * 1024, V, lane, nxt, nv);
      fold_block32(cur, cv, c, lp);
      if (blk + 1 < kChunk / 1024) {
#pragma unroll
        for (int t = 0; t < 32; ++t) cur[t] = nxt[t];
        cv = nv;
      }
    }
    const Partial wp = warp_merge(lp);
    if (lane == 0) {
      StatPart out;
      out.k = wp.k;
      out.s_hi = wp.s.hi;
      out.s_lo = wp.s.lo;
      out.bad = wp.bad;
      if (row < M)
        tpart[static_cast<size_t>(row) * P + chunk] = out;
      else
        dpart[static_cast<size_t>(row - M) * P + chunk] = out;
    }
  }
}

// The same partials from a bulk-copy stream (V % 4 == 0, 16-byte aligned
// rows): one persistent CTA per SM; lane 0 of warp 0 copies whole
// (row, 4096-token) units -- 16 KB, contiguous -- into a ring of S <= 12
// shared-memory stages with cp.async.bulk.  Two consumer warps own each stage
// s: they fold units s, s + S, s + 2S, ... of the CTA's sequence in order
// (one warp the unit's first two 1024-token blocks, the other the last two,
// merged through shared memory), so neither waits on its stage's barrier more
// than one phase ahead (a parity wait two phases ahead would pass on the older
// phase).  The fold's exp2 chains need many warps to keep the SM busy:
// twelve warps folding whole units ran at ~4.4 TB/s, the stream alone ~7.5.  Each SM keeps up to S units (~190 KB) in flight, which a
// register double buffer (one 4 KB block per warp) cannot; the fold reads
// shared memory four values at a time, so a thread needs few registers.
constexpr int kBulkConsumers = 24;  // two per stage (S <= 12)
constexpr int kBulkThreads = 32 * (1 + kBulkConsumers);
constexpr uint32_t kBulkUnitBytes = kChunk * 4;

// Folds the lane's 32 values of one 1024-token block of a shared-memory stage
// (the same lane layout as load_block32: tokens 4(32j + lane) .. +3) into its
// running partial, reading four values at a time, so that a thread needs few
// registers and sixteen warps per SM fit.  `nv` is the number of the block's
// tokens inside the row (a multiple of 4; <= 0: none).  Same rules as
// fold_block32: a non-finite value adds nothing and marks the partial; the
// terms are summed in four chains of eight.
__device__ __forceinline__ void fold_smem32(const float* blk, int nv, int lane, Expo c, Partial& lp) {
  if (nv >= 1024) {
    float zm = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 f = *reinterpret_cast<const float4*>(blk + (j * 32 + lane) * 4);
      zm = fmaxf(fmaxf(zm, fmaxf(f.x, f.y)), fmaxf(f.z, f.w));
    }
    const float hm = expo_hi(zm, c);
    if (isfinite(hm)) {
      const float kn = ceilf(hm);
      const float k = lp.k == -INFINITY ? kn : fmaxf(lp.k, kn);
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 f = *reinterpret_cast<const float4*>(blk + (j * 32 + lane) * 4);
        a0 += pow2_rel(f.x, c, k);
        a1 += pow2_rel(f.y, c, k);
        a2 += pow2_rel(f.z, c, k);
        a3 += pow2_rel(f.w, c, k);
      }
      const float sum = (a0 + a1) + (a2 + a3);
      if (isfinite(sum)) {
        if (lp.k != -INFINITY && kn > lp.k) {
          const float sc = pow2_nonpos(lp.k - kn);
          lp.s = {lp.s.hi * sc, lp.s.lo * sc};
        }
        lp.k = k;
        lp.s = ff_add_f(lp.s, sum);
        return;
      }
    }
  }
  // a partial block, or one with a non-finite value: the masked form
  float hm = -INFINITY;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int e = (j * 32 + lane) * 4;
    if (e < nv) {
      const float4 f = *reinterpret_cast<const float4*>(blk + e);
      const float v[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float h = expo_hi(v[t], c);
        if (isfinite(h))
          hm = fmaxf(hm, h);
        else
          lp.bad = 1;
      }
    }
  }
  if (hm == -INFINITY) return;
  const float kn = ceilf(hm);
  if (lp.k == -INFINITY) {
    lp.k = kn;
  } else if (kn > lp.k) {
    const float sc = pow2_nonpos(lp.k - kn);
    lp.s = {lp.s.hi * sc, lp.s.lo * sc};
    lp.k = kn;
  }
  float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int e = (j * 32 + lane) * 4;
    if (e < nv) {
      const float4 f = *reinterpret_cast<const float4*>(blk + e);
      const float v[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float h = expo_hi(v[t], c);
        if (isfinite(h)) a[t] += exp2f((h - lp.k) + expo_lo(v[t], h, c));
      }
    }
  }
  lp.s = ff_add_f(lp.s, (a[0] + a[1]) + (a[2] + a[3]));
}

__global__ void __launch_bounds__(kBulkThreads, 1)
    row_stats_bulk_kernel(const float* __restrict__ zp, const float* __restrict__ zq, int M, int V, long long ldp,
                          Expo c, StatPart* tpart, StatPart* dpart, int P, long long units, int* err,
                          unsigned* tickets, int n_tickets, int S, int zero_err) {
  extern __shared__ __align__(16) uint8_t bulk_smem[];
  float* ring = reinterpret_cast<float*>(bulk_smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(bulk_smem + static_cast<size_t>(S) * kBulkUnitBytes);
  uint64_t* empty = full + S;
  float4* handoff = reinterpret_cast<float4*>(empty + S);  // [S] the second half's partial, per stage
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (blockIdx.x == 0) {
    if (zero_err && err && threadIdx.x == 0) *err = 0;
    for (int i = threadIdx.x; i < n_tickets; i += kBulkThreads) tickets[i] = 0u;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 2);
    }
    fence_barrier_init();
  }
  __syncthreads();
  // this CTA's units: u = blockIdx.x + i * gridDim.x
  const long long mine = units > blockIdx.x ? (units - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  auto unit_src = [&](long long u, int& row, int& chunk, int& n) -> const float* {
    row = static_cast<int>(u / P);
    chunk = static_cast<int>(u - static_cast<long long>(row) * P);
    n = min(kChunk, V - chunk * kChunk);
    const float* z = row < M ? zp + static_cast<size_t>(row) * ldp : zq + static_cast<size_t>(row - M) * V;
    return z + static_cast<size_t>(chunk) * kChunk;
  };
  if (warp == 0) {
    if (lane == 0) {
      long long issued = 0;
      for (long long i = 0; i < mine; ++i) {
        const int s = static_cast<int>(i % S);
        const uint32_t ph = static_cast<uint32_t>((i / S) & 1);
        if (!mbar_wait(&empty[s], ph ^ 1u)) {
          if (err) atomicOr(err, kErrTimeout);
          break;
        }
        int row, chunk, n;
        const float* src = unit_src(blockIdx.x + i * gridDim.x, row, chunk, n);
        const uint32_t bytes = static_cast<uint32_t>(n) * 4u;
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_load(ring + static_cast<size_t>(s) * kChunk, src, bytes, &full[s]);
        ++issued;
      }
      // the copies in flight land before the CTA may exit
      for (long long i = issued > S ? issued - S : 0; i < issued; ++i)
        if (!mbar_wait(&full[i % S], static_cast<uint32_t>((i / S) & 1))) {
          if (err) atomicOr(err, kErrTimeout);
          break;
        }
    }
  } else if ((warp - 1) / 2 < S) {
    const int st = (warp - 1) / 2;  // this warp's stage
    const int half = (warp - 1) & 1;  // 0: blocks 0-1 of a unit, 1: blocks 2-3
    for (long long i = st; i < mine; i += S) {
      // both warps of the pair take the wait's outcome together (a barrier
      // with an AND reduction that both always reach), so that neither can
      // be left at the pair's barriers below by the other's timeout
      const uint32_t got = mbar_wait(&full[st], static_cast<uint32_t>((i / S) & 1)) ? 1u : 0u;
      uint32_t both;
      asm volatile(
          "{\n\t.reg .pred pin, pout;\n\t"
          "setp.ne.u32 pin, %1, 0;\n\t"
          "bar.red.and.pred pout, %2, 64, pin;\n\t"
          "selp.u32 %0, 1, 0, pout;\n\t}\n"
          : "=r"(both)
          : "r"(got), "r"(1 + st)
          : "memory");
      if (!both) {
        if (lane == 0 && err) atomicOr(err, kErrTimeout);
        break;
      }
      int row, chunk, n;
      unit_src(blockIdx.x + i * gridDim.x, row, chunk, n);
      const float* stage = ring + static_cast<size_t>(st) * kChunk;
      Partial lp = partial_empty();
#pragma unroll 1
      for (int blk = 2 * half; blk < 2 * half + 2; ++blk)
        fold_smem32(stage + blk * 1024, n - blk * 1024, lane, c, lp);
      const Partial wp = warp_merge(lp);
      // the pair meets on a named barrier of its own (1 + stage): the second
      // half's partial goes through shared memory to the first
      if (half == 1 && lane == 0) handoff[st] = make_float4(wp.k, wp.s.hi, wp.s.lo, __int_as_float(wp.bad));
      asm volatile("bar.sync %0, 64;" ::"r"(1 + st) : "memory");
      if (half == 0 && lane == 0) {
        const float4 o = handoff[st];
        Partial other;
        other.k = o.x;
        other.s = {o.y, o.z};
        other.bad = __float_as_int(o.w);
        const Partial m = partial_merge(wp, other);
        StatPart out;
        out.k = m.k;
        out.s_hi = m.s.hi;
        out.s_lo = m.s.lo;
        out.bad = m.bad;
        if (row < M)
          tpart[static_cast<size_t>(row) * P + chunk] = out;
        else
          dpart[static_cast<size_t>(row - M) * P + chunk] = out;
      }
      // both warps' reads of the stage and of the hand-off are done
      asm volatile("bar.sync %0, 64;" ::"r"(1 + st) : "memory");
      if (lane == 0) mbar_arrive(&empty[st]);
    }
  }
}

// ---------------------------------------------------------------- decision
// The decision of one sequence, computed by every CTA of that sequence with
// identical arithmetic (so identically): merge the softmax partials of its
// 2K+1 rows, run the accept tests left to right, take the accepted prefix.
struct Decision {
  int n, bad, badtok, rowbad;
  float k_p, k_q;
  ff S_p, S_q, kappa;
};

struct DecideSmem {
  float rk[2 * kMaxK + 1];
  ff rS[2 * kMaxK + 1];
  int rbad[2 * kMaxK + 1];
  int xj[kMaxK];
  float zqx[kMaxK];
  float zpx[kMaxK];
  float uj[kMaxK + 1];
  float pj[kMaxK], qj[kMaxK], aj[kMaxK];
  Decision d;
};

// Loads the sequence's inputs that no preceding kernel writes (drafts,
// uniforms, draft logits at the drafts); may run before griddep_wait.
__device__ void load_inputs(const VerifyArgs& a, int b, DecideSmem& ds) {
  const int lane = threadIdx.x & 31;
  if (threadIdx.x >= 32) return;
  const int K = a.K;
  if (lane < K) {
    const int x = a.x[b * K + lane];
    const bool ok = x >= 0 && x < a.V;
    ds.xj[lane] = x;
    ds.zqx[lane] = ok ? a.zq[static_cast<size_t>(b * K + lane) * a.V + x] : 0.f;
  }
  for (int j = lane; j <= K; j += 32) ds.uj[j] = a.u[b * (K + 1) + j];
}

// Merge the partials of every row of sequence b (one warp per row over all
// the block's warps, two passes: the row's largest reference, then the
// exact-scaled compensated sum), then warp 0 decides.  Ends with a
// __syncthreads.
__device__ void decide(const VerifyArgs& a, int b, DecideSmem& ds) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = static_cast<int>(blockDim.x >> 5);
  const int K = a.K;
  const int nrows = 2 * K + 1;
  // the target logit at each draft, issued now so its latency overlaps the merge
  float zpx = 0.f;
  if (warp == nw - 1 && lane < K) {
    const int xj = ds.xj[lane];
    if (xj >= 0 && xj < a.V) zpx = __ldcg(&a.zp[static_cast<size_t>(b * (K + 1) + lane) * a.ldp + xj]);
  }
  for (int r = warp; r < nrows; r += nw) {
    const StatPart* pp = r <= K ? a.tpart + static_cast<size_t>(b * (K + 1) + r) * a.Pt
                                : a.dpart + static_cast<size_t>(b * K + (r - K - 1)) * a.Pd;
    const int np = r <= K ? a.Pt : a.Pd;
    // batches of kBatch partials per lane, all loads issued before use; a
    // row of up to 32*kBatch partials stays in registers for both passes
    constexpr int kBatch = 8;
    float4 w[kBatch];
    float kmax = -INFINITY;
    int bad = 0;
    for (int i0 = 0; i0 < np; i0 += 32 * kBatch) {
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = i0 + j * 32 + lane;
        w[j] = i < np ? __ldcg(reinterpret_cast<const float4*>(pp + i)) : make_float4(-INFINITY, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (w[j].y != 0.f || w[j].z != 0.f) kmax = fmaxf(kmax, w[j].x);
        bad |= __float_as_int(w[j].w);
      }
    }
    kmax = warp_max_f(kmax);
    bad = __any_sync(0xffffffffu, bad != 0) ? 1 : 0;
    float sh = 0.f, sl = 0.f;
    if (kmax != -INFINITY) {
      for (int i0 = 0; i0 < np; i0 += 32 * kBatch) {
        if (np > 32 * kBatch) {  // more than one batch: reload (L2-resident)
#pragma unroll
          for (int j = 0; j < kBatch; ++j) {
            const int i = i0 + j * 32 + lane;
            w[j] = i < np ? __ldcg(reinterpret_cast<const float4*>(pp + i)) : make_float4(-INFINITY, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          if (w[j].y != 0.f || w[j].z != 0.f) {
            const float sc = pow2_int(w[j].x - kmax);
            ff_accumulate(sh, sl, w[j].y * sc);
            ff_accumulate(sh, sl, w[j].z * sc);
          }
        }
      }
    }
    const ff s = warp_sum_ff(ff_norm(sh, sl));
    if (lane == 0) {
      ds.rk[r] = kmax;
      ds.rS[r] = s;
      ds.rbad[r] = bad || !(s.hi > 0.f) || !isfinite(s.hi) || !isfinite(kmax);
    }
  }
  if (warp == nw - 1 && lane < K) ds.zpx[lane] = zpx;
  __syncthreads();
  if (warp == 0) {
    const Expo c{a.c_hi, a.c_lo};
    bool tok_ok = true, acc = false;
    float pj = 0.f, qj = 0.f, aj = 0.f;
    if (lane < K) {
      const int xj = ds.xj[lane];
      tok_ok = xj >= 0 && xj < a.V;
      if (tok_ok) {
        const float zp = ds.zpx[lane];
        const float zq = ds.zqx[lane];
        const float hp = expo_hi(zp, c), hq = expo_hi(zq, c);
        const float lp = (hp - ds.rk[lane]) + expo_lo(zp, hp, c);          // log2 of S_p * p(x)
        const float lq = (hq - ds.rk[K + 1 + lane]) + expo_lo(zq, hq, c);  // log2 of S_q * q(x)
        const float Sp = ds.rS[lane].hi, Sq = ds.rS[K + 1 + lane].hi;
        pj = exp2f(lp) / Sp;
        qj = exp2f(lq) / Sq;
        aj = fminf(1.f, exp2f(lp - lq) * (Sq / Sp));
        acc = ds.uj[lane] < aj;
      }
      ds.pj[lane] = pj;
      ds.qj[lane] = qj;
      ds.aj[lane] = aj;
    }
    const unsigned acc_mask = __ballot_sync(0xffffffffu, acc);
    const unsigned badtok = __ballot_sync(0xffffffffu, lane < K && !tok_ok);
    int rowbad = 0;
    for (int r = lane; r < nrows; r += 32) rowbad |= ds.rbad[r];
    rowbad = __any_sync(0xffffffffu, rowbad != 0) ? 1 : 0;
    int n = (acc_mask == 0xffffffffu) ? 32 : (__ffs(~acc_mask) - 1);
    n = min(n, K);
    if (lane == 0) {
      Decision d;
      d.n = n;
      d.badtok = badtok != 0u;
      d.rowbad = rowbad;
      d.bad = d.badtok || d.rowbad;
      d.k_p = ds.rk[n];
      d.S_p = ds.rS[n];
      if (n < K) {
        d.k_q = ds.rk[K + 1 + n];
        d.S_q = ds.rS[K + 1 + n];
        d.kappa = ff_div(ds.rS[n], ds.rS[K + 1 + n]);
      } else {
        d.k_q = 0.f;
        d.S_q = {0.f, 0.f};
        d.kappa = {0.f, 0.f};
      }
      ds.d = d;
    }
  }
  __syncthreads();
}

// The accepted prefix, the -1 padding after the drawn token, the accept
// count and the debug fields 0-4 (written once per sequence, by the CTA of
// chunk 0).
__device__ void write_prefix(const VerifyArgs& a, int b, const DecideSmem& ds) {
  const int lane = threadIdx.x & 31;
  if (threadIdx.x >= 32) return;
  const int K = a.K;
  const Decision& d = ds.d;
  for (int j = lane; j <= K; j += 32) {
    const bool slot = j < K;
    // position n belongs to the drawn token, written by the sequence's last
    // CTA (only an invalid sequence gets -1 there)
    if (d.bad || j != d.n) a.out_tokens[b * (K + 1) + j] = (!d.bad && j < d.n) ? ds.xj[j] : -1;
    if (a.out_debug) {
      float* dbg = a.out_debug + static_cast<size_t>(b * (K + 1) + j) * 6;
      dbg[0] = slot ? ds.pj[j] : 0.f;
      dbg[1] = slot ? ds.qj[j] : 0.f;
      dbg[2] = slot ? ds.aj[j] : 0.f;
      // log sum_v exp(z_v / T) = ln 2 * (k + log2 S)
      dbg[3] = 0.6931471805599453f * (ds.rk[j] + log2f(ds.rS[j].hi));
      dbg[4] = slot ? 0.6931471805599453f * (ds.rk[K + 1 + j] + log2f(ds.rS[K + 1 + j].hi)) : 0.f;
      if (d.bad || j != d.n) dbg[5] = 0.f;  // field 5 at n: the last CTA's residual mass
    }
  }
  if (lane == 0) {
    a.out_n[b] = d.bad ? -1 : d.n;
    if (d.bad) atomicOr(a.err, (d.badtok ? kErrTokenRange : 0) | (d.rowbad ? kErrNonFinite : 0));
  }
}

// ---------------------------------------------------------------- residual
struct ResRow {
  const float* zp;
  const float* zq;
  Expo c;
  float k_p, k_q, kh, kl;
  int V;
  bool rej;
};

// S_p * max(0, p - q) = max(0, e_p - kappa * e_q) for one token, kappa =
// S_p / S_q as a float pair; for the bonus row (no rejection) S_p * p = e_p.
__device__ __forceinline__ float residual_term(float zp, float zq, const ResRow& R) {
  const float ep = pow2_rel(zp, R.c, R.k_p);
  if (!R.rej) return ep;
  const float eq = pow2_rel(zq, R.c, R.k_q);
  return fmaxf(0.f, ep - fmaf(R.kh, eq, R.kl * eq));
}

// The row pair's 16 logits of tokens e0 .. e0+15 (the draft row only at a
// rejection), and their residual terms.
template <bool kVec>
__device__ __forceinline__ void load_pair(const ResRow& R, int e0, float (&zp)[kPer], float (&zq)[kPer],
                                          unsigned& valid) {
  unsigned vq;
  load16<kVec>(R.zp, e0, R.V, zp, valid);
  if (R.rej) {
    load16<kVec>(R.zq, e0, R.V, zq, vq);
  } else {
#pragma unroll
    for (int i = 0; i < kPer; ++i) zq[i] = 0.f;
  }
}

__device__ __forceinline__ void pair_terms(const ResRow& R, const float (&zp)[kPer], const float (&zq)[kPer],
                                           unsigned valid, float (&r)[kPer]) {
#pragma unroll
  for (int i = 0; i < kPer; ++i) r[i] = ((valid >> i) & 1u) ? residual_term(zp[i], zq[i], R) : 0.f;
}

template <bool kVec>
__device__ __forceinline__ void residual_segment(const ResRow& R, int e0, float (&r)[kPer]) {
  float zp[kPer], zq[kPer];
  unsigned valid;
  load_pair<kVec>(R, e0, zp, zq, valid);
  pair_terms(R, zp, zq, valid, r);
}

__device__ __forceinline__ float segment_total(const float (&r)[kPer]) {
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kPer; ++i) s += r[i];
  return s;
}

// The smallest token of `chunk` whose cumulative mass base + (prefix through
// it) exceeds t, or INT_MAX; and the chunk's last token with positive mass
// (or -1) for the rounding fallback.
__device__ void locate_from_terms(const float (&r)[kPer], int e0, ff base, ff t, int& y, int& last_pos, ff* sm_ff,
                                  int* sm_i) {
  const int lane = threadIdx.x & 31, warp = chunk_warp();
  ff excl, total;
  block_excl_scan_ff({segment_total(r), 0.f}, excl, total, sm_ff);
  const ff tb = ff_add(base, excl);
  int found = INT_MAX, lastp = -1;
  float run = 0.f;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    run += r[i];
    if (found == INT_MAX && ff_gt(ff_add_f(tb, run), t)) found = e0 + i;
    if (r[i] > 0.f) lastp = e0 + i;
  }
  found = warp_min_i(found);
  lastp = warp_max_i(lastp);
  if (lane == 0) {
    sm_i[warp] = found;
    sm_i[kWarps + warp] = lastp;
  }
  chunk_sync();
  y = sm_i[0];
  last_pos = sm_i[kWarps];
  for (int w = 1; w < kWarps; ++w) {
    y = min(y, sm_i[w]);
    last_pos = max(last_pos, sm_i[kWarps + w]);
  }
  chunk_sync();
}

template <bool kVec>
__device__ void locate_in_chunk(const ResRow& R, int chunk, ff base, ff t, int& y, int& last_pos, ff* sm_ff,
                                int* sm_i) {
  const int e0 = chunk * kChunk + threadIdx.x * kPer;
  float r[kPer];
  residual_segment<kVec>(R, e0, r);
  locate_from_terms(r, e0, base, t, y, last_pos, sm_ff, sm_i);
}

// grid (sequences) x (groups of a.G consecutive chunks of 4096 tokens, G
// sized at launch so that the grid fits the SMs at once): the decision
// (redundantly per CTA), the residual mass of the row pair at the first
// rejection (or of the bonus row) per chunk, and, in the last CTA of the
// sequence, the inverse-CDF draw.
template <bool kVec>
__global__ void __launch_bounds__(kThreads) finish_kernel(const VerifyArgs a) {
  __shared__ DecideSmem ds;
  __shared__ ff sm_ff[kWarps];
  __shared__ ff sm_w[2][kWarps];  // per-chunk warp masses, alternating buffers
  __shared__ int sm_i[2 * kWarps];
  __shared__ ff s_base, s_t, s_S;
  __shared__ int s_chunk;
  const int b = blockIdx.x, grp = blockIdx.y;
  const int c0 = grp * a.G, c1 = min(a.CB, c0 + a.G);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  load_inputs(a, b, ds);
  __syncthreads();  // the drafts in shared memory are read by other warps below
  griddep_wait();
  griddep_launch_dependents();  // the next kernel may start; the LM head grid is complete
  decide(a, b, ds);
  if (grp == 0) write_prefix(a, b, ds);
  const Decision& d = ds.d;
  if (d.bad) return;
  const int K = a.K;
  const int n = d.n;
  ResRow R;
  R.rej = n < K;
  R.zp = a.zp + static_cast<size_t>(b * (K + 1) + n) * a.ldp;
  R.zq = R.rej ? a.zq + static_cast<size_t>(b * K + n) * a.V : nullptr;
  R.c = {a.c_hi, a.c_lo};
  R.k_p = d.k_p;
  R.k_q = d.k_q;
  R.kh = d.kappa.hi;
  R.kl = d.kappa.lo;
  R.V = a.V;

  {
    // chunk by chunk; the next chunk's loads are in flight while this
    // chunk's terms are reduced
    const int t0 = threadIdx.x * kPer;
    float zp[kPer], zq[kPer];
    unsigned valid;
    load_pair<kVec>(R, c0 * kChunk + t0, zp, zq, valid);
    for (int c = c0; c < c1; ++c) {
      float r[kPer];
      pair_terms(R, zp, zq, valid, r);
      if (c + 1 < c1) load_pair<kVec>(R, (c + 1) * kChunk + t0, zp, zq, valid);
      const ff ws = warp_sum_ff({segment_total(r), 0.f});
      ff* sw = sm_w[(c - c0) & 1];
      if (lane == 0) sw[warp] = ws;
      __syncthreads();
      if (threadIdx.x == 0) {
        ff total = sw[0];
        for (int w = 1; w < kWarps; ++w) total = ff_add(total, sw[w]);
        a.res_sums[static_cast<size_t>(b) * a.CB + c] = make_float2(total.hi, total.lo);
      }
    }
  }
  if (!last_block_ticket(&a.tickets[b], gridDim.y, sm_i)) return;

  const float2* sums = a.res_sums + static_cast<size_t>(b) * a.CB;
  const float u = ds.uj[K];
  // total residual mass (warp 0, lanes over chunks); the first 64 chunk sums
  // stay in registers for the search below
  ff cached[2] = {{0.f, 0.f}, {0.f, 0.f}};
  if (threadIdx.x < 32) {
    ff s{0.f, 0.f};
    for (int i = lane; i < a.CB; i += 32) {
      const float2 v = __ldcg(&sums[i]);
      const ff fv{v.x, v.y};
      if (i < 64) cached[i >> 5] = fv;
      s = ff_add(s, fv);
    }
    s = warp_sum_ff(s);
    if (lane == 0) s_S = s;
  }
  __syncthreads();
  bool refilled = false;
  if (!(s_S.hi > 0.f) && R.rej) {
    refilled = true;
    // A rejection whose residual has no mass in f32 (impossible in exact
    // arithmetic): draw from p at that position instead.
    R.rej = false;
    R.zq = nullptr;
    ff P{0.f, 0.f};
    for (int i = 0; i < a.CB; ++i) {
      float r[kPer];
      residual_segment<kVec>(R, i * kChunk + threadIdx.x * kPer, r);
      ff excl, total;
      block_excl_scan_ff({segment_total(r), 0.f}, excl, total, sm_ff);
      if (threadIdx.x == 0) a.res_sums[static_cast<size_t>(b) * a.CB + i] = make_float2(total.hi, total.lo);
      P = ff_add(P, total);
    }
    __syncthreads();
    if (threadIdx.x == 0) s_S = P;
    __syncthreads();
  }
  // the chunk holding t = u * S: warp 0 scans the chunk sums 32 at a time
  if (threadIdx.x < 32) {
    const ff t = ff_mul_f(s_S, u);
    ff carry{0.f, 0.f};
    int cs = -1, last = -1;
    ff base{0.f, 0.f}, base_last{0.f, 0.f};
    for (int i0 = 0; i0 < a.CB && cs < 0; i0 += 32) {
      const int i = i0 + lane;
      ff v{0.f, 0.f};
      if (i < a.CB) {
        if (i0 < 64 && !refilled) {
          v = cached[i0 >> 5];
        } else {
          const float2 w = __ldcg(&sums[i]);
          v = {w.x, w.y};
        }
      }
      ff incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        ff o{__shfl_up_sync(0xffffffffu, incl.hi, off), __shfl_up_sync(0xffffffffu, incl.lo, off)};
        if (lane >= off) incl = ff_add(o, incl);
      }
      ff ex{__shfl_up_sync(0xffffffffu, incl.hi, 1), __shfl_up_sync(0xffffffffu, incl.lo, 1)};
      if (lane == 0) ex = {0.f, 0.f};
      const ff excl_w = ff_add(carry, ex);
      const ff incl_w = ff_add(carry, incl);
      const unsigned hit = __ballot_sync(0xffffffffu, i < a.CB && ff_gt(incl_w, t));
      const unsigned pos = __ballot_sync(0xffffffffu, i < a.CB && v.hi > 0.f);
      if (hit) {
        const int src = __ffs(hit) - 1;
        cs = i0 + src;
        base = {__shfl_sync(0xffffffffu, excl_w.hi, src), __shfl_sync(0xffffffffu, excl_w.lo, src)};
      }
      if (pos) {
        const int src = 31 - __clz(pos);
        last = i0 + src;
        base_last = {__shfl_sync(0xffffffffu, excl_w.hi, src), __shfl_sync(0xffffffffu, excl_w.lo, src)};
      }
      carry = {__shfl_sync(0xffffffffu, incl_w.hi, 31), __shfl_sync(0xffffffffu, incl_w.lo, 31)};
    }
    if (cs < 0) {  // rounding left t at the very end: the last chunk with mass
      cs = last < 0 ? 0 : last;
      base = base_last;
    }
    if (lane == 0) {
      s_chunk = cs;
      s_base = base;
      s_t = t;
    }
  }
  __syncthreads();
  int y, last_pos;
  locate_in_chunk<kVec>(R, s_chunk, s_base, s_t, y, last_pos, sm_ff, sm_i);
  if (threadIdx.x == 0) {
    if (y == INT_MAX) y = last_pos >= 0 ? last_pos : 0;
    a.out_tokens[b * (K + 1) + n] = y;
    if (a.out_debug) {
      const ff mass = R.rej ? ff_div(s_S, d.S_p) : ff{1.f, 0.f};
      a.out_debug[static_cast<size_t>(b * (K + 1) + n) * 6 + 5] = mass.hi;
    }
  }
}

// Rows of at most kMaxClusterChunks chunks (V <= 131072): one cluster per
// sequence, kCPC chunks per CTA (kCPC * kThreads threads; chunk h of a CTA
// owns warps h*kWarps .. h*kWarps+kWarps-1).  The chunk masses meet through
// distributed shared memory after one cluster barrier instead of a global
// array and a last-CTA ticket, every CTA finds the chunk holding t = u * S,
// and the warps owning it locate the token from the residual terms they
// still hold in registers (no second read of the row pair).  Arithmetic
// identical to finish_kernel: the same chunk masses in the same order, the
// same search.  Clusters above 8 CTAs are a non-portable size; the launch
// checks that one fits and otherwise takes finish_kernel.
constexpr int kMaxClusterCtas = 16;
constexpr int kMaxClusterChunks = 2 * kMaxClusterCtas;
static_assert(kMaxClusterChunks <= 32, "one lane per chunk in the chunk search");

// The cluster's chunk masses of exchange `round` (warp 0): total S, the
// chunk holding t = S * u, the mass before it, and t.  Chunk j's mass is
// slot round*kCPC + j%kCPC of CTA j/kCPC.
template <int kCPC>
__device__ void cluster_chunk_search(float4* s_mass, int round, int C, float u, ff& S, int& cs, ff& base, ff& t) {
  const int lane = threadIdx.x & 31;
  ff v{0.f, 0.f};
  if (lane < C) {
    const float4 f = ld_cluster_f4(cluster_map(&s_mass[round * kCPC + lane % kCPC], static_cast<uint32_t>(lane / kCPC)));
    v = {f.x, f.y};
  }
  // the same sequential order as the chunk-sum search of finish_kernel: a
  // warp inclusive scan, lane j holding chunks 0..j
  ff incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    ff o{__shfl_up_sync(0xffffffffu, incl.hi, off), __shfl_up_sync(0xffffffffu, incl.lo, off)};
    if (lane >= off) incl = ff_add(o, incl);
  }
  ff ex{__shfl_up_sync(0xffffffffu, incl.hi, 1), __shfl_up_sync(0xffffffffu, incl.lo, 1)};
  if (lane == 0) ex = {0.f, 0.f};
  // S as finish_kernel forms it: the warp sum of the chunk masses
  S = warp_sum_ff(v);
  t = ff_mul_f(S, u);
  const unsigned hit = __ballot_sync(0xffffffffu, lane < C && ff_gt(incl, t));
  const unsigned pos = __ballot_sync(0xffffffffu, lane < C && v.hi > 0.f);
  if (hit) {
    cs = __ffs(hit) - 1;
  } else {  // rounding left t at the very end: the last chunk with mass
    cs = pos ? 31 - __clz(pos) : 0;
  }
  base = {__shfl_sync(0xffffffffu, ex.hi, cs), __shfl_sync(0xffffffffu, ex.lo, cs)};
}

template <bool kVec, int kCPC>
__global__ void __launch_bounds__(kThreads * kCPC, 2) finish_cluster_kernel(const VerifyArgs a) {
  __shared__ DecideSmem ds;
  __shared__ ff sm_ff[kWarps * kCPC];
  __shared__ int sm_i[2 * kWarps];
  __shared__ float4 s_mass[2 * kCPC];  // this CTA's chunk masses, per exchange round (hi, lo)
  __shared__ ff s_base, s_t, s_S;
  __shared__ int s_chunk;
  const int C = a.CB;                         // chunks per row
  const int ctas = (C + kCPC - 1) / kCPC;     // CTAs per cluster
  const int b = blockIdx.x / ctas;
  const int rank = static_cast<int>(cluster_ctarank());
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = rank * kCPC + warp / kWarps;  // C itself (no tokens) in the second half of an odd row's last CTA
  load_inputs(a, b, ds);
  __syncthreads();  // the drafts in shared memory are read by other warps below
  griddep_wait();
  griddep_launch_dependents();  // the next kernel may start; the LM head grid is complete
  decide(a, b, ds);
  if (rank == 0) write_prefix(a, b, ds);
  const Decision& d = ds.d;
  if (d.bad) return;  // every CTA of the cluster decided the same: none waits at a barrier below
  const int K = a.K;
  const int n = d.n;
  ResRow R;
  R.rej = n < K;
  R.zp = a.zp + static_cast<size_t>(b * (K + 1) + n) * a.ldp;
  R.zq = R.rej ? a.zq + static_cast<size_t>(b * K + n) * a.V : nullptr;
  R.c = {a.c_hi, a.c_lo};
  R.k_p = d.k_p;
  R.k_q = d.k_q;
  R.kh = d.kappa.hi;
  R.kl = d.kappa.lo;
  R.V = a.V;
  const float u = ds.uj[K];
  const int e0 = chunk * kChunk + (threadIdx.x % kThreads) * kPer;
  float r[kPer];
  auto chunk_mass = [&](int round) {
    residual_segment<kVec>(R, e0, r);
    const ff ws = warp_sum_ff({segment_total(r), 0.f});
    if (lane == 0) sm_ff[warp] = ws;
    __syncthreads();
    if (threadIdx.x < kCPC) {
      const ff* w8 = sm_ff + threadIdx.x * kWarps;
      ff total = w8[0];
      for (int w = 1; w < kWarps; ++w) total = ff_add(total, w8[w]);
      s_mass[round * kCPC + threadIdx.x] = make_float4(total.hi, total.lo, 0.f, 0.f);
    }
    cluster_sync();  // every CTA's masses of this round are readable
    if (threadIdx.x < 32) {
      ff S, base, t;
      int cs;
      cluster_chunk_search<kCPC>(s_mass, round, C, u, S, cs, base, t);
      if (lane == 0) {
        s_S = S;
        s_chunk = cs;
        s_base = base;
        s_t = t;
      }
    }
    __syncthreads();
  };
  chunk_mass(0);
  if (!(s_S.hi > 0.f) && R.rej) {
    // A rejection whose residual has no mass in f32 (impossible in exact
    // arithmetic): draw from p at that position instead.
    R.rej = false;
    R.zq = nullptr;
    chunk_mass(1);
  }
  const int owner = s_chunk;
  cluster_sync();  // every CTA has read the others' masses: none leaves before
  if (chunk != owner) return;
  // the owning chunk's kThreads threads alone from here (named barrier 1)
  int y, last_pos;
  locate_from_terms(r, e0, s_base, s_t, y, last_pos, sm_ff, sm_i);
  if (threadIdx.x % kThreads == 0) {
    if (y == INT_MAX) y = last_pos >= 0 ? last_pos : 0;
    a.out_tokens[b * (K + 1) + n] = y;
    if (a.out_debug) {
      const ff mass = R.rej ? ff_div(s_S, d.S_p) : ff{1.f, 0.f};
      a.out_debug[static_cast<size_t>(b * (K + 1) + n) * 6 + 5] = mass.hi;
    }
  }
}

// ---------------------------------------------------------------- greedy
// One CTA per sequence: reduce the per-(row, partition) (max, lowest argmax)
// partials of rows b*(K+1) .. b*(K+1)+K, then compare with the drafts.
__global__ void __launch_bounds__(kThreads) greedy_finish_kernel(const GreedyArgs a) {
  __shared__ float sv[kWarps];
  __shared__ int si[kWarps];
  __shared__ int sb[kWarps];
  __shared__ int g_arg[kMaxK + 1];
  __shared__ float g_val[kMaxK + 1];
  __shared__ int g_bad[kMaxK + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = blockIdx.x;
  const int K = a.K;
  griddep_wait();
  griddep_launch_dependents();  // the next kernel may start; the LM head grid is complete
  for (int j = 0; j <= K; ++j) {
    const size_t row = static_cast<size_t>(b) * (K + 1) + j;
    const float* pv = a.part_max + row * a.P;
    const int* pi = a.part_idx + row * a.P;
    float bv = -INFINITY;
    int bi = INT_MAX;
    int bad = 0;
    constexpr int kBatch = 4;
    for (int p0 = 0; p0 < a.P; p0 += kThreads * kBatch) {
      float v[kBatch];
      int ix[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int p = p0 + j * kThreads + threadIdx.x;
        v[j] = p < a.P ? __ldcg(&pv[p]) : -INFINITY;
        ix[j] = p < a.P ? __ldcg(&pi[p]) : INT_MAX;
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (ix[j] == -2) {
          bad = 1;
        } else if (v[j] > bv || (v[j] == bv && ix[j] < bi)) {
          bv = v[j];
          bi = ix[j];
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    bad = __any_sync(0xffffffffu, bad != 0) ? 1 : 0;
    if (lane == 0) {
      sv[warp] = bv;
      si[warp] = bi;
      sb[warp] = bad;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float v0 = sv[0];
      int i0 = si[0];
      int b0 = sb[0];
      for (int w = 1; w < kWarps; ++w) {
        b0 |= sb[w];
        if (sv[w] > v0 || (sv[w] == v0 && si[w] < i0)) {
          v0 = sv[w];
          i0 = si[w];
        }
      }
      g_arg[j] = i0;
      g_val[j] = v0;
      g_bad[j] = b0 || i0 == INT_MAX;
    }
    __syncthreads();
  }
  if (warp != 0) return;
  int xj = -1;
  bool tok_ok = true;
  if (lane < K) {
    xj = a.x[b * K + lane];
    tok_ok = xj >= 0 && xj < a.V;
  }
  const unsigned match = __ballot_sync(0xffffffffu, lane < K && xj == g_arg[lane]);
  const unsigned badtok = __ballot_sync(0xffffffffu, lane < K && !tok_ok);
  int rowbad = 0;
  for (int j = lane; j <= K; j += 32) rowbad |= g_bad[j];
  rowbad = __any_sync(0xffffffffu, rowbad != 0) ? 1 : 0;
  const bool bad = badtok != 0u || rowbad != 0;
  int n = (match == 0xffffffffu) ? 32 : (__ffs(~match) - 1);
  n = min(n, K);
  for (int j = lane; j <= K; j += 32) {
    int tok = -1;
    if (!bad) tok = j < n ? xj : (j == n ? g_arg[n] : -1);
    a.out_tokens[b * (K + 1) + j] = tok;
    if (a.out_debug) {
      float* dbg = a.out_debug + (static_cast<size_t>(b) * (K + 1) + j) * 6;
      dbg[0] = g_val[j];
      dbg[1] = static_cast<float>(g_arg[j] == INT_MAX ? -1 : g_arg[j]);
      dbg[2] = dbg[3] = dbg[4] = dbg[5] = 0.f;
    }
  }
  if (lane == 0) {
    a.out_n[b] = bad ? -1 : n;
    if (bad) atomicOr(a.err, (badtok ? kErrTokenRange : 0) | (rowbad ? kErrNonFinite : 0));
  }
}

// Per (row, chunk) max and lowest argmax of given logits: [M][P] partials.
template <bool kVec>
__global__ void __launch_bounds__(kThreads) row_argmax_kernel(const float* __restrict__ logits, int M, int V, int P,
                                                             float* part_max, int* part_idx, int* err) {
  __shared__ float sv[kWarps];
  __shared__ int si[kWarps];
  __shared__ int sb[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int row = blockIdx.x, chunk = blockIdx.y;
  if (row == 0 && chunk == 0 && threadIdx.x == 0) *err = 0;
  const int e0 = chunk * kChunk + threadIdx.x * kPer;
  float z[kPer];
  unsigned valid;
  load16<kVec>(logits + static_cast<size_t>(row) * V, e0, V, z, valid);
  float bv = -INFINITY;
  int bi = INT_MAX;
  bool bad = false;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {  // ascending ids: strict > keeps the lowest on ties
    if (!((valid >> i) & 1u)) continue;
    if (!isfinite(z[i])) {
      bad = true;
    } else if (z[i] > bv) {
      bv = z[i];
      bi = e0 + i;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
    if (ov > bv || (ov == bv && oi < bi)) {
      bv = ov;
      bi = oi;
    }
  }
  const bool wbad = __any_sync(0xffffffffu, bad);
  if (lane == 0) {
    sv[warp] = bv;
    si[warp] = bi;
    sb[warp] = wbad;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float v = sv[0];
    int i0 = si[0];
    bool b0 = sb[0];
    for (int w = 1; w < kWarps; ++w) {
      b0 |= sb[w] != 0;
      if (sv[w] > v || (sv[w] == v && si[w] < i0)) {
        v = sv[w];
        i0 = si[w];
      }
    }
    part_max[static_cast<size_t>(row) * P + chunk] = v;
    part_idx[static_cast<size_t>(row) * P + chunk] = b0 ? -2 : i0;
  }
}

}  // namespace

void exponent_constant(float temperature, float* c_hi, float* c_lo) {
  const double c = 1.4426950408889634073599246810019 / static_cast<double>(temperature);
  *c_hi = static_cast<float>(c);
  *c_lo = static_cast<float>(c - static_cast<double>(*c_hi));
}

cudaError_t launch_row_stats(const float* zp, const float* zq, int M, int draft_rows, int V, float c_hi, float c_lo,
                             StatPart* tpart, StatPart* dpart, int* err, unsigned* tickets, int n_tickets,
                             cudaStream_t stream, long long ldp, bool zero_err) {
  const int P = (V + kChunk - 1) / kChunk;
  const long long units = static_cast<long long>(M + draft_rows) * P;
  if (units == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // warps take whole units; as many blocks as fit on the SMs at once
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, row_stats_kernel<true>, kStatThreads, 0);
  if (e != cudaSuccess) return e;
  const int grid = static_cast<int>(
      std::min<long long>((units + kStatThreads / 32 - 1) / (kStatThreads / 32), static_cast<long long>(std::max(per_sm, 1)) * sms));
  const Expo c{c_hi, c_lo};
  if (ldp <= 0) ldp = V;
  const bool vec = V % 4 == 0 && ldp % 4 == 0 && (reinterpret_cast<uintptr_t>(zp) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(zq) & 15u) == 0;
  // large passes (a few units per SM at least) stream through the bulk-copy
  // ring; small ones are latency-bound and keep the many-warp form
  if (vec && units >= 4ll * sms) {
    int smem_optin = 0;
    e = cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    const int S = std::min(12, (smem_optin - 1024) / static_cast<int>(kBulkUnitBytes + 32));
    if (S >= 4) {
      const size_t smem = static_cast<size_t>(S) * (kBulkUnitBytes + 32);
      static bool attr_done[64] = {false};
      if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
      if (!attr_done[dev]) {
        e = cudaFuncSetAttribute(row_stats_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
      }
      const int bgrid = static_cast<int>(std::min<long long>(units, sms));
      row_stats_bulk_kernel<<<bgrid, kBulkThreads, smem, stream>>>(zp, zq, M, V, ldp, c, tpart, dpart, P, units,
                                                                    err, tickets, n_tickets, S, zero_err ? 1 : 0);
      return cudaGetLastError();
    }
  }
  if (vec)
    row_stats_kernel<true><<<grid, kStatThreads, 0, stream>>>(zp, zq, M, V, ldp, c, tpart, dpart, P, units, err,
                                                              tickets, n_tickets, zero_err ? 1 : 0);
  else
    row_stats_kernel<false><<<grid, kStatThreads, 0, stream>>>(zp, zq, M, V, ldp, c, tpart, dpart, P, units, err,
                                                               tickets, n_tickets, zero_err ? 1 : 0);
  return cudaGetLastError();
}

namespace {

// One cluster of `ctas` CTAs of finish_cluster_kernel<kVec, kCPC> per
// sequence, a programmatic dependent of the preceding kernel.  `probe`
// asks instead how many such clusters can be resident at once.
template <bool kVec, int kCPC>
cudaError_t cluster_finish(const VerifyArgs& a, int ctas, cudaStream_t stream, int* probe) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.B) * static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(kThreads * kCPC);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(ctas);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (probe) {
    if (ctas > 8) {
      cudaError_t e = cudaFuncSetAttribute(finish_cluster_kernel<kVec, kCPC>,
                                           cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) {
        (void)cudaGetLastError();
        *probe = 0;
        return cudaSuccess;
      }
    }
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.numAttrs = 1;
    int clusters = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&clusters, finish_cluster_kernel<kVec, kCPC>, &cfg);
    if (e != cudaSuccess) (void)cudaGetLastError();
    *probe = e == cudaSuccess ? clusters : 0;
    return cudaSuccess;
  }
  return cudaLaunchKernelEx(&cfg, finish_cluster_kernel<kVec, kCPC>, a);
}

template <int kCPC>
cudaError_t cluster_finish_any(const VerifyArgs& a, bool vec, int ctas, cudaStream_t stream, int* probe) {
  return vec ? cluster_finish<true, kCPC>(a, ctas, stream, probe) : cluster_finish<false, kCPC>(a, ctas, stream, probe);
}

// How many clusters of `ctas` CTAs (kCPC = 2 when above 8) are resident on
// this device at once, probed once per (size, load width) and process:
// stored plus one (0 unknown).
std::atomic<int> g_cluster_fits[kMaxClusterCtas + 1][2];

// CTAs of finish_kernel<kVec> resident on the device at once (0 unknown).
std::atomic<int> g_finish_resident[2];

}  // namespace

cudaError_t launch_verify_sampling(const VerifyArgs& a, cudaStream_t stream) {
  // 16-byte loads need every target row 16-byte aligned
  const bool vec = a.V % 4 == 0 && a.ldp % 4 == 0 && (reinterpret_cast<uintptr_t>(a.zp) & 15u) == 0;
  if (a.CB <= kMaxClusterChunks) {
    // up to 8 chunks: one CTA per chunk; above: two chunks per CTA
    const bool two = a.CB > kMaxClusterChunks / 4;
    const int ctas = two ? (a.CB + 1) / 2 : a.CB;
    std::atomic<int>& fits = g_cluster_fits[ctas][vec ? 1 : 0];
    int f = fits.load(std::memory_order_relaxed);
    if (f == 0) {
      int n = 0;
      if (two) cluster_finish_any<2>(a, vec, ctas, stream, &n);
      else cluster_finish_any<1>(a, vec, ctas, stream, &n);
      f = n + 1;
      fits.store(f, std::memory_order_relaxed);
    }
    // only while every sequence's cluster is resident at once: clusters in
    // waves cost more than the grid kernel's single wave
    if (a.B <= f - 1) {
      if (two) return cluster_finish_any<2>(a, vec, ctas, stream, nullptr);
      return cluster_finish_any<1>(a, vec, ctas, stream, nullptr);
    }
  }
  // chunks per CTA: as few as let the whole grid be resident at once
  std::atomic<int>& resident = g_finish_resident[vec ? 1 : 0];
  int res = resident.load(std::memory_order_relaxed);
  if (res == 0) {
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = vec ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, finish_kernel<true>, kThreads, 0)
              : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, finish_kernel<false>, kThreads, 0);
    if (e != cudaSuccess) return e;
    res = std::max(1, per_sm * sms);
    resident.store(res, std::memory_order_relaxed);
  }
  VerifyArgs g_args = a;
  const long long units = static_cast<long long>(a.B) * a.CB;
  int G = static_cast<int>(std::min<long long>(a.CB, std::max<long long>(1, (units + res - 1) / res)));
  while (G < a.CB && static_cast<long long>(a.B) * ((a.CB + G - 1) / G) > res) ++G;  // whole groups per row
  g_args.G = G;
  const dim3 g(a.B, (a.CB + G - 1) / G);
  if (vec) return launch_dependent(finish_kernel<true>, g, dim3(kThreads), stream, g_args);
  return launch_dependent(finish_kernel<false>, g, dim3(kThreads), stream, g_args);
}

cudaError_t launch_greedy_finish(const GreedyArgs& a, cudaStream_t stream) {
  return launch_dependent(greedy_finish_kernel, dim3(a.B), dim3(kThreads), stream, a);
}

cudaError_t launch_row_argmax(const float* logits, int M, int V, float* part_max, int* part_idx, int* err,
                              cudaStream_t stream) {
  const int P = (V + kChunk - 1) / kChunk;
  const dim3 g(M, P);
  if (V % 4 == 0)
    row_argmax_kernel<true><<<g, kThreads, 0, stream>>>(logits, M, V, P, part_max, part_idx, err);
  else
    row_argmax_kernel<false><<<g, kThreads, 0, stream>>>(logits, M, V, P, part_max, part_idx, err);
  return cudaGetLastError();
}

}  // namespace sv
