// Vocabulary-parallel verify-and-accept kernels (sm_103a, CUDA cores).
//
// Sampling path (T > 0), two launches after the LM head:
//
//  1. row_stats_kernel, grid (chunks of 8192 tokens) x (rows): every target
//     row z_p[b,j] (j = 0..K) and draft row z_q[b,j] (j < K) is read once
//     with 128-bit loads; each CTA reduces its chunk to (max of z/T,
//     sum exp(z/T - max)) (the online max / sum-exp of softmax(z/T), page
//     "quochung.cyou" A.I article, section "Forward pass": the scores are a
//     distribution summing to 100%).  The last CTA of a sequence (atomic
//     ticket, no grid-wide wait) combines the partials, gathers p_j(x_j)
//     and q_j(x_j), runs the accept test u_j < min(1, p_j(x_j)/q_j(x_j))
//     (section "Modified rejection sampling / Giải pháp"), takes the
//     accepted prefix with one warp ballot (section "Áp dụng thuật toán":
//     left to right, stop at the first rejection) and writes the accepted
//     tokens.
//  2. residual_kernel, grid (chunks of 4096 tokens) x (sequences): the row
//     pair at the first rejection n_b is read once more and reduced to the
//     residual mass of max(0, p - q) per chunk (section "Khi reject thì lấy
//     token từ đâu?"), or of p_K for the bonus token when n_b = K.  The last
//     CTA of the sequence finds the chunk that holds u*S and rescans it
//     with a block-wide prefix scan to pick the smallest token whose
//     cumulative mass exceeds u*S (inverse CDF, ascending token id).
//
// Greedy path (T = 0): the LM head writes per-(vocabulary tile, row)
// (max, lowest argmax) partials; greedy_finish_kernel reduces them and
// compares the drafts with the argmax left to right (section "Một vòng
// speculative decoding", Bước 3).
//
// Arithmetic: z/T is an IEEE f32 division, exp is expf; row normalisers and
// the residual's prefix sums are accumulated in f64 across threads (f32
// inside a thread's 16 or 32 elements) so that the draw's decision is
// limited by the logits, not by the summation.
#include <cfloat>
#include <climits>

#include "internal.h"

namespace sv {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowPerThread = kRowChunk / kThreads;  // 32
constexpr int kResPerThread = kResChunk / kThreads;  // 16
static_assert(kRowPerThread % 4 == 0 && kResPerThread % 4 == 0, "vector width");

__device__ __forceinline__ float scaled(float z, float T) { return __fdiv_rn(z, T); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Max over the block; every thread gets the result.  Uses sm[kWarps].
__device__ float block_max(float v, float* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max(v);
  if (lane == 0) sm[warp] = v;
  __syncthreads();
  float r = sm[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) r = fmaxf(r, sm[w]);
  __syncthreads();
  return r;
}

// Sum over the block in a fixed order; every thread gets the result.
__device__ double block_sum_d(double v, double* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_d(v);
  if (lane == 0) sm[warp] = v;
  __syncthreads();
  double r = 0.0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) r += sm[w];
  __syncthreads();
  return r;
}

// Exclusive prefix sum over the block's threads (thread order) and the total.
__device__ void block_excl_scan_d(double v, double& excl, double& total, double* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const double o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  double ex = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) ex = 0.0;
  if (lane == 31) sm[warp] = incl;
  __syncthreads();
  double woff = 0.0, tot = 0.0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    if (w == warp) woff = tot;
    tot += sm[w];
  }
  __syncthreads();
  excl = woff + ex;
  total = tot;
}

__device__ int block_min_i(int v, int* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, off));
  if (lane == 0) sm[warp] = v;
  __syncthreads();
  int r = sm[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) r = min(r, sm[w]);
  __syncthreads();
  return r;
}

__device__ int block_max_i(int v, int* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, off));
  if (lane == 0) sm[warp] = v;
  __syncthreads();
  int r = sm[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) r = max(r, sm[w]);
  __syncthreads();
  return r;
}

// Ticket: returns true in every thread of the block that arrives last among
// `expected` blocks counted on *counter.  Writes made by the earlier blocks
// before their ticket are visible to the last one afterwards.
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

// ---------------------------------------------------------------- decision
// Run by the whole block of the last row-statistics CTA of sequence b.
__device__ void decide_sequence(const VerifyArgs& a, int b) {
  __shared__ float rm[2 * kMaxK + 1];
  __shared__ double rS[2 * kMaxK + 1];
  __shared__ int rbad[2 * kMaxK + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int K = a.K;
  const int M = a.B * (K + 1);
  const int nrows = 2 * K + 1;

  // combine the chunk partials of every row of the sequence, one warp per row
  for (int r = warp; r < nrows; r += kWarps) {
    const int grow = r <= K ? b * (K + 1) + r : M + b * K + (r - K - 1);
    const RowPart* pp = a.parts + static_cast<size_t>(grow) * a.CA;
    float m = -INFINITY;
    int bad = 0;
    for (int c = lane; c < a.CA; c += 32) {
      m = fmaxf(m, __ldcg(&pp[c].m));
      bad |= __ldcg(&pp[c].bad);
    }
    m = warp_max(m);
    bad = __any_sync(0xffffffffu, bad != 0) ? 1 : 0;
    double s = 0.0;
    for (int c = lane; c < a.CA; c += 32) {
      const float mc = __ldcg(&pp[c].m);
      const double sc = __ldcg(&pp[c].s);
      if (sc > 0.0) s += sc * exp(static_cast<double>(mc) - static_cast<double>(m));
    }
    s = warp_sum_d(s);
    if (lane == 0) {
      rm[r] = m;
      rS[r] = s;
      rbad[r] = bad || !(s > 0.0) || !isfinite(s);
    }
  }
  __syncthreads();

  if (warp != 0) return;
  const float T = a.T;
  bool tok_ok = true, acc = false;
  int xj = -1;
  double pj = 0.0, qj = 0.0, aj = 0.0;
  if (lane < K) {
    xj = a.x[b * K + lane];
    tok_ok = xj >= 0 && xj < a.V;
    if (tok_ok) {
      const float zp = a.zp[static_cast<size_t>(b * (K + 1) + lane) * a.V + xj];
      const float zq = a.zq[static_cast<size_t>(b * K + lane) * a.V + xj];
      const double lp = static_cast<double>(scaled(zp, T)) - static_cast<double>(rm[lane]);
      const double lq = static_cast<double>(scaled(zq, T)) - static_cast<double>(rm[K + 1 + lane]);
      const double Sp = rS[lane], Sq = rS[K + 1 + lane];
      pj = exp(lp) / Sp;
      qj = exp(lq) / Sq;
      aj = fmin(1.0, exp(lp - lq) * (Sq / Sp));
      acc = static_cast<double>(a.u[b * (K + 1) + lane]) < aj;
    }
  }
  const unsigned acc_mask = __ballot_sync(0xffffffffu, acc);
  const unsigned badtok = __ballot_sync(0xffffffffu, lane < K && !tok_ok);
  int rowbad = 0;
  for (int r = lane; r < nrows; r += 32) rowbad |= rbad[r];
  rowbad = __any_sync(0xffffffffu, rowbad != 0) ? 1 : 0;
  const bool bad = badtok != 0u || rowbad != 0;
  int n = (acc_mask == 0xffffffffu) ? 32 : (__ffs(~acc_mask) - 1);
  n = min(n, K);

  if (lane <= K) {
    int tok = -1;
    if (!bad && lane < n) tok = xj;
    a.out_tokens[b * (K + 1) + lane] = tok;
    if (a.out_debug) {
      float* dbg = a.out_debug + static_cast<size_t>(b * (K + 1) + lane) * 6;
      dbg[0] = lane < K ? static_cast<float>(pj) : 0.f;
      dbg[1] = lane < K ? static_cast<float>(qj) : 0.f;
      dbg[2] = lane < K ? static_cast<float>(aj) : 0.f;
      dbg[3] = static_cast<float>(static_cast<double>(rm[lane]) + log(rS[lane]));
      dbg[4] = lane < K ? static_cast<float>(static_cast<double>(rm[K + 1 + lane]) + log(rS[K + 1 + lane])) : 0.f;
      dbg[5] = 0.f;
    }
  }
  if (lane == 0) {
    a.out_n[b] = bad ? -1 : n;
    if (bad) atomicOr(a.err, (badtok ? kErrTokenRange : 0) | (rowbad ? kErrNonFinite : 0));
    SeqState st;
    st.n = n;
    st.bad = bad ? 1 : 0;
    st.m_p = rm[n];
    st.S_p = rS[n];
    if (n < K) {
      st.m_q = rm[K + 1 + n];
      st.S_q = rS[K + 1 + n];
      st.kappa = rS[n] / rS[K + 1 + n];
    } else {
      st.m_q = 0.f;
      st.S_q = 0.0;
      st.kappa = 0.0;
    }
    a.seq[b] = st;
  }
}

// ---------------------------------------------------------------- pass 1
template <bool kVec>
__global__ void __launch_bounds__(kThreads) row_stats_kernel(const VerifyArgs a) {
  __shared__ float sm_f[kWarps];
  __shared__ double sm_d[kWarps];
  __shared__ int sm_i[1];
  const int row = blockIdx.y, c = blockIdx.x;
  const int M = a.B * (a.K + 1);
  const bool target = row < M;
  const float* z = target ? a.zp + static_cast<size_t>(row) * a.V : a.zq + static_cast<size_t>(row - M) * a.V;
  const int b = target ? row / (a.K + 1) : (row - M) / a.K;
  const int v0 = c * kRowChunk;
  const int v1 = min(a.V, v0 + kRowChunk);
  const float T = a.T;

  float x[kRowPerThread];
  int bad = 0;
  if (kVec) {
#pragma unroll
    for (int i = 0; i < kRowPerThread / 4; ++i) {
      const int e = v0 + (i * kThreads + threadIdx.x) * 4;
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e + 3 < v1) {
        f = __ldg(reinterpret_cast<const float4*>(z + e));
      } else {
        if (e + 0 < v1) f.x = z[e + 0];
        if (e + 1 < v1) f.y = z[e + 1];
        if (e + 2 < v1) f.z = z[e + 2];
      }
      const float fv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const bool valid = e + k < v1;
        bad |= valid && !isfinite(fv[k]);
        x[4 * i + k] = valid ? scaled(fv[k], T) : -INFINITY;
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < kRowPerThread; ++i) {
      const int e = v0 + i * kThreads + threadIdx.x;
      const bool valid = e < v1;
      const float zv = valid ? z[e] : 0.f;
      bad |= valid && !isfinite(zv);
      x[i] = valid ? scaled(zv, T) : -INFINITY;
    }
  }
  float tmax = -INFINITY;
#pragma unroll
  for (int i = 0; i < kRowPerThread; ++i) tmax = fmaxf(tmax, x[i]);
  const float m = block_max(tmax, sm_f);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kRowPerThread; ++i) s += expf(x[i] - m);
  const double S = block_sum_d(static_cast<double>(s), sm_d);
  const int any_bad = __syncthreads_or(bad);
  if (threadIdx.x == 0) {
    RowPart part;
    part.m = m;
    part.bad = any_bad;
    part.s = S;
    a.parts[static_cast<size_t>(row) * a.CA + c] = part;
  }
  const unsigned expected = static_cast<unsigned>((2 * a.K + 1) * a.CA);
  if (!last_block_ticket(&a.tickets_a[b], expected, sm_i)) return;
  decide_sequence(a, b);
}

// ---------------------------------------------------------------- pass 2
struct ResRow {
  const float* zp;
  const float* zq;
  float T, m_p, m_q, kh, kl;
  int V;
  bool rej;
};

// Residual mass of one token, scaled by S_p:  S_p * max(0, p - q)
// = max(0, e_p - kappa * e_q), with kappa = S_p / S_q carried as a pair of
// floats so that no rounded copy of it biases every term the same way.  For
// the bonus row (no rejection) it is e_p = S_p * p.
__device__ __forceinline__ float residual_term(float zp, float zq, const ResRow& R) {
  const float ep = expf(scaled(zp, R.T) - R.m_p);
  if (!R.rej) return ep;
  const float eq = expf(scaled(zq, R.T) - R.m_q);
  return fmaxf(0.f, ep - fmaf(R.kh, eq, R.kl * eq));
}

template <bool kVec>
__device__ __forceinline__ void residual_segment(const ResRow& R, int e0, float (&r)[kResPerThread]) {
  float zp[kResPerThread], zq[kResPerThread];
  if (kVec && e0 + kResPerThread - 1 < R.V) {
#pragma unroll
    for (int i = 0; i < kResPerThread / 4; ++i) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(R.zp + e0) + i);
      zp[4 * i] = f.x;
      zp[4 * i + 1] = f.y;
      zp[4 * i + 2] = f.z;
      zp[4 * i + 3] = f.w;
      if (R.rej) {
        const float4 g = __ldg(reinterpret_cast<const float4*>(R.zq + e0) + i);
        zq[4 * i] = g.x;
        zq[4 * i + 1] = g.y;
        zq[4 * i + 2] = g.z;
        zq[4 * i + 3] = g.w;
      } else {
        zq[4 * i] = zq[4 * i + 1] = zq[4 * i + 2] = zq[4 * i + 3] = 0.f;
      }
    }
#pragma unroll
    for (int i = 0; i < kResPerThread; ++i) r[i] = residual_term(zp[i], zq[i], R);
  } else {
#pragma unroll
    for (int i = 0; i < kResPerThread; ++i) {
      const int e = e0 + i;
      if (e < R.V) {
        const float a = R.zp[e];
        const float q = R.rej ? R.zq[e] : 0.f;
        r[i] = residual_term(a, q, R);
      } else {
        r[i] = 0.f;
      }
    }
  }
}

__device__ __forceinline__ float segment_total(const float (&r)[kResPerThread]) {
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kResPerThread; ++i) s += r[i];
  return s;
}

// Within one chunk: the smallest token whose cumulative mass base + (prefix
// through it) exceeds t; INT_MAX if none does.  Also returns the last token
// of the chunk with positive mass (or -1) for the rounding fallback.
template <bool kVec>
__device__ void locate_in_chunk(const ResRow& R, int chunk, double base, double t, int& y, int& last_pos,
                                double* sm_d, int* sm_i) {
  const int e0 = chunk * kResChunk + threadIdx.x * kResPerThread;
  float r[kResPerThread];
  residual_segment<kVec>(R, e0, r);
  double excl, total;
  block_excl_scan_d(static_cast<double>(segment_total(r)), excl, total, sm_d);
  const double tb = base + excl;
  int found = INT_MAX, lastp = -1;
  float run = 0.f;
#pragma unroll
  for (int i = 0; i < kResPerThread; ++i) {
    run += r[i];
    if (found == INT_MAX && tb + static_cast<double>(run) > t) found = e0 + i;
    if (r[i] > 0.f) lastp = e0 + i;
  }
  y = block_min_i(found, sm_i);
  last_pos = block_max_i(lastp, sm_i);
}

template <bool kVec>
__global__ void __launch_bounds__(kThreads) residual_kernel(const VerifyArgs a) {
  __shared__ double sm_d[kWarps];
  __shared__ int sm_i[kWarps];
  __shared__ SeqState st;
  __shared__ double s_base, s_t, s_S;
  __shared__ int s_chunk;
  const int b = blockIdx.y, c = blockIdx.x;
  if (threadIdx.x == 0) {
    const SeqState* g = &a.seq[b];
    st.n = __ldcg(&g->n);
    st.bad = __ldcg(&g->bad);
    st.m_p = __ldcg(&g->m_p);
    st.m_q = __ldcg(&g->m_q);
    st.S_p = __ldcg(&g->S_p);
    st.S_q = __ldcg(&g->S_q);
    st.kappa = __ldcg(&g->kappa);
  }
  __syncthreads();
  if (st.bad) return;
  const int K = a.K;
  const int n = st.n;
  ResRow R;
  R.rej = n < K;
  R.zp = a.zp + static_cast<size_t>(b * (K + 1) + n) * a.V;
  R.zq = R.rej ? a.zq + static_cast<size_t>(b * K + n) * a.V : nullptr;
  R.T = a.T;
  R.m_p = st.m_p;
  R.m_q = st.m_q;
  R.kh = static_cast<float>(st.kappa);
  R.kl = static_cast<float>(st.kappa - static_cast<double>(R.kh));
  R.V = a.V;

  {
    float r[kResPerThread];
    residual_segment<kVec>(R, c * kResChunk + threadIdx.x * kResPerThread, r);
    double excl, total;
    block_excl_scan_d(static_cast<double>(segment_total(r)), excl, total, sm_d);
    if (threadIdx.x == 0) a.res_sums[static_cast<size_t>(b) * a.CB + c] = total;
  }
  if (!last_block_ticket(&a.tickets_b[b], static_cast<unsigned>(a.CB), sm_i)) return;

  const double u = static_cast<double>(a.u[b * (K + 1) + K]);
  const double* sums = a.res_sums + static_cast<size_t>(b) * a.CB;
  if (threadIdx.x == 0) {
    double S = 0.0;
    for (int i = 0; i < a.CB; ++i) S += __ldcg(&sums[i]);
    s_S = S;
  }
  __syncthreads();
  if (!(s_S > 0.0) && R.rej) {
    // A rejection whose residual has no mass in f32: draw from p at that
    // position instead (never happens in exact arithmetic).
    R.rej = false;
    R.zq = nullptr;
    double P = 0.0;
    for (int i = 0; i < a.CB; ++i) {
      float r[kResPerThread];
      residual_segment<kVec>(R, i * kResChunk + threadIdx.x * kResPerThread, r);
      double excl, total;
      block_excl_scan_d(static_cast<double>(segment_total(r)), excl, total, sm_d);
      if (threadIdx.x == 0) a.res_sums[static_cast<size_t>(b) * a.CB + i] = total;
      P += total;
    }
    __syncthreads();
    if (threadIdx.x == 0) s_S = P;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double S = s_S;
    const double t = u * S;
    double P = 0.0;
    int cs = -1;
    for (int i = 0; i < a.CB; ++i) {
      const double Si = __ldcg(&sums[i]);
      if (P + Si > t) {
        cs = i;
        break;
      }
      P += Si;
    }
    if (cs < 0) {
      // rounding left t at the very end: the last chunk with mass
      P = 0.0;
      int last = -1;
      double Pl = 0.0;
      for (int i = 0; i < a.CB; ++i) {
        const double Si = __ldcg(&sums[i]);
        if (Si > 0.0) {
          last = i;
          Pl = P;
        }
        P += Si;
      }
      cs = last < 0 ? 0 : last;
      P = Pl;
    }
    s_chunk = cs;
    s_base = P;
    s_t = t;
  }
  __syncthreads();
  int y, last_pos;
  locate_in_chunk<kVec>(R, s_chunk, s_base, s_t, y, last_pos, sm_d, sm_i);
  if (threadIdx.x == 0) {
    if (y == INT_MAX) y = last_pos >= 0 ? last_pos : 0;
    a.out_tokens[b * (K + 1) + n] = y;
    if (a.out_debug) {
      a.out_debug[static_cast<size_t>(b * (K + 1) + n) * 6 + 5] =
          static_cast<float>(R.rej ? s_S / st.S_p : 1.0);
    }
  }
}

// ---------------------------------------------------------------- greedy
constexpr int kGreedyRows = 32;    // rows per CTA (one per lane)
constexpr int kGreedySlices = 8;   // partition slices (grid.y)

// Partials of the greedy reduction: per (slice, row) best value and index.
__global__ void __launch_bounds__(kThreads) greedy_finish_kernel(const GreedyArgs a, float* slice_max,
                                                                 int* slice_idx, int* row_arg,
                                                                 unsigned* ticket) {
  __shared__ float sv_[kWarps][kGreedyRows];
  __shared__ int si_[kWarps][kGreedyRows];
  __shared__ int sm_i[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int M = a.B * (a.K + 1);
  const int m = blockIdx.x * kGreedyRows + lane;
  const int slice = blockIdx.y;
  float bv = -INFINITY;
  int bi = INT_MAX;
  bool bad = false;
  if (m < M) {
    for (int p = slice * kWarps + warp; p < a.P; p += kWarps * kGreedySlices) {
      const float v = __ldcg(&a.part_max[static_cast<size_t>(p) * M + m]);
      const int i = __ldcg(&a.part_idx[static_cast<size_t>(p) * M + m]);
      if (i == -2) {
        bad = true;
      } else if (v > bv || (v == bv && i < bi)) {
        bv = v;
        bi = i;
      }
    }
  }
  sv_[warp][lane] = bv;
  si_[warp][lane] = bad ? -2 : bi;
  __syncthreads();
  if (warp == 0 && m < M) {
    float v0 = sv_[0][lane];
    int i0 = si_[0][lane];
    bool b0 = i0 == -2;
    for (int w = 1; w < kWarps; ++w) {
      const float v = sv_[w][lane];
      const int i = si_[w][lane];
      if (i == -2) {
        b0 = true;
      } else if (v > v0 || (v == v0 && i < i0) || i0 == -2) {
        v0 = v;
        i0 = i;
      }
    }
    slice_max[static_cast<size_t>(slice) * M + m] = v0;
    slice_idx[static_cast<size_t>(slice) * M + m] = b0 ? -2 : i0;
  }
  if (!last_block_ticket(ticket, gridDim.x * gridDim.y, sm_i)) return;

  // the last CTA: combine the slices of every row, then decide every sequence
  for (int r = threadIdx.x; r < M; r += kThreads) {
    float v0 = -INFINITY;
    int i0 = INT_MAX;
    bool b0 = false;
    for (int s = 0; s < kGreedySlices; ++s) {
      const float v = __ldcg(&slice_max[static_cast<size_t>(s) * M + r]);
      const int i = __ldcg(&slice_idx[static_cast<size_t>(s) * M + r]);
      if (i == -2) {
        b0 = true;
      } else if (v > v0 || (v == v0 && i < i0)) {
        v0 = v;
        i0 = i;
      }
    }
    row_arg[r] = (b0 || i0 == INT_MAX) ? -2 : i0;
    if (a.out_debug) {
      float* dbg = a.out_debug + static_cast<size_t>(r) * 6;
      dbg[0] = v0;
      dbg[1] = static_cast<float>(i0 == INT_MAX ? -1 : i0);
      dbg[2] = dbg[3] = dbg[4] = dbg[5] = 0.f;
    }
  }
  __syncthreads();
  __threadfence_block();
  const int K = a.K;
  for (int b = threadIdx.x; b < a.B; b += kThreads) {
    bool badrow = false, badtok = false;
    for (int j = 0; j <= K; ++j) badrow |= row_arg[b * (K + 1) + j] == -2;
    int n = K;
    for (int j = 0; j < K; ++j) {
      const int x = a.x[b * K + j];
      if (x < 0 || x >= a.V) badtok = true;
    }
    for (int j = 0; j < K; ++j) {
      if (a.x[b * K + j] != row_arg[b * (K + 1) + j]) {
        n = j;
        break;
      }
    }
    const bool bad = badrow || badtok;
    for (int j = 0; j <= K; ++j) {
      int tok = -1;
      if (!bad) tok = j < n ? a.x[b * K + j] : (j == n ? row_arg[b * (K + 1) + n] : -1);
      a.out_tokens[b * (K + 1) + j] = tok;
    }
    a.out_n[b] = bad ? -1 : n;
    if (bad) atomicOr(a.err, (badtok ? kErrTokenRange : 0) | (badrow ? kErrNonFinite : 0));
  }
}

// Per (chunk, row) max and lowest argmax of given logits: [P][M] partials.
template <bool kVec>
__global__ void __launch_bounds__(kThreads) row_argmax_kernel(const float* __restrict__ logits, int M, int V,
                                                             float* part_max, int* part_idx) {
  __shared__ float sv_[kWarps];
  __shared__ int si_[kWarps];
  __shared__ int sb_[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int row = blockIdx.y, c = blockIdx.x;
  const float* z = logits + static_cast<size_t>(row) * V;
  const int v0 = c * kRowChunk, v1 = min(V, v0 + kRowChunk);
  float bv = -INFINITY;
  int bi = INT_MAX;
  bool bad = false;
  // ascending element order per thread, so "first seen wins" keeps the lowest id on ties
  for (int i = 0; i < kRowPerThread; ++i) {
    const int e = v0 + i * kThreads + threadIdx.x;
    if (e < v1) {
      const float v = z[e];
      if (!isfinite(v)) {
        bad = true;
      } else if (v > bv) {
        bv = v;
        bi = e;
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
  const bool wbad = __any_sync(0xffffffffu, bad);
  if (lane == 0) {
    sv_[warp] = bv;
    si_[warp] = bi;
    sb_[warp] = wbad;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float v = sv_[0];
    int i0 = si_[0];
    bool b0 = sb_[0];
    for (int w = 1; w < kWarps; ++w) {
      b0 |= sb_[w] != 0;
      if (sv_[w] > v || (sv_[w] == v && si_[w] < i0)) {
        v = sv_[w];
        i0 = si_[w];
      }
    }
    part_max[static_cast<size_t>(c) * M + row] = v;
    part_idx[static_cast<size_t>(c) * M + row] = b0 ? -2 : i0;
  }
}

}  // namespace

cudaError_t launch_verify_sampling(const VerifyArgs& a, cudaStream_t stream) {
  const int M = a.B * (a.K + 1);
  const int R = M + a.B * a.K;
  const bool vec = (a.V % 4) == 0;
  dim3 g1(a.CA, R);
  if (vec)
    row_stats_kernel<true><<<g1, kThreads, 0, stream>>>(a);
  else
    row_stats_kernel<false><<<g1, kThreads, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 g2(a.CB, a.B);
  if (vec)
    residual_kernel<true><<<g2, kThreads, 0, stream>>>(a);
  else
    residual_kernel<false><<<g2, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

// Workspace for the greedy finish: slice partials [kGreedySlices][M] (f32 + i32)
// and row results [M]; the caller provides them after the partition partials.
size_t greedy_scratch_bytes(int M) {
  return static_cast<size_t>(kGreedySlices) * M * 8 + static_cast<size_t>(M) * 4;
}

cudaError_t launch_greedy_finish_ws(const GreedyArgs& a, void* scratch, unsigned* ticket, cudaStream_t stream) {
  const int M = a.B * (a.K + 1);
  float* slice_max = static_cast<float*>(scratch);
  int* slice_idx = reinterpret_cast<int*>(slice_max + static_cast<size_t>(kGreedySlices) * M);
  int* row_arg = slice_idx + static_cast<size_t>(kGreedySlices) * M;
  dim3 g((M + kGreedyRows - 1) / kGreedyRows, kGreedySlices);
  greedy_finish_kernel<<<g, kThreads, 0, stream>>>(a, slice_max, slice_idx, row_arg, ticket);
  return cudaGetLastError();
}

cudaError_t launch_row_argmax(const float* logits, int M, int V, float* part_max, int* part_idx,
                              cudaStream_t stream) {
  dim3 g((V + kRowChunk - 1) / kRowChunk, M);
  row_argmax_kernel<false><<<g, kThreads, 0, stream>>>(logits, M, V, part_max, part_idx);
  return cudaGetLastError();
}

}  // namespace sv
