// Vocabulary-parallel verify-and-accept kernels (sm_103a, CUDA cores).
//
// Sampling path (T > 0), two launches after the LM head:
//
//  1. stats_kernel, grid (rows) x (chunks of 4096 tokens): every target row
//     z_p[b,j] (j = 0..K) and draft row z_q[b,j] (j < K) is read once with
//     128-bit loads and reduced to its softmax(z/T) normaliser (page
//     "quochung.cyou" A.I article, section "Forward pass": the scores form a
//     distribution summing to 100%).  The last CTA of each sequence (atomic
//     ticket; no CTA ever waits for another) combines the chunks, gathers
//     p_j(x_j) and q_j(x_j), runs the accept test u_j < min(1, p_j(x_j) /
//     q_j(x_j)) (section "Modified rejection sampling / Giải pháp"), takes
//     the accepted prefix with one warp ballot (section "Áp dụng thuật
//     toán": left to right, stop at the first rejection) and writes the
//     accepted tokens.
//  2. residual_kernel, grid (sequences) x (chunks of 4096 tokens): the row
//     pair at the first rejection n_b is read once more and reduced to the
//     mass of max(0, p - q) per chunk (section "Khi reject thì lấy token từ
//     đâu?"), or of p_K for the bonus token when n_b = K.  The last CTA of
//     the sequence finds the chunk holding u*S and rescans it with a
//     block-wide prefix scan for the smallest token whose cumulative mass
//     exceeds u*S (inverse CDF, ascending token id).
//
// Arithmetic.  exp(z/T) is evaluated as 2^(z*c) with c = log2(e)/T carried
// as a pair of floats, so z*c is exact to ~1e-14 and no rounded temperature
// or log2(e) scales every exponent the same way.  Each chunk sums
// 2^(z*c - k_c) against an integer reference k_c (the ceiling of its largest
// exponent): rescaling chunks to a common reference is then an exact power
// of two.  Sums are compensated (float-float), so the normalisers, their
// ratio kappa = S_p / S_q and the residual's prefix sums carry no
// systematic error larger than ~1e-12; the only per-token error left is the
// f32 rounding of one exponent and one exp2f, which is random across tokens.
// Nothing here uses f64 (slow on this part).
//
// Greedy path (T = 0): the LM head writes per-(row, vocabulary tile)
// (max, lowest argmax) partials; greedy_finish_kernel reduces them and
// compares the drafts with the argmax left to right (section "Một vòng
// speculative decoding", Bước 3).
#include <cfloat>
#include <climits>

#include "internal.h"

namespace sv {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPer = kChunk / kThreads;  // 16 tokens per thread
static_assert(kPer == 16, "load16 handles 16 tokens per thread");

// ------------------------------------------------------------ float-float
struct ff {
  float hi, lo;
};

// a + b exactly as hi + lo (Knuth's TwoSum).
__device__ __forceinline__ ff two_sum(float a, float b) {
  const float s = a + b;
  const float bb = s - a;
  const float e = (a - (s - bb)) + (b - bb);
  return {s, e};
}

__device__ __forceinline__ ff ff_norm(float hi, float lo) {
  const float s = hi + lo;
  return {s, lo - (s - hi)};
}

__device__ __forceinline__ ff ff_add(ff a, ff b) {
  const ff s = two_sum(a.hi, b.hi);
  return ff_norm(s.hi, s.lo + a.lo + b.lo);
}

__device__ __forceinline__ ff ff_add_f(ff a, float b) {
  const ff s = two_sum(a.hi, b);
  return ff_norm(s.hi, s.lo + a.lo);
}

// a > b for normalised pairs.
__device__ __forceinline__ bool ff_gt(ff a, ff b) { return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo); }

__device__ __forceinline__ ff ff_scale2(ff a, int e) { return {ldexpf(a.hi, e), ldexpf(a.lo, e)}; }

__device__ __forceinline__ ff ff_mul_f(ff a, float b) {
  const float p = a.hi * b;
  const float e = fmaf(a.hi, b, -p);
  return ff_norm(p, e + a.lo * b);
}

// a / b to ~1e-14 (one correction step of the f32 quotient).
__device__ __forceinline__ ff ff_div(ff a, ff b) {
  const float q1 = a.hi / b.hi;
  const ff qb = ff_mul_f(b, q1);
  const ff r = ff_add(a, {-qb.hi, -qb.lo});
  const float q2 = r.hi / b.hi;
  return ff_norm(q1, q2);
}

__device__ __forceinline__ ff shfl_xor_ff(ff v, int off) {
  return {__shfl_xor_sync(0xffffffffu, v.hi, off), __shfl_xor_sync(0xffffffffu, v.lo, off)};
}

__device__ __forceinline__ ff warp_sum_ff(ff v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = ff_add(v, shfl_xor_ff(v, off));
  return v;
}

// ------------------------------------------------------------ exponent map
// z * c as a float pair, c = log2(e) / T given as (ch, cl).
struct Expo {
  float ch, cl;
};

__device__ __forceinline__ ff expo(float z, Expo c) {
  const float h = z * c.ch;
  const float l = fmaf(z, c.ch, -h) + z * c.cl;
  return ff_norm(h, l);
}

// 2^(y - k) for an integer-valued float k.
__device__ __forceinline__ float pow2_rel(ff y, float k) { return exp2f((y.hi - k) + y.lo); }

// ------------------------------------------------------------ block helpers
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

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

// Exclusive prefix sum (thread order) of a float-float value over the block,
// and the block total.  sm: kWarps pairs.
__device__ void block_excl_scan_ff(ff v, ff& excl, ff& total, ff* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  ff incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    ff o{__shfl_up_sync(0xffffffffu, incl.hi, off), __shfl_up_sync(0xffffffffu, incl.lo, off)};
    if (lane >= off) incl = ff_add(o, incl);
  }
  ff ex{__shfl_up_sync(0xffffffffu, incl.hi, 1), __shfl_up_sync(0xffffffffu, incl.lo, 1)};
  if (lane == 0) ex = {0.f, 0.f};
  if (lane == 31) sm[warp] = incl;
  __syncthreads();
  ff off{0.f, 0.f}, tot{0.f, 0.f};
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    if (w == warp) off = tot;
    tot = ff_add(tot, sm[w]);
  }
  __syncthreads();
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

// ---------------------------------------------------------------- decision
// Run by the whole block of the last statistics CTA of sequence b.
__device__ void decide_sequence(const VerifyArgs& a, int b) {
  __shared__ float rk[2 * kMaxK + 1];
  __shared__ ff rS[2 * kMaxK + 1];
  __shared__ int rbad[2 * kMaxK + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int K = a.K;
  const int M = a.B * (K + 1);
  const int nrows = 2 * K + 1;

  // combine the chunk partials of every row of the sequence, one warp per row
  for (int r = warp; r < nrows; r += kWarps) {
    const int grow = r <= K ? b * (K + 1) + r : M + b * K + (r - K - 1);
    const ChunkStat* pp = a.stats + static_cast<size_t>(grow) * a.CA;
    float kmax = -INFINITY;
    int bad = 0;
    for (int c = lane; c < a.CA; c += 32) {
      kmax = fmaxf(kmax, __ldcg(&pp[c].k));
      bad |= __ldcg(&pp[c].bad);
    }
    kmax = warp_max(kmax);
    ff s{0.f, 0.f};
    for (int c = lane; c < a.CA; c += 32) {
      const float kc = __ldcg(&pp[c].k);
      const ff sc{__ldcg(&pp[c].s_hi), __ldcg(&pp[c].s_lo)};
      if (sc.hi > 0.f) s = ff_add(s, ff_scale2(sc, static_cast<int>(kc - kmax)));
    }
    s = warp_sum_ff(s);
    bad = __any_sync(0xffffffffu, bad != 0) ? 1 : 0;
    if (lane == 0) {
      rk[r] = kmax;
      rS[r] = s;
      rbad[r] = bad || !(s.hi > 0.f) || !isfinite(s.hi) || !isfinite(kmax);
    }
  }
  __syncthreads();

  if (warp != 0) return;
  const Expo c{a.c_hi, a.c_lo};
  bool tok_ok = true, acc = false;
  int xj = -1;
  float pj = 0.f, qj = 0.f, aj = 0.f;
  if (lane < K) {
    xj = a.x[b * K + lane];
    tok_ok = xj >= 0 && xj < a.V;
    if (tok_ok) {
      const float zp = a.zp[static_cast<size_t>(b * (K + 1) + lane) * a.V + xj];
      const float zq = a.zq[static_cast<size_t>(b * K + lane) * a.V + xj];
      const ff yp = expo(zp, c), yq = expo(zq, c);
      const float lp = (yp.hi - rk[lane]) + yp.lo;          // log2 of S_p * p(x)
      const float lq = (yq.hi - rk[K + 1 + lane]) + yq.lo;  // log2 of S_q * q(x)
      const float Sp = rS[lane].hi, Sq = rS[K + 1 + lane].hi;
      pj = exp2f(lp) / Sp;
      qj = exp2f(lq) / Sq;
      aj = fminf(1.f, exp2f(lp - lq) * (Sq / Sp));
      acc = a.u[b * (K + 1) + lane] < aj;
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

  // positions 0..K (K + 1 <= 33 may exceed the warp: a second pass covers j = 32)
  for (int j = lane; j <= K; j += 32) {
    const bool slot = j < K;  // j == lane whenever slot is true
    a.out_tokens[b * (K + 1) + j] = (!bad && j < n) ? xj : -1;
    if (a.out_debug) {
      float* dbg = a.out_debug + static_cast<size_t>(b * (K + 1) + j) * 6;
      dbg[0] = slot ? pj : 0.f;
      dbg[1] = slot ? qj : 0.f;
      dbg[2] = slot ? aj : 0.f;
      // log sum_v exp(z_v / T) = ln 2 * (k + log2 S)
      dbg[3] = 0.6931471805599453f * (rk[j] + log2f(rS[j].hi));
      dbg[4] = slot ? 0.6931471805599453f * (rk[K + 1 + j] + log2f(rS[K + 1 + j].hi)) : 0.f;
      dbg[5] = 0.f;
    }
  }
  if (lane == 0) {
    a.out_n[b] = bad ? -1 : n;
    if (bad) atomicOr(a.err, (badtok ? kErrTokenRange : 0) | (rowbad ? kErrNonFinite : 0));
    SeqState st;
    st.n = n;
    st.bad = bad ? 1 : 0;
    st.k_p = rk[n];
    st.S_p = make_float2(rS[n].hi, rS[n].lo);
    if (n < K) {
      st.k_q = rk[K + 1 + n];
      st.S_q = make_float2(rS[K + 1 + n].hi, rS[K + 1 + n].lo);
      const ff kap = ff_div(rS[n], rS[K + 1 + n]);
      st.kappa = make_float2(kap.hi, kap.lo);
    } else {
      st.k_q = 0.f;
      st.S_q = make_float2(0.f, 0.f);
      st.kappa = make_float2(0.f, 0.f);
    }
    a.seq[b] = st;
  }
}

// ---------------------------------------------------------------- pass 1
template <bool kVec>
__global__ void __launch_bounds__(kThreads) stats_kernel(const VerifyArgs a) {
  __shared__ float sm_f[kWarps];
  __shared__ ff sm_ff[kWarps];
  __shared__ int sm_i[1];
  const int row = blockIdx.x, chunk = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int M = a.B * (a.K + 1);
  const bool target = row < M;
  const float* z = target ? a.zp + static_cast<size_t>(row) * a.V : a.zq + static_cast<size_t>(row - M) * a.V;
  const int b = target ? row / (a.K + 1) : (row - M) / a.K;
  const Expo c{a.c_hi, a.c_lo};

  float v[kPer];
  unsigned valid;
  load16<kVec>(z, chunk * kChunk + threadIdx.x * kPer, a.V, v, valid);
  ff y[kPer];
  float ymax = -INFINITY;
  int bad = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const bool in = (valid >> i) & 1u;
    bad |= in && !isfinite(v[i]);
    y[i] = expo(v[i], c);
    if (in) ymax = fmaxf(ymax, y[i].hi);
  }
  ymax = warp_max(ymax);
  if (lane == 0) sm_f[warp] = ymax;
  __syncthreads();
  float kc = sm_f[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) kc = fmaxf(kc, sm_f[w]);
  kc = ceilf(kc);
  ff s{0.f, 0.f};
#pragma unroll
  for (int i = 0; i < kPer; ++i)
    if ((valid >> i) & 1u) s = ff_add_f(s, pow2_rel(y[i], kc));
  s = warp_sum_ff(s);
  const int any_bad = __syncthreads_or(bad);
  if (lane == 0) sm_ff[warp] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    ff t = sm_ff[0];
    for (int w = 1; w < kWarps; ++w) t = ff_add(t, sm_ff[w]);
    ChunkStat cs;
    cs.k = kc;
    cs.bad = any_bad;
    cs.s_hi = t.hi;
    cs.s_lo = t.lo;
    a.stats[static_cast<size_t>(row) * a.CA + chunk] = cs;
  }
  const unsigned expected = static_cast<unsigned>((2 * a.K + 1) * a.CA);
  if (!last_block_ticket(&a.tickets_a[b], expected, sm_i)) return;
  decide_sequence(a, b);
}

// ---------------------------------------------------------------- pass 2
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
  const float ep = pow2_rel(expo(zp, R.c), R.k_p);
  if (!R.rej) return ep;
  const float eq = pow2_rel(expo(zq, R.c), R.k_q);
  return fmaxf(0.f, ep - fmaf(R.kh, eq, R.kl * eq));
}

template <bool kVec>
__device__ __forceinline__ void residual_segment(const ResRow& R, int e0, float (&r)[kPer]) {
  float zp[kPer], zq[kPer];
  unsigned valid, vq;
  load16<kVec>(R.zp, e0, R.V, zp, valid);
  if (R.rej) {
    load16<kVec>(R.zq, e0, R.V, zq, vq);
  } else {
#pragma unroll
    for (int i = 0; i < kPer; ++i) zq[i] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) r[i] = ((valid >> i) & 1u) ? residual_term(zp[i], zq[i], R) : 0.f;
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
template <bool kVec>
__device__ void locate_in_chunk(const ResRow& R, int chunk, ff base, ff t, int& y, int& last_pos, ff* sm_ff,
                                int* sm_i) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e0 = chunk * kChunk + threadIdx.x * kPer;
  float r[kPer];
  residual_segment<kVec>(R, e0, r);
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
  __syncthreads();
  y = sm_i[0];
  last_pos = sm_i[kWarps];
  for (int w = 1; w < kWarps; ++w) {
    y = min(y, sm_i[w]);
    last_pos = max(last_pos, sm_i[kWarps + w]);
  }
  __syncthreads();
}

template <bool kVec>
__global__ void __launch_bounds__(kThreads) residual_kernel(const VerifyArgs a) {
  __shared__ ff sm_ff[kWarps];
  __shared__ int sm_i[2 * kWarps];
  __shared__ SeqState st;
  __shared__ ff s_base, s_t, s_S;
  __shared__ int s_chunk;
  const int b = blockIdx.x, chunk = blockIdx.y;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    const SeqState* g = &a.seq[b];
    st.n = __ldcg(&g->n);
    st.bad = __ldcg(&g->bad);
    st.k_p = __ldcg(&g->k_p);
    st.k_q = __ldcg(&g->k_q);
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
  R.c = {a.c_hi, a.c_lo};
  R.k_p = st.k_p;
  R.k_q = st.k_q;
  R.kh = st.kappa.x;
  R.kl = st.kappa.y;
  R.V = a.V;

  {
    float r[kPer];
    residual_segment<kVec>(R, chunk * kChunk + threadIdx.x * kPer, r);
    ff excl, total;
    block_excl_scan_ff({segment_total(r), 0.f}, excl, total, sm_ff);
    if (threadIdx.x == 0) a.res_sums[static_cast<size_t>(b) * a.CB + chunk] = make_float2(total.hi, total.lo);
  }
  if (!last_block_ticket(&a.tickets_b[b], static_cast<unsigned>(a.CB), sm_i)) return;

  const float2* sums = a.res_sums + static_cast<size_t>(b) * a.CB;
  const float u = a.u[b * (K + 1) + K];
  // total residual mass (warp 0, lanes over chunks)
  if (threadIdx.x < 32) {
    ff s{0.f, 0.f};
    for (int i = lane; i < a.CB; i += 32) {
      const float2 v = __ldcg(&sums[i]);
      s = ff_add(s, {v.x, v.y});
    }
    s = warp_sum_ff(s);
    if (lane == 0) s_S = s;
  }
  __syncthreads();
  if (!(s_S.hi > 0.f) && R.rej) {
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
        const float2 w = __ldcg(&sums[i]);
        v = {w.x, w.y};
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
      const ff mass = R.rej ? ff_div(s_S, {st.S_p.x, st.S_p.y}) : ff{1.f, 0.f};
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
  for (int j = 0; j <= K; ++j) {
    const size_t row = static_cast<size_t>(b) * (K + 1) + j;
    const float* pv = a.part_max + row * a.P;
    const int* pi = a.part_idx + row * a.P;
    float bv = -INFINITY;
    int bi = INT_MAX;
    int bad = 0;
    for (int p = threadIdx.x; p < a.P; p += kThreads) {
      const float v = __ldcg(&pv[p]);
      const int i = __ldcg(&pi[p]);
      if (i == -2) {
        bad = 1;
      } else if (v > bv || (v == bv && i < bi)) {
        bv = v;
        bi = i;
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
                                                             float* part_max, int* part_idx) {
  __shared__ float sv[kWarps];
  __shared__ int si[kWarps];
  __shared__ int sb[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int row = blockIdx.x, chunk = blockIdx.y;
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

cudaError_t launch_verify_sampling(const VerifyArgs& a, cudaStream_t stream) {
  const int M = a.B * (a.K + 1);
  const int R = M + a.B * a.K;
  const bool vec = (a.V % 4) == 0;
  const dim3 g1(R, a.CA);
  if (vec)
    stats_kernel<true><<<g1, kThreads, 0, stream>>>(a);
  else
    stats_kernel<false><<<g1, kThreads, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 g2(a.B, a.CB);
  if (vec)
    residual_kernel<true><<<g2, kThreads, 0, stream>>>(a);
  else
    residual_kernel<false><<<g2, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_greedy_finish(const GreedyArgs& a, cudaStream_t stream) {
  greedy_finish_kernel<<<a.B, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_row_argmax(const float* logits, int M, int V, float* part_max, int* part_idx,
                              cudaStream_t stream) {
  const int P = (V + kChunk - 1) / kChunk;
  const dim3 g(M, P);
  if (V % 4 == 0)
    row_argmax_kernel<true><<<g, kThreads, 0, stream>>>(logits, M, V, P, part_max, part_idx);
  else
    row_argmax_kernel<false><<<g, kThreads, 0, stream>>>(logits, M, V, P, part_max, part_idx);
  return cudaGetLastError();
}

}  // namespace sv
