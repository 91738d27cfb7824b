// Tree-shaped candidate verification ("Speculative Decoding: Memverifikasi
// Token Draft secara Paralel", section "Sampling eksak memerlukan aturan
// koreksi").  Declared in include/spec_tree.h.
//
// Sampling: one thread-block cluster of kC CTAs per sequence: 16 or 12 (a
// non-portable size) when that many clusters of all B trees are resident at
// once, else 8.  CTA r owns
// the vocabulary slice [r*S, (r+1)*S) and keeps the current node's target and
// draft rows of that slice in shared memory, as probabilities.  Every
// reduction of the walk -- a node's two softmax normalisers, the residual
// mass after a rejection, the slice masses of the final draw -- is a block
// reduction followed by an exchange of one value per CTA through distributed
// shared memory; every CTA merges the kC values in rank order, so all of
// them reach the same decisions and walk the tree in lockstep.  A rejection
// costs one pass over shared memory and one cluster barrier; the rows of a
// node are read from HBM / L2 once, when the walk reaches it.
//
// The residual after k rejections against the same draft row q is
// max(0, p - lambda_k q) / S'_k with lambda_1 = 1, lambda_{k+1} =
// lambda_k + S'_k and S'_k = sum(max(0, p - lambda_k q)): one scalar per
// rejection instead of a rewritten row.
//
// Greedy: one CTA per sequence reduces the LM head's per-tile argmax
// partials of the rows it visits.
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdlib>

#include "internal.h"
#include "sm103_ptx.cuh"
#include "spec_tree.h"
#include "verify_math.cuh"

namespace sv {
namespace {

constexpr int kTC = 8;            // CTAs per cluster (one cluster per sequence): the portable size
constexpr int kTCMax = 16;        // the largest (non-portable) size
constexpr int kTT = 512;          // threads per CTA
constexpr int kTW = kTT / 32;
constexpr int kMaxSlice = 24576;  // vocabulary entries per CTA
constexpr int kMaxNodes = 256;

struct TreeArgs {
  int B, N, V, S;
  int bulk;  // rows start on 16-byte boundaries (V % 4 == 0): node rows come in by TMA bulk copies
  float c_hi, c_lo;
  const float* zp;  // [B*N][V]
  const float* zq;  // [B*N][V]
  const int32_t* tok;
  const int32_t* par;
  const float* u;
  int32_t* out_tok;
  int32_t* out_path;
  int32_t* out_n;
  int* err;
  const float* pmax;  // greedy: [B*N][P]
  const int* pidx;
  int P;
};

struct TreeShared {
  float4 ex[2][2][kTW];  // cluster exchange: up to two values per warp [pass parity][value][warp]
  int par[kMaxNodes];
  int tok[kMaxNodes];
  int path[kMaxNodes];
  float czp[kMaxNodes], czq[kMaxNodes];  // target / draft logit of each child of the node being loaded
  float4 res, res2;                      // a cluster reduction's result, broadcast to the block
  int res_slot, res_last;
  int flag;
  uint64_t bar;  // completion of the node-row bulk copies
};

// Every cluster reduction of the walk: lane 0 of each warp publishes its
// warp's value in exchange slot [ph][warp], one cluster barrier makes every
// slot of every CTA readable, and warp 0 of each CTA reads all kC * kTW
// values, lane l the consecutive slots l*kPL .. l*kPL + kPL - 1 in (rank,
// warp) order, and merges them in that fixed order: every CTA computes the
// same result.  The barrier of the next reduction (the other parity)
// orders the reuse of the slots and of sh.res.
__device__ __forceinline__ void publish_warp(TreeShared& sh, int ph, float4 v) {
  if ((threadIdx.x & 31) == 0) sh.ex[ph][0][threadIdx.x >> 5] = v;
  cluster_sync();
}

template <int kC>
__device__ __forceinline__ void fetch_lane_slots(TreeShared& sh, int ph, float4 (&f)[kC * kTW / 32], int which = 0) {
  constexpr int kPL = kC * kTW / 32;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < kPL; ++j) {
    const int i = lane * kPL + j;
    f[j] = ld_cluster_f4(cluster_map(&sh.ex[ph][which][i % kTW], static_cast<uint32_t>(i / kTW)));
  }
}

// Warp w's contiguous block [w0, w1) of a slice of cnt entries: every pass
// over a node's rows uses this mapping, so a warp's own scale factors apply
// to everything it reads.
__device__ __forceinline__ void warp_block(int cnt, int& w0, int& w1) {
  const int blk = ((cnt + kTW - 1) / kTW + 31) / 32 * 32;
  w0 = min(cnt, static_cast<int>(threadIdx.x >> 5) * blk);
  w1 = min(cnt, w0 + blk);
}

__device__ __forceinline__ float4 max4(float4 a, float4 b) {
  return make_float4(fmaxf(a.x, b.x), fmaxf(a.y, b.y), fmaxf(a.z, b.z), fmaxf(a.w, b.w));
}

__device__ __forceinline__ float4 warp_max4(float4 v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float4 o{__shfl_xor_sync(0xffffffffu, v.x, off), __shfl_xor_sync(0xffffffffu, v.y, off),
                   __shfl_xor_sync(0xffffffffu, v.z, off), __shfl_xor_sync(0xffffffffu, v.w, off)};
    v = max4(v, o);
  }
  return v;
}

// Cluster-wide componentwise maximum of one float4 per thread.
template <int kC>
__device__ float4 cluster_max4(TreeShared& sh, int ph, float4 v) {
  publish_warp(sh, ph, warp_max4(v));
  if (threadIdx.x < 32) {
    constexpr int kPL = kC * kTW / 32;
    float4 f[kPL];
    fetch_lane_slots<kC>(sh, ph, f);
    float4 m = f[0];
#pragma unroll
    for (int j = 1; j < kPL; ++j) m = max4(m, f[j]);
    m = warp_max4(m);
    if (threadIdx.x == 0) sh.res = m;
  }
  __syncthreads();
  return sh.res;
}

// Cluster-wide float-float sums of two values per thread: (sum a, sum b).
template <int kC>
__device__ void cluster_sum2(TreeShared& sh, int ph, ff& a, ff& b) {
  a = warp_sum_ff(a);
  b = warp_sum_ff(b);
  publish_warp(sh, ph, make_float4(a.hi, a.lo, b.hi, b.lo));
  if (threadIdx.x < 32) {
    constexpr int kPL = kC * kTW / 32;
    float4 f[kPL];
    fetch_lane_slots<kC>(sh, ph, f);
    ff x{f[0].x, f[0].y}, y{f[0].z, f[0].w};
#pragma unroll
    for (int j = 1; j < kPL; ++j) {
      x = ff_add(x, ff{f[j].x, f[j].y});
      y = ff_add(y, ff{f[j].z, f[j].w});
    }
    x = warp_sum_ff(x);
    y = warp_sum_ff(y);
    if (threadIdx.x == 0) sh.res = make_float4(x.hi, x.lo, y.hi, y.lo);
  }
  __syncthreads();
  a = ff{sh.res.x, sh.res.y};
  b = ff{sh.res.z, sh.res.w};
}

struct NodeStats {
  float kp, inv_p, kq, inv_q;  // the row's reference exponents and 1 / normaliser (cluster-wide)
  float ip_w, iq_w;            // this warp's factors: p_v = sp[v] * ip_w, q_v = sq[v] * iq_w
  int bad;
};

// Loads node `node`'s target row (and draft row if need_q) of this CTA's
// slice into shared memory as 2^(z*c - k_w), k_w = ceil of the largest z*c
// of warp w's block (no barrier: each warp reduces its own block), sums the
// block, and merges the (k_w, sum_w) pairs of every warp of the cluster
// into K = max k_w and S = sum of sum_w * 2^(k_w - K) (exact powers of two).
// A non-finite logit, or a row without mass, marks the node bad in every CTA.
template <int kC>
__device__ NodeStats load_node(const TreeArgs& a, TreeShared& sh, float* sp, float* sq, int b, int node, bool need_q,
                               int rank, int& ph, uint32_t& bar_phase, Expo c) {
  const int lane = threadIdx.x & 31;
  const int base = rank * a.S;
  const int cnt = max(0, min(a.S, a.V - base));
  const size_t row = (static_cast<size_t>(b) * a.N + node) * a.V + base;
  int bad_p = 0, bad_q = 0;
  if (a.bulk) {
    // the slice of both rows by TMA; every thread of the CTA finished with the
    // previous node's rows at the cluster barrier that ended its last pass
    if (cnt > 0) {
      if (threadIdx.x == 0) {
        const uint32_t bytes = static_cast<uint32_t>(cnt) * 4u;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&sh.bar, need_q ? 2u * bytes : bytes);
        bulk_load(sp, a.zp + row, bytes, &sh.bar);
        if (need_q) bulk_load(sq, a.zq + row, bytes, &sh.bar);
      }
      if (!mbar_wait(&sh.bar, bar_phase)) {
        bad_p = 1;  // reported through the cluster exchange, so every CTA sees it
        if (threadIdx.x == 0) atomicOr(a.err, kErrTimeout);
        (void)mbar_wait(&sh.bar, bar_phase);  // one more bounded wait for the copies in flight
      }
      bar_phase ^= 1u;
    }
  } else {
    for (int i = threadIdx.x; i < cnt; i += kTT) {
      sp[i] = __ldcg(a.zp + row + i);
      if (need_q) sq[i] = __ldcg(a.zq + row + i);
    }
  }
  __syncthreads();
  int w0, w1;
  warp_block(cnt, w0, w1);
  // the block's largest exponent per row
  float mp = -INFINITY, mq = -INFINITY;
  if (!bad_p) {
    for (int i = w0 + lane; i < w1; i += 32) {
      const float h = expo_hi(sp[i], c);
      if (!isfinite(h)) bad_p = 1; else mp = fmaxf(mp, h);
      if (need_q) {
        const float g = expo_hi(sq[i], c);
        if (!isfinite(g)) bad_q = 1; else mq = fmaxf(mq, g);
      }
    }
  }
  const float kp_w = ceilf(warp_max_f(mp)), kq_w = ceilf(warp_max_f(mq));
  // 2^(z*c - k_w) in place and the block sums
  float ph_ = 0.f, pl = 0.f, qh = 0.f, ql = 0.f;
  if (kp_w != -INFINITY) {
    for (int i = w0 + lane; i < w1; i += 32) {
      const float e = pow2_rel(sp[i], c, kp_w);
      sp[i] = e;
      ff_accumulate(ph_, pl, e);
    }
  }
  if (need_q && kq_w != -INFINITY) {
    for (int i = w0 + lane; i < w1; i += 32) {
      const float f = pow2_rel(sq[i], c, kq_w);
      sq[i] = f;
      ff_accumulate(qh, ql, f);
    }
  }
  const ff sp_w = warp_sum_ff(ff_norm(ph_, pl)), sq_w = warp_sum_ff(ff_norm(qh, ql));
  const int bp = __any_sync(0xffffffffu, bad_p != 0), bq = __any_sync(0xffffffffu, bad_q != 0);
  if (lane == 0) {
    sh.ex[ph][0][threadIdx.x >> 5] = make_float4(kp_w, sp_w.hi, sp_w.lo, bp ? 1.f : 0.f);
    sh.ex[ph][1][threadIdx.x >> 5] = make_float4(kq_w, sq_w.hi, sq_w.lo, bq ? 1.f : 0.f);
  }
  cluster_sync();
  if (threadIdx.x < 32) {
    constexpr int kPL = kC * kTW / 32;
    float4 fp[kPL], fq[kPL];
    fetch_lane_slots<kC>(sh, ph, fp, 0);
    fetch_lane_slots<kC>(sh, ph, fq, 1);
    float4 m = make_float4(fp[0].x, fq[0].x, fp[0].w, fq[0].w);
#pragma unroll
    for (int j = 1; j < kPL; ++j) m = max4(m, make_float4(fp[j].x, fq[j].x, fp[j].w, fq[j].w));
    m = warp_max4(m);
    ff Sp{0.f, 0.f}, Sq{0.f, 0.f};
#pragma unroll
    for (int j = 0; j < kPL; ++j) {
      const float a_ = pow2_nonpos(fp[j].x - m.x), b_ = pow2_nonpos(fq[j].x - m.y);
      Sp = ff_add(Sp, ff{fp[j].y * a_, fp[j].z * a_});
      Sq = ff_add(Sq, ff{fq[j].y * b_, fq[j].z * b_});
    }
    Sp = warp_sum_ff(Sp);
    Sq = warp_sum_ff(Sq);
    if (threadIdx.x == 0) {
      sh.res = m;
      sh.res2 = make_float4(Sp.hi, Sp.lo, Sq.hi, Sq.lo);
    }
  }
  __syncthreads();
  ph ^= 1;
  const float4 m = sh.res, S = sh.res2;
  NodeStats st;
  st.bad = m.z != 0.f || m.x == -INFINITY || !(S.x > 0.f) || !isfinite(S.x) ||
           (need_q && (m.w != 0.f || m.y == -INFINITY || !(S.z > 0.f) || !isfinite(S.z)));
  st.kp = m.x;
  st.kq = need_q ? m.y : 0.f;
  st.inv_p = st.bad ? 0.f : 1.f / (S.x + S.y);
  st.inv_q = (st.bad || !need_q) ? 0.f : 1.f / (S.z + S.w);
  st.ip_w = st.inv_p * pow2_nonpos(kp_w - st.kp);
  st.iq_w = need_q ? st.inv_q * pow2_nonpos(kq_w - st.kq) : 0.f;
  return st;
}

// r_v = max(0, p_v - lam q_v) (lam = 0: p_v), p_v = sp[v]*ip, q_v = sq[v]*iq.
__device__ __forceinline__ float rval(float e_p, float e_q, float ip, float iq, float lam) {
  return lam > 0.f ? fmaxf(0.f, e_p * ip - lam * (e_q * iq)) : e_p * ip;
}

// Mass of max(0, p - lam q) over the whole row.
template <int kC>
__device__ ff residual_mass(const TreeArgs& a, TreeShared& sh, const float* sp, const float* sq, const NodeStats& st,
                            float lam, int rank, int& ph) {
  const int cnt = max(0, min(a.S, a.V - rank * a.S));
  int w0, w1;
  warp_block(cnt, w0, w1);
  float hi = 0.f, lo = 0.f;
  for (int i = w0 + static_cast<int>(threadIdx.x & 31); i < w1; i += 32)
    ff_accumulate(hi, lo, rval(sp[i], sq[i], st.ip_w, st.iq_w, lam));
  ff tot = ff_norm(hi, lo), none{0.f, 0.f};
  cluster_sum2<kC>(sh, ph, tot, none);
  ph ^= 1;
  return tot;
}

__device__ __forceinline__ int warp_max_i(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

// Inverse-CDF draw over max(0, p - lam q) (lam = 0: over p) with uniform u,
// written to out_tok[b][pos] by the warp that finds it.  Warp w of each CTA
// covers the contiguous block [w*blk, (w+1)*blk) of its slice, so the
// (rank, warp) block masses in that order are coarse steps of the CDF: one
// cluster reduction scans them for the block holding t = u*S, and the warp
// owning that block scans it 32 tokens at a time.
template <int kC>
__device__ void draw(const TreeArgs& a, TreeShared& sh, const float* sp, const float* sq, const NodeStats& st,
                     float lam, float u, int rank, int& ph, int b, int pos) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int base = rank * a.S;
  const int cnt = max(0, min(a.S, a.V - base));
  const float ip = st.ip_w, iq = st.iq_w;
  int w0, w1;
  warp_block(cnt, w0, w1);
  float hi = 0.f, lo = 0.f;
  int lastp = -1;
  for (int i = w0 + lane; i < w1; i += 32) {
    const float d = rval(sp[i], lam > 0.f ? sq[i] : 0.f, ip, iq, lam);
    if (d > 0.f) {
      ff_accumulate(hi, lo, d);
      lastp = base + i;
    }
  }
  const ff wsum = warp_sum_ff(ff_norm(hi, lo));
  lastp = warp_max_i(lastp);
  publish_warp(sh, ph, make_float4(wsum.hi, wsum.lo, __int_as_float(lastp), 0.f));
  if (threadIdx.x < 32) {
    constexpr int kPL = kC * kTW / 32;
    float4 f[kPL];
    fetch_lane_slots<kC>(sh, ph, f);
    ff tot{0.f, 0.f};
    int last = -1;
#pragma unroll
    for (int j = 0; j < kPL; ++j) {
      tot = ff_add(tot, ff{f[j].x, f[j].y});
      last = max(last, __float_as_int(f[j].z));
    }
    // exclusive prefix of the lanes' totals; S the total
    ff incl = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const ff o{__shfl_up_sync(0xffffffffu, incl.hi, off), __shfl_up_sync(0xffffffffu, incl.lo, off)};
      if (lane >= off) incl = ff_add(o, incl);
    }
    ff ex{__shfl_up_sync(0xffffffffu, incl.hi, 1), __shfl_up_sync(0xffffffffu, incl.lo, 1)};
    if (lane == 0) ex = {0.f, 0.f};
    const ff S{__shfl_sync(0xffffffffu, incl.hi, 31), __shfl_sync(0xffffffffu, incl.lo, 31)};
    const ff t = ff_mul_f(S, u);
    // this lane's first slot whose inclusive prefix exceeds t, and the prefix before it
    ff run = ex, pre{0.f, 0.f};
    int hit = -1;
#pragma unroll
    for (int j = 0; j < kPL; ++j) {
      const ff nxt = ff_add(run, ff{f[j].x, f[j].y});
      if (hit < 0 && ff_gt(nxt, t)) {
        hit = j;
        pre = run;
      }
      run = nxt;
    }
    const unsigned hm = __ballot_sync(0xffffffffu, hit >= 0);
    last = warp_max_i(last);
    int slot = -1;
    float4 r = make_float4(0.f, 0.f, t.hi, t.lo);
    if (hm) {
      const int src = __ffs(hm) - 1;
      slot = src * kPL + __shfl_sync(0xffffffffu, hit, src);
      r.x = __shfl_sync(0xffffffffu, pre.hi, src);
      r.y = __shfl_sync(0xffffffffu, pre.lo, src);
    }
    if (lane == 0) {
      sh.res_slot = slot;
      sh.res_last = last;
      sh.res = r;
    }
  }
  __syncthreads();
  int32_t* out = a.out_tok + static_cast<size_t>(b) * a.N + pos;
  const int slot = sh.res_slot;
  if (slot < 0) {  // rounding left t past every block: the last token with mass
    if (rank == 0 && threadIdx.x == 0) *out = sh.res_last;
    return;
  }
  if (rank != slot / kTW || warp != slot % kTW) return;
  const ff tl = ff_add(ff{sh.res.z, sh.res.w}, ff{-sh.res.x, -sh.res.y});
  ff run{0.f, 0.f};
  int y = -1;
  for (int i0 = w0; i0 < w1 && y < 0; i0 += 32) {
    const int i = i0 + lane;
    const float d = i < w1 ? rval(sp[i], lam > 0.f ? sq[i] : 0.f, ip, iq, lam) : 0.f;
    ff incl{d, 0.f};
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const ff o{__shfl_up_sync(0xffffffffu, incl.hi, off), __shfl_up_sync(0xffffffffu, incl.lo, off)};
      if (lane >= off) incl = ff_add(o, incl);
    }
    const unsigned h = __ballot_sync(0xffffffffu, i < w1 && ff_gt(ff_add(run, incl), tl));
    if (h) y = base + i0 + __ffs(h) - 1;
    const ff tot{__shfl_sync(0xffffffffu, incl.hi, 31), __shfl_sync(0xffffffffu, incl.lo, 31)};
    run = ff_add(run, tot);
  }
  // (rounding left t past this block's last step: its last token with mass)
  if (lane == 0) *out = y >= 0 ? y : lastp;
}

template <int kC>
__global__ void __launch_bounds__(kTT, 1) tree_sample_kernel(const TreeArgs a) {
  __shared__ TreeShared sh;
  extern __shared__ float4 dyn[];
  float* sp = reinterpret_cast<float*>(dyn);
  float* sq = sp + a.S;
  const int rank = static_cast<int>(cluster_ctarank());
  const int b = blockIdx.x / kC;
  const Expo c{a.c_hi, a.c_lo};
  griddep_wait();
  // tree structure and validity
  if (threadIdx.x == 0) {
    sh.flag = 0;
    mbar_init(&sh.bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  uint32_t bar_phase = 0;
  for (int i = threadIdx.x; i < a.N; i += kTT) {
    const int p = a.par[static_cast<size_t>(b) * a.N + i];
    const int t = a.tok[static_cast<size_t>(b) * a.N + i];
    sh.par[i] = p;
    sh.tok[i] = t;
    const bool ok = i == 0 ? p == -1 : (p >= 0 && p < i && t >= 0 && t < a.V);
    if (!ok) atomicOr(&sh.flag, kErrTokenRange);
  }
  __syncthreads();
  int bad = sh.flag;
  int ph = 0;
  int cur = 0, n = 0;
  auto next_child = [&](int node, int after) {
    for (int i = after + 1; i < a.N; ++i)
      if (sh.par[i] == node) return i;
    return -1;
  };
  while (!bad) {
    const int first = next_child(cur, 0);
    {
      // the children's logits for their acceptance tests, in flight while
      // the node's rows arrive (load_node's barrier publishes them)
      const size_t crow = (static_cast<size_t>(b) * a.N + cur) * a.V;
      for (int i = threadIdx.x; i < a.N; i += kTT) {
        if (sh.par[i] == cur) {
          sh.czp[i] = __ldcg(a.zp + crow + sh.tok[i]);
          sh.czq[i] = __ldcg(a.zq + crow + sh.tok[i]);
        }
      }
    }
    const NodeStats st = load_node<kC>(a, sh, sp, sq, b, cur, first >= 0, rank, ph, bar_phase, c);
    if (st.bad) {
      bad = kErrNonFinite;
      break;
    }
    float lam = 0.f;       // 0: r = p
    ff sres = {1.f, 0.f};  // mass of max(0, p - lam q) (1 for r = p)
    int accepted = -1;
    for (int ch = first; ch >= 0; ch = next_child(cur, ch)) {
      const float px = pow2_rel(sh.czp[ch], c, st.kp) * st.inv_p;
      const float qx = pow2_rel(sh.czq[ch], c, st.kq) * st.inv_q;
      const float rx = lam > 0.f ? fmaxf(0.f, px - lam * qx) / (sres.hi + sres.lo) : px;
      const float acc = qx > 0.f ? fminf(1.f, rx / qx) : (rx > 0.f ? 1.f : 0.f);
      if (__ldcg(a.u + static_cast<size_t>(b) * a.N + ch) < acc) {
        accepted = ch;
        break;
      }
      const float lam_new = lam > 0.f ? lam + (sres.hi + sres.lo) : 1.f;
      const ff s_new = residual_mass<kC>(a, sh, sp, sq, st, lam_new, rank, ph);
      if (s_new.hi > 0.f) {
        lam = lam_new;
        sres = s_new;
      }  // no mass left: the working distribution stays as it was
    }
    const float u0 = __ldcg(a.u + static_cast<size_t>(b) * a.N);
    if (accepted < 0) {
      draw<kC>(a, sh, sp, sq, st, lam, u0, rank, ph, b, n);
      break;
    }
    sh.path[n++] = accepted;  // every thread writes the same value
    cur = accepted;
    if (next_child(cur, 0) < 0) {
      const NodeStats sb = load_node<kC>(a, sh, sp, sq, b, cur, false, rank, ph, bar_phase, c);
      if (sb.bad) {
        bad = kErrNonFinite;
        break;
      }
      draw<kC>(a, sh, sp, sq, sb, 0.f, u0, rank, ph, b, n);
      break;
    }
  }
  __syncthreads();
  if (rank == 0) {
    const size_t o = static_cast<size_t>(b) * a.N;
    for (int i = threadIdx.x; i < a.N; i += kTT) {
      int tv = -1, pv = -1;
      if (!bad && i < n) {
        pv = sh.path[i];
        tv = sh.tok[pv];
      }
      if (bad || i != n) a.out_tok[o + i] = tv;  // position n: the drawn token, written by the warp that drew it
      a.out_path[o + i] = pv;
    }
    if (threadIdx.x == 0) {
      a.out_n[b] = bad ? -1 : n;
      if (bad) atomicOr(a.err, bad);
    }
  }
  cluster_sync();  // no CTA leaves while another may still read its shared memory
}

// ---------------------------------------------------------------- greedy
__global__ void __launch_bounds__(kTT) tree_greedy_kernel(const TreeArgs a) {
  __shared__ TreeShared sh;
  __shared__ float sv_[kTW];
  __shared__ int si_[kTW], sb_[kTW];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = blockIdx.x;
  griddep_wait();
  if (threadIdx.x == 0) sh.flag = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < a.N; i += kTT) {
    const int p = a.par[static_cast<size_t>(b) * a.N + i];
    const int t = a.tok[static_cast<size_t>(b) * a.N + i];
    sh.par[i] = p;
    sh.tok[i] = t;
    const bool ok = i == 0 ? p == -1 : (p >= 0 && p < i && t >= 0 && t < a.V);
    if (!ok) atomicOr(&sh.flag, kErrTokenRange);
  }
  __syncthreads();
  int bad = sh.flag;
  int cur = 0, n = 0, y = -1;
  while (!bad) {
    const size_t row = static_cast<size_t>(b) * a.N + cur;
    const float* pv = a.pmax + row * a.P;
    const int* pi = a.pidx + row * a.P;
    float bv = -INFINITY;
    int bi = INT_MAX, bb = 0;
    for (int p = threadIdx.x; p < a.P; p += kTT) {
      const float v = __ldcg(pv + p);
      const int ix = __ldcg(pi + p);
      if (ix == -2) bb = 1;
      else if (v > bv || (v == bv && ix < bi)) {
        bv = v;
        bi = ix;
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
    bb = __any_sync(0xffffffffu, bb) ? 1 : 0;
    if (lane == 0) {
      sv_[warp] = bv;
      si_[warp] = bi;
      sb_[warp] = bb;
    }
    __syncthreads();
    float v0 = sv_[0];
    int i0 = si_[0], b0 = sb_[0];
    for (int w = 1; w < kTW; ++w) {
      b0 |= sb_[w];
      if (sv_[w] > v0 || (sv_[w] == v0 && si_[w] < i0)) {
        v0 = sv_[w];
        i0 = si_[w];
      }
    }
    __syncthreads();
    if (b0 || i0 == INT_MAX) {
      bad = kErrNonFinite;
      break;
    }
    int nxt = -1;
    for (int i = 1; i < a.N; ++i)
      if (sh.par[i] == cur && sh.tok[i] == i0) {
        nxt = i;
        break;
      }
    if (nxt < 0) {
      y = i0;
      break;
    }
    sh.path[n++] = nxt;
    cur = nxt;
  }
  __syncthreads();
  const size_t o = static_cast<size_t>(b) * a.N;
  for (int i = threadIdx.x; i < a.N; i += kTT) {
    int tv = -1, pv = -1;
    if (!bad) {
      if (i < n) {
        pv = sh.path[i];
        tv = sh.tok[pv];
      } else if (i == n) {
        tv = y;
      }
    }
    a.out_tok[o + i] = tv;
    a.out_path[o + i] = pv;
  }
  if (threadIdx.x == 0) {
    a.out_n[b] = bad ? -1 : n;
    if (bad) atomicOr(a.err, bad);
  }
}

// ---------------------------------------------------------------- host side
size_t round_up(size_t x) { return (x + 255) / 256 * 256; }

bool tree_dims_ok(const spec_tree_dims& d, bool need_head) {
  if (d.B < 1 || d.N < 1 || d.N > kMaxNodes || d.V < 1 || d.V > kTC * kMaxSlice) return false;
  if (static_cast<long long>(d.B) * d.N > (1ll << 24)) return false;
  if (need_head && (d.d < 8 || d.d % 8 != 0 || d.d > (1 << 20))) return false;
  return true;
}

struct TreeLayout {
  size_t logits = 0, pmax = 0, pidx = 0, total = 0;
  int P = 0;
};

// [0, 256): error word; then the logits (sampling, when kept here) or the
// argmax partials (greedy).
TreeLayout tree_layout(const spec_tree_dims& d, bool greedy, bool logits_in_ws, bool from_logits) {
  TreeLayout L;
  size_t off = 256;
  const size_t M = static_cast<size_t>(d.B) * d.N;
  if (greedy) {
    L.P = from_logits ? (d.V + kChunk - 1) / kChunk : (d.V + kHeadTileV - 1) / kHeadTileV;
    L.pmax = off;
    off += round_up(sizeof(float) * M * L.P);
    L.pidx = off;
    off += round_up(sizeof(int) * M * L.P);
  } else if (logits_in_ws) {
    L.logits = off;
    off += round_up(sizeof(float) * M * d.V);
  }
  L.total = off;
  return L;
}

bool aligned(const void* p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

spec_status check_tree_args(const spec_tree_dims& d, float T, const float* draft_logits, const int32_t* tokens,
                            const int32_t* parents, const float* uniforms, const int32_t* out_tokens,
                            const int32_t* out_path, const int32_t* out_n) {
  if (!(T >= 0.f) || !std::isfinite(T)) return SPEC_ERR_ARG;
  if (!tokens || !parents || !out_tokens || !out_path || !out_n) return SPEC_ERR_ARG;
  if (T > 0.f && (!draft_logits || !uniforms)) return SPEC_ERR_ARG;
  if (draft_logits && !aligned(draft_logits, 16)) return SPEC_ERR_ALIGN;
  const uintptr_t any4 = reinterpret_cast<uintptr_t>(tokens) | reinterpret_cast<uintptr_t>(parents) |
                         reinterpret_cast<uintptr_t>(out_tokens) | reinterpret_cast<uintptr_t>(out_path) |
                         reinterpret_cast<uintptr_t>(out_n) | reinterpret_cast<uintptr_t>(uniforms);
  if (any4 & 3u) return SPEC_ERR_ALIGN;
  return SPEC_OK;
}

TreeArgs tree_args(const spec_tree_dims& d, float T, const float* zp, const float* zq, const int32_t* tokens,
                   const int32_t* parents, const float* uniforms, int32_t* out_tokens, int32_t* out_path,
                   int32_t* out_n, int* err) {
  TreeArgs a;
  a.B = d.B;
  a.N = d.N;
  a.V = d.V;
  a.S = ((d.V + kTC - 1) / kTC + 3) / 4 * 4;
  a.bulk = d.V % 4 == 0 && (reinterpret_cast<uintptr_t>(zp) & 15u) == 0 && (reinterpret_cast<uintptr_t>(zq) & 15u) == 0;
  if (T > 0.f) exponent_constant(T, &a.c_hi, &a.c_lo); else a.c_hi = a.c_lo = 0.f;
  a.zp = zp;
  a.zq = zq;
  a.tok = tokens;
  a.par = parents;
  a.u = uniforms;
  a.out_tok = out_tokens;
  a.out_path = out_path;
  a.out_n = out_n;
  a.err = err;
  a.pmax = nullptr;
  a.pidx = nullptr;
  a.P = 0;
  return a;
}

// One cluster of kC CTAs per tree, a programmatic dependent of the LM head;
// `probe` asks instead how many such clusters can be resident at once.
template <int kC>
cudaError_t tree_sample_launch(TreeArgs a, cudaStream_t s, int* probe) {
  a.S = ((a.V + kC - 1) / kC + 3) / 4 * 4;  // slice per CTA, whole 16-byte units
  const size_t smem = 2u * sizeof(float) * static_cast<size_t>(a.S);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B * kC);
  cfg.blockDim = dim3(kTT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (probe) {
    *probe = 0;
    const int max_smem = 2 * static_cast<int>(sizeof(float)) * kMaxSlice;
    cudaError_t e = cudaFuncSetAttribute(tree_sample_kernel<kC>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (e == cudaSuccess && kC > 8)
      e = cudaFuncSetAttribute(tree_sample_kernel<kC>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      return kC > 8 ? cudaSuccess : e;  // the portable size must work
    }
    cfg.gridDim = dim3(kC);
    cfg.numAttrs = 1;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, tree_sample_kernel<kC>, &cfg);
    if (e != cudaSuccess) (void)cudaGetLastError();
    *probe = e == cudaSuccess ? clusters : 0;
    return cudaSuccess;
  }
  return cudaLaunchKernelEx(&cfg, tree_sample_kernel<kC>, a);
}

cudaError_t launch_tree_sample(const TreeArgs& a, const DeviceInfo& dev, cudaStream_t s) {
  // per device: resident clusters of 16, 12 and 8 CTAs (probed once, at the
  // largest slices any call asks for); ready[] set after the probe
  static int fit[64][3];
  static bool ready[64] = {false};
  if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
  if (!ready[dev.device]) {
    TreeArgs pa = a;
    pa.V = kTC * kMaxSlice;
    cudaError_t e = tree_sample_launch<kTCMax>(pa, s, &fit[dev.device][0]);
    if (e == cudaSuccess) e = tree_sample_launch<12>(pa, s, &fit[dev.device][1]);
    if (e == cudaSuccess) e = tree_sample_launch<kTC>(pa, s, &fit[dev.device][2]);
    if (e != cudaSuccess) return e;
    ready[dev.device] = true;
  }
  // SPEC_TREE_CLUSTER_CTAS = 8, 12 or 16 forces that size where one such
  // cluster fits (the tests run every size against the oracle this way)
  if (const char* force = std::getenv("SPEC_TREE_CLUSTER_CTAS")) {
    const int f = std::atoi(force);
    if (f == 16 && fit[dev.device][0] > 0) return tree_sample_launch<kTCMax>(a, s, nullptr);
    if (f == 12 && fit[dev.device][1] > 0) return tree_sample_launch<12>(a, s, nullptr);
    if (f == 8) return tree_sample_launch<kTC>(a, s, nullptr);
  }
  // the largest cluster of which all B trees are resident at once (a tree
  // that waits for another tree's walk to end costs a whole walk); the
  // portable 8 otherwise
  if (a.B <= fit[dev.device][0]) return tree_sample_launch<kTCMax>(a, s, nullptr);
  if (a.B <= fit[dev.device][1]) return tree_sample_launch<12>(a, s, nullptr);
  return tree_sample_launch<kTC>(a, s, nullptr);
}

}  // namespace
}  // namespace sv

extern "C" {

size_t spec_tree_workspace_bytes(spec_tree_dims dims, float temperature, int32_t logits_in_workspace) {
  if (!sv::tree_dims_ok(dims, false) || !(temperature >= 0.f) || !std::isfinite(temperature)) return 0;
  return sv::tree_layout(dims, temperature == 0.f, logits_in_workspace != 0, false).total;
}

spec_status spec_tree_verify(const void* hidden, const void* W_lm, const float* draft_logits, const int32_t* tokens,
                             const int32_t* parents, const float* uniforms, float temperature, int32_t* out_tokens,
                             int32_t* out_path, int32_t* out_num_accepted, spec_tree_dims dims, void* workspace,
                             size_t workspace_bytes, float* out_target_logits, spec_stream_t stream) {
  using namespace sv;
  if (!tree_dims_ok(dims, true)) return SPEC_ERR_DIMS;
  if (!hidden || !W_lm) return SPEC_ERR_ARG;
  if (!aligned(hidden, 16) || !aligned(W_lm, 16)) return SPEC_ERR_ALIGN;
  spec_status st = check_tree_args(dims, temperature, draft_logits, tokens, parents, uniforms, out_tokens, out_path,
                                   out_num_accepted);
  if (st != SPEC_OK) return st;
  const bool greedy = temperature == 0.f;
  if (greedy && out_target_logits) return SPEC_ERR_ARG;
  if (out_target_logits && !aligned(out_target_logits, 16)) return SPEC_ERR_ALIGN;
  const TreeLayout L = tree_layout(dims, greedy, !greedy && !out_target_logits, false);
  if (!workspace || workspace_bytes < L.total) return SPEC_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return SPEC_ERR_ALIGN;
  DeviceInfo dev;
  const int ds = current_device(dev);
  if (ds != SPEC_OK) return static_cast<spec_status>(ds);
  char* ws = static_cast<char*>(workspace);
  int* err = reinterpret_cast<int*>(ws);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int M = dims.B * dims.N;
  bool enc_fail = false;
  if (greedy) {
    float* pmax = reinterpret_cast<float*>(ws + L.pmax);
    int* pidx = reinterpret_cast<int*>(ws + L.pidx);
    const cudaError_t e = launch_head(hidden, W_lm, M, dims.d, dims.V, HeadOut::kArgmax, nullptr, pmax, pidx, nullptr,
                                      err, true, dev, s, &enc_fail);
    if (enc_fail || e != cudaSuccess) return SPEC_ERR_CUDA;
    TreeArgs a = tree_args(dims, 0.f, nullptr, nullptr, tokens, parents, nullptr, out_tokens, out_path,
                           out_num_accepted, err);
    a.pmax = pmax;
    a.pidx = pidx;
    a.P = L.P;
    return launch_dependent(tree_greedy_kernel, dim3(dims.B), dim3(kTT), s, a) == cudaSuccess ? SPEC_OK
                                                                                              : SPEC_ERR_CUDA;
  }
  float* logits = out_target_logits ? out_target_logits : reinterpret_cast<float*>(ws + L.logits);
  const cudaError_t e = launch_head(hidden, W_lm, M, dims.d, dims.V, HeadOut::kLogits, logits, nullptr, nullptr,
                                    nullptr, err, true, dev, s, &enc_fail);
  if (enc_fail || e != cudaSuccess) return SPEC_ERR_CUDA;
  const TreeArgs a = tree_args(dims, temperature, logits, draft_logits, tokens, parents, uniforms, out_tokens,
                               out_path, out_num_accepted, err);
  return launch_tree_sample(a, dev, s) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status spec_tree_verify_from_logits(const float* target_logits, const float* draft_logits,
                                         const int32_t* tokens, const int32_t* parents, const float* uniforms,
                                         float temperature, int32_t* out_tokens, int32_t* out_path,
                                         int32_t* out_num_accepted, spec_tree_dims dims, void* workspace,
                                         size_t workspace_bytes, spec_stream_t stream) {
  using namespace sv;
  if (!tree_dims_ok(dims, false)) return SPEC_ERR_DIMS;
  if (!target_logits) return SPEC_ERR_ARG;
  if (!aligned(target_logits, 16)) return SPEC_ERR_ALIGN;
  spec_status st = check_tree_args(dims, temperature, draft_logits, tokens, parents, uniforms, out_tokens, out_path,
                                   out_num_accepted);
  if (st != SPEC_OK) return st;
  const bool greedy = temperature == 0.f;
  const TreeLayout L = tree_layout(dims, greedy, false, true);
  if (!workspace || workspace_bytes < L.total) return SPEC_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return SPEC_ERR_ALIGN;
  DeviceInfo dev;
  const int ds = current_device(dev);
  if (ds != SPEC_OK) return static_cast<spec_status>(ds);
  char* ws = static_cast<char*>(workspace);
  int* err = reinterpret_cast<int*>(ws);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int M = dims.B * dims.N;
  if (greedy) {
    float* pmax = reinterpret_cast<float*>(ws + L.pmax);
    int* pidx = reinterpret_cast<int*>(ws + L.pidx);
    if (launch_row_argmax(target_logits, M, dims.V, pmax, pidx, err, s) != cudaSuccess) return SPEC_ERR_CUDA;
    TreeArgs a = tree_args(dims, 0.f, target_logits, nullptr, tokens, parents, nullptr, out_tokens, out_path,
                           out_num_accepted, err);
    a.pmax = pmax;
    a.pidx = pidx;
    a.P = L.P;
    return launch_dependent(tree_greedy_kernel, dim3(dims.B), dim3(kTT), s, a) == cudaSuccess ? SPEC_OK
                                                                                              : SPEC_ERR_CUDA;
  }
  if (cudaMemsetAsync(err, 0, sizeof(int), s) != cudaSuccess) return SPEC_ERR_CUDA;
  const TreeArgs a = tree_args(dims, temperature, target_logits, draft_logits, tokens, parents, uniforms, out_tokens,
                               out_path, out_num_accepted, err);
  return launch_tree_sample(a, dev, s) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // extern "C"
