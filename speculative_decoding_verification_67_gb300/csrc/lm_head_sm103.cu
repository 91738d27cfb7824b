// LM-head contraction on the 5th-generation tensor cores (sm_103a).
//
// logits[m][v] = sum_k hidden[m][k] * W[v][k]   (bf16 in, f32 accumulate)
//
// The step this serves scores all drafted positions of all sequences in one
// pass over the LM-head weight (page "quochung.cyou" A.I article, sections
// "Hidden state" and "Tại sao target kiểm tra được nhiều vị trí trong một
// lần?": the weight is read once and used for every candidate position).
// With M = B*(K+1) small, the weight stream is the whole cost, so the kernel
// is organised around reading W exactly once at HBM speed:
//
//  * swap-AB: a tile is 128 vocabulary rows (the MMA's M = 128 operand, A)
//    times N positions (the MMA's N operand, B, N = M rounded up, at most
//    256 per position chunk); the f32 accumulator lives in TMEM;
//  * persistent CTAs, one per SM; each walks tiles tile = blockIdx.x +
//    i*gridDim.x; position chunks of one vocabulary tile are adjacent in
//    that order so that, when M needs several chunks, the CTAs reading the
//    same W rows run together and share them through L2;
//  * warp roles: warp 0 issues TMA loads (W tile 128x64 with an evict-first
//    L2 hint, hidden tile Nx64 with evict-last), warp 1 allocates TMEM and
//    issues tcgen05.mma from one thread, the epilogue warps drain TMEM
//    (tcgen05.ld) and write the f32 logits, per-tile (max, lowest argmax)
//    partials for the greedy path, or the logits plus the softmax(z/T)
//    normaliser partials of every target row (the epilogue holds each logit
//    in a register already, so the statistics cost no extra pass over the
//    logits), while two side warps reduce the draft logits to the same
//    partials, hidden under the weight stream (or under the MMAs, above 64
//    positions, when they fit the head's run);
//  * precise accumulation everywhere: the tensor core never accumulates
//    over the whole hidden size.  Up to 64 positions (head_kernel) every
//    four 64-wide hidden blocks go into a fresh TMEM slot (4 slots rotate)
//    and the epilogue adds the slot results in f32 registers, so the tensor
//    core's own accumulation spans 256 products; above 64 positions
//    (head_large_kernel, further down) groups of 32 blocks (2048 products)
//    alternate between two slots.  An accumulator over the whole hidden size
//    moved ~0.24 % of the sampling step's inverse-CDF draws at d = 8192
//    against fp64 logits; 1024-product groups kept that ~0.02 %, 2048-product
//    groups (2.5 % faster on the tensor-bound shapes) ~0.03 %;
//  * every wait is bounded; a timeout sets the error word, drains the copies
//    in flight and frees TMEM before returning.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <mutex>

#include "internal.h"
#include "sm103_ptx.cuh"
#include "verify_math.cuh"

namespace sv {
namespace {

constexpr int kThreads = 256;  // 8 warps: producer, MMA, 4 epilogue, 2 draft statistics
constexpr uint32_t kABytes = kHeadTileV * kHeadTileK * 2;  // 16 KB W tile per stage
constexpr uint32_t kBarrierBytes = 512;
constexpr uint32_t kArgmaxSmallBytes = 2 * 4 * 256 * 4;    // greedy scratch: [4 warps][256] values and indices
constexpr int kSlotsPrecise = 4;
constexpr int kGroupPrecise = 4;  // hidden blocks accumulated per TMEM slot (precise scheme)

constexpr int kModeLogits = static_cast<int>(HeadOut::kLogits);
constexpr int kModeArgmax = static_cast<int>(HeadOut::kArgmax);
constexpr int kModeStats = static_cast<int>(HeadOut::kStats);

struct HeadParams {
  int M, d, V;
  int streamk, groups;          // stream-K schedule; units (slot groups) per tile
  int gkb;                      // hidden blocks per TMEM slot (precise schemes)
  float* fix;                   // [grid][64][128] partial sums handed to a tile's first CTA
  unsigned long long* flags;    // [grid][4] = epoch once the CTA's quadrant's sums are stored
  unsigned long long epoch;     // unique per launch
  int N, num_chunks, num_vt, num_tiles, num_kb, stages;
  int kbs;                      // hidden blocks per pipeline stage (large-batch kernel: 1 or 2)
  uint32_t tmem_cols;
  float* logits;
  long long ldz;       // row stride of logits in floats
  float* part_max;
  int* part_idx;
  int* err;
  int zero_err;
  // sampling statistics
  float c_hi, c_lo;
  StatPart* tpart;
  int tparts;          // partials per target row (one per CTA)
  const float* zq;
  int draft_rows;
  StatPart* dpart;
  int dparts;          // partials per draft row = ceil(V / kChunk)
  unsigned* tickets;   // zeroed here for the kernel that follows
  int n_tickets;
};

// Timeouts of calls without a workspace (the bare LM head) latch here.
__device__ int g_head_timeout_word = 0;

__device__ __forceinline__ void report_timeout(int* err) {
  atomicOr(err ? err : &g_head_timeout_word, kErrTimeout);
}

// The work of one CTA as items (tile, groups [g0, g1)).  Tile mode: whole
// tiles blockIdx.x, blockIdx.x + gridDim.x, ...; stream-K: the CTA's equal
// contiguous share of the num_tiles * groups units, split at tile ends.  Every
// warp role walks the same items.
struct WorkCursor {
  long long u, end;
};

__device__ __forceinline__ long long streamk_start(const HeadParams& p, int cta) {
  return static_cast<long long>(p.num_tiles) * p.groups * cta / gridDim.x;
}

__device__ __forceinline__ WorkCursor work_begin(const HeadParams& p) {
  if (p.streamk) return {streamk_start(p, blockIdx.x), streamk_start(p, blockIdx.x + 1)};
  return {static_cast<long long>(blockIdx.x), static_cast<long long>(p.num_tiles)};
}

__device__ __forceinline__ bool work_next(const HeadParams& p, WorkCursor& c, int& tile, int& g0, int& g1) {
  if (c.u >= c.end) return false;
  if (p.streamk) {
    tile = static_cast<int>(c.u / p.groups);
    g0 = static_cast<int>(c.u - static_cast<long long>(tile) * p.groups);
    g1 = static_cast<int>(min(static_cast<long long>(p.groups), g0 + (c.end - c.u)));
    c.u += g1 - g0;
  } else {
    tile = static_cast<int>(c.u);
    g0 = 0;
    g1 = p.groups;
    c.u += gridDim.x;
  }
  return true;
}

// Greedy partials of the kCols (16 or 32) columns [c0, c0 + kCols) over the
// warp's 32 rows, by warp collectives (the small-batch scheme, whose epilogue
// has time to spare): per column the largest value and the lowest row
// holding it.
// Values map to order-preserving unsigned keys (-0 taken as +0 first, so
// that equal floats give equal keys); one warp max reduction finds the
// largest key and a ballot the lowest lane with it (the lowest token id).
// Rows past V and non-finite values take key 0, below every finite value's
// key; a non-finite value marks the column (index -2).  Lane l keeps column
// c0 + l's result, so the warp writes the scratch once per array.
template <int kCols>
__device__ __forceinline__ void argmax_redux(const HeadParams& p, const float* val, int c0, int v, int q, int lane,
                                            float* scr) {
  float* red_val = scr;
  int* red_idx = reinterpret_cast<int*>(scr + 1024);
  const bool in = v < p.V;
  const int v0 = v - lane;  // the warp's first row
  float my_val = -INFINITY;
  int my_idx = 0x7fffffff;
#pragma unroll
  for (int i = 0; i < kCols; ++i) {
    const float x = val[i] + 0.f;
    const bool bad = in && !isfinite(x);
    const uint32_t u = __float_as_uint(x);
    const uint32_t key = (in && !bad) ? ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) : 0u;
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
    const uint32_t win = __ballot_sync(0xffffffffu, key == kmax);
    const bool any_bad = __any_sync(0xffffffffu, bad);
    if (lane == i) {
      my_val = kmax == 0u ? -INFINITY : __uint_as_float((kmax & 0x80000000u) ? (kmax & 0x7fffffffu) : ~kmax);
      my_idx = any_bad ? -2 : (kmax == 0u ? 0x7fffffff : v0 + __ffs(win) - 1);
    }
  }
  if (lane < kCols) {
    red_val[q * 256 + c0 + lane] = my_val;
    red_idx[q * 256 + c0 + lane] = my_idx;
  }
}

// Output of 16 columns [c0, c0+16) of this thread's vocabulary row v: the
// logits, or the greedy partials of the small-batch scheme.  Scratch layout
// (per lane quadrant q and column): argmax uses [0] value, [1] index;
// statistics use [0] reference k, [1] sum hi, [2] sum lo.
template <int kMode>
__device__ __forceinline__ void emit16(const HeadParams& p, const float (&val)[16], int c0, int m0, int v, int q,
                                       int lane, float* scr) {
  if (kMode != kModeArgmax) {
    if (v < p.V) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int m = m0 + c0 + i;
        if (m < p.M) p.logits[static_cast<size_t>(m) * p.ldz + v] = val[i];
      }
    }
  }
  if (kMode == kModeArgmax) argmax_redux<16>(p, val, c0, v, q, lane, scr);
}

__device__ __forceinline__ void store_part(StatPart* dst, const Partial& a) {
  StatPart sp;
  sp.k = a.k;
  sp.s_hi = a.s.hi;
  sp.s_lo = a.s.lo;
  sp.bad = a.bad;
  *dst = sp;
}

// One lane's share of a 1024-token block of a draft row, 32 values: the
// largest finite h = z c, an integer reference k above it (ref_above), the 32
// terms 2^(z c - k) <= 1 summed in f32, and that sum added to the lane's
// float-float partial after bringing both to the larger reference (exact
// powers of two).  `valid` marks the values inside the row; a non-finite value
// marks the partial and is left out of it.
template <bool kAll>
__device__ __forceinline__ void draft_block(const float (&x)[32], unsigned valid, Expo c, Partial& lp) {
  float hm = -INFINITY;
  int bad = 0;
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    const float h = expo_hi(x[t], c);
    const bool in = kAll || ((valid >> t) & 1u);
    const bool fin = fabsf(h) < INFINITY;
    bad |= (in && !fin) ? 1 : 0;
    hm = (in && fin) ? fmaxf(hm, h) : hm;
  }
  lp.bad |= bad;
  if (hm == -INFINITY) return;
  const float k = ref_above(hm);
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int t = 0; t < 32; t += 2) {
    const float h0 = expo_hi(x[t], c), h1 = expo_hi(x[t + 1], c);
    const float e0 = exp2f((h0 - k) + expo_lo(x[t], h0, c));
    const float e1 = exp2f((h1 - k) + expo_lo(x[t + 1], h1, c));
    const bool u0 = (kAll || ((valid >> t) & 1u)) && fabsf(h0) < INFINITY;
    const bool u1 = (kAll || ((valid >> (t + 1)) & 1u)) && fabsf(h1) < INFINITY;
    s0 += u0 ? e0 : 0.f;
    s1 += u1 ? e1 : 0.f;
  }
  const float sb = s0 + s1;
  if (lp.k == -INFINITY) {
    lp.k = k;
    lp.s = {sb, 0.f};
  } else {
    const float kn = fmaxf(lp.k, k);
    const float fa = pow2_nonpos(lp.k - kn);
    lp.s = ff_add_f({lp.s.hi * fa, lp.s.lo * fa}, sb * pow2_nonpos(k - kn));
    lp.k = kn;
  }
}

// Draft-row statistics by two side warps (6-7 of the small-batch head, 10-11
// of the large-batch one): units of (draft row, 4096-token chunk) taken
// round-robin over CTAs, each streamed as four blocks of 1024 tokens (eight
// float4 per lane), the next block's loads in flight while the current one is
// summed (draft_block); the warp merges its lanes per unit.  (Two blocks ahead,
// or loads that skip L2 retention, measured no faster.)  Rows whose
// length is not a multiple of 4 floats are read with scalar loads.
__device__ void draft_stats(const HeadParams& p, int side_warp, int lane) {
  constexpr int kBlocks = kChunk / 1024;
  const Expo c{p.c_hi, p.c_lo};
  const long long units = static_cast<long long>(p.draft_rows) * p.dparts;
  const long long stride = 2LL * gridDim.x;
  long long u = blockIdx.x + static_cast<long long>(side_warp) * gridDim.x;
  if (u >= units) return;
  if (p.V % 4 != 0) {
    for (; u < units; u += stride) {
      const int row = static_cast<int>(u / p.dparts);
      const int chunk = static_cast<int>(u - static_cast<long long>(row) * p.dparts);
      const float* z = p.zq + static_cast<size_t>(row) * p.V;
      Partial lp = partial_empty();
#pragma unroll 1
      for (int blk = 0; blk < kBlocks; ++blk) {
        const int base = chunk * kChunk + blk * 1024;
        float x[32];
        unsigned valid = 0;
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          const int e = base + t * 32 + lane;
          x[t] = e < p.V ? z[e] : 0.f;
          valid |= e < p.V ? (1u << t) : 0u;
        }
        draft_block<false>(x, valid, c, lp);
      }
      const Partial wp = warp_merge(lp);
      if (lane == 0) store_part(&p.dpart[u], wp);
    }
    return;
  }
  auto load = [&](long long uu, int blk, float4 (&dst)[8], unsigned& valid) {
    const int row = static_cast<int>(uu / p.dparts);
    const int chunk = static_cast<int>(uu - static_cast<long long>(row) * p.dparts);
    const float* z = p.zq + static_cast<size_t>(row) * p.V;
    const int base = chunk * kChunk + blk * 1024;
    valid = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = base + (j * 32 + lane) * 4;
      const bool in = e < p.V;
      dst[j] = in ? __ldg(reinterpret_cast<const float4*>(z + e)) : make_float4(0.f, 0.f, 0.f, 0.f);
      valid |= in ? (0xfu << (4 * j)) : 0u;
    }
  };
  float4 cur[8], nxt[8];
  unsigned vcur, vnxt = 0;
  int blk = 0;
  load(u, 0, cur, vcur);
  Partial lp = partial_empty();
  while (true) {
    long long nu = u;
    int nb = blk + 1;
    if (nb == kBlocks) {
      nb = 0;
      nu += stride;
    }
    const bool more = nu < units;
    if (more) load(nu, nb, nxt, vnxt);
    float x[32];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      x[4 * j] = cur[j].x;
      x[4 * j + 1] = cur[j].y;
      x[4 * j + 2] = cur[j].z;
      x[4 * j + 3] = cur[j].w;
    }
    if (vcur == 0xffffffffu)
      draft_block<true>(x, vcur, c, lp);
    else
      draft_block<false>(x, vcur, c, lp);
    if (blk == kBlocks - 1) {
      const Partial wp = warp_merge(lp);
      if (lane == 0) store_part(&p.dpart[u], wp);
      lp = partial_empty();
    }
    if (!more) break;
#pragma unroll
    for (int j = 0; j < 8; ++j) cur[j] = nxt[j];
    vcur = vnxt;
    u = nu;
    blk = nb;
  }
}

// Greedy partials of one tile: combine the four lane quadrants per column.
__device__ __forceinline__ void argmax_finish(const HeadParams& p, int N, int vt, int m0, int et, const float* scr) {
  const float* red_val = scr;
  const int* red_idx = reinterpret_cast<const int*>(scr + 1024);
  for (int c = et; c < N; c += 128) {
    const int m = m0 + c;
    if (m >= p.M) continue;
    float bv = red_val[c];
    int bi = red_idx[c];
    bool bad = bi == -2;
#pragma unroll
    for (int qq = 1; qq < 4; ++qq) {
      const float ov = red_val[qq * 256 + c];
      const int oi = red_idx[qq * 256 + c];
      bad |= oi == -2;
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    p.part_max[static_cast<size_t>(m) * p.num_vt + vt] = bv;
    p.part_idx[static_cast<size_t>(m) * p.num_vt + vt] = bad ? -2 : bi;
  }
}

// Up to 64 positions: precise accumulation with N == kPrecN (16, 32, 48 or
// 64) positions per tile.  kMode: HeadOut as int.
template <int kPrecN, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    head_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_h,
                const HeadParams p) {
  constexpr int kSlots = kSlotsPrecise;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int S = p.stages;
  const int N = kPrecN;
  const uint32_t b_bytes = static_cast<uint32_t>(N) * 128u;
  const uint32_t stage_bytes = kABytes + b_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * stage_bytes);
  uint64_t* full = bars;              // [S] TMA landed
  uint64_t* empty = bars + S;         // [S] MMAs reading the stage are done
  uint64_t* afull = bars + 2 * S;     // [4] accumulator (slot) ready
  uint64_t* afree = afull + 4;        // [4] accumulator (slot) drained
  uint64_t* mma_done = afree + 4;     // [1] teardown
  uint64_t* red_full = mma_done + 1;  // [1] argmax scratch written by the 4 epilogue warps
  uint64_t* red_free = red_full + 1;  // [1] argmax scratch consumed
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(red_free + 1);
  float* scr = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + kBarrierBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&afull[i], 1);
      mbar_init(&afree[i], 4);
    }
    mbar_init(mma_done, 1);
    mbar_init(red_full, 4);
    mbar_init(red_free, 4);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensor_map(&tmap_w);
    prefetch_tensor_map(&tmap_h);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, p.tmem_cols);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_h = l2_policy_evict_last();
      int s = 0;
      uint32_t ph = 0;
      long long issued = 0;
      bool ok = true;
      WorkCursor wc = work_begin(p);
      int tile, g0, g1;
      while (ok && work_next(p, wc, tile, g0, g1)) {
        const int vt = tile / p.num_chunks;
        const int pc = tile - vt * p.num_chunks;
        const int kb0 = g0 * p.gkb;
        const int kb1 = min(g1 * p.gkb, p.num_kb);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1u)) {
            report_timeout(p.err);
            ok = false;
            break;
          }
          uint8_t* a_dst = smem + static_cast<size_t>(s) * stage_bytes;
          mbar_arrive_expect_tx(&full[s], stage_bytes);
          tma_load_2d(a_dst, &tmap_w, &full[s], kb * kHeadTileK, vt * kHeadTileV, pol_w);
          tma_load_2d(a_dst + kABytes, &tmap_h, &full[s], kb * kHeadTileK, pc * N, pol_h);
          ++issued;
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      griddep_launch_dependents();
      // Let the last copies land before the CTA can exit (they complete the
      // `full` phase they were issued for; in a normal run that phase has
      // long completed and the waits return at once).
      const long long tail = issued < S ? issued : S;
      for (long long i = 0; i < tail; ++i) {
        if (--s < 0) {
          s = S - 1;
          ph ^= 1u;
        }
        if (!mbar_wait(&full[s], ph)) {
          report_timeout(p.err);
          break;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kHeadTileV, static_cast<uint32_t>(N));
      int s = 0;
      uint32_t ph = 0;
      int slot = 0;
      uint32_t sph = 0;
      bool ok = true;
      WorkCursor wc = work_begin(p);
      int tile, g0, g1;
      while (ok && work_next(p, wc, tile, g0, g1)) {
        const int kb0 = g0 * p.gkb;
        const int kb1 = min(g1 * p.gkb, p.num_kb);
        // position in the current slot group (kb0 starts one); a counter, not
        // kb % gkb: an integer division per hidden block in this one issuing
        // thread held the tensor pipe back (a 128-position head: 275 vs 212 us
        // per call)
        int gpos = 0;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[s], ph)) {
            report_timeout(p.err);
            ok = false;
            break;
          }
          const bool group_first = gpos == 0;
          const bool group_last = gpos == p.gkb - 1 || kb + 1 == p.num_kb;
          gpos = group_last ? 0 : gpos + 1;
          if (group_first) {
            if (!mbar_wait(&afree[slot], sph ^ 1u)) {
              report_timeout(p.err);
              ok = false;
              break;
            }
          }
          tc_fence_after_sync();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(slot * N);
          const uint32_t a_addr = smem_u32(smem + static_cast<size_t>(s) * stage_bytes);
          const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
          for (int k = 0; k < kHeadTileK / 16; ++k) {
            const bool acc = !(group_first && k == 0);
            mma_bf16_ss(d_tmem, smem_desc_k_sw128(a_addr + k * 32), smem_desc_k_sw128(b_addr + k * 32), idesc,
                        acc ? 1u : 0u);
          }
          mma_commit(&empty[s]);
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
          if (group_last) {
            mma_commit(&afull[slot]);
            if (++slot == kSlots) {
              slot = 0;
              sph ^= 1u;
            }
          }
        }
        if (!ok) break;
      }
      // Every MMA issued by this thread has retired once this arrives.
      mma_commit(mma_done);
      if (!mbar_wait(mma_done, 0)) report_timeout(p.err);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;            // TMEM lane quadrant this warp may read
    const int et = threadIdx.x - 64;   // 0..127 among the epilogue threads
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    // This grid may start while the kernel before it in the stream (the
    // previous step's finishing kernel) still runs: the producer and the MMA
    // warp only read the weight and the hidden states, which that kernel does
    // not write, but everything the epilogue writes (logits, partials, the
    // error word and tickets) may still be read by it, so the epilogue waits
    // for it before its first such write.
    bool waited = false;
    auto wait_prev = [&]() {
      if (waited) return;
      griddep_wait();
      waited = true;
      if (blockIdx.x == 0) {
        if (p.zero_err && et == 0) *p.err = 0;
        for (int i = et; i < p.n_tickets; i += 128) p.tickets[i] = 0u;
      }
    };
    // statistics keep per-thread running partials (one per column), merged
    // across the CTA's threads once at the end; greedy partials are reduced
    // across the quadrants per tile through the scratch
    constexpr bool run_stats = kMode == kModeStats;
    constexpr bool reduce = kMode == kModeArgmax;
    constexpr int kRun = run_stats ? kPrecN : 1;
    float rk[kRun], rs[kRun];
#pragma unroll
    for (int i = 0; i < kRun; ++i) {
      rk[i] = -INFINITY;
      rs[i] = 0.f;
    }
    int slot = 0;
    uint32_t sph = 0, rph = 0;
    bool ok = true;
    WorkCursor wc = work_begin(p);
    int tile, g0, g1;
    while (ok && work_next(p, wc, tile, g0, g1)) {
      const int vt = tile / p.num_chunks;
      const int pc = tile - vt * p.num_chunks;
      const int v = vt * kHeadTileV + q * 32 + lane;
      const int m0 = pc * N;
      if (reduce && !mbar_wait(red_free, rph ^ 1u)) {  // previous tile's scratch consumed
        report_timeout(p.err);
        break;
      }
      {
        float acc[kPrecN];
#pragma unroll
        for (int i = 0; i < kPrecN; ++i) acc[i] = 0.f;
        if (g0 == 0 && g1 < p.groups) {
          // (stream-K)
          // The first part of a tile whose other groups belong to the next
          // CTA(s), each of which stored them before anything else: start
          // from their sums (the loads' latency then hides behind this tile's
          // own MMAs instead of following them; the order of the additions
          // is fixed by the schedule, so results stay deterministic).
          for (int c2 = blockIdx.x + 1; c2 < static_cast<int>(gridDim.x); ++c2) {
            if (streamk_start(p, c2) >= static_cast<long long>(tile + 1) * p.groups) break;
            bool got = true;
            if (lane == 0) {
              const unsigned long long* fl = &p.flags[c2 * 4 + q];
              if (ld_acquire_u64(fl) != p.epoch) {
                const uint64_t t0 = global_timer_ns();
                while (ld_acquire_u64(fl) != p.epoch) {
                  if (global_timer_ns() - t0 > kWaitLimitNs) {
                    got = false;
                    break;
                  }
                }
              }
            }
            got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
            if (!got) {
              report_timeout(p.err);
              continue;
            }
            const float* f = p.fix + static_cast<size_t>(c2) * kFixupFloatsPerCta + et;
#pragma unroll
            for (int i = 0; i < kPrecN; ++i) acc[i] += __ldcg(f + i * 128);
          }
        }
        for (int g = g0; g < g1; ++g) {
          if (!mbar_wait(&afull[slot], sph)) {
            report_timeout(p.err);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          if constexpr (kPrecN == 16) {
            float val[16];
            tmem_load_16(t_lane + static_cast<uint32_t>(slot * kPrecN), val);
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] += val[i];
          } else if constexpr (kPrecN == 48) {
            float val[48];
            tmem_load_48(t_lane + static_cast<uint32_t>(slot * kPrecN), val);
#pragma unroll
            for (int i = 0; i < 48; ++i) acc[i] += val[i];
          } else {
#pragma unroll
            for (int c0 = 0; c0 < kPrecN; c0 += 32) {
              float val[32];
              tmem_load_32(t_lane + static_cast<uint32_t>(slot * kPrecN + c0), val);
#pragma unroll
              for (int i = 0; i < 32; ++i) acc[c0 + i] += val[i];
            }
          }
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&afree[slot]);
          if (++slot == kSlots) {
            slot = 0;
            sph ^= 1u;
          }
        }
        if (!ok) break;
        if (g0 > 0) {
          // a later part of a tile: hand this quadrant's sums to the CTA that
          // owns the tile's first group, and emit nothing
          float* f = p.fix + static_cast<size_t>(blockIdx.x) * kFixupFloatsPerCta + et;
#pragma unroll
          for (int i = 0; i < kPrecN; ++i) f[i * 128] = acc[i];
          __syncwarp();
          if (lane == 0) {
            __threadfence();
            st_release_u64(&p.flags[blockIdx.x * 4 + q], p.epoch);
          }
          continue;
        }
        wait_prev();
        if constexpr (run_stats) {
          // logits out, and fold this row's value of every column into the
          // thread's running partial of that column (exact rescaling)
          const Expo c{p.c_hi, p.c_lo};
          const bool in = v < p.V;  // rows past V (last tile) hold zeros and fold nothing
          // Columns in chunks of 8 with no branch inside a chunk, so that the
          // chunk's independent chains interleave; columns past M in the last
          // chunk only see zeros and are never stored or merged.  The
          // reference of each running partial is an integer >= every value
          // folded so far and only rises; a rise rescales the sum by an exact
          // power of two.  Reference and rescale use float adds and integer
          // ops only (ceilf and float-to-int conversions issue ~12x slower
          // than an add), and no per-column predicate: a non-finite value
          // turns its column's sum into NaN, which the merge flags.
#pragma unroll
          for (int i0 = 0; i0 < kPrecN; i0 += 8) {
            if (i0 >= p.M) break;
#pragma unroll
            for (int i = i0; i < i0 + 8; ++i) {
              const float z = acc[i];
              if (in && i < p.M) p.logits[static_cast<size_t>(i) * p.ldz + v] = z;
              const float h = expo_hi(z, c);
              const float rn = fmaxf(rk[i], in ? ref_above(h) : -INFINITY);
              rs[i] *= pow2_nonpos(rk[i] - rn);
              rk[i] = rn;
              const float t = exp2f((h - rn) + expo_lo(z, h, c));
              rs[i] += in ? t : 0.f;
            }
          }
        } else {
#pragma unroll
          for (int c0 = 0; c0 < kPrecN; c0 += 16) {
            float val[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) val[i] = acc[c0 + i];
            emit16<kMode>(p, val, c0, m0, v, q, lane, scr);
          }
        }
      }
      if (reduce) {
        __syncwarp();
        if (lane == 0) mbar_arrive(red_full);
        if (!mbar_wait(red_full, rph)) {
          report_timeout(p.err);
          break;
        }
        argmax_finish(p, N, vt, m0, et, scr);
        __syncwarp();
        if (lane == 0) mbar_arrive(red_free);
        rph ^= 1u;
      }
    }
    wait_prev();  // (a CTA that finished no tile still writes its partials and clears the tickets)
    if constexpr (run_stats) {
      // Merge the 128 threads' running partials per column through shared
      // memory (the pipeline stages are idle now: every load has been
      // consumed), several threads per column, then one partial per CTA.
      // [column][thread]: thread et's writes are consecutive words; a column
      // reader takes every kTpc-th float4 of its column, and the pitch of
      // 128 + 4 kTpc words puts the 8 float4 reads of each quarter-warp
      // phase in distinct banks.
      constexpr int kTpc = kPrecN == 16 ? 8 : (kPrecN == 32 ? 4 : 2);  // threads per column
      constexpr int kPitch = 128 + 4 * kTpc;
      constexpr int kVecs = 128 / 4 / kTpc;                    // float4 reads per thread and array
      float* trk = reinterpret_cast<float*>(smem);             // references
      float* trs = trk + kPrecN * kPitch;                      // sums
#pragma unroll
      for (int i = 0; i < kPrecN; ++i) {
        trk[i * kPitch + et] = rk[i];
        trs[i * kPitch + et] = rs[i];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(red_full);
      if (!mbar_wait(red_full, 0)) {
        report_timeout(p.err);
      } else {
        const int col = et / kTpc, part = et % kTpc;
        const bool active = col < kPrecN;
        const int ccol = active ? col : 0;
        const float4* rk4 = reinterpret_cast<const float4*>(trk + ccol * kPitch) + part;
        const float4* rs4 = reinterpret_cast<const float4*>(trs + ccol * kPitch) + part;
        // pass 1: the column's reference = the largest of the 128 references
        float kmax = -INFINITY;
#pragma unroll
        for (int j = 0; j < kVecs; ++j) {
          const float4 r = rk4[j * kTpc];
          kmax = fmaxf(kmax, fmaxf(fmaxf(r.x, r.y), fmaxf(r.z, r.w)));
        }
#pragma unroll
        for (int off = 1; off < kTpc; off <<= 1) kmax = fmaxf(kmax, __shfl_xor_sync(0xffffffffu, kmax, off));
        // pass 2: exact power-of-two scaling to that reference, compensated
        // sum in four independent chains
        float sh[4] = {0.f, 0.f, 0.f, 0.f}, sl[4] = {0.f, 0.f, 0.f, 0.f};
        if (kmax != -INFINITY) {
#pragma unroll
          for (int j = 0; j < kVecs; ++j) {
            const float4 r = rk4[j * kTpc];
            const float4 s = rs4[j * kTpc];
            ff_accumulate(sh[0], sl[0], s.x * pow2_nonpos(r.x - kmax));
            ff_accumulate(sh[1], sl[1], s.y * pow2_nonpos(r.y - kmax));
            ff_accumulate(sh[2], sl[2], s.z * pow2_nonpos(r.z - kmax));
            ff_accumulate(sh[3], sl[3], s.w * pow2_nonpos(r.w - kmax));
          }
        }
        ff sum = ff_norm(sh[0], sl[0]);
#pragma unroll
        for (int i = 1; i < 4; ++i) sum = ff_add(sum, ff_norm(sh[i], sl[i]));
#pragma unroll
        for (int off = 1; off < kTpc; off <<= 1) sum = ff_add(sum, shfl_xor_ff(sum, off));
        Partial acc;
        acc.k = kmax;
        acc.s = sum;
        // a non-finite logit made its thread's sum NaN (or the reference +inf)
        acc.bad = !isfinite(sum.hi) || kmax == INFINITY;
        if (part == 0 && col < kPrecN && col < p.M)
          store_part(&p.tpart[static_cast<size_t>(col) * p.tparts + blockIdx.x], acc);
      }
    }
  } else if (kMode == kModeStats) {
    // ------------------------------------------------------------ draft statistics
    griddep_wait();  // the draft partials may still be read by the kernel before this one
    draft_stats(p, warp - 6, lane);
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, p.tmem_cols);
}

// ---------------------------------------------------------------- large batches
// Above 64 positions.  A tile is 128 vocabulary rows times a position chunk of
// N <= 256 columns (a multiple of 32; B = 64, K = 8 gives three chunks of 192,
// B = 256, K = 4 five of 256), the same operand shapes as one accumulator over
// the whole hidden size would use, so the tensor core sees the same operand
// traffic per product.  The accumulation is precise: groups of kLargeGroup
// hidden blocks (2048 products) go into two TMEM slots of N columns in turn,
// and the epilogue adds the slots in f32 registers.  Eight epilogue warps
// share the work: warp w reads TMEM lane quadrant w % 4 and one half of the
// columns, so that a thread keeps N/2 <= 128 running sums; while it drains one
// slot the MMAs fill the other.
constexpr int kLargeWarps = 10;                  // producer, MMA, 8 epilogue warps
constexpr int kLargeThreads = 32 * kLargeWarps;
// With sampling statistics two side warps reduce the draft rows: 384 threads
// still leave a thread the 168 registers the 320-thread forms use.
__host__ __device__ constexpr int large_threads(int mode) {
  return mode == kModeStats ? kLargeThreads + 64 : kLargeThreads;
}
constexpr int kLargeGroup = 32;                  // hidden blocks per TMEM slot (2048 products)
constexpr int kLargeHalfMax = 128;               // columns per epilogue thread at N = 256
constexpr int kLargePitch = 20;                  // floats per row of a warp's 32 x 16 transpose block
// a warp's transpose block: 32 rows at a pitch of kLargePitch, rows 16-31
// shifted by 16 more floats (for the statistics' column reads)
constexpr int kLargeTbFloats = 32 * kLargePitch + 16;
// greedy and statistics scratch: [4 quadrants][256 columns] twice (values and
// indices, or references and sums), then one transpose block per epilogue warp
constexpr uint32_t kLargeScratchBytes = (2 * 4 * 256 + 8 * kLargeTbFloats) * 4;

// Greedy partials of 16 columns [col, col + 16) over the warp's 32 rows: the
// block goes through the warp's own transpose block (128-bit stores at a pitch
// of 20 floats: conflict-free stores and column reads), then lane c < 16 scans
// column col + c for the first row holding the largest finite value.  Rows
// past V are skipped; a non-finite value marks the column (index -2).
__device__ __forceinline__ void argmax_large16(const HeadParams& p, const float (&val)[16], int col, int v, int q,
                                               int lane, float* tb, float* red_val, int* red_idx) {
  __syncwarp();  // every lane's reads of the previous block are done
#pragma unroll
  for (int j = 0; j < 16; j += 4)
    *reinterpret_cast<float4*>(tb + lane * kLargePitch + j) = make_float4(val[j], val[j + 1], val[j + 2], val[j + 3]);
  __syncwarp();
  const int v0 = v - lane;             // the warp's first row
  const int rows = min(32, p.V - v0);  // of which inside the vocabulary (may be <= 0)
  if (lane < 16) {
    float best = -INFINITY;
    int br = -1;
    bool bad = false;
#pragma unroll 8
    for (int r = 0; r < 32; ++r) {
      const float x = tb[r * kLargePitch + lane];
      const bool use = r < rows;
      const bool fin = isfinite(x);
      bad |= use && !fin;
      if (use && fin && x > best) {
        best = x;
        br = r;
      }
    }
    red_val[q * 256 + col + lane] = best;
    red_idx[q * 256 + col + lane] = bad ? -2 : (br < 0 ? 0x7fffffff : v0 + br);
  }
}

// The tile's greedy partial per column: the four lane quadrants merged (the
// lower quadrant holds the lower token ids, so equal values keep the lower).
__device__ __forceinline__ void argmax_merge_large(const HeadParams& p, int N, int vt, int m0, int et,
                                                   const float* red_val, const int* red_idx) {
  if (vt >= p.num_vt) return;  // the peer half of a pair's last tile lies past V
  for (int c = et; c < N; c += 256) {
    const int m = m0 + c;
    if (m >= p.M) continue;
    float bv = red_val[c];
    int bi = red_idx[c];
    bool bad = bi == -2;
#pragma unroll
    for (int qq = 1; qq < 4; ++qq) {
      const float ov = red_val[qq * 256 + c];
      const int oi = red_idx[qq * 256 + c];
      bad |= oi == -2;
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    p.part_max[static_cast<size_t>(m) * p.num_vt + vt] = bv;
    p.part_idx[static_cast<size_t>(m) * p.num_vt + vt] = bad ? -2 : bi;
  }
}

// Softmax-normaliser partials of 16 columns [col, col + 16) over the warp's 32
// rows (the target statistics of a tile).  The block goes through the warp's
// transpose block (rows 16-31 16 floats further on, which puts the two halves'
// column reads in distinct banks); lane L then takes column L % 16 over the 16
// rows of its half L / 16.  Two passes over the block: the largest h = z c of
// the column, then the sum of 2^(z c - k) against the integer reference
// k = ref_above(that maximum), shared by both halves.  Rows past V are
// skipped; a non-finite logit marks the column (reference +inf).
__device__ __forceinline__ void stats_large16(const HeadParams& p, const float (&val)[16], int col, int v, int q,
                                              int lane, float* tb, float* red_k, float* red_s) {
  __syncwarp();  // every lane's reads of the previous block are done
  float* row_ptr = tb + lane * kLargePitch + (lane >= 16 ? 16 : 0);
#pragma unroll
  for (int j = 0; j < 16; j += 4)
    *reinterpret_cast<float4*>(row_ptr + j) = make_float4(val[j], val[j + 1], val[j + 2], val[j + 3]);
  __syncwarp();
  const Expo c{p.c_hi, p.c_lo};
  const int cc = lane & 15, hf = lane >> 4;
  const int nrow = min(32, p.V - (v - lane)) - 16 * hf;  // rows of this lane's half inside the vocabulary
  const float* col_ptr = tb + hf * (16 * kLargePitch + 16) + cc;
  float hm = -INFINITY;
  int bad = 0;
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const float h = expo_hi(col_ptr[r * kLargePitch], c);
    const bool use = r < nrow;
    bad |= (use && !(fabsf(h) < INFINITY)) ? 1 : 0;
    hm = use ? fmaxf(hm, h) : hm;
  }
  hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, 16));
  bad |= __shfl_xor_sync(0xffffffffu, bad, 16);
  const float k = hm == -INFINITY ? -INFINITY : ref_above(hm);
  float s = 0.f;
#pragma unroll
  for (int r = 0; r < 16; ++r) {  // (the values are read again: 16 registers fewer)
    const float z = col_ptr[r * kLargePitch];
    const float h = expo_hi(z, c);
    const float t = exp2f((h - k) + expo_lo(z, h, c));
    s += r < nrow ? t : 0.f;
  }
  s += __shfl_xor_sync(0xffffffffu, s, 16);
  if (lane < 16) {
    red_k[q * 256 + col + lane] = bad ? INFINITY : k;
    red_s[q * 256 + col + lane] = s;
  }
}

// The tile's partial of column et (one column per epilogue thread): the four
// lane quadrants brought to their largest reference (exact powers of two) and
// added, then merged into this CTA's running partial of the row, which only
// this thread reads and writes during the launch.
__device__ __forceinline__ void stats_merge_large(const HeadParams& p, int N, int vt, int m0, int et,
                                                  const float* red_k, const float* red_s) {
  if (vt >= p.num_vt || et >= N) return;  // (the peer half of a pair's last tile lies past V)
  const int m = m0 + et;
  if (m >= p.M) return;
  float k = red_k[et];
#pragma unroll
  for (int qq = 1; qq < 4; ++qq) k = fmaxf(k, red_k[qq * 256 + et]);
  Partial t = partial_empty();
  t.bad = k == INFINITY ? 1 : 0;
  if (!t.bad && k != -INFINITY) {
    float sum = 0.f;
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) sum += red_s[qq * 256 + et] * pow2_nonpos(red_k[qq * 256 + et] - k);
    t.k = k;
    t.s = {sum, 0.f};
  }
  StatPart* dst = &p.tpart[static_cast<size_t>(m) * p.tparts + blockIdx.x];
  const StatPart old = *dst;
  const Partial run{old.k, {old.s_hi, old.s_lo}, old.bad};
  store_part(dst, partial_merge(run, t));
}

// kMode: kModeLogits (f32 logits), kModeArgmax (per-tile greedy partials) or
// kModeStats (f32 logits, one softmax partial per CTA and target row, and the
// draft rows' partials from two side warps).
// kPair: the MMAs run over a CTA pair (a cluster of two on neighbouring SMs,
// tcgen05 cta_group::2): a tile is 256 vocabulary rows, each CTA loads its
// 128 rows of W and half of the chunk's hidden rows, the leader (even rank)
// issues M = 256 MMAs that read both CTAs' shared memory and write both CTAs'
// tensor memory, and each CTA's epilogue drains its own 128 rows.  Per SM
// that halves the hidden-state operand traffic of a product, the part of
// shared-memory and L2 bandwidth that bounds the single-CTA MMAs.
template <int kMode, bool kPair>
__global__ void __launch_bounds__(large_threads(kMode), 1)
    head_large_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_h,
                      const HeadParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int S = p.stages;
  const int N = p.N;
  const int NH = N >> 1;                 // columns per epilogue half
  const int NB = kPair ? NH : N;         // hidden rows of this CTA's B tile
  // a stage holds kbs hidden blocks: [A_0 .. A_{kbs-1}][B_0 .. B_{kbs-1}]
  const int kbs = p.kbs;
  const uint32_t b_bytes = static_cast<uint32_t>(NB) * 128u;
  const uint32_t stage_bytes = static_cast<uint32_t>(kbs) * (kABytes + b_bytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * stage_bytes);
  uint64_t* full = bars;              // [S] TMA landed (pair: both CTAs' bytes, on the leader)
  uint64_t* empty = bars + S;         // [S] MMAs reading the stage are done
  uint64_t* afull = bars + 2 * S;     // [2] slot holds a finished group
  uint64_t* afree = afull + 2;        // [2] slot drained by the epilogue warps (pair: of both CTAs, on the leader)
  uint64_t* mma_done = afree + 2;     // [1] teardown
  uint64_t* red_full = mma_done + 1;  // [1] greedy scratch written by the 8 epilogue warps
  uint64_t* red_free = red_full + 1;  // [1] greedy scratch consumed
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(red_free + 1);
  float* scr = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + kBarrierBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;  // 0: the pair's leader
  const int unit0 = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int units = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  constexpr int kRowsPerTile = kPair ? 2 * kHeadTileV : kHeadTileV;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&afull[i], 1);
      mbar_init(&afree[i], kPair ? 16 : 8);
    }
    mbar_init(mma_done, 1);
    mbar_init(red_full, 8);
    mbar_init(red_free, 8);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensor_map(&tmap_w);
    prefetch_tensor_map(&tmap_h);
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(tmem_holder, p.tmem_cols);
      tmem_relinquish_alloc_permit_pair();
    } else {
      tmem_alloc(tmem_holder, p.tmem_cols);
      tmem_relinquish_alloc_permit();
    }
  }
  tc_fence_before_sync();
  if constexpr (kPair)
    cluster_sync();  // both CTAs' barriers initialised and tensor memory allocated
  else
    __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_h = l2_policy_evict_last();
      int s = 0;
      uint32_t ph = 0;
      long long issued = 0;
      bool ok = true;
      for (int tile = unit0; ok && tile < p.num_tiles; tile += units) {
        const int vt = tile / p.num_chunks;
        const int pc = tile - vt * p.num_chunks;
        const int w_row = vt * kRowsPerTile + static_cast<int>(rank) * kHeadTileV;
        const int h_row = pc * N + static_cast<int>(rank) * NB;
        for (int kb = 0; kb < p.num_kb; kb += kbs) {
          if (!mbar_wait(&empty[s], ph ^ 1u)) {
            report_timeout(p.err);
            ok = false;
            break;
          }
          uint8_t* a_dst = smem + static_cast<size_t>(s) * stage_bytes;
          uint8_t* b_dst = a_dst + static_cast<size_t>(kbs) * kABytes;
          if constexpr (kPair) {
            // both CTAs' bytes complete on the leader's barrier, which
            // expects them all
            if (rank == 0) mbar_arrive_expect_tx(&full[s], 2u * stage_bytes);
            const uint32_t bar = cluster_map(&full[s], 0);
            for (int j = 0; j < kbs; ++j) {
              tma_load_2d_pair(a_dst + j * kABytes, &tmap_w, bar, (kb + j) * kHeadTileK, w_row, pol_w);
              tma_load_2d_pair(b_dst + j * b_bytes, &tmap_h, bar, (kb + j) * kHeadTileK, h_row, pol_h);
            }
          } else {
            mbar_arrive_expect_tx(&full[s], stage_bytes);
            for (int j = 0; j < kbs; ++j) {
              tma_load_2d(a_dst + j * kABytes, &tmap_w, &full[s], (kb + j) * kHeadTileK, w_row, pol_w);
              tma_load_2d(b_dst + j * b_bytes, &tmap_h, &full[s], (kb + j) * kHeadTileK, h_row, pol_h);
            }
          }
          ++issued;
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      griddep_launch_dependents();
      // the last copies land before the CTA may exit (a pair's peer cannot
      // see its bytes land: the leader waits for both CTAs' here, and the
      // peer stays until the leader reaches the final cluster barrier)
      if (!kPair || rank == 0) {
        const long long tail = issued < S ? issued : S;
        for (long long i = 0; i < tail; ++i) {
          if (--s < 0) {
            s = S - 1;
            ph ^= 1u;
          }
          if (!mbar_wait(&full[s], ph)) {
            report_timeout(p.err);
            break;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (the leader's)
    if (lane == 0 && rank == 0) {
      const uint32_t idesc = idesc_bf16_f32(kPair ? 2 * kHeadTileV : kHeadTileV, static_cast<uint32_t>(N));
      // The tensor pipe idles whenever this one thread falls behind, so its
      // loop is kept short: the operand descriptors of stage 0 are built once
      // and stepped by adding to their start-address field (address >> 4; the
      // stages are 1024-byte aligned and below 256 KB, so the field never
      // carries): + stage_bytes >> 4 per stage, + 2 per 16-wide K step.
      const uint64_t a_desc0 = smem_desc_k_sw128(smem_u32(smem));
      const uint64_t b_desc0 = smem_desc_k_sw128(smem_u32(smem) + static_cast<uint32_t>(kbs) * kABytes);
      const uint64_t stage_step = stage_bytes >> 4;
      int s = 0;
      uint32_t ph = 0;
      uint64_t soff = 0;  // stage s's offset in descriptor units
      int slot = 0;
      uint32_t sph = 0;
      bool ok = true;
      for (int tile = unit0; ok && tile < p.num_tiles; tile += units) {
        int gpos = 0;  // position in the current group (a counter: no division in this thread)
        for (int kb = 0; kb < p.num_kb; kb += kbs) {
          if (!mbar_wait(&full[s], ph)) {
            report_timeout(p.err);
            ok = false;
            break;
          }
          // groups are whole stages (kLargeGroup is a multiple of kbs)
          const bool group_first = gpos == 0;
          const bool group_last = gpos + kbs == kLargeGroup || kb + kbs >= p.num_kb;
          gpos = group_last ? 0 : gpos + kbs;
          if (group_first) {
            // the slot the group overwrites has been drained by the epilogue
            if (!(kPair ? mbar_wait_cluster(&afree[slot], sph ^ 1u) : mbar_wait(&afree[slot], sph ^ 1u))) {
              report_timeout(p.err);
              ok = false;
              break;
            }
            tc_fence_after_sync();
          }
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(slot * N);
          const uint64_t a_desc = a_desc0 + soff, b_desc = b_desc0 + soff;
          for (int j = 0; j < kbs; ++j) {
            const uint64_t aj = a_desc + j * (kABytes >> 4), bj = b_desc + j * (b_bytes >> 4);
#pragma unroll
            for (int k = 0; k < kHeadTileK / 16; ++k) {
              const uint32_t accumulate = (group_first && j == 0 && k == 0) ? 0u : 1u;
              if constexpr (kPair)
                mma_bf16_ss_pair(d_tmem, aj + 2 * k, bj + 2 * k, idesc, accumulate);
              else
                mma_bf16_ss(d_tmem, aj + 2 * k, bj + 2 * k, idesc, accumulate);
            }
          }
          if constexpr (kPair)
            mma_commit_pair(&empty[s], 0x3);  // frees the stage in both CTAs
          else
            mma_commit(&empty[s]);
          soff += stage_step;
          if (++s == S) {
            s = 0;
            soff = 0;
            ph ^= 1u;
          }
          if (group_last) {
            if constexpr (kPair)
              mma_commit_pair(&afull[slot], 0x3);  // both CTAs' epilogues
            else
              mma_commit(&afull[slot]);
            slot ^= 1;
            if (slot == 0) sph ^= 1u;
          }
        }
      }
      // every MMA issued by this thread has retired once this arrives
      if constexpr (kPair)
        mma_commit_pair(mma_done, 0x1);
      else
        mma_commit(mma_done);
      if (!mbar_wait(mma_done, 0)) report_timeout(p.err);
    }
  } else if (kMode != kModeStats || warp < kLargeWarps) {
    // ------------------------------------------------------------ epilogue (warps 2..9)
    const int q = warp & 3;               // TMEM lane quadrant this warp may read
    const int half = (warp - 2) >> 2;     // which half of the tile's columns
    const int et = threadIdx.x - 64;      // 0..255 among the epilogue threads
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(half * NH);
    float* red_val = scr;                                // greedy: values; statistics: references
    int* red_idx = reinterpret_cast<int*>(scr + 1024);   // greedy: indices
    float* red_s = scr + 1024;                           // statistics: sums
    float* tb = scr + 2048 + (warp - 2) * kLargeTbFloats;
    // a drained slot is reported to the MMA issuer, in the leader CTA
    const uint32_t afree_leader0 = kPair ? cluster_map(&afree[0], 0) : 0u;
    const uint32_t afree_leader1 = kPair ? cluster_map(&afree[1], 0) : 0u;
    // with programmatic launch this grid may start while the kernel before it
    // still runs: the first write (logits, partials, the error word) waits
    bool waited = false;
    auto wait_prev = [&]() {
      if (waited) return;
      griddep_wait();
      waited = true;
      if (blockIdx.x == 0) {
        if (p.zero_err && et == 0) *p.err = 0;
        for (int i = et; i < p.n_tickets; i += 256) p.tickets[i] = 0u;
      }
      if constexpr (kMode == kModeStats) {
        // this CTA's running partials start empty (thread et owns column et
        // of every chunk)
        if (et < N)
          for (int pc = 0; pc < p.num_chunks; ++pc) {
            const int m = pc * N + et;
            if (m < p.M) store_part(&p.tpart[static_cast<size_t>(m) * p.tparts + blockIdx.x], partial_empty());
          }
      }
    };
    const int groups = (p.num_kb + kLargeGroup - 1) / kLargeGroup;
    int slot = 0;
    uint32_t sph = 0, rph = 0;
    bool ok = true;
    for (int tile = unit0; ok && tile < p.num_tiles; tile += units) {
      const int vt2 = tile / p.num_chunks;
      const int pc = tile - vt2 * p.num_chunks;
      const int vt = kPair ? 2 * vt2 + static_cast<int>(rank) : vt2;  // this CTA's 128-row vocabulary tile
      const int v = vt * kHeadTileV + q * 32 + lane;
      const int m0 = pc * N;
      const int c0 = half * NH;  // this thread's first column of the tile
      float acc[kLargeHalfMax];
#pragma unroll
      for (int i = 0; i < kLargeHalfMax; ++i) acc[i] = 0.f;
      for (int g = 0; g < groups; ++g) {
        if (!(kPair ? mbar_wait_cluster(&afull[slot], sph) : mbar_wait(&afull[slot], sph))) {
          report_timeout(p.err);
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t t_slot = t_lane + static_cast<uint32_t>(slot * N);
        // 16 columns per load: 128 sums and 16 loaded values stay within the
        // 168 registers a thread of a 320-thread block may hold
#pragma unroll
        for (int j = 0; j < kLargeHalfMax; j += 16) {
          if (j < NH) {
            float val[16];
            tmem_load_16(t_slot + j, val);
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[j + i] += val[i];
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          if constexpr (kPair)
            mbar_arrive_remote(slot == 0 ? afree_leader0 : afree_leader1);
          else
            mbar_arrive(&afree[slot]);
        }
        slot ^= 1;
        if (slot == 0) sph ^= 1u;
      }
      if (!ok) break;
      wait_prev();
      if constexpr (kMode == kModeLogits) {
        if (v < p.V) {
#pragma unroll
          for (int i = 0; i < kLargeHalfMax; ++i) {
            const int m = m0 + c0 + i;
            if (i < NH && m < p.M) p.logits[static_cast<size_t>(m) * p.ldz + v] = acc[i];
          }
        }
      } else {
        if (!mbar_wait(red_free, rph ^ 1u)) {  // the previous tile's scratch consumed
          report_timeout(p.err);
          break;
        }
        // 16 columns at a time (statistics: their logits are stored first),
        // so that each block's sums die after it
#pragma unroll
        for (int j = 0; j < kLargeHalfMax; j += 16) {
          if (j < NH) {
            float v16[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v16[i] = acc[j + i];
            if constexpr (kMode == kModeArgmax) {
              argmax_large16(p, v16, c0 + j, v, q, lane, tb, red_val, red_idx);
            } else {
              if (v < p.V) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  const int m = m0 + c0 + j + i;
                  if (m < p.M) p.logits[static_cast<size_t>(m) * p.ldz + v] = v16[i];
                }
              }
              stats_large16(p, v16, c0 + j, v, q, lane, tb, red_val, red_s);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(red_full);
        if (!mbar_wait(red_full, rph)) {
          report_timeout(p.err);
          break;
        }
        if constexpr (kMode == kModeArgmax)
          argmax_merge_large(p, N, vt, m0, et, red_val, red_idx);
        else
          stats_merge_large(p, N, vt, m0, et, red_val, red_s);
        __syncwarp();
        if (lane == 0) mbar_arrive(red_free);
        rph ^= 1u;
      }
    }
    wait_prev();  // (a CTA that finished no tile still clears the error word and writes its partials)
  } else {
    // ------------------------------------------------------------ draft statistics (warps 10, 11)
    if constexpr (kMode == kModeStats) {
      griddep_wait();  // the draft partials may still be read by the kernel before this one
      draft_stats(p, warp - kLargeWarps, lane);
    }
  }

  tc_fence_before_sync();
  if constexpr (kPair) {
    // every MMA of the pair has retired (the leader's MMA thread waited for
    // them) and both epilogues are done before either CTA frees its tensor
    // memory; neither CTA exits while the other may still reach it
    cluster_sync();
    tc_fence_after_sync();
    if (warp == 1) tmem_dealloc_pair(tmem_base, p.tmem_cols);
    cluster_sync();
  } else {
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

template <int kMode, bool kPair>
cudaError_t launch_large(const CUtensorMap& map_w, const CUtensorMap& map_h, const HeadParams& p, const HeadPlan& h,
                         const DeviceInfo& dev, cudaStream_t stream) {
  static bool attr_done[64] = {false};
  if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev.device]) {
    const cudaError_t e = cudaFuncSetAttribute(head_large_kernel<kMode, kPair>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, dev.max_smem_optin);
    if (e != cudaSuccess) return e;
    attr_done[dev.device] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(h.grid);
  cfg.blockDim = dim3(large_threads(kMode));
  cfg.dynamicSmemBytes = h.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = kPair ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, head_large_kernel<kMode, kPair>, map_w, map_h, p);
}

// Clusters of two large-batch CTAs that fit the device at once (0 if the
// pair form cannot be resident), probed once per device and block size.
template <int kMode>
int large_pair_clusters(const DeviceInfo& dev, size_t smem_bytes) {
  static int cached[64] = {0};
  static size_t cached_smem[64] = {0};
  static std::mutex mu;
  if (dev.device < 0 || dev.device >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cached_smem[dev.device] == smem_bytes) return cached[dev.device];
  int n = 0;
  if (cudaFuncSetAttribute(head_large_kernel<kMode, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           dev.max_smem_optin) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * static_cast<unsigned>(dev.sm_count / 2));
    cfg.blockDim = dim3(large_threads(kMode));
    cfg.dynamicSmemBytes = smem_bytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, head_large_kernel<kMode, true>, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();  // a failed probe leaves no sticky error
  cached[dev.device] = n;
  cached_smem[dev.device] = smem_bytes;
  return n;
}

// A 64-bit value unique to each launch in this process (the stream-K flags
// compare against it, so a workspace needs no clearing between calls).
unsigned long long next_epoch() {
  static std::atomic<unsigned long long> counter{
      static_cast<unsigned long long>(std::chrono::steady_clock::now().time_since_epoch().count()) * 0x9E3779B97F4A7C15ull};
  unsigned long long e;
  do {
    e = counter.fetch_add(1ull) + 1ull;
  } while (e == 0ull);
  return e;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Row-major bf16 matrix [rows][inner] as a 2-D tensor map with boxes of
// box_rows x 64 elements, 128-byte swizzle, zero fill outside the matrix.
bool encode_bf16_rows(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kHeadTileK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int kPrecN, int kMode>
cudaError_t launch_variant(const CUtensorMap& map_w, const CUtensorMap& map_h, const HeadParams& p,
                           const HeadPlan& h, const DeviceInfo& dev, cudaStream_t stream) {
  static bool attr_done[64] = {false};
  if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev.device]) {
    const cudaError_t e = cudaFuncSetAttribute(head_kernel<kPrecN, kMode>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, dev.max_smem_optin);
    if (e != cudaSuccess) return e;
    attr_done[dev.device] = true;
  }
  // the small precise scheme is launched as a programmatic dependent of the
  // kernel before it (see the epilogue's wait): at B=8, V=128256 this hides
  // most of the previous step's finishing kernel (177 vs 185 us per step);
  // the large batches measured slightly slower with it, so they launch
  // plainly
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(h.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = h.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, head_kernel<kPrecN, kMode>, map_w, map_h, p);
}

template <int kPrecN>
cudaError_t launch_mode(HeadOut mode, const CUtensorMap& map_w, const CUtensorMap& map_h, const HeadParams& p,
                        const HeadPlan& h, const DeviceInfo& dev, cudaStream_t stream) {
  switch (mode) {
    case HeadOut::kLogits: return launch_variant<kPrecN, kModeLogits>(map_w, map_h, p, h, dev, stream);
    case HeadOut::kArgmax: return launch_variant<kPrecN, kModeArgmax>(map_w, map_h, p, h, dev, stream);
    case HeadOut::kStats: return launch_variant<kPrecN, kModeStats>(map_w, map_h, p, h, dev, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

HeadPlan plan_head(int M, int d, int V, HeadOut mode, const DeviceInfo& dev, bool streamk) {
  HeadPlan h;
  if (M <= 64) {
    h.precise = true;
    h.N = M <= 16 ? 16 : (M <= 32 ? 32 : (M <= 48 ? 48 : 64));
    h.num_chunks = 1;
    h.gkb = kGroupPrecise;
    // tcgen05.alloc takes a power of two >= 32 columns
    uint32_t cols = 32;
    while (cols < static_cast<uint32_t>(kSlotsPrecise * h.N)) cols <<= 1;
    h.tmem_cols = cols;
  } else {
    // above 64 positions: chunks of at most 256 positions, as even as
    // multiples of 32 allow, two TMEM slots of N columns (large-batch kernel)
    h.large = true;
    const int chunks = (M + 255) / 256;
    const int per = (M + chunks - 1) / chunks;
    h.N = (per + 31) / 32 * 32;
    h.num_chunks = (M + h.N - 1) / h.N;
    h.gkb = kLargeGroup;
    uint32_t cols = 32;
    while (cols < static_cast<uint32_t>(2 * h.N)) cols <<= 1;
    h.tmem_cols = cols;
  }
  h.num_vt = (V + kHeadTileV - 1) / kHeadTileV;
  h.num_tiles = h.num_vt * h.num_chunks;
  h.num_kb = (d + kHeadTileK - 1) / kHeadTileK;
  // cross-quadrant scratch: the greedy epilogues, and the large-batch
  // statistics epilogue
  size_t scratch = 0;
  if (mode == HeadOut::kArgmax) scratch = h.large ? kLargeScratchBytes : kArgmaxSmallBytes;
  if (mode == HeadOut::kStats && h.large) scratch = kLargeScratchBytes;
  const size_t fixed = 1024 + kBarrierBytes + scratch;
  const size_t budget = static_cast<size_t>(dev.max_smem_optin);
  auto fit = [&](size_t stage) {
    h.stages = std::min(12, std::max(2, static_cast<int>((budget - fixed) / stage)));
    h.smem_bytes = fixed + static_cast<size_t>(h.stages) * stage;
  };
  fit(kABytes + static_cast<size_t>(h.N) * 128);
  h.streamk = streamk && h.precise;
  h.groups = (h.num_kb + h.gkb - 1) / h.gkb;
  const long long units = h.streamk ? static_cast<long long>(h.num_tiles) * h.groups : h.num_tiles;
  h.grid = static_cast<int>(std::min<long long>(units, std::min(dev.sm_count, kMaxHeadGrid)));
  if (h.large) {
    // two hidden blocks a stage when the blocks pair up: one barrier wait
    // and one commit of the MMA thread for every eight MMAs
    h.kbs = h.num_kb % 2 == 0 ? 2 : 1;
    fit(static_cast<size_t>(h.kbs) * (kABytes + static_cast<size_t>(h.N) * 128));
    h.grid = static_cast<int>(std::min<long long>(h.num_tiles, std::min(dev.sm_count, kMaxHeadGrid)));
    // CTA pairs where their clusters fit: tiles of 256 vocabulary rows, each
    // CTA holding half of the chunk's hidden rows
    fit(static_cast<size_t>(h.kbs) * (kABytes + static_cast<size_t>(h.N / 2) * 128));
    const int clusters = mode == HeadOut::kStats ? large_pair_clusters<kModeStats>(dev, h.smem_bytes)
                                                 : large_pair_clusters<kModeLogits>(dev, h.smem_bytes);
    if (clusters > 0) {
      h.pair = true;
      h.num_tiles = ((V + 2 * kHeadTileV - 1) / (2 * kHeadTileV)) * h.num_chunks;
      h.grid = 2 * std::min(std::min(clusters, h.num_tiles), kMaxHeadGrid / 2);  // (target partials: one per CTA)
    } else {
      fit(static_cast<size_t>(h.kbs) * (kABytes + static_cast<size_t>(h.N) * 128));
    }
  }
  // the statistics: one running partial per CTA and target row
  h.target_parts = h.grid;
  return h;
}

cudaError_t launch_head(const void* hidden, const void* W, int M, int d, int V, HeadOut mode, float* logits,
                        float* part_max, int* part_idx, const HeadStats* stats, int* err, bool zero_err,
                        const DeviceInfo& dev, cudaStream_t stream, bool* encode_failed, long long ldz,
                        void* fixup) {
  *encode_failed = false;
  const HeadPlan h = plan_head(M, d, V, mode, dev, fixup != nullptr);
  CUtensorMap map_w, map_h;
  if (!encode_bf16_rows(&map_w, W, static_cast<uint64_t>(d), static_cast<uint64_t>(V), kHeadTileV) ||
      !encode_bf16_rows(&map_h, hidden, static_cast<uint64_t>(d), static_cast<uint64_t>(M),
                        static_cast<uint32_t>(h.pair ? h.N / 2 : h.N))) {
    *encode_failed = true;
    return cudaErrorInvalidValue;
  }
  HeadParams p = {};
  p.M = M;
  p.d = d;
  p.V = V;
  p.N = h.N;
  p.num_chunks = h.num_chunks;
  p.num_vt = h.num_vt;
  p.num_tiles = h.num_tiles;
  p.num_kb = h.num_kb;
  p.kbs = h.kbs;
  p.stages = h.stages;
  p.tmem_cols = h.tmem_cols;
  p.logits = logits;
  p.ldz = ldz > 0 ? ldz : V;
  p.streamk = h.streamk ? 1 : 0;
  p.groups = h.groups;
  p.gkb = h.gkb;
  p.fix = h.streamk ? static_cast<float*>(fixup) : nullptr;
  p.flags = h.streamk ? reinterpret_cast<unsigned long long*>(static_cast<char*>(fixup) +
                                                              kMaxHeadGrid * kFixupFloatsPerCta * 4)
                      : nullptr;
  p.epoch = next_epoch();
  p.part_max = part_max;
  p.part_idx = part_idx;
  p.err = err;
  p.zero_err = (zero_err && err) ? 1 : 0;
  if (mode == HeadOut::kStats) {
    if (!stats) return cudaErrorInvalidValue;
    p.c_hi = stats->c_hi;
    p.c_lo = stats->c_lo;
    p.tpart = stats->tpart;
    p.tparts = h.target_parts;
    p.zq = stats->zq;
    p.draft_rows = stats->draft_rows;
    p.dpart = stats->dpart;
    p.dparts = (V + kChunk - 1) / kChunk;
    p.tickets = stats->tickets;
    p.n_tickets = stats->n_tickets;
  }
  if (h.large) {
    if (mode == HeadOut::kStats)
      return h.pair ? launch_large<kModeStats, true>(map_w, map_h, p, h, dev, stream)
                    : launch_large<kModeStats, false>(map_w, map_h, p, h, dev, stream);
    if (mode == HeadOut::kLogits)
      return h.pair ? launch_large<kModeLogits, true>(map_w, map_h, p, h, dev, stream)
                    : launch_large<kModeLogits, false>(map_w, map_h, p, h, dev, stream);
    return h.pair ? launch_large<kModeArgmax, true>(map_w, map_h, p, h, dev, stream)
                  : launch_large<kModeArgmax, false>(map_w, map_h, p, h, dev, stream);
  }
  if (h.N == 16) return launch_mode<16>(mode, map_w, map_h, p, h, dev, stream);
  if (h.N == 32) return launch_mode<32>(mode, map_w, map_h, p, h, dev, stream);
  if (h.N == 48) return launch_mode<48>(mode, map_w, map_h, p, h, dev, stream);
  return launch_mode<64>(mode, map_w, map_h, p, h, dev, stream);
}

}  // namespace sv
