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
//    issues tcgen05.mma from one thread, warps 2-5 drain TMEM (tcgen05.ld)
//    and write either the f32 logits or per-tile (max, lowest argmax)
//    partials for the greedy path;
//  * two accumulation schemes.  Standard (any N): one TMEM accumulator per
//    tile over the whole hidden size, double-buffered so the epilogue of a
//    tile overlaps the next tile's MMAs.  Precise (N <= 64, the small-batch
//    regime): every 64-wide hidden block is accumulated into a fresh TMEM
//    slot (4 slots rotate) and the epilogue adds the block results in f32
//    registers with round-to-nearest, so the tensor core's own accumulation
//    only ever spans 64 products; this cuts the logits' error against exact
//    arithmetic several-fold at no cost to the weight stream;
//  * every wait is bounded; a timeout sets the error word, drains the copies
//    in flight and frees TMEM before returning.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace sv {
namespace {

constexpr int kThreads = 192;
constexpr uint32_t kABytes = kHeadTileV * kHeadTileK * 2;  // 16 KB W tile per stage
constexpr uint32_t kBarrierBytes = 512;
constexpr uint32_t kReduceBytes = 2 * 4 * 256 * 4;         // argmax scratch
constexpr int kSlotsPrecise = 4;

struct HeadParams {
  int M, d, V;
  int N, num_chunks, num_vt, num_tiles, num_kb, stages;
  uint32_t tmem_cols;
  int mode;
  float* logits;
  float* part_max;
  int* part_idx;
  int* err;
};

// Timeouts of calls without a workspace (the bare LM head) latch here.
__device__ int g_head_timeout_word = 0;

__device__ __forceinline__ void report_timeout(int* err) {
  atomicOr(err ? err : &g_head_timeout_word, kErrTimeout);
}

// Output of 16 columns [c0, c0+16) of this thread's vocabulary row v.
template <bool kArgmax>
__device__ __forceinline__ void emit16(const HeadParams& p, const float (&val)[16], int c0, int m0, int v, int q,
                                       int lane, float* red_val, int* red_idx) {
  if (!kArgmax) {
    if (v < p.V) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int m = m0 + c0 + i;
        if (m < p.M) p.logits[static_cast<size_t>(m) * p.V + v] = val[i];
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float bv = val[i];
      int bi = v;
      const bool bad = (v < p.V) && !isfinite(bv);
      if (v >= p.V || bad) {
        bv = -INFINITY;
        bi = 0x7fffffff;
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
      const bool any_bad = __any_sync(0xffffffffu, bad);
      if (lane == 0) {
        red_val[q * 256 + c0 + i] = bv;
        red_idx[q * 256 + c0 + i] = any_bad ? -2 : bi;
      }
    }
  }
}

// Greedy partials of one tile: combine the four lane quadrants per column.
__device__ __forceinline__ void argmax_finish(const HeadParams& p, int N, int vt, int m0, int et,
                                              const float* red_val, const int* red_idx) {
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

// kPrecN == 0: standard accumulation; kPrecN == 32 or 64: precise
// accumulation with N == kPrecN.  kArgmax selects the greedy partials
// epilogue instead of the logits one.
template <int kPrecN, bool kArgmax>
__global__ void __launch_bounds__(kThreads, 1)
    head_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_h,
                const HeadParams p) {
  constexpr bool kPrecise = kPrecN > 0;
  constexpr int kSlots = kPrecise ? kSlotsPrecise : 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int S = p.stages;
  const int N = kPrecise ? kPrecN : p.N;
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
  float* red_val = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + kBarrierBytes);
  int* red_idx = reinterpret_cast<int*>(red_val + 4 * 256);

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
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        const int vt = tile / p.num_chunks;
        const int pc = tile - vt * p.num_chunks;
        for (int kb = 0; kb < p.num_kb; ++kb) {
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
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        if (!kPrecise) {
          if (!mbar_wait(&afree[slot], sph ^ 1u)) {
            report_timeout(p.err);
            break;
          }
          tc_fence_after_sync();
        }
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(&full[s], ph)) {
            report_timeout(p.err);
            ok = false;
            break;
          }
          if (kPrecise) {
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
            const bool acc = kPrecise ? (k != 0) : ((kb | k) != 0);
            mma_bf16_ss(d_tmem, smem_desc_k_sw128(a_addr + k * 32), smem_desc_k_sw128(b_addr + k * 32), idesc,
                        acc ? 1u : 0u);
          }
          mma_commit(&empty[s]);
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
          if (kPrecise) {
            mma_commit(&afull[slot]);
            if (++slot == kSlots) {
              slot = 0;
              sph ^= 1u;
            }
          }
        }
        if (!ok) break;
        if (!kPrecise) {
          mma_commit(&afull[slot]);
          if (++slot == kSlots) {
            slot = 0;
            sph ^= 1u;
          }
        }
      }
      // Every MMA issued by this thread has retired once this arrives.
      mma_commit(mma_done);
      if (!mbar_wait(mma_done, 0)) report_timeout(p.err);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;            // TMEM lane quadrant this warp may read
    const int et = threadIdx.x - 64;   // 0..127 among the epilogue threads
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    constexpr bool argmax = kArgmax;
    int slot = 0;
    uint32_t sph = 0, rph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      const int vt = tile / p.num_chunks;
      const int pc = tile - vt * p.num_chunks;
      const int v = vt * kHeadTileV + q * 32 + lane;
      const int m0 = pc * N;
      if (argmax && !mbar_wait(red_free, rph ^ 1u)) {  // previous tile's scratch consumed
        report_timeout(p.err);
        break;
      }
      if constexpr (kPrecise) {
        float acc[kPrecN];
#pragma unroll
        for (int i = 0; i < kPrecN; ++i) acc[i] = 0.f;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(&afull[slot], sph)) {
            report_timeout(p.err);
            ok = false;
            break;
          }
          tc_fence_after_sync();
#pragma unroll
          for (int c0 = 0; c0 < kPrecN; c0 += 32) {
            float val[32];
            tmem_load_32(t_lane + static_cast<uint32_t>(slot * kPrecN + c0), val);
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[c0 + i] += val[i];
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
#pragma unroll
        for (int c0 = 0; c0 < kPrecN; c0 += 16) {
          float val[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) val[i] = acc[c0 + i];
          emit16<kArgmax>(p, val, c0, m0, v, q, lane, red_val, red_idx);
        }
      } else {
        if (!mbar_wait(&afull[slot], sph)) {
          report_timeout(p.err);
          break;
        }
        tc_fence_after_sync();
        const uint32_t t_row = t_lane + static_cast<uint32_t>(slot * N);
        for (int c0 = 0; c0 < N; c0 += 16) {
          float val[16];
          tmem_load_16(t_row + c0, val);
          emit16<kArgmax>(p, val, c0, m0, v, q, lane, red_val, red_idx);
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&afree[slot]);
        if (++slot == kSlots) {
          slot = 0;
          sph ^= 1u;
        }
      }
      if (argmax) {
        __syncwarp();
        if (lane == 0) mbar_arrive(red_full);
        if (!mbar_wait(red_full, rph)) {
          report_timeout(p.err);
          break;
        }
        argmax_finish(p, N, vt, m0, et, red_val, red_idx);
        __syncwarp();
        if (lane == 0) mbar_arrive(red_free);
        rph ^= 1u;
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, p.tmem_cols);
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

template <int kPrecN, bool kArgmax>
cudaError_t launch_variant(const CUtensorMap& map_w, const CUtensorMap& map_h, const HeadParams& p,
                           const HeadPlan& h, const DeviceInfo& dev, cudaStream_t stream) {
  static bool attr_done[64] = {false};
  if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev.device]) {
    const cudaError_t e = cudaFuncSetAttribute(head_kernel<kPrecN, kArgmax>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, dev.max_smem_optin);
    if (e != cudaSuccess) return e;
    attr_done[dev.device] = true;
  }
  head_kernel<kPrecN, kArgmax><<<h.grid, kThreads, h.smem_bytes, stream>>>(map_w, map_h, p);
  return cudaGetLastError();
}

}  // namespace

HeadPlan plan_head(int M, int d, int V, const DeviceInfo& dev) {
  HeadPlan h;
  if (M <= 64) {
    h.precise = true;
    h.N = M <= 32 ? 32 : 64;
    h.num_chunks = 1;
    h.tmem_cols = static_cast<uint32_t>(kSlotsPrecise * h.N);
  } else {
    const int chunks = (M + 255) / 256;
    const int per = (M + chunks - 1) / chunks;
    h.N = std::max(16, (per + 15) / 16 * 16);
    h.num_chunks = (M + h.N - 1) / h.N;
    uint32_t cols = 32;
    while (cols < static_cast<uint32_t>(2 * h.N)) cols <<= 1;
    h.tmem_cols = cols;
  }
  h.num_vt = (V + kHeadTileV - 1) / kHeadTileV;
  h.num_tiles = h.num_vt * h.num_chunks;
  h.num_kb = (d + kHeadTileK - 1) / kHeadTileK;
  const size_t stage = kABytes + static_cast<size_t>(h.N) * 128;
  const size_t fixed = 1024 + kBarrierBytes + kReduceBytes;
  const size_t budget = static_cast<size_t>(dev.max_smem_optin);
  int stages = static_cast<int>((budget - fixed) / stage);
  stages = std::min(12, std::max(2, stages));
  h.stages = stages;
  h.smem_bytes = fixed + static_cast<size_t>(stages) * stage;
  h.grid = std::min(h.num_tiles, dev.sm_count);
  return h;
}

cudaError_t launch_head(const void* hidden, const void* W, int M, int d, int V, HeadOut mode, float* logits,
                        float* part_max, int* part_idx, int* err, const DeviceInfo& dev, cudaStream_t stream,
                        bool* encode_failed) {
  *encode_failed = false;
  const HeadPlan h = plan_head(M, d, V, dev);
  CUtensorMap map_w, map_h;
  if (!encode_bf16_rows(&map_w, W, static_cast<uint64_t>(d), static_cast<uint64_t>(V), kHeadTileV) ||
      !encode_bf16_rows(&map_h, hidden, static_cast<uint64_t>(d), static_cast<uint64_t>(M),
                        static_cast<uint32_t>(h.N))) {
    *encode_failed = true;
    return cudaErrorInvalidValue;
  }
  HeadParams p;
  p.M = M;
  p.d = d;
  p.V = V;
  p.N = h.N;
  p.num_chunks = h.num_chunks;
  p.num_vt = h.num_vt;
  p.num_tiles = h.num_tiles;
  p.num_kb = h.num_kb;
  p.stages = h.stages;
  p.tmem_cols = h.tmem_cols;
  p.mode = static_cast<int>(mode);
  p.logits = logits;
  p.part_max = part_max;
  p.part_idx = part_idx;
  p.err = err;
  const bool am = mode == HeadOut::kArgmax;
  if (!h.precise) return am ? launch_variant<0, true>(map_w, map_h, p, h, dev, stream)
                            : launch_variant<0, false>(map_w, map_h, p, h, dev, stream);
  if (h.N == 32) return am ? launch_variant<32, true>(map_w, map_h, p, h, dev, stream)
                           : launch_variant<32, false>(map_w, map_h, p, h, dev, stream);
  return am ? launch_variant<64, true>(map_w, map_h, p, h, dev, stream)
            : launch_variant<64, false>(map_w, map_h, p, h, dev, stream);
}

}  // namespace sv
