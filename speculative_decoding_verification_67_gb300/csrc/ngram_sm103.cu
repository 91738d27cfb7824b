// Prompt-lookup (n-gram) drafter (quochung.cyou A.I article on speculative
// decoding, section "Vấn đề 3: Làm sao khi không muốn train drafter?").
// Declared in include/spec_ngram.h.
//
// One kernel.  A CTA takes one chunk of candidate end positions e of one
// sequence (up to kNgMaxChunk; smaller chunks when there are few sequences,
// so that the grid still covers the SMs).  Thread 0 reads the length and
// brings the chunk, plus the kNgMaxN tokens before it, into shared memory
// with two TMA bulk copies; every thread then scans its positions there, four
// per 16-byte load, for the number of the history's last tokens ending at e,
// up to n_max.  The best (length, -e) key of the CTA
// goes to the sequence's slot with one 64-bit atomicMax; the last CTA of the
// sequence (a ticket) reads the key, resets slot and ticket, and writes the
// proposal.  The history is read from HBM once.
#include <cstdint>

#include "internal.h"
#include "sm103_ptx.cuh"
#include "spec_ngram.h"

namespace {

constexpr int kNgThreads = 256;
constexpr int kNgMaxChunk = 8192;
constexpr int kNgMinChunk = 1024;
constexpr int kNgHalf = kNgMaxChunk / 2;  // positions in the first of the two staging copies
constexpr int kNgMaxN = 16;
constexpr int kNgMaxK = 32;
constexpr size_t kCtrlBytes = 256;  // [0] error accumulator, [1] error word, [2] sequences finished

struct NgArgs {
  const int32_t* hist;
  const int32_t* len;
  int32_t* drafts;
  int32_t* count;
  int B, max_len, K, n_min, n_max, chunk;
  int* ctrl;
  unsigned long long* key;  // [B] best (length << 32 | ~e) so far, 0 = none
  unsigned* ticket;         // [B]
};

__global__ void __launch_bounds__(kNgThreads) ngram_kernel(const NgArgs a) {
  __shared__ __align__(128) int s_tok[kNgMaxN + kNgMaxChunk + 4];  // [0, kNgMaxN): the tokens before the chunk
  __shared__ int s_suf[kNgMaxN];                                     // s_suf[t] = h[L-1-t]
  __shared__ unsigned long long s_red[kNgThreads / 32];
  __shared__ __align__(8) uint64_t s_bar[2];  // the two halves of the chunk landed
  __shared__ int s_L, s_last;
  __shared__ unsigned long long s_key;
  const int b = blockIdx.y;
  const long long row = static_cast<long long>(b) * a.max_len;
  const int c0 = blockIdx.x * a.chunk;

  // The chunk's tokens [c0, e_end) come in as two bulk copies (the first
  // kNgHalf positions with the kNgMaxN tokens before c0, then the rest), so
  // that the scan of the first half overlaps the second half's transfer.
  if (threadIdx.x == 0) {
    const int L = a.len[b];
    s_L = L;
    const bool valid = L >= 0 && L <= a.max_len;
    const int e_end = valid ? min(c0 + a.chunk, L - 1) : 0;
    if (e_end > c0) {
      // rounded up to whole 16-byte words (rows are whole words long)
      const int n4 = (e_end - c0 + 3) & ~3;
      const uint32_t body0 = static_cast<uint32_t>(min(n4, kNgHalf)) * 4u;
      const uint32_t body1 = static_cast<uint32_t>(max(n4 - kNgHalf, 0)) * 4u;
      const uint32_t halo = c0 > 0 ? kNgMaxN * 4u : 0u;
      sv::mbar_init(&s_bar[0], 1);
      sv::mbar_init(&s_bar[1], 1);
      sv::fence_barrier_init();
      sv::mbar_arrive_expect_tx(&s_bar[0], body0 + halo);
      sv::bulk_load(s_tok + kNgMaxN, a.hist + row + c0, body0, &s_bar[0]);
      if (halo) sv::bulk_load(s_tok, a.hist + row + c0 - kNgMaxN, halo, &s_bar[0]);
      if (body1) {
        sv::mbar_arrive_expect_tx(&s_bar[1], body1);
        sv::bulk_load(s_tok + kNgMaxN + kNgHalf, a.hist + row + c0 + kNgHalf, body1, &s_bar[1]);
      }
    }
  }
  if (threadIdx.x < a.n_max) {
    const int L = a.len[b];
    s_suf[threadIdx.x] = (L >= 0 && L <= a.max_len && static_cast<int>(threadIdx.x) < L)
                             ? a.hist[row + L - 1 - threadIdx.x] : 0;
  }
  __syncthreads();  // the barriers exist; s_L and s_suf are written
  const int L = s_L;
  const bool valid = L >= 0 && L <= a.max_len;
  const int e_end = valid ? min(c0 + a.chunk, L - 1) : 0;
  // four positions per 16-byte shared load (consecutive threads, consecutive
  // words: conflict-free): one mask of the positions holding the last token (a
  // group without one leaves at once), and for the others the masks of the
  // three preceding tokens, whose ANDs give the match lengths of all four;
  // only a match of four or more tokens when n_max > 4 looks further back.  A
  // thread's positions increase, so it keeps its longest match and, for equal
  // lengths, the earliest, and stops once it has one of n_max tokens.
  const int n_e = max(e_end - c0, 0);
  const int s0 = s_suf[0], s1 = s_suf[min(1, kNgMaxN - 1)], s2 = s_suf[min(2, kNgMaxN - 1)],
            s3 = s_suf[min(3, kNgMaxN - 1)];
  const int nmax4 = min(a.n_max, 4);
  int best_l = 0, best_e = 0;
  bool done = false;
  int timed_out = 0;
  // every thread waits for each half it scans, and for both halves in any case
  // before the CTA can leave (no copy may still be writing its shared memory)
  auto wait_half = [&](int h) {
    if (!sv::mbar_wait(&s_bar[h], 0)) {
      timed_out = 1;
      (void)sv::mbar_wait(&s_bar[h], 0);  // one more bounded wait for the copies in flight
    }
  };
  auto scan = [&](int qa, int qb) {
    for (int q0 = qa + 4 * static_cast<int>(threadIdx.x); q0 < qb && !done; q0 += 4 * kNgThreads) {
      const int4 v = *reinterpret_cast<const int4*>(s_tok + kNgMaxN + q0);
      const int rem = n_e - q0;
      const unsigned live = rem >= 4 ? 0xfu : ((1u << rem) - 1u);
      const unsigned B0 = ((v.x == s0) | ((v.y == s0) << 1) | ((v.z == s0) << 2) | ((v.w == s0) << 3)) & live;
      if (B0 == 0u) continue;
      const int4 pv = *reinterpret_cast<const int4*>(s_tok + kNgMaxN + q0 - 4);
      // bit q of Bl: h[e - l] == s_l for e = c0 + q0 + q
      const unsigned B1 = (pv.w == s1) | ((v.x == s1) << 1) | ((v.y == s1) << 2) | ((v.z == s1) << 3);
      const unsigned B2 = (pv.z == s2) | ((pv.w == s2) << 1) | ((v.x == s2) << 2) | ((v.y == s2) << 3);
      const unsigned B3 = (pv.y == s3) | ((pv.z == s3) << 1) | ((pv.w == s3) << 2) | ((v.x == s3) << 3);
      // a match of j tokens needs j <= e + 1 (only at the history's start)
      const bool head = c0 + q0 == 0;
      const unsigned M1 = B0 & B1 & (head ? 0xeu : 0xfu);
      const unsigned M2 = M1 & B2 & (head ? 0xcu : 0xfu);
      const unsigned M3 = M2 & B3 & (head ? 0x8u : 0xfu);
      int top;
      unsigned tm;
      if (nmax4 >= 4 && M3) {
        top = 4;
        tm = M3;
      } else if (nmax4 >= 3 && M2) {
        top = 3;
        tm = M2;
      } else if (nmax4 >= 2 && M1) {
        top = 2;
        tm = M1;
      } else {
        top = 1;
        tm = B0;
      }
      if (top < a.n_min) continue;
      int l = top;
      int e = c0 + q0 + __ffs(tm) - 1;  // the earliest position at that length
      if (top == 4 && a.n_max > 4) {
        for (unsigned mm = M3; mm; mm &= mm - 1u) {
          const int q = __ffs(mm) - 1;
          const int ee = c0 + q0 + q;
          const int lim = min(a.n_max, ee + 1);
          const int* t = s_tok + kNgMaxN + q0 + q;  // t[-l] = h[ee - l]
          int ll = 4;
          while (ll < lim && t[-ll] == s_suf[ll]) ++ll;
          if (ll > l) {
            l = ll;
            e = ee;
          }
        }
      }
      if (l > best_l) {
        best_l = l;
        best_e = e;
        if (l == a.n_max) done = true;  // this thread's later positions cannot do better
      }
    }
  };
  if (n_e > 0) {
    wait_half(0);
    if (!timed_out) scan(0, min(n_e, kNgHalf));
    if (n_e > kNgHalf) {
      wait_half(1);
      if (!timed_out) scan(kNgHalf, n_e);
    }
  }
  if (timed_out) atomicOr(a.ctrl, SPEC_NGRAM_DEVERR_TIMEOUT);
  unsigned long long best =
      best_l ? (static_cast<unsigned long long>(best_l) << 32) | (0xffffffffu - static_cast<unsigned>(best_e)) : 0ull;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
    best = o > best ? o : best;
  }
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long m = 0ull;
    for (int w = 0; w < kNgThreads / 32; ++w) m = s_red[w] > m ? s_red[w] : m;
    if (m) atomicMax(a.key + b, m);
    __threadfence();
    s_last = atomicAdd(a.ticket + b, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;

  // the last CTA of sequence b writes its proposal
  if (threadIdx.x == 0) {
    __threadfence();
    s_key = atomicExch(a.key + b, 0ull);
    a.ticket[b] = 0u;
  }
  __syncthreads();
  const unsigned long long k = s_key;
  int32_t* out = a.drafts + static_cast<long long>(b) * a.K;
  if (!valid) {
    if (threadIdx.x < a.K) out[threadIdx.x] = -1;
    if (threadIdx.x == 0) {
      a.count[b] = -1;
      atomicOr(a.ctrl, SPEC_NGRAM_DEVERR_LENGTH);
    }
  } else if (k == 0ull) {
    const int fill = L > 0 ? s_suf[0] : 0;
    if (threadIdx.x < a.K) out[threadIdx.x] = fill;
    if (threadIdx.x == 0) a.count[b] = 0;
  } else {
    const int e = static_cast<int>(0xffffffffu - static_cast<unsigned>(k & 0xffffffffull));
    const int cnt = min(a.K, L - 1 - e);
    if (threadIdx.x < a.K) out[threadIdx.x] = a.hist[row + e + 1 + min(static_cast<int>(threadIdx.x), cnt - 1)];
    if (threadIdx.x == 0) a.count[b] = cnt;
  }
  // the last sequence to finish publishes the call's error word
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(reinterpret_cast<unsigned*>(a.ctrl + 2), 1u) == static_cast<unsigned>(a.B) - 1) {
      __threadfence();
      a.ctrl[1] = atomicExch(a.ctrl, 0);
      a.ctrl[2] = 0;
    }
  }
}

bool dims_ok(const spec_ngram_dims& d) {
  return d.B >= 1 && d.B <= 65535 && d.max_len >= 4 && d.max_len <= (1 << 30) && d.max_len % 4 == 0 && d.K >= 1 &&
         d.K <= kNgMaxK && d.n_min >= 1 && d.n_min <= d.n_max && d.n_max <= kNgMaxN;
}

size_t workspace_bytes(const spec_ngram_dims& d) {
  const size_t keys = (8u * static_cast<size_t>(d.B) + 255) / 256 * 256;
  const size_t tickets = (4u * static_cast<size_t>(d.B) + 255) / 256 * 256;
  return kCtrlBytes + keys + tickets;
}

}  // namespace

extern "C" {

size_t spec_ngram_workspace_bytes(spec_ngram_dims dims) { return dims_ok(dims) ? workspace_bytes(dims) : 0; }

spec_status spec_ngram_propose(const int32_t* history, const int32_t* lengths, int32_t* out_drafts,
                               int32_t* out_count, spec_ngram_dims dims, void* workspace, size_t workspace_bytes_given,
                               spec_stream_t stream) {
  if (!history || !lengths || !out_drafts || !out_count || !workspace) return SPEC_ERR_ARG;
  if (!dims_ok(dims)) return SPEC_ERR_DIMS;
  const uintptr_t any4 = reinterpret_cast<uintptr_t>(history) | reinterpret_cast<uintptr_t>(lengths) |
                         reinterpret_cast<uintptr_t>(out_drafts) | reinterpret_cast<uintptr_t>(out_count);
  if ((any4 & 3u) || (reinterpret_cast<uintptr_t>(workspace) & 15u) || (reinterpret_cast<uintptr_t>(history) & 15u))
    return SPEC_ERR_ALIGN;
  if (workspace_bytes_given < workspace_bytes(dims)) return SPEC_ERR_WORKSPACE;
  sv::DeviceInfo dev;
  const int st = sv::current_device(dev);
  if (st != SPEC_OK) return static_cast<spec_status>(st);
  NgArgs a;
  a.hist = history;
  a.len = lengths;
  a.drafts = out_drafts;
  a.count = out_count;
  a.B = dims.B;
  a.max_len = dims.max_len;
  a.K = dims.K;
  a.n_min = dims.n_min;
  a.n_max = dims.n_max;
  a.ctrl = static_cast<int*>(workspace);
  char* p = static_cast<char*>(workspace) + kCtrlBytes;
  a.key = reinterpret_cast<unsigned long long*>(p);
  a.ticket = reinterpret_cast<unsigned*>(p + (8u * static_cast<size_t>(dims.B) + 255) / 256 * 256);
  // the largest chunk that still gives two CTAs per SM
  int chunk = kNgMaxChunk;
  while (chunk > kNgMinChunk &&
         static_cast<long long>(dims.B) * ((dims.max_len + chunk - 1) / chunk) < 2ll * dev.sm_count)
    chunk >>= 1;
  a.chunk = chunk;
  const dim3 grid((dims.max_len + chunk - 1) / chunk, dims.B);
  ngram_kernel<<<grid, kNgThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status spec_ngram_read_error(void* workspace, int32_t* error_word, spec_stream_t stream) {
  if (!workspace || !error_word) return SPEC_ERR_ARG;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess ||
      cudaMemcpy(error_word, static_cast<int*>(workspace) + 1, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

}  // extern "C"
