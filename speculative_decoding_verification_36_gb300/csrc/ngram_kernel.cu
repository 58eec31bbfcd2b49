// ngram_kernel.cu -- n-gram (prompt-lookup) drafting on the device.
//
// Implements the drafter that copies candidate continuations from the prompt
// or the output so far through an n-gram lookup (pages: "Speculative Decoding
// for LLM Inference ..." sections "The variant landscape" and "Support in
// production systems", and the FAQ "Do all variants require a separate draft
// model?").  The pages fix no rule; the one built here: for each sequence
// with history h[0 .. L-1], the longest match length m in [n_min, n_max] for
// which the last m tokens occurred earlier wins, and among its occurrences the
// latest one whose end e (exclusive) is at most L - 1; the drafts are
// h[e .. e + d - 1], d = min(K, L - e).
//
// Two launches.
//
// Scan.  The candidate match ends of sequence b are cut into chunks of
// kNgramChunk (chunk c: ends c0 + 1 .. c0 + kNgramChunk, c0 = c kNgramChunk,
// whose last compared tokens h[e - 1] are the chunk's own); the (sequence,
// chunk) entries form one flat list.  A persistent grid takes entry
// blockIdx.x first and then claims one entry at a time from a counter, so
// CTAs that draw short or empty chunks simply claim more.  A CTA is one
// producer warp and kNgramConsumers consumer warps around a ring of
// kNgramStages stage buffers in shared memory.
//   The producer publishes each entry's chunk (c0, the range of its ends,
// the suffix's place in the stage) with the stage and, when the chunk holds
// candidate ends, starts two bulk asynchronous copies (TMA) into it: the
// chunk's tokens with the kNgramHalo tokens before them, and the
// 16-byte-aligned window over the history's last kNgramMaxN tokens; both
// complete on the stage's "full" mbarrier.
//   Each consumer warp takes a quarter of the ends four at a time (one
// 16-byte shared-memory load holds the tokens before four ends; most ends
// fail on that first token), measures how many tokens before each surviving
// end agree with the history's suffix (at most n_max), reduces its best end
// to one 32-bit key (m << 16) | r (r = e - c0: the largest key is the longest
// match and, for that length, the latest end), folds it into the stage's key
// with a shared-memory atomicMax and releases the stage with its own arrival
// on the "empty" mbarrier; no consumer waits for another.
//   Before the producer refills a stage it turns the stage's key into the
// entry's slot ((m << 32) | e), so each CTA keeps up to kNgramStages - 1
// chunks in flight while its consumers compare one, and no CTA ever waits for
// another.  Waiting warps are suspended in mbarrier.try_wait, not polling.
//   Rows that do not start on a 16-byte boundary are read by the consumers
// straight from global memory (the producer then only hands out entries).
//
// Finish.  One warp per sequence takes the largest key over the sequence's
// slots and copies the drafts.  It is launched with programmatic stream
// serialisation: its CTAs may become resident while the scan runs and wait
// in griddepcontrol.wait for the scan's completion and memory, so the second
// launch adds no launch gap.
//
// Every history token is read from HBM once.
#include "sv_common.cuh"
#include "sv_kernels.h"

#include <string.h>

namespace sv {

constexpr int kNgramConsumers = 8;  // consumer warps per CTA
constexpr int kNgramConsumerThreads = 32 * kNgramConsumers;
constexpr int kNgramThreads = kNgramConsumerThreads + 32;  // and the producer warp
constexpr int kNgramPerThread = 16;
constexpr int kNgramChunk = kNgramConsumerThreads * kNgramPerThread;  // candidate ends per entry
constexpr int kNgramStages = 3;
constexpr int kNgramHalo = kNgramMaxN;      // tokens staged before a chunk
constexpr int kNgramWin = kNgramMaxN + 4;   // the aligned window over the last kNgramMaxN tokens
constexpr int kNgramWinOff = kNgramHalo + kNgramChunk;
constexpr int kNgramStageInts = kNgramWinOff + kNgramWin;
constexpr size_t kNgramSmem = (size_t)kNgramStages * kNgramStageInts * sizeof(int32_t);
constexpr int kNgramFinishWarps = 8;
// bulk copies start and end on 16-byte boundaries of global and shared memory
static_assert(kNgramPerThread % 4 == 0, "ends are compared four at a time");
static_assert((kNgramHalo * 4) % 16 == 0 && (kNgramWinOff * 4) % 16 == 0 && (kNgramStageInts * 4) % 16 == 0,
              "stage layout must keep 16-byte alignment");

// ---------------------------------------------------------------------------
// mbarrier and bulk-copy primitives (shared memory of this CTA)
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned smem_addr(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(unsigned long long* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// arrive and add `bytes` to the transaction count the phase waits for
__device__ __forceinline__ void mbar_arrive_tx(unsigned long long* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
// Has the phase with this parity completed?  The thread may be suspended up
// to about kNgramSuspendNs while the phase is still open (no instructions
// issue meanwhile).  Acquire: the completing arrivals and copies are visible
// afterwards.
constexpr unsigned kNgramSuspendNs = 128;
__device__ __forceinline__ bool mbar_try(unsigned long long* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(kNgramSuspendNs)
      : "memory");
  return ok != 0;
}
// One bulk copy global -> shared, completing `bytes` on the mbarrier.  Both
// addresses and the size are multiples of 16 bytes.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, unsigned bytes, unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// Warp-uniform bounded wait: every lane tries, and the warp leaves together
// once all lanes have seen the phase; false after `limit` further tries
// (each suspends for at most about kNgramSuspendNs).
__device__ __forceinline__ bool warp_wait(unsigned long long* bar, unsigned parity, unsigned limit) {
  if (__all_sync(0xffffffffu, mbar_try(bar, parity))) return true;
  for (unsigned it = 0; it < limit; ++it)
    if (__all_sync(0xffffffffu, mbar_try(bar, parity))) return true;
  return false;
}

// First token of the window staged over h[L - kNgramMaxN .. L - 1]: a
// multiple of 4, so that the window's copy starts on a 16-byte boundary.
__device__ __forceinline__ int ngram_win_lo(int L) { return L >= kNgramMaxN ? (L - kNgramMaxN) & ~3 : 0; }

// An entry as the producer publishes it with its stage.
struct NgramStage {
  int g;           // entry index, -1: no entries left
  int b, c0;       // sequence and first token of the chunk
  int r_lo, r_hi;  // candidate ends e = c0 + r, r in [r_lo, r_hi] (empty when r_lo > r_hi)
  int L;           // the sequence's length
};

// Entry g of a sequence of length L: chunk-local ends r in [r_lo, r_hi], a
// subset of [1, kNgramChunk], with e = c0 + r in [n_min, L - 1].
__device__ __forceinline__ NgramStage ngram_stage_of(const NgramArgs& a, int g, int L) {
  NgramStage k;
  k.g = g;
  k.b = g / a.chunks;
  k.c0 = (g - k.b * a.chunks) * kNgramChunk;
  const bool bad = L < 0 || (long long)L > a.stride;
  k.r_lo = max(1, a.n_min - k.c0);
  k.r_hi = bad ? -1 : min(L - 1 - k.c0, kNgramChunk);
  k.L = L;
  return k;
}

// The producer's drain waits this long for its own copies whatever limit the
// other waits have, so that no CTA leaves with a copy into its shared memory
// still in flight.
constexpr unsigned kNgramDrainLimit = kSpinLimit;

// One consumer warp's best key (m << 16) | r over its ends of the chunk in
// `k` (0: none).  kVec: the tokens come from the stage (tok[x] = h[c0 + x]
// for x in [-kNgramHalo, kNgramChunk), win[tail - t] = h[L - 1 - t]);
// otherwise straight from the row in global memory.
template <bool kVec>
__device__ __forceinline__ unsigned ngram_scan_chunk(const NgramArgs& a, const NgramStage& k, const int32_t* st,
                                                     int tid) {
  const int32_t* h = a.tokens + (long long)k.b * a.stride;
  const int32_t* tok = st + kNgramHalo;
  const int32_t* win = st + kNgramWinOff;
  const int tail = k.L - 1 - ngram_win_lo(k.L);
  const int last = kVec ? win[tail] : __ldg(h + k.L - 1);
  const int n_max = a.n_max, n_min = a.n_min;
  unsigned best = 0;
#pragma unroll
  for (int q = 0; q < kNgramPerThread / 4; ++q) {
    // ends r = 4y + 1 .. 4y + 4: the tokens before them are h[c0 + 4y + t]
    const int y = q * kNgramConsumerThreads + tid;
    const int rb = 4 * y + 1;
    if (rb > k.r_hi || rb + 3 < k.r_lo) continue;
    int4 v;
    if (kVec) {
      v = *(const int4*)(tok + 4 * y);  // consecutive lanes, consecutive 16 bytes
    } else {
      const int32_t* p = h + k.c0 + 4 * y;  // only ends in range are read
      v.x = rb >= k.r_lo && rb <= k.r_hi ? __ldg(p) : ~last;
      v.y = rb + 1 >= k.r_lo && rb + 1 <= k.r_hi ? __ldg(p + 1) : ~last;
      v.z = rb + 2 >= k.r_lo && rb + 2 <= k.r_hi ? __ldg(p + 2) : ~last;
      v.w = rb + 3 >= k.r_lo && rb + 3 <= k.r_hi ? __ldg(p + 3) : ~last;
    }
    unsigned hit = (unsigned)(v.x == last) | (unsigned)(v.y == last) << 1 | (unsigned)(v.z == last) << 2 |
                   (unsigned)(v.w == last) << 3;
    while (hit) {
      const int t = __ffs(hit) - 1;
      hit &= hit - 1;
      const int r = rb + t;
      if (r < k.r_lo || r > k.r_hi) continue;
      // tokens before e = c0 + r that agree with the suffix, backwards; at
      // most e of them exist
      const int mlim = min(n_max, k.c0 + r);
      int m = 1;
      if (kVec) {
        while (m < mlim && tok[r - 1 - m] == win[tail - m]) ++m;
      } else {
        while (m < mlim && __ldg(h + k.c0 + r - 1 - m) == __ldg(h + k.L - 1 - m)) ++m;
      }
      if (m >= n_min) {
        const unsigned key = ((unsigned)m << 16) | (unsigned)r;
        best = key > best ? key : best;
      }
    }
  }
  return __reduce_max_sync(0xffffffffu, best);
}

__global__ void __launch_bounds__(kNgramThreads) ngram_scan_kernel(const __grid_constant__ NgramArgs a) {
  // stage s: st[kNgramHalo + i] = h[c0 + i], st[kNgramHalo - t] = h[c0 - t]
  // (t <= kNgramHalo, chunks after the first), st[kNgramWinOff + j] = h[lo + j]
  extern __shared__ __align__(128) int32_t s_stage[];
  __shared__ __align__(8) unsigned long long s_full[kNgramStages], s_empty[kNgramStages];
  __shared__ NgramStage s_meta[kNgramStages];
  __shared__ unsigned s_key[kNgramStages];  // the stage's best (m << 16) | r, folded by the consumer warps
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the finishing launch may become resident now; it waits for this grid
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int s = 0; s < kNgramStages; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], kNgramConsumers);
      s_key[s] = 0;
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();  // the only block-wide barrier
  const int total = a.B * a.chunks;

  if (warp == kNgramConsumers) {
    // ---------------- producer warp (lane 0 acts) ----------------
    // The key of a stage's last round, turned into the entry's slot.
    auto collect = [&](int s) {
      const unsigned key = s_key[s];
      s_key[s] = 0;
      const NgramStage& m = s_meta[s];
      if (m.g >= 0 && key) a.slot[m.g] = ((unsigned long long)(key >> 16) << 32) | (unsigned)(m.c0 + (key & 0xffffu));
    };
    // Entries in the order this CTA takes them: blockIdx.x first, then
    // claims from the counter (which start at G, the CTA count).  The order
    // only grows, so the round that meets an entry >= total drops no entry
    // below total.  Lane 0 claims two rounds ahead and loads lengths one round
    // ahead, so that neither latency lies between a released stage and its
    // next copy.
    const int G = (int)gridDim.x;
    int e0 = blockIdx.x, e1 = 0, L0 = 0;
    if (lane == 0) {
      e1 = G + atomicAdd(a.counter, 1);
      L0 = e0 < total ? __ldg(a.lengths + e0 / a.chunks) : 0;
    }
    int i = 0;  // stage rounds handed to the consumers
    bool ok = true;
    for (;; ++i) {
      const int s = i % kNgramStages;
      if (i >= kNgramStages) {
        // the consumers have released the stage's previous round
        ok = warp_wait(&s_empty[s], ((i / kNgramStages) & 1) ^ 1, spin_limit());
        if (!ok) break;
        if (lane == 0) collect(s);
      }
      const bool closing = __shfl_sync(0xffffffffu, e0, 0) >= total;  // lane 0's entry
      if (lane == 0) {
        if (closing) {
          s_meta[s].g = -1;
          mbar_arrive(&s_full[s]);
        } else {
          const int L = L0;
          const NgramStage k = ngram_stage_of(a, e0, L);
          s_meta[s] = k;
          if (a.vec && k.r_lo <= k.r_hi) {
            const int32_t* h = a.tokens + (long long)k.b * a.stride;
            int32_t* st = s_stage + (size_t)s * kNgramStageInts;
            // the chunk's tokens below L rounded up to 4 (still inside the
            // row: stride is a multiple of 4), after the halo for chunks
            // after the first
            const int n4 = (min(L - k.c0, kNgramChunk) + 3) & ~3;
            const int halo = k.c0 > 0 ? kNgramHalo : 0;
            const int lo = ngram_win_lo(L), hi = (L + 3) & ~3;
            const unsigned main_bytes = (unsigned)(halo + n4) * 4u, win_bytes = (unsigned)(hi - lo) * 4u;
            mbar_arrive_tx(&s_full[s], main_bytes + win_bytes);
            bulk_load(st + kNgramHalo - halo, h + k.c0 - halo, main_bytes, &s_full[s]);
            bulk_load(st + kNgramWinOff, h + lo, win_bytes, &s_full[s]);
          } else {
            mbar_arrive(&s_full[s]);
          }
          const int e2 = G + atomicAdd(a.counter, 1);  // first needed next round
          L0 = e1 < total ? __ldg(a.lengths + e1 / a.chunks) : 0;
          e0 = e1;
          e1 = e2;
        }
      }
      if (closing) {
        ++i;
        break;
      }
    }
    if (!ok && lane == 0) atomicOr(a.status, kStatusTimeout);  // consumers gave up: nothing more handed out
    // Drain: every round not yet collected has landed (copies done) before
    // the warp, and so the CTA, leaves; its key goes to its slot once the
    // consumers release it.
    for (int r = i > kNgramStages ? i - kNgramStages : 0; r < i; ++r) {
      const int s = r % kNgramStages;
      if (!warp_wait(&s_full[s], (r / kNgramStages) & 1, kNgramDrainLimit)) {
        if (lane == 0) atomicOr(a.status, kStatusTimeout);
        continue;
      }
      // the closing round: no consumer releases it
      if (__shfl_sync(0xffffffffu, lane == 0 ? (int)(s_meta[s].g < 0) : 0, 0)) continue;
      if (!warp_wait(&s_empty[s], (r / kNgramStages) & 1, spin_limit())) {
        if (lane == 0) atomicOr(a.status, kStatusTimeout);
        continue;
      }
      if (lane == 0) collect(s);
    }
    return;
  }

  // ---------------- consumer warps ----------------
  for (int i = 0;; ++i) {
    const int s = i % kNgramStages;
    if (!warp_wait(&s_full[s], (i / kNgramStages) & 1, spin_limit())) {
      if (lane == 0) atomicOr(a.status, kStatusTimeout);
      break;
    }
    const NgramStage k = s_meta[s];
    if (k.g < 0) break;
    unsigned best = 0;
    if (k.r_lo <= k.r_hi) {
      const int32_t* st = s_stage + (size_t)s * kNgramStageInts;
      best = a.vec ? ngram_scan_chunk<true>(a, k, st, tid) : ngram_scan_chunk<false>(a, k, st, tid);
    }
    __syncwarp();  // every lane's reads of the stage come before the release
    if (lane == 0) {
      if (best) atomicMax(&s_key[s], best);
      mbar_arrive(&s_empty[s]);
    }
  }
}

// One warp per sequence, once the scan grid has completed.
__global__ void __launch_bounds__(32 * kNgramFinishWarps) ngram_finish_kernel(const __grid_constant__ NgramArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.x * kNgramFinishWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= a.B) return;
  const int32_t* h = a.tokens + (long long)b * a.stride;
  const int L = a.lengths[b];
  int32_t* out = a.drafts + (long long)b * a.K;
  if (L < 0 || (long long)L > a.stride) {
    for (int i = lane; i < a.K; i += 32) out[i] = -1;
    if (lane == 0) {
      a.n_drafts[b] = -1;
      a.match_len[b] = -1;
      atomicOr(a.status, kStatusBadData);
    }
    return;
  }
  unsigned long long key = 0;
  for (int c = lane; c < a.chunks; c += 32) {
    const unsigned long long v = __ldcg(a.slot + (long long)b * a.chunks + c);
    key = v > key ? v : key;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, key, off);
    key = o > key ? o : key;
  }
  int m = (int)(key >> 32);
  const long long e = (long long)(key & 0xffffffffull);
  // a key the scan cannot produce (a slot left unwritten after an expired
  // wait) reads as no match
  if (m < a.n_min || m > a.n_max || e < m || e > (long long)L - 1) m = 0;
  const long long room = m ? L - e : 0;
  const int d = (int)(room < a.K ? room : a.K);
  for (int i = lane; i < a.K; i += 32) out[i] = i < d ? __ldg(h + e + i) : -1;
  if (lane == 0) {
    a.n_drafts[b] = d;
    a.match_len[b] = m;
  }
}

int ngram_chunk() { return kNgramChunk; }

int ngram_blocks_per_sm() {
  if (cudaFuncSetAttribute(ngram_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kNgramSmem) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, ngram_scan_kernel, kNgramThreads, kNgramSmem) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t ngram_set_spin_limit(unsigned n) { return set_spin_limit_here(n); }

cudaError_t launch_ngram(const NgramArgs& a, int grid, cudaStream_t s) {
  if (a.B <= 0 || grid <= 0) return cudaSuccess;
  ngram_scan_kernel<<<(unsigned)grid, kNgramThreads, kNgramSmem, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)((a.B + kNgramFinishWarps - 1) / kNgramFinishWarps));
  cfg.blockDim = dim3(32 * kNgramFinishWarps);
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, ngram_finish_kernel, a);
}

}  // namespace sv
