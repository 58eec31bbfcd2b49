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
// Work decomposition: CTA (b, c) scans candidate ends e in chunk c of
// sequence b (kNgramChunk ends).  It stages the chunk's tokens and n_max
// tokens before it in shared memory with coalesced loads, and every thread
// measures, for the ends it owns, how many tokens before e agree with the
// history's suffix (at most n_max).  The best end of the CTA is packed as
// (m << 32) | e, so that the largest key is the longest match and, for that
// length, the latest end; one atomic per CTA folds it into the sequence's key
// (stored complemented: atomicMin, so that the all-ones workspace fill is the
// empty key), then takes the sequence's ticket; nothing waits for either, so
// a CTA retires right after, except the one that takes the sequence's last
// ticket, whose first warp then writes the drafts.  Every history token is
// read from HBM once.
#include "sv_common.cuh"
#include "sv_kernels.h"

namespace sv {

constexpr int kNgramThreads = 256;
constexpr int kNgramPerThread = 16;
constexpr int kNgramChunk = kNgramThreads * kNgramPerThread;  // candidate ends per CTA

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// The drafts of sequence b (one warp), once every CTA of the sequence has
// folded its best end into the key.
__device__ __noinline__ void ngram_finish(const NgramArgs& a, int b, int lane) {
  const int32_t* h = a.tokens + (long long)b * a.stride;
  const long long L = a.lengths[b];
  int32_t* out = a.drafts + (long long)b * a.K;
  if (L < 0 || L > a.stride) {
    for (int i = lane; i < a.K; i += 32) out[i] = -1;
    if (lane == 0) {
      a.n_drafts[b] = -1;
      a.match_len[b] = -1;
      atomicOr(a.status, kStatusBadData);
    }
    return;
  }
  const unsigned long long key = ~ld_relaxed_u64(a.key + b);
  const int m = (int)(key >> 32);
  const long long e = (long long)(key & 0xffffffffull);
  const long long room = m ? L - e : 0;
  const int d = (int)(room < a.K ? room : a.K);
  for (int i = lane; i < a.K; i += 32) out[i] = i < d ? __ldg(h + e + i) : -1;
  if (lane == 0) {
    a.n_drafts[b] = d;
    a.match_len[b] = m;
  }
}

__global__ void __launch_bounds__(kNgramThreads) ngram_kernel(const __grid_constant__ NgramArgs a) {
  // s_tok[kNgramMaxN + i] holds h[c0 + i] (16-byte aligned, for vector
  // stores); the n_max tokens before the chunk sit just below it
  __shared__ __align__(16) int32_t s_tok[kNgramMaxN + kNgramChunk];
  __shared__ int32_t s_suf[kNgramMaxN];  // h[L - n_max + t]
  __shared__ unsigned long long s_best[kNgramThreads / 32];
  const int b = blockIdx.x / a.chunks;
  const int c = blockIdx.x - b * a.chunks;
  const int tid = threadIdx.x;
  const int32_t* h = a.tokens + (long long)b * a.stride;
  const int L = a.lengths[b];
  const bool bad = L < 0 || (long long)L > a.stride;
  unsigned long long best = 0;  // (m << 32) | e of the best end seen, 0 for none
  const int c0 = c * kNgramChunk;
  // candidate ends of this chunk, chunk-local: r = e - c0 in [r_lo, r_hi]
  // with e in [n_min, L - 1]
  const int r_lo = a.n_min > c0 ? a.n_min - c0 : 0;
  const int r_hi = bad ? -1 : min(L - 1 - c0, kNgramChunk - 1);
  if (r_lo <= r_hi) {
    // the chunk's tokens below L (only h[.. L - 2] is ever compared: a match
    // ending at e <= L - 1 reads h[e - m .. e - 1]), in 16-byte vectors with
    // all of a thread's loads issued before its stores when rows are aligned
    const int n_main = min(L - c0, kNgramChunk);
    if (a.vec) {
      constexpr int kV = kNgramChunk / 4 / kNgramThreads;  // 16-byte vectors per thread
      int4 v[kV];
#pragma unroll
      for (int q = 0; q < kV; ++q) {
        const int i = 4 * (q * kNgramThreads + tid);
        if (i + 3 < n_main) v[q] = __ldg((const int4*)(h + c0 + i));
      }
#pragma unroll
      for (int q = 0; q < kV; ++q) {
        const int i = 4 * (q * kNgramThreads + tid);
        if (i + 3 < n_main) {
          *(int4*)&s_tok[kNgramMaxN + i] = v[q];
        } else {
          for (int t = 0; t < 4 && i + t < n_main; ++t) s_tok[kNgramMaxN + i + t] = __ldg(h + c0 + i + t);
        }
      }
    } else {
      for (int i = tid; i < n_main; i += kNgramThreads) s_tok[kNgramMaxN + i] = __ldg(h + c0 + i);
    }
    if (tid < a.n_max) {
      const int g = c0 - a.n_max + tid;
      s_tok[kNgramMaxN - a.n_max + tid] = g >= 0 ? __ldg(h + g) : 0;
      const int gs = L - a.n_max + tid;
      s_suf[tid] = gs >= 0 ? __ldg(h + gs) : 0;
    }
  }
  __syncthreads();
  if (r_lo <= r_hi) {
    const int n_max = a.n_max, n_min = a.n_min;
    const int last = s_suf[n_max - 1];  // h[L - 1]
    // end e = c0 + r, r = k * threads + tid: consecutive threads read
    // consecutive shared-memory words.  Most ends fail on the first token.
#pragma unroll 4
    for (int k = 0; k < kNgramPerThread; ++k) {
      const int r = k * kNgramThreads + tid;
      if (r < r_lo || r > r_hi) continue;
      const int j = kNgramMaxN + r - 1;  // shared index of h[e - 1]
      if (s_tok[j] != last) continue;
      // tokens before e that agree with the suffix, backwards; at most e of
      // them exist
      const int mlim = min(n_max, c0 + r);
      int m = 1;
      while (m < mlim && s_tok[j - m] == s_suf[n_max - 1 - m]) ++m;
      if (m >= n_min) {
        const unsigned long long key = ((unsigned long long)m << 32) | (unsigned)(c0 + r);
        best = key > best ? key : best;
      }
    }
  }
  // block maximum, then one atomic per CTA (nothing waits for its result)
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
    best = o > best ? o : best;
  }
  if ((tid & 31) == 0) s_best[tid >> 5] = best;
  __syncthreads();
  __shared__ int s_last;
  if (tid == 0) {
    for (int w = 1; w < kNgramThreads / 32; ++w) best = s_best[w] > best ? s_best[w] : best;
    if (best) atomicMin(a.key + b, ~best);
    // the key update is visible before this CTA's ticket: the CTA taking
    // the last ticket sees every CTA's key
    __threadfence();
    s_last = ticket_take(a.ticket + b) == a.chunks - 1;
  }
  __syncthreads();
  if (s_last && tid < 32) {
    __threadfence();
    ngram_finish(a, b, tid);
  }
}

int ngram_chunk() { return kNgramChunk; }

cudaError_t launch_ngram(const NgramArgs& a, cudaStream_t s) {
  const long long grid = (long long)a.B * a.chunks;
  if (grid <= 0) return cudaSuccess;
  ngram_kernel<<<(unsigned)grid, kNgramThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace sv
