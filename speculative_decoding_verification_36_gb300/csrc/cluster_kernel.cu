// cluster_kernel.cu -- fused speculative-sampling verify streamed by
// thread-block clusters, so that every logit is read from HBM once.
//
// The method (pages: "Speculative Decoding & Draft Model Topologies ..." sec. 2;
// "Speculative Decoding for LLM Inference ..." sections "The draft-and-verify
// loop" and "The correctness guarantee"; "Speculative Decoding at Scale ..."
// sec. 1; "Speculative Decoding in Production ..." sec. 2), per sequence b:
// softmax statistics of target rows 0..K and draft rows 0..K-1 at temperature
// tau, the acceptance test u_i < p_i(x_i) / q_i(x_i), the first rejection n,
// and one inverse-CDF draw from max(0, p_n - q_n) (n < K) or p_K (n = K).
//
// Work decomposition.  Position unit (b, i) is target row i and draft row i of
// sequence b (target row K alone for i = K).  One thread-block cluster of C
// CTAs reads a unit together: CTA r owns elements [r LC, (r+1) LC) of both
// rows.  Units are taken in position-major order (u = i B + b, unit u by
// cluster u mod G).  Each CTA has four kinds of warps:
//   * producer (one thread): bulk asynchronous copies (the TMA engine) of the
//     CTA's sub-chunks (SB elements of each row) into a ring of S shared-memory
//     buffers, as the compute warps free them;
//   * 16 compute warps: the ring's items in order.  A statistics item adds its
//     elements to each lane's online (max, sum of exp2) pair; after a unit's
//     last sub-chunk the last warp to finish merges the warps' pairs and
//     pushes the CTA's record into the shared memory of every CTA of the
//     cluster (st.async, counted by a transaction barrier).  A draw item
//     computes the weights of a replacement or bonus distribution and their
//     masses, which are pushed the same way;
//   * decider: merges the C records of each unit in rank order (so every CTA
//     holds the same statistics and takes the same decisions), tests the
//     position, and when a token must be drawn there (the position can be the
//     sequence's first rejection, or the bonus row with no rejection known)
//     asks the producer to stream the unit's sub-chunks through the ring once
//     more.  Those copies follow the first read within microseconds and are
//     served by L2 (rows of positions 0 and 1 are copied with an evict_last
//     policy).  Once every CTA's masses are in, the CTA holding the CDF
//     crossing finds the token (CTA, sub-chunk, warp, warp step, lane,
//     element);
//   * service: stores verdicts and draws, counts each sequence's finished
//     units and writes a sequence's outputs when its last unit is in.
// Units are decided in position-major order, so when unit (b, i) is decided
// the positions before i of sequence b have normally been resolved: whether a
// draw is needed is read from the sequence's first-rejection word.  A draw
// made while that was not yet known stays in its position's slot, unused if an
// earlier position rejects.
//
// Progress.  No cluster waits for another cluster.  Inside a cluster the
// compute warps wait only for their own copies and for credits that the
// deciders return after consuming older records and draws; the deciders poll
// and never wait for a later item, and the producer gives draw items priority
// over statistics items, which bounds the draws in flight.  Every wait has an
// iteration limit after which the kernel flags SPEC_FLAG_TIMEOUT.
#include "sv_common.cuh"
#include "sv_kernels.h"

#include <math.h>

namespace sv {

namespace {

// ---------------------------------------------------------------------------
// cluster, mbarrier, bulk-copy and distributed-shared-memory primitives
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ int cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return (int)r;
}
__device__ __forceinline__ int cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return (int)r;
}
__device__ __forceinline__ int cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return (int)r;
}
// every thread of every CTA of the cluster
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
// One arrival that also raises the bytes the current phase waits for.
__device__ __forceinline__ void mbar_arrive_expect(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// Has the phase of parity `parity` completed?  (no waiting; cluster-scope
// acquire, so data the other CTAs pushed before completing it is visible.)
// Lane 0's answer, for the whole warp.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}
// Wait for that phase for about `ns` nanoseconds at most, suspended in
// hardware (no instruction issue) meanwhile.  Lane 0's answer, for the warp.
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, unsigned parity, unsigned ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
      : "memory");
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}
// Bounded wait for a phase of one of this CTA's ring barriers (completed by
// its own copies and warps: CTA-scope acquire); false when the limit ran out.
__device__ __forceinline__ bool mbar_wait_local(uint64_t* bar, unsigned parity) {
  const uint32_t a = smem_addr(bar);
  for (unsigned it = 0; it < kSpinLimit; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}
// Bounded wait for that phase (cluster-scope acquire); false when the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity) {
  const uint32_t a = smem_addr(bar);
  for (unsigned it = 0; it < kSpinLimit; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}
// The address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t remote_addr(const void* p, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}
// Arrival on CTA `rank`'s copy of `bar`, releasing this thread's earlier
// accesses at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint64_t* bar, int rank) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_addr(bar, rank))
               : "memory");
}
// 16 bytes into CTA `rank`'s copy of `dst`, counted as transaction bytes on
// its copy of `bar`.
__device__ __forceinline__ void push16(void* dst, uint64_t* bar, int rank, uint4 v) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1,%2,%3,%4}, [%5];" ::"r"(
                   remote_addr(dst, rank)),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(remote_addr(bar, rank))
               : "memory");
}
// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from
// global memory into this CTA's shared memory; completion is counted on `bar`.
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, unsigned bytes, uint64_t* bar,
                                          uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ int ld_volatile(const int* p) { return *(const volatile int*)p; }
__device__ __forceinline__ void st_volatile(int* p, int v) { *(volatile int*)p = v; }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }
__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

// ---------------------------------------------------------------------------
// shared-memory control block (after the S ring buffers)
// ---------------------------------------------------------------------------
constexpr int kItemStats = 0, kItemDraw = 1, kItemEnd = 2;

struct alignas(16) Rec {  // one CTA's statistics of a unit (48 bytes)
  float mT, sT, tT, zT;   // target row: max, sum, entropy accumulator, logit at x_i (marker: not here)
  float mD, sD, tD, zD;   // draft row
  uint32_t fr;            // rank 0: the sequence's first-rejection word read during the unit
  uint32_t pad[3];
};
struct Desc {  // what a ring buffer holds
  int type, k, j, d;  // item type, unit (cluster-local index), sub-chunk, draw index
  int b, i;           // sequence and position of the unit
  int x;              // drafted token of the position (statistics items)
  uint32_t fr;        // rank 0: the sequence's first-rejection word, read one unit ahead
};
struct alignas(16) DrawReq {  // a draw the decider asked for
  TailConsts kc;              // weights (residual or bonus)
  double w;                   // resampling uniform
  int k, b, i, verdict;
  float st8[8];               // merged mT, sT, tT, zT, mD, sD, tD, zD (for the hand-off)
};
struct DoneEntry {  // a finished unit, for the service warp (64 bytes)
  int b, i, verdict, drawn;
  int token;
  float zratio;  // Z / sT of the draw
  float mT, sT, tT, zT, mD, sD, tD, zD;
  int pad[2];
};
struct Ctl {
  uint64_t full[kClMaxStages];    // ring buffer: copies landed (producer arrival + bytes)
  uint64_t empty[kClMaxStages];   // ring buffer: every compute warp is done with it
  uint64_t xb[kClSlots];          // unit records of all C CTAs are in (decider arrival + bytes)
  uint64_t xfree[kClSlots];       // every CTA's decider consumed the records in this slot
  uint64_t db[kClDrawSlots];      // draw masses of all C CTAs are in
  uint64_t dfree[kClDrawSlots];   // every CTA's decider consumed the masses in this slot
  Rec rec[kClSlots][kClMaxC];
  double dmass[kClDrawSlots][kClMaxC][2];  // per CTA: (the draw's mass, its bonus mass)
  Desc desc[kClMaxStages];
  DrawReq dreq[kClDrawSlots];
  float wp[kClSlots][kClCompute][6];  // per unit: each warp's (mT, sT, tT, mD, sD, tD)
  float zx[kClSlots][2];              // logits at x_i, written by the warp that holds them
  int ucnt[kClSlots];                 // compute warps done with the unit in this slot
  float wsub[kClDrawSlots][kClMaxSub][kClCompute];  // draw: mass of each (sub-chunk, warp)
  float wbon[kClDrawSlots][kClCompute];             // draw: each warp's bonus mass
  int dcnt[kClDrawSlots];             // compute warps done with the draw in this slot
  DoneEntry ring[kClRing];
  int ring_head, ring_tail;
  int posted;        // draws posted by the decider
  int finished;      // draws the decider has finished
  int decider_done;  // every unit decided and every draw finished
};

// (m, s) of two rows over the 32 lanes at once (warp_ms on both, interleaved:
// the same operations in the same order, so the results are those of two
// separate warp_ms calls).
__device__ __forceinline__ void warp_ms2(float& m1, float& s1, float& m2, float& s2, float c) {
  float x1 = m1, x2 = m2;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, off));
    x2 = fmaxf(x2, __shfl_xor_sync(0xffffffffu, x2, off));
  }
  const float b1 = (x1 == neg_inf()) ? 0.f : x1, b2 = (x2 == neg_inf()) ? 0.f : x2;
  float t1 = s1 * ex2((m1 - b1) * c), t2 = s2 * ex2((m2 - b2) * c);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    t1 += __shfl_xor_sync(0xffffffffu, t1, off);
    t2 += __shfl_xor_sync(0xffffffffu, t2, off);
  }
  m1 = x1;
  s1 = t1;
  m2 = x2;
  s2 = t2;
}

__device__ __forceinline__ bool row_usable(float m, float s) {
  return s > 0.f && s < INFINITY && m < INFINITY && m > neg_inf();
}

template <class E>
__device__ __forceinline__ float smem_elem(const typename E::storage* p) {
  if constexpr (sizeof(typename E::storage) == 2)
    return __uint_as_float(((uint32_t)*p) << 16);
  else
    return *p;
}

template <class E>
__device__ __forceinline__ uint4 neg_inf_vec() {
  return make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
}

// One sub-chunk of a warp, both rows: each lane's kClMaxStepsW vectors of the
// target row (zt) and of the draft row (zd) go into the lane's running
// (max, sum of exp2) pairs.  One maximum per row over all of the lane's
// vectors, one rescale of the running sum if it rose (branch-free), then every
// exponential independent of the others, into two partial sums per row, the
// two rows interleaved: no dependence chain longer than a few operations.
// With ENT the entropy accumulators (sum of 2^d d, d <= 0) follow the sums.
template <class E, int VEC, bool ENT>
__device__ __forceinline__ float vec_max(const Raw<E, VEC> (&z)[kClMaxStepsW]) {
  if constexpr (VEC == 8) {
    uint32_t w[kClMaxStepsW];
#pragma unroll
    for (int u = 0; u < kClMaxStepsW; ++u)
      w[u] = bf16x2_max(bf16x2_max(z[u].w.x, z[u].w.y), bf16x2_max(z[u].w.z, z[u].w.w));
#pragma unroll
    for (int h = kClMaxStepsW / 2; h > 0; h >>= 1)
#pragma unroll
      for (int u = 0; u < h; ++u) w[u] = bf16x2_max(w[u], w[u + h]);
    return fmaxf(bf16_lo(w[0]), bf16_hi(w[0]));
  } else {
    float m0 = neg_inf(), m1 = neg_inf();
#pragma unroll
    for (int u = 0; u < kClMaxStepsW; ++u) {
      m0 = fmaxf(m0, fmaxf(elem(z[u], 0), elem(z[u], 1)));
      m1 = fmaxf(m1, fmaxf(elem(z[u], 2), elem(z[u], 3)));
    }
    return fmaxf(m0, m1);
  }
}
// Raise the running maximum m to cover bm; the running sums follow (exponents
// are always taken relative to the current maximum).
template <bool ENT>
__device__ __forceinline__ float raise_max(float& m, float bm, f2_t& acc, f2_t& tacc, float cc) {
  const float mn = fmaxf(m, bm);
  const float delta = (m == mn) ? 0.f : (m - mn) * cc;  // <= 0; -inf when m was empty
  const float f = ex2(delta);
  if constexpr (ENT) {
    // t' = 2^delta (t + delta s); an empty accumulator stays empty
    tacc = (m == neg_inf()) ? f2(0.f, 0.f) : f2mul(f2(f, f), f2fma(f2(delta, delta), acc, tacc));
  }
  acc = (m == neg_inf()) ? f2(0.f, 0.f) : f2mul(acc, f2(f, f));
  m = mn;
  return (mn == neg_inf()) ? 0.f : mn;
}
// 2^{(z - base) c} of both elements of a pair, added into s (and 2^d d into t):
// float2 arithmetic on register pairs, each operation rounding as its scalar
// counterpart.
__device__ __forceinline__ void exp_acc2(float2& s, float2& t, float2 z, float2 nb, float2 c2, bool ent) {
  const float2 d = __fmul2_rn(__fadd2_rn(z, nb), c2);
  const float2 e = make_float2(ex2(d.x), ex2(d.y));
  s = __fadd2_rn(s, e);
  if (ent) t = __ffma2_rn(e, make_float2(fmaxf(d.x, -126.f), fmaxf(d.y, -126.f)), t);
}
template <class E, int VEC>
__device__ __forceinline__ float2 pair2(const Raw<E, VEC>& r, int p) {
  if constexpr (VEC == 8) {
    const uint32_t w = word_of(r.w, p);
    return make_float2(bf16_lo(w), bf16_hi(w));
  } else {
    return make_float2(__uint_as_float(word_of(r.w, 2 * p)), __uint_as_float(word_of(r.w, 2 * p + 1)));
  }
}
template <class E, int VEC, bool ENT>
__device__ __forceinline__ void item_stats(const Raw<E, VEC> (&zt)[kClMaxStepsW], const Raw<E, VEC> (&zd)[kClMaxStepsW],
                                           int nv, bool pair, float& mT, f2_t& aT, f2_t& eT, float& mD, f2_t& aD,
                                           f2_t& eD, float cc) {
  const float baseT = raise_max<ENT>(mT, vec_max<E, VEC, ENT>(zt), aT, eT, cc);
  const float baseD = pair ? raise_max<ENT>(mD, vec_max<E, VEC, ENT>(zd), aD, eD, cc) : 0.f;
  const float2 nT = make_float2(-baseT, -baseT), nD = make_float2(-baseD, -baseD), c2 = make_float2(cc, cc);
  float2 sT0 = make_float2(0.f, 0.f), sT1 = sT0, sD0 = sT0, sD1 = sT0, tT0 = sT0, tT1 = sT0, tD0 = sT0, tD1 = sT0;
#pragma unroll
  for (int u = 0; u < kClMaxStepsW; ++u) {
    if (u >= nv) break;  // this warp's steps only (warp-uniform)
#pragma unroll
    for (int p = 0; p < VEC / 2; ++p) {
      exp_acc2((p & 1) ? sT1 : sT0, (p & 1) ? tT1 : tT0, pair2<E, VEC>(zt[u], p), nT, c2, ENT);
      if (pair) exp_acc2((p & 1) ? sD1 : sD0, (p & 1) ? tD1 : tD0, pair2<E, VEC>(zd[u], p), nD, c2, ENT);
    }
  }
  const float2 sT = __fadd2_rn(sT0, sT1), sD = __fadd2_rn(sD0, sD1);
  aT = f2add(aT, f2(sT.x, sT.y));
  if constexpr (ENT) {
    const float2 tT = __fadd2_rn(tT0, tT1);
    eT = f2add(eT, f2(tT.x, tT.y));
  }
  if (pair) {
    aD = f2add(aD, f2(sD.x, sD.y));
    if constexpr (ENT) {
      const float2 tD = __fadd2_rn(tD0, tD1);
      eD = f2add(eD, f2(tD.x, tD.y));
    }
  }
}

// Acceptance of x_i: q(x_i) = 0, or u < p(x_i) / q(x_i) = 2^{(zT - mT) c - (zD - mD) c} sD / sT.
// The ratio is first formed in fp32.  Its relative error is below
// (|lp| + |lq|) 1.7e-7 + 6e-7 (the two exponents rounded three times each, the
// ex2.approx error, the quotient and the product); the decision is taken
// from it only when u lies outside twice that band, else the fp64 form
// decides (the ratio from exact differences, exp2 in double).
__device__ __forceinline__ int accept_verdict(float zT, float mT, float sT, float zD, float mD, float sD,
                                              double u, float c_hi, double c64) {
  if (zD == neg_inf()) return kVerdictAccept;  // q(x) = 0 <= p(x)
  const float lp = (zT - mT) * c_hi, lq = (zD - mD) * c_hi;
  const float r = ex2(lp - lq) * (sD / sT);
  const float tol = r * ((fabsf(lp) + fabsf(lq)) * 4e-7f + 2e-6f);
  const float uf = (float)u;
  if (uf < r - tol) return kVerdictAccept;
  if (uf > r + tol) return kVerdictReject;
  const double lp64 = ((double)zT - (double)mT) * c64, lq64 = ((double)zD - (double)mD) * c64;
  return u < exp2(lp64 - lq64) * ((double)sD / (double)sT) ? kVerdictAccept : kVerdictReject;
}

// Commit of sequence b (the service warp): every unit of b has handed in its
// verdict, so n is the first position that is not an accept; the token drawn
// there is in the position's slot.  Bad data in any row flags the sequence.
__device__ void commit_seq(const ClusterArgs& a, int b) {
  const int lane = threadIdx.x & 31;
  const int K = a.K;
  int n = K;
  bool bad = false, missing = false;
  for (int j0 = 0; j0 <= K; j0 += 32) {
    const int j = j0 + lane;
    const int v = j <= K ? ld_relaxed_s32(a.verdict + (size_t)b * (K + 1) + j) : kVerdictAccept;
    bad |= __any_sync(0xffffffffu, v == kVerdictBad) != 0;
    missing |= __any_sync(0xffffffffu, v == (int)kMarker) != 0;
    const unsigned rej = __ballot_sync(0xffffffffu, j < K && v != kVerdictAccept);
    if (n == K && rej) n = j0 + __ffs(rej) - 1;
  }
  uint2 res = make_uint2(kMarker, kMarker);
  if (!bad && !missing && lane == 0) res = ld_relaxed_u2(a.slot + (size_t)b * (K + 1) + n);
  res.x = __shfl_sync(0xffffffffu, res.x, 0);
  res.y = __shfl_sync(0xffffffffu, res.y, 0);
  // a missing verdict or draw can only follow an expired wait
  const bool lost = !bad && (missing || res.x == kMarker);
  int32_t* out = a.out_tokens + (size_t)b * (K + 1);
  const int32_t* x = a.tokens + (size_t)b * K;
  if (bad || lost) {
    for (int j = lane; j <= K; j += 32) out[j] = -1;
    if (lane == 0) {
      a.out_n[b] = -1;
      atomicOr(a.status, bad ? kStatusBadData : kStatusTimeout);
      if (a.out_resid) a.out_resid[b] = NAN;
    }
  } else {
    const int token = (int)res.x;
    for (int j = lane; j <= K; j += 32) out[j] = j < n ? __ldg(x + j) : (j == n ? token : -1);
    if (lane == 0) {
      a.out_n[b] = n;
      if (a.out_resid) a.out_resid[b] = __uint_as_float(res.y);
    }
  }
  __syncwarp();
}

// The service warp: stores what the decider hands over (verdicts, draws, the
// optional statistics outputs), counts every sequence's finished units and
// commits the sequences whose last unit it sees.  Up to 32 entries are
// handled at once, one per lane, so their atomics overlap.
template <bool ENT>
__device__ void service_loop(const ClusterArgs& a, Ctl& ctl) {
  const int lane = threadIdx.x & 31;
  const int K = a.K, R = 2 * K + 1;
  int tail = 0;
  unsigned idle = 0, nap = 64;
  for (;;) {
    const int head = __shfl_sync(0xffffffffu, ld_volatile(&ctl.ring_head), 0);
    if (head == tail) {
      const int done = __shfl_sync(0xffffffffu, ld_volatile(&ctl.decider_done), 0);
      if (done && __shfl_sync(0xffffffffu, ld_volatile(&ctl.ring_head), 0) == tail) break;
      if (++idle >= kSpinLimit) {  // the decider stopped handing over: give up
        if (lane == 0) atomicOr(a.status, kStatusTimeout);
        break;
      }
      __nanosleep(nap);
      if (nap < 2048) nap <<= 1;
      continue;
    }
    idle = 0;
    nap = 64;
    __threadfence_block();
    const int cnt = min(head - tail, 32);
    const bool mine = lane < cnt;
    DoneEntry e;
    if (mine) e = ctl.ring[(tail + lane) % kClRing];
    __threadfence_block();
    __syncwarp();
    if (lane == 0) st_volatile(&ctl.ring_tail, tail + cnt);  // the slots may be refilled
    tail += cnt;
    bool last = false;
    if (mine) {
      const int b = e.b, i = e.i;
      const bool pair = i < K;
      st_relaxed_s32(a.verdict + (size_t)b * (K + 1) + i, e.verdict);
      if (e.drawn) st_relaxed_u2(a.slot + (size_t)b * (K + 1) + i, (uint32_t)e.token, f2u(e.zratio));
      if (a.out_row_stats) {
        float* rs = a.out_row_stats + ((size_t)b * R + i) * 2;
        rs[0] = (float)((double)e.mT * a.inv_tau);
        rs[1] = e.sT;
        if (pair) {
          float* rd = a.out_row_stats + ((size_t)b * R + K + 1 + i) * 2;
          rd[0] = (float)((double)e.mD * a.inv_tau);
          rd[1] = e.sD;
        }
      }
      if constexpr (ENT) {
        // nats: ln s - ln 2 * t / s (NaN for a row without mass or with NaN)
        a.out_entropy[(size_t)b * R + i] =
            (float)(log((double)e.sT) - 0.69314718055994530942 * (double)e.tT / (double)e.sT);
        if (pair)
          a.out_entropy[(size_t)b * R + K + 1 + i] =
              (float)(log((double)e.sD) - 0.69314718055994530942 * (double)e.tD / (double)e.sD);
      }
      if (a.out_pq && pair && e.verdict != kVerdictBad) {
        const double lp = ((double)e.zT - (double)e.mT) * a.c64;
        const double lq = ((double)e.zD - (double)e.mD) * a.c64;
        a.out_pq[((size_t)b * K + i) * 2 + 0] = (float)(exp2(lp) / (double)e.sT);
        a.out_pq[((size_t)b * K + i) * 2 + 1] = (float)(exp2(lq) / (double)e.sD);
      }
      // the (K+1)-th arrival (the count starts at -1) finds every other unit in
      last = atom_add_acq_rel(a.arrive + b, 1) == K - 1;
    }
    unsigned lm = __ballot_sync(0xffffffffu, last);
    __syncwarp();
    while (lm) {
      const int L = __ffs(lm) - 1;
      lm &= lm - 1;
      commit_seq(a, __shfl_sync(0xffffffffu, e.b, L));
    }
  }
}

// The decider's hand-off of a finished unit to the service warp (lane 0).
__device__ __forceinline__ void hand_off(const ClusterArgs& a, Ctl& ctl, int& head, int b, int i, int verdict,
                                         int drawn, int token, float zratio, const float* st8) {
  unsigned it = 0;
  while (head - ld_volatile(&ctl.ring_tail) >= kClRing && ++it < kSpinLimit) __nanosleep(64);
  if (head - ld_volatile(&ctl.ring_tail) >= kClRing) {
    atomicOr(a.status, kStatusTimeout);
    return;
  }
  DoneEntry& e = ctl.ring[head % kClRing];
  e.b = b;
  e.i = i;
  e.verdict = verdict;
  e.drawn = drawn;
  e.token = token < 0 ? (int)kMarker : token;
  e.zratio = zratio;
  e.mT = st8[0]; e.sT = st8[1]; e.tT = st8[2]; e.zT = st8[3];
  e.mD = st8[4]; e.sD = st8[5]; e.tD = st8[6]; e.zD = st8[7];
  __threadfence_block();
  ++head;
  st_volatile(&ctl.ring_head, head);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <class E, bool ENT>
__global__ void __launch_bounds__(kClThreads, 1) cluster_kernel(const __grid_constant__ ClusterArgs a) {
  using Sto = typename E::storage;
  constexpr int VEC = E::kVec;
  constexpr int STEPW = 32 * VEC;  // elements per warp step (32 lanes x 16 bytes)
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = cluster_rank(), g = cluster_index(), G = cluster_count();
  const int C = a.C, S = a.S, K = a.K, B = a.B, NSC = a.NSC, SB = a.SB;
  const int rows = K > 0 ? 2 : 1;
  const size_t rowb = (size_t)SB * sizeof(Sto);  // bytes of one row's sub-chunk
  const size_t bufb = (size_t)rows * rowb;
  Ctl& ctl = *reinterpret_cast<Ctl*>(smem + ((S * bufb + 127) / 128) * 128);
  const int v0 = rank * a.LC;
  const int nvalid = max(0, min(a.V, v0 + a.LC) - v0);  // elements of this CTA's chunk
  const int nk = g < a.U ? (a.U - 1 - g) / G + 1 : 0;   // units of this cluster

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.empty[s], kClCompute);
    }
    for (int q = 0; q < kClSlots; ++q) {
      mbar_init(&ctl.xb[q], 1);
      mbar_init(&ctl.xfree[q], (unsigned)C);
      ctl.ucnt[q] = 0;
      ctl.zx[q][0] = ctl.zx[q][1] = u2f(kMarker);
    }
    for (int q = 0; q < kClDrawSlots; ++q) {
      mbar_init(&ctl.db[q], 1);
      mbar_init(&ctl.dfree[q], (unsigned)C);
      ctl.dcnt[q] = 0;
    }
    ctl.ring_head = ctl.ring_tail = 0;
    ctl.posted = ctl.finished = ctl.decider_done = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  cluster_sync_all();  // no CTA pushes into another before its barriers exist

  // elements [e0, e1) of this CTA's chunk that sub-chunk j covers
  auto sub_range = [&](int j, int& e0, int& e1) {
    e0 = min(j * SB, nvalid);
    e1 = min(e0 + SB, nvalid);
  };
  auto unit_of = [&](int k, int& b, int& i) {
    const int u = g + k * G;
    i = fdiv(u, a.div_b);
    b = u - i * B;
  };

  if (warp == kClProducer) {
    // ------------------------------------------------------------------
    // producer (lane 0): the ring's items in order; a posted draw's
    // sub-chunks go before any further statistics sub-chunk
    // ------------------------------------------------------------------
    if (lane == 0) {
      const uint64_t pol_keep = l2_policy_evict_last();   // rows a draw may read again soon
      const uint64_t pol_once = l2_policy_evict_first();  // rows read once
      const int nstats = nk * NSC;
      int sq = 0, dj = 0, dissued = 0;
      // token and first-rejection word of the next statistics unit, loaded one
      // unit ahead so that no copy waits for them
      int xk = 0, xn = 0;
      uint32_t frk = 0xffffffffu, frn = 0xffffffffu;
      auto fetch_unit = [&](int k, int& xv, uint32_t& fv) {
        xv = 0;
        fv = 0xffffffffu;
        if (k >= nk) return;
        int b, i;
        unit_of(k, b, i);
        if (i < K) xv = __ldg(a.tokens + (size_t)b * K + i);
        if (rank == 0) fv = (uint32_t)ld_relaxed_s32((const int*)a.firstrej + b);
      };
      fetch_unit(0, xn, frn);
      for (int t = 0;; ++t) {
        const int s = t % S;
        if (t >= S && !mbar_wait_local(&ctl.empty[s], (unsigned)(((t / S) - 1) & 1))) atomicOr(a.status, kStatusTimeout);
        Desc dsc;
        dsc.type = kItemEnd;
        dsc.k = dsc.j = dsc.d = dsc.b = dsc.i = dsc.x = 0;
        dsc.fr = 0xffffffffu;
        bool draw_pair = false;
        for (unsigned it = 0;; ++it) {
          const int posted = ld_volatile(&ctl.posted);
          __threadfence_block();  // the request is read after its count
          if (dissued < posted) {
            const DrawReq& r = ctl.dreq[dissued % kClDrawSlots];
            dsc.type = kItemDraw;
            dsc.d = dissued;
            dsc.k = r.k;
            dsc.j = dj;
            dsc.b = r.b;
            dsc.i = r.i;
            draw_pair = r.kc.residual != 0;
            if (++dj == NSC) {
              dj = 0;
              ++dissued;
            }
            break;
          }
          if (sq < nstats) {
            dsc.type = kItemStats;
            dsc.k = sq / NSC;
            dsc.j = sq - dsc.k * NSC;
            unit_of(dsc.k, dsc.b, dsc.i);
            if (dsc.j == 0) {  // a new unit: take the prefetched words, fetch the next unit's
              xk = xn;
              frk = frn;
              fetch_unit(dsc.k + 1, xn, frn);
            }
            dsc.x = xk;
            dsc.fr = frk;
            ++sq;
            break;
          }
          if (ld_volatile(&ctl.decider_done)) break;  // the end of the ring
          if (it >= kSpinLimit) {
            atomicOr(a.status, kStatusTimeout);
            break;
          }
          __nanosleep(128);
        }
        // the buffer's previous contents were read by generic loads before now
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        ctl.desc[s] = dsc;
        if (dsc.type == kItemEnd) {
          mbar_arrive_expect(&ctl.full[s], 0);
          break;
        }
        int e0, e1;
        sub_range(dsc.j, e0, e1);
        const int nrows = dsc.type == kItemDraw ? (draw_pair ? 2 : 1) : (dsc.i < K ? 2 : 1);
        const unsigned bytes = (unsigned)((size_t)(e1 - e0) * sizeof(Sto));
        mbar_arrive_expect(&ctl.full[s], bytes * (unsigned)nrows);
        if (bytes) {
          const uint64_t pol = (dsc.type == kItemStats && dsc.i <= 1) ? pol_keep : pol_once;
          unsigned char* dst = smem + (size_t)s * bufb;
          const size_t off = (size_t)v0 + (size_t)e0;
          bulk_copy(dst, (const Sto*)a.target + ((size_t)dsc.b * (K + 1) + dsc.i) * (size_t)a.V + off, bytes,
                    &ctl.full[s], pol);
          if (nrows == 2)
            bulk_copy(dst + rowb, (const Sto*)a.draft + ((size_t)dsc.b * K + dsc.i) * (size_t)a.V + off, bytes,
                      &ctl.full[s], pol);
        }
      }
    }
  } else if (warp == kClDecider) {
    // ------------------------------------------------------------------
    // decider: units in order and draws in order, polling both
    // ------------------------------------------------------------------
    int kd = 0;          // next unit to decide
    int df = 0;          // oldest draw not yet finished
    int posted = 0;      // draws posted
    int head = 0;        // service ring head (lane 0)
    bool armed = false;  // the next unit's record barrier carries its expectation
    double ubuf = 0.0;   // this lane's uniform of the current batch (16 units x 2 streams)
    int ubase = -16;     // first unit of the batch
    int xnext = 0;       // drafted token of unit kd (lane 0, loaded one unit ahead)
    unsigned idle = 0;
    if (lane == 0 && nk > 0) {
      int b, i;
      unit_of(0, b, i);
      xnext = i < K ? __ldg(a.tokens + (size_t)b * K + i) : 0;
    }
    while (kd < nk || df < posted) {
      bool progress = false;
      // -- the next unit's records --
      if (kd < nk) {
        const int q = kd % kClSlots;
        if (!armed) {
          if (lane == 0) mbar_arrive_expect(&ctl.xb[q], (unsigned)(C * sizeof(Rec)));
          armed = true;
        }
        // a suspended wait when no draw is in flight, a quick look otherwise
        const bool ready = df < posted ? mbar_test(&ctl.xb[q], (unsigned)((kd / kClSlots) & 1))
                                       : mbar_wait_for(&ctl.xb[q], (unsigned)((kd / kClSlots) & 1), 2000u);
        if (ready) {
          progress = true;
          armed = false;
          int b, i;
          unit_of(kd, b, i);
          const bool pair = i < K;
          if (kd >= ubase + 16) {  // uniforms of units kd .. kd+15, one per lane
            ubase = kd;
            const int kk = kd + (lane >> 1);
            ubuf = 0.0;
            if (kk < nk) {
              int bb, ii;
              unit_of(kk, bb, ii);
              ubuf = uniform_draw(a.seed, (uint64_t)bb, (uint64_t)ii, (uint64_t)(lane & 1));
            }
          }
          const double u_acc = __shfl_sync(0xffffffffu, ubuf, 2 * (kd - ubase));
          const double u_res = __shfl_sync(0xffffffffu, ubuf, 2 * (kd - ubase) + 1);
          // every CTA's record, merged in rank order (lane = rank)
          float rm1 = neg_inf(), rs1 = 0.f, rt1 = 0.f, rz1 = u2f(kMarker);
          float rm2 = neg_inf(), rs2 = 0.f, rt2 = 0.f, rz2 = u2f(kMarker);
          uint32_t rfr = 0xffffffffu;
          if (lane < C) {
            const Rec& r = ctl.rec[q][lane];
            rm1 = r.mT; rs1 = r.sT; rt1 = r.tT; rz1 = r.zT;
            rm2 = r.mD; rs2 = r.sD; rt2 = r.tD; rz2 = r.zD;
            rfr = r.fr;
          }
          __syncwarp();
          // the slot may be refilled once every CTA's decider has read it
          if (lane < C) mbar_arrive_remote(&ctl.xfree[q], lane);
          const unsigned owner = __ballot_sync(0xffffffffu, f2u(rz1) != kMarker);
          const int ol = owner ? __ffs(owner) - 1 : 0;
          const float zT = __shfl_sync(0xffffffffu, rz1, ol), zD = __shfl_sync(0xffffffffu, rz2, ol);
          rfr = __shfl_sync(0xffffffffu, rfr, 0);
          if constexpr (ENT) {
            warp_mst(rm1, rs1, rt1, a.c_hi);
            warp_mst(rm2, rs2, rt2, a.c_hi);
          } else {
            warp_ms2(rm1, rs1, rm2, rs2, a.c_hi);
          }
          const int x = __shfl_sync(0xffffffffu, xnext, 0);
          if (lane == 0 && kd + 1 < nk) {  // the next unit's token
            int b2, i2;
            unit_of(kd + 1, b2, i2);
            xnext = i2 < K ? __ldg(a.tokens + (size_t)b2 * K + i2) : 0;
          }
          if (lane == 0) {
            bool bad = !row_usable(rm1, rs1);
            if (pair) bad = bad || !row_usable(rm2, rs2) || x < 0 || x >= a.V;
            int verdict = bad ? kVerdictBad : kVerdictAccept;
            if (pair && !bad) {
              if (!owner) {  // a valid token always has an owner: only an expired wait gets here
                atomicOr(a.status, kStatusTimeout);
                verdict = kVerdictBad;
              } else {
                verdict = accept_verdict(zT, rm1, rs1, zD, rm2, rs2, u_acc, a.c_hi, a.c64);
              }
            }
            if (rank == 0 && verdict != kVerdictAccept) atomicMin(a.firstrej + b, (unsigned)i);
            const bool earlier = rfr != 0xffffffffu && (int)rfr < i;  // a known rejection before i
            const bool need = verdict != kVerdictBad && !earlier && (pair ? verdict == kVerdictReject : true);
            const float st8[8] = {rm1, rs1, rt1, zT, rm2, rs2, rt2, zD};
            if (!need) {
              if (kd % C == rank) hand_off(a, ctl, head, b, i, verdict, 0, -1, 0.f, st8);
            } else {
              // slot `posted` is free once draw posted - kClDrawSlots is finished
              // (the producer's priority keeps far fewer draws in flight)
              unsigned it = 0;
              while (posted - ld_volatile(&ctl.finished) >= kClDrawSlots && ++it < kSpinLimit) __nanosleep(64);
              if (posted - ld_volatile(&ctl.finished) >= kClDrawSlots) atomicOr(a.status, kStatusTimeout);
              DrawReq& r = ctl.dreq[posted % kClDrawSlots];
              r.kc.mT = rm1;
              r.kc.mD = rm2;
              r.kc.c_hi = a.c_hi;
              r.kc.c_lo = a.c_lo;
              r.kc.residual = pair ? 1 : 0;
              r.kc.lam_hi = r.kc.lam_lo = 0.f;
              if (pair) {
                const double lam = log2((double)rs1) - log2((double)rs2);  // log2(sT / sD)
                r.kc.lam_hi = (float)lam;
                r.kc.lam_lo = (float)(lam - (double)r.kc.lam_hi);
              }
              r.w = u_res;
              r.k = kd;
              r.b = b;
              r.i = i;
              r.verdict = verdict;
              for (int q2 = 0; q2 < 8; ++q2) r.st8[q2] = st8[q2];
              mbar_arrive_expect(&ctl.db[posted % kClDrawSlots], (unsigned)(C * 16));
              __threadfence_block();
              st_volatile(&ctl.posted, posted + 1);
            }
          }
          posted = __shfl_sync(0xffffffffu, ld_volatile(&ctl.posted), 0);
          ++kd;
        }
      }
      // -- the oldest draw's masses --
      if (df < posted && (kd < nk ? mbar_test(&ctl.db[df % kClDrawSlots], (unsigned)((df / kClDrawSlots) & 1))
                                  : mbar_wait_for(&ctl.db[df % kClDrawSlots], (unsigned)((df / kClDrawSlots) & 1),
                                                  2000u))) {
        progress = true;
        const int ds = df % kClDrawSlots;
        const DrawReq& r = ctl.dreq[ds];
        double mres = 0.0, mbon = 0.0;
        if (lane < C) {
          mres = ctl.dmass[ds][lane][0];
          mbon = ctl.dmass[ds][lane][1];
        }
        __syncwarp();
        if (lane < C) mbar_arrive_remote(&ctl.dfree[ds], lane);
        double Z = warp_sum_f64(mres);
        TailConsts kc = r.kc;
        bool by_bonus = false;
        if (kc.residual && !(Z > 0.0)) {
          // a rejection always leaves positive residual mass; zero can only come
          // from rounding: draw from p_i itself, with the bonus masses
          kc.residual = 0;
          by_bonus = true;
          mres = mbon;
          Z = warp_sum_f64(mbon);
        }
        const double theta = r.w * Z;
        double before = 0.0;
        // the CTA holding the crossing (values one per lane: C <= 16)
        const int rsel = warp_cdf_search(C, theta, 0.0, [&](int) { return mres; }, &before);
        int token = -1;
        if (rsel == rank) {
          // steps to rescan: the chosen warp's steps of the chosen sub-chunk, or
          // (drawing from p_i after an empty residual) every step of the chunk
          int q0 = 0, q1 = (nvalid + STEPW - 1) / STEPW;
          double run = before;
          if (!by_bonus) {
            const float* flat = &ctl.wsub[ds][0][0];  // [sub-chunk][warp], vocabulary order
            double bf = before;
            const int fsel = warp_cdf_search(NSC * kClCompute, theta, before,
                                             [&](int f) { return (double)flat[f]; }, &bf);
            if (fsel >= 0) {
              const int jsel = fsel / kClCompute, wsel = fsel % kClCompute;
              int e0, e1;
              sub_range(jsel, e0, e1);
              const int nst = (e1 - e0 + STEPW - 1) / STEPW;
              q0 = e0 / STEPW + (wsel * nst) / kClCompute;
              q1 = e0 / STEPW + ((wsel + 1) * nst) / kClCompute;
              run = bf;
            } else {
              q1 = q0;  // no mass: only an expired wait gets here
            }
          }
          const Sto* rowT = (const Sto*)a.target + ((size_t)r.b * (K + 1) + r.i) * (size_t)a.V + v0;
          const Sto* rowD = (const Sto*)a.draft + ((size_t)r.b * K + r.i) * (size_t)a.V + v0;
          int last_tok = -1;
          for (int q2 = q0; q2 < q1 && token < 0; ++q2) {
            const int e = (q2 * 32 + lane) * VEC;
            Raw<E, VEC> zt, zd;
            zt.w = e < nvalid ? ld_stream16(rowT + e) : neg_inf_vec<E>();
            zd.w = (kc.residual && e < nvalid) ? ld_stream16(rowD + e) : zt.w;
            float wv[VEC];
            lane_weights<E, VEC>(zt, zd, kc, wv);
            float ls = 0.f;
#pragma unroll
            for (int q3 = 0; q3 < VEC; ++q3) ls = __fadd_rn(ls, wv[q3]);
            const float ps = warp_sum(ls);  // the step's mass, as the compute warps formed it
            double incl = (double)ls;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
              const double o = __shfl_up_sync(0xffffffffu, incl, off);
              if (lane >= off) incl += o;
            }
            const double excl = incl - (double)ls;
            const unsigned has = __ballot_sync(0xffffffffu, ls > 0.f);
            const bool step_hit = ps > 0.f && run + (double)ps > theta;
            const unsigned cb = __ballot_sync(0xffffffffu, ls > 0.f && run + excl + (double)ls > theta);
            if (has) {
              const int L = (step_hit && cb) ? __ffs(cb) - 1 : 31 - __clz(has);
              int tk = -1;
              if (lane == L) {
                float part = 0.f;
                int pick = -1, lastpos = -1;
#pragma unroll
                for (int q3 = 0; q3 < VEC; ++q3) {
                  part = __fadd_rn(part, wv[q3]);
                  if (wv[q3] > 0.f) {
                    lastpos = q3;
                    if (pick < 0 && run + excl + (double)part > theta) pick = q3;
                  }
                }
                if (pick < 0) pick = lastpos;
                tk = v0 + e + pick;
              }
              tk = __shfl_sync(0xffffffffu, tk, L);
              if (step_hit) token = tk;
              last_tok = tk;  // rounding may leave theta past every step: the last with mass
            }
            run += (double)ps;
          }
          if (token < 0) token = last_tok;
        }
        if (lane == 0) {
          if (rsel < 0 || (rsel == rank && token < 0)) atomicOr(a.status, kStatusTimeout);  // no mass: expired wait
          if (rsel == rank || (rsel < 0 && r.k % C == rank))
            hand_off(a, ctl, head, r.b, r.i, r.verdict, 1, token, (float)(Z / (double)r.st8[1]), r.st8);
          __threadfence_block();
          st_volatile(&ctl.finished, df + 1);
        }
        ++df;
        __syncwarp();
      }
      if (progress) {
        idle = 0;
      } else {
        if (++idle >= kSpinLimit) {
          if (lane == 0) atomicOr(a.status, kStatusTimeout);
          break;
        }
        if (df < posted) __nanosleep(256);
      }
    }
    if (lane == 0) {
      __threadfence_block();
      st_volatile(&ctl.decider_done, 1);
    }
  } else if (warp == kClService) {
    service_loop<ENT>(a, ctl);
  } else {
    // ------------------------------------------------------------------
    // compute warps: the ring's items in order
    // ------------------------------------------------------------------
    float mT = neg_inf(), mD = neg_inf();
    f2_t aT = f2(0.f, 0.f), aD = f2(0.f, 0.f), eT = f2(0.f, 0.f), eD = f2(0.f, 0.f);
    float dwb = 0.f;  // draw: this warp's bonus mass over the sub-chunks so far
    for (int t = 0;; ++t) {
      const int s = t % S;
      if (!mbar_wait_local(&ctl.full[s], (unsigned)((t / S) & 1)) && lane == 0) atomicOr(a.status, kStatusTimeout);
      const Desc dsc = ctl.desc[s];
      if (dsc.type == kItemEnd) break;
      const Sto* bufT = (const Sto*)(smem + (size_t)s * bufb);
      const Sto* bufD = (const Sto*)(smem + (size_t)s * bufb + rowb);
      int e0, e1;
      sub_range(dsc.j, e0, e1);
      const int len = e1 - e0;
      const int nst = (len + STEPW - 1) / STEPW;
      const int q0 = (warp * nst) / kClCompute, q1 = ((warp + 1) * nst) / kClCompute;
      if (dsc.type == kItemStats) {
        const int q = dsc.k % kClSlots;
        const bool pair = dsc.i < K;
        if (dsc.j == 0) {  // a new unit: fresh running statistics
          mT = mD = neg_inf();
          aT = aD = eT = eD = f2(0.f, 0.f);
        }
        // this warp's steps of the sub-chunk, all loaded before the arithmetic
        // (steps past the warp's share are skipped warp-uniformly; only the
        // chunk's last step can hold elements past its end)
        Raw<E, VEC> zt[kClMaxStepsW], zd[kClMaxStepsW];
#pragma unroll
        for (int w2 = 0; w2 < kClMaxStepsW; ++w2) {
          zt[w2].w = neg_inf_vec<E>();
          zd[w2].w = neg_inf_vec<E>();
          if (q0 + w2 < q1) {
            const int e = ((q0 + w2) * 32 + lane) * VEC;
            if (e < len) {
              zt[w2].w = ld_shared16(bufT + e);
              if (pair) zd[w2].w = ld_shared16(bufD + e);
            }
          }
        }
        // the logits at x_i, if this warp's steps hold them
        if (lane == 0 && pair) {
          const int xe = dsc.x - v0 - e0;  // element within the sub-chunk
          if (xe >= q0 * STEPW && xe < q1 * STEPW && xe < len && xe >= 0) {
            ctl.zx[q][0] = smem_elem<E>(bufT + xe);
            ctl.zx[q][1] = smem_elem<E>(bufD + xe);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.empty[s]);  // done with the buffer
        item_stats<E, VEC, ENT>(zt, zd, q1 - q0, pair, mT, aT, eT, mD, aD, eD, a.c_hi);
        if (dsc.j == NSC - 1) {
          // the unit is done for this warp: its (m, s) pairs into the slot
          float sT = f2lo(aT) + f2hi(aT), sD = f2lo(aD) + f2hi(aD);
          float tT = 0.f, tD = 0.f;
          if constexpr (ENT) {
            tT = f2lo(eT) + f2hi(eT);
            tD = f2lo(eD) + f2hi(eD);
            warp_mst(mT, sT, tT, a.c_hi);
            warp_mst(mD, sD, tD, a.c_hi);
          } else {
            warp_ms2(mT, sT, mD, sD, a.c_hi);
          }
          int last = 0;
          if (lane == 0) {
            float* w6 = ctl.wp[q][warp];
            w6[0] = mT; w6[1] = sT; w6[2] = tT; w6[3] = mD; w6[4] = sD; w6[5] = tD;
            __threadfence_block();
            last = atomicAdd(&ctl.ucnt[q], 1) == kClCompute - 1;
          }
          last = __shfl_sync(0xffffffffu, last, 0);
          if (last) {
            // merge the 16 warps in order and push the CTA's record to every CTA
            __threadfence_block();
            float m1 = neg_inf(), s1 = 0.f, t1 = 0.f, m2 = neg_inf(), s2 = 0.f, t2 = 0.f;
            if (lane < kClCompute) {
              const float* w6 = ctl.wp[q][lane];
              m1 = w6[0]; s1 = w6[1]; t1 = w6[2]; m2 = w6[3]; s2 = w6[4]; t2 = w6[5];
            }
            if constexpr (ENT) {
              warp_mst(m1, s1, t1, a.c_hi);
              warp_mst(m2, s2, t2, a.c_hi);
            } else {
              warp_ms2(m1, s1, m2, s2, a.c_hi);
            }
            const float z1 = ctl.zx[q][0], z2 = ctl.zx[q][1];
            const uint32_t frv = rank == 0 ? dsc.fr : 0xffffffffu;
            __syncwarp();
            if (lane == 0) {  // the slot's next unit starts from scratch
              ctl.ucnt[q] = 0;
              ctl.zx[q][0] = ctl.zx[q][1] = u2f(kMarker);
            }
            // every CTA's copy of the slot is free once all deciders consumed
            // unit k - kClSlots
            if (dsc.k >= kClSlots && !mbar_wait(&ctl.xfree[q], (unsigned)(((dsc.k / kClSlots) - 1) & 1)) &&
                lane == 0)
              atomicOr(a.status, kStatusTimeout);
            if (lane < C) {
              Rec* dst = &ctl.rec[q][rank];
              push16(&dst->mT, &ctl.xb[q], lane, make_uint4(f2u(m1), f2u(s1), f2u(t1), f2u(z1)));
              push16(&dst->mD, &ctl.xb[q], lane, make_uint4(f2u(m2), f2u(s2), f2u(t2), f2u(z2)));
              push16(&dst->fr, &ctl.xb[q], lane, make_uint4(frv, 0u, 0u, 0u));
            }
          }
          __syncwarp();
        }
      } else {
        // draw item: the replacement / bonus weights of this warp's steps
        const int ds = dsc.d % kClDrawSlots;
        const TailConsts kc = ctl.dreq[ds].kc;
        Raw<E, VEC> zt[kClMaxStepsW], zd[kClMaxStepsW];
#pragma unroll
        for (int w2 = 0; w2 < kClMaxStepsW; ++w2) {
          zt[w2].w = neg_inf_vec<E>();
          if (q0 + w2 < q1) {
            const int e = ((q0 + w2) * 32 + lane) * VEC;
            if (e < len) zt[w2].w = ld_shared16(bufT + e);
          }
          zd[w2].w = zt[w2].w;
          if (kc.residual && q0 + w2 < q1) {
            const int e = ((q0 + w2) * 32 + lane) * VEC;
            if (e < len) zd[w2].w = ld_shared16(bufD + e);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.empty[s]);  // done with the buffer
        if (dsc.j == 0) dwb = 0.f;
        // step masses as the decider's rescan forms them (a warp sum per step);
        // the bonus mass is only needed as a total
        float wm = 0.f, lbs = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kClMaxStepsW; ++w2) {
          if (q0 + w2 < q1) {
            float lb;
            const float ls = lane_mass_both<E, VEC>(zt[w2], zd[w2], kc, lb);
            wm += warp_sum(ls);
            lbs += lb;
          }
        }
        dwb += kc.residual ? warp_sum(lbs) : wm;
        if (lane == 0) ctl.wsub[ds][dsc.j][warp] = wm;
        if (dsc.j == NSC - 1) {
          int last = 0;
          if (lane == 0) {
            ctl.wbon[ds][warp] = dwb;
            __threadfence_block();
            last = atomicAdd(&ctl.dcnt[ds], 1) == kClCompute - 1;
          }
          last = __shfl_sync(0xffffffffu, last, 0);
          if (last) {
            __threadfence_block();
            // the CTA's masses in fixed order: sub-chunks, then warps
            double cm = 0.0;
            for (int j = 0; j < NSC; ++j)
              cm += warp_sum_f64(lane < kClCompute ? (double)ctl.wsub[ds][j][lane] : 0.0);
            const double cb = warp_sum_f64(lane < kClCompute ? (double)ctl.wbon[ds][lane] : 0.0);
            __syncwarp();
            if (lane == 0) ctl.dcnt[ds] = 0;
            if (dsc.d >= kClDrawSlots &&
                !mbar_wait(&ctl.dfree[ds], (unsigned)(((dsc.d / kClDrawSlots) - 1) & 1)) && lane == 0)
              atomicOr(a.status, kStatusTimeout);
            if (lane < C) {
              const unsigned long long cmb = (unsigned long long)__double_as_longlong(cm);
              const unsigned long long cbb = (unsigned long long)__double_as_longlong(cb);
              push16(&ctl.dmass[ds][rank][0], &ctl.db[ds], lane,
                     make_uint4((uint32_t)cmb, (uint32_t)(cmb >> 32), (uint32_t)cbb, (uint32_t)(cbb >> 32)));
            }
          }
          __syncwarp();
        }
      }
    }
  }
  // no CTA leaves while another may still push into its shared memory
  __syncwarp();
  cluster_sync_all();
}

}  // namespace

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static size_t cl_align(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t cluster_smem_bytes(int S, size_t buf_bytes) {
  return cl_align((size_t)S * buf_bytes, 128) + sizeof(Ctl);
}

// Workspace: arrive [B], firstrej [B], verdict [B, K+1], slot [B, K+1]; one
// 0xff fill starts the counts at -1, the first-rejection words at "none" and
// the slots at the marker.
static void cluster_layout(int B, int K, size_t* off) {
  size_t o = 0;
  off[0] = o; o += cl_align((size_t)B * 4, 256);
  off[1] = o; o += cl_align((size_t)B * 4, 256);
  off[2] = o; o += cl_align((size_t)B * (K + 1) * 4, 256);
  off[3] = o; o += cl_align((size_t)B * (K + 1) * 8, 256);
  off[4] = o;
}

WsLayout cluster_workspace(int B, int K) {
  size_t off[5];
  cluster_layout(B, K, off);
  WsLayout l;
  l.total = off[4];
  l.zero_bytes = 0;
  l.marker_off = 0;
  l.marker_bytes = off[4];
  return l;
}

void cluster_bind_workspace(ClusterArgs& a, void* ws) {
  size_t off[5];
  cluster_layout(a.B, a.K, off);
  char* p = (char*)ws;
  a.arrive = (int*)(p + off[0]);
  a.firstrej = (unsigned*)(p + off[1]);
  a.verdict = (int*)(p + off[2]);
  a.slot = (uint2*)(p + off[3]);
}

template <class E, bool ENT>
static cudaError_t prepare_t(int smem_max) {
  auto* k = cluster_kernel<E, ENT>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

cudaError_t cluster_prepare(int smem_max) {
  cudaError_t e = prepare_t<BF16, false>(smem_max);
  if (e == cudaSuccess) e = prepare_t<BF16, true>(smem_max);
  if (e == cudaSuccess) e = prepare_t<F32, false>(smem_max);
  if (e == cudaSuccess) e = prepare_t<F32, true>(smem_max);
  return e;
}

template <class E, bool ENT>
static cudaError_t launch_t(const ClusterArgs& a, int clusters, size_t smem, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(clusters * a.C), 1, 1);
  cfg.blockDim = dim3(kClThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)a.C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, cluster_kernel<E, ENT>, a);
}

cudaError_t launch_cluster(const ClusterArgs& a, bool bf16, bool ent, int clusters, size_t smem,
                           cudaStream_t s) {
  if (bf16) return ent ? launch_t<BF16, true>(a, clusters, smem, s) : launch_t<BF16, false>(a, clusters, smem, s);
  return ent ? launch_t<F32, true>(a, clusters, smem, s) : launch_t<F32, false>(a, clusters, smem, s);
}

template <class E, bool ENT>
static int max_active_t(int C, size_t smem) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)C, 1, 1);
  cfg.blockDim = dim3(kClThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, cluster_kernel<E, ENT>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

int cluster_max_active(bool bf16, bool ent, int C, size_t smem) {
  if (bf16) return ent ? max_active_t<BF16, true>(C, smem) : max_active_t<BF16, false>(C, smem);
  return ent ? max_active_t<F32, true>(C, smem) : max_active_t<F32, false>(C, smem);
}

}  // namespace sv
