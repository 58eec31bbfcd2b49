// sample_kernel.cu -- fused speculative-sampling verify kernel (temperature > 0).
//
// Implements, for every sequence b (pages: "Speculative Decoding & Draft Model
// Topologies ..." sec. 2; "Speculative Decoding for LLM Inference ..." sections
// "The draft-and-verify loop" and "The correctness guarantee"; "Speculative
// Decoding at Scale ..." sec. 1; "Speculative Decoding in Production ..." sec. 2):
//   1. temperature-softmax statistics of the K+1 target rows and K draft rows,
//   2. the gather of p_i(x_i) and q_i(x_i) at the drafted tokens,
//   3. the acceptance test u_i < min(1, p_i(x_i) / q_i(x_i)),
//   4. the first-rejection scan giving n,
//   5. the replacement distribution max(0, p_n - q_n) (n < K) or the bonus
//      distribution p_K (n == K), and
//   6. an inverse-CDF draw from it.
//
// Work decomposition: one persistent grid of independent warps (sv_kernels.h).
//   * statistics slice = SL elements of one row: an online (max, sum of
//     exp2) pass with 16-byte streaming loads and packed f32x2 arithmetic,
//     reduced to one (m, s) pair in the workspace.  Slices are streamed by
//     draft position (position-major, with position 0 spread through the
//     first part of the stream).  The warp that takes the last ticket of a
//     position's row pair merges both rows, runs steps 2-3 for that position
//     (the ratio from error-free fp32 differences, see accept_draw) and
//     records the verdict; the verdict that completes the prefix
//     0..n fixes n (step 4) and appends the sequence's decision to the
//     decision queue, without waiting for the rows after the first rejection.
//   * tail slice = a segment of the tail row (pair) of a decided sequence:
//     the mass of every warp step ("piece") of the replacement / bonus
//     distribution, streamed through a per-warp shared-memory ring.  Tail
//     items are owned by fixed warps; a warp polls its next item's queue entry
//     while it streams statistics slices and takes the item once the entry is
//     there, so no warp ever waits for a decision while statistics work is
//     left.  The warp that takes the last tail ticket finds the CDF crossing
//     from the slice and piece masses and rescans one piece (step 6).
//   * commit: a sequence's outputs are written once its token is drawn and
//     every one of its rows has been checked for bad data.
// Every reduction runs in a fixed order, so results are run-to-run identical.
#include "sv_common.cuh"
#include "sv_kernels.h"

#include <math.h>

namespace sv {

template <class E>
__device__ __forceinline__ const typename E::storage* target_row(const SampleArgs& a, int b, int r) {
  return (const typename E::storage*)a.target + ((size_t)b * (a.K + 1) + r) * (size_t)a.V;
}
template <class E>
__device__ __forceinline__ const typename E::storage* draft_row(const SampleArgs& a, int b, int r) {
  return (const typename E::storage*)a.draft + ((size_t)b * a.K + r) * (size_t)a.V;
}

__device__ __forceinline__ TailConsts tail_consts(const SampleArgs& a, const SeqInfo& si) {
  TailConsts k;
  k.mT = si.mT;
  k.mD = si.mD;
  k.c_hi = a.c_hi;
  k.c_lo = a.c_lo;
  k.lam_hi = si.lam_hi;
  k.lam_lo = si.lam_lo;
  k.residual = si.mode == kModeResidual;
  return k;
}

// ---------------------------------------------------------------------------
// decision queue.  The decider of a sequence takes the next queue position
// and writes its SeqInfo there with two relaxed 16-byte stores; a reader
// validates each field against kMarker (a NaN no field ever holds).
// ---------------------------------------------------------------------------
// Lane 0 takes the next queue position (a predicated atomic: nothing waits
// for it until the entry is written).
__device__ __forceinline__ int reserve_decision(const SampleArgs& a, int lane) {
  int v = -1;
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.eq.s32 p, %1, 0;\n\t"
      "@p atom.relaxed.gpu.global.add.s32 %0, [%2], 1;\n\t}"
      : "+r"(v)
      : "r"(lane), "l"(a.qcount)
      : "memory");
  return v + 1;
}

__device__ __forceinline__ void publish_decision(const SampleArgs& a, int pos, const SeqInfo& si) {
  uint32_t* e = (uint32_t*)(a.queue + pos);
  st_relaxed_v4(e, (uint32_t)si.b, (uint32_t)si.n, (uint32_t)si.mode, __float_as_uint(si.mT));
  st_relaxed_v4(e + 4, __float_as_uint(si.mD), __float_as_uint(si.lam_hi), __float_as_uint(si.lam_lo),
                __float_as_uint(si.sT));
}

__device__ __forceinline__ bool word_set(uint32_t v) { return v != kMarker; }

// First word (the sequence id) of queue entry pos, loaded by lane 0 when
// `pred` holds (kMarker elsewhere); nothing waits for it until it is read.
__device__ __forceinline__ uint32_t poll_decision(const SampleArgs& a, bool pred, int pos) {
  return ld_relaxed_if(pred, a.queue + pos, kMarker);
}

// Lane 0's bounded wait for the first word of queue entry pos (kMarker if the
// wait ran out, which is flagged).
__device__ __forceinline__ uint32_t wait_decision(const SampleArgs& a, int pos) {
  unsigned it = 0, nap = 64;
  uint32_t seen = poll_decision(a, true, pos);
  while (!word_set(seen) && ++it < spin_limit()) {
    __nanosleep(nap);
    if (nap < 256) nap <<= 1;  // (a 1 us cap cost c1 0.8 us per call)
    seen = poll_decision(a, true, pos);
  }
  if (!word_set(seen)) atomicOr(a.status, kStatusTimeout);
  return seen;
}

// The whole entry, once its first word has been seen; the other fields were
// stored at the same moment, so the bounded wait is at most a few round trips.
__device__ __noinline__ SeqInfo read_decision(const SampleArgs& a, int pos) {
  const uint32_t* e = (const uint32_t*)(a.queue + pos);
  uint4 x = ld_relaxed_v4(e), y = ld_relaxed_v4(e + 4);
  unsigned it = 0;
  bool ok;
  while (!(ok = word_set(x.x) && word_set(x.y) && word_set(x.z) && word_set(x.w) && word_set(y.x) &&
                word_set(y.y) && word_set(y.z) && word_set(y.w)) &&
         ++it < spin_limit()) {
    __nanosleep(64);
    x = ld_relaxed_v4(e);
    y = ld_relaxed_v4(e + 4);
  }
  SeqInfo si;
  if (!ok) {
    atomicOr(a.status, kStatusTimeout);
    si.mode = kModeBad;  // treated as undecided: the tail slices do nothing
  } else {
    si.mode = (int)x.z;
  }
  si.b = (int)x.x;
  si.n = (int)x.y;
  si.mT = __uint_as_float(x.w);
  si.mD = __uint_as_float(y.x);
  si.lam_hi = __uint_as_float(y.y);
  si.lam_lo = __uint_as_float(y.z);
  si.sT = __uint_as_float(y.w);
  return si;
}

// ---------------------------------------------------------------------------
// Position units.  Unit (b, i) is the row pair of draft position i of
// sequence b (target row i and draft row i), or target row K alone for i = K.
// The warp that takes a unit's last slice ticket merges the slice partials of
// its rows, tests position i and records the verdict in the sequence's
// resolution word.  A sequence is decided as soon as positions 0..n are
// resolved with 0..n-1 accepted and n rejected (or 0..K resolved and all K
// accepted): the rows of the positions after n never delay the decision.
// Its outputs are committed once every row has also been checked for bad data.
// ---------------------------------------------------------------------------
constexpr int kUnitBad = 0x10000;   // added to the sequence's unit count by a unit with bad data
constexpr uint32_t kResultBad = 0x7ffffffeu;  // result slot field: no value (never kMarker)

__device__ __forceinline__ int unit_slices(const SampleArgs& a, int i) { return i < a.K ? 2 * a.CS : a.CS; }

// Lane 0: record the verdict of position i of sequence b.  Returns n (lane 0)
// if this resolution is the one that decides the sequence, else -1.  With
// K <= 31 the resolved and rejected positions live in one 64-bit word per
// sequence (stored complemented, so that the all-ones fill is the empty set)
// and the one atomic whose result crosses into "decided" identifies the
// decider.  With larger K the sequence is decided by its last resolution,
// which scans the verdicts in position order.
__device__ __forceinline__ int resolve_position(const SampleArgs& a, int b, int i, int verdict) {
  if (a.K <= kMaskMaxK) {
    unsigned long long bits = 1ull << i;
    if (verdict != kVerdictAccept && i < a.K) bits |= 1ull << (32 + i);
    const unsigned long long old_set = ~atomicAnd(a.resword + b, ~bits);
    const int was = decided_n(old_set, a.K), now = decided_n(old_set | bits, a.K);
    return (was < 0 && now >= 0) ? now : -1;
  }
  return ticket_take(a.posticket + b) == a.K ? a.K + 1 : -1;  // K + 1: scan the verdicts
}

// The suggested next draft length of sequence b, decided at n (one warp): the
// mean entropy of target rows 0..n (fp64 sum of the stored fp32 values)
// against the two thresholds, one step from K, clamped to [k_min, k_max].
__device__ __noinline__ void commit_khint(const SampleArgs& a, int b, int n) {
  const int lane = threadIdx.x & 31;
  const float* h = a.hrow + (size_t)b * (a.K + 1);
  double sum = 0.0;
  for (int i = lane; i <= n; i += 32) sum += (double)wait_f32(h + i, a.status);
  sum = warp_sum_f64(sum);
  if (lane == 0) {
    const double hbar = sum / (double)(n + 1);
    int k = a.K;
    if (hbar < a.h_lo)
      k = a.K + 1;
    else if (hbar > a.h_hi)
      k = a.K - 1;
    a.out_khint[b] = max(a.k_min, min(a.k_max, k));
    if (a.out_hmean) a.out_hmean[b] = (float)hbar;
  }
}

// Commit (one warp): writes out_tokens, out_n and out_resid (and the draft
// length suggestion when asked for).  A sequence's
// commit count gathers K + 2 arrivals: one per position unit (with kUnitBad
// added when the unit saw bad data) and one for the result (the drawn token,
// or a bad decision).  Whichever arrives last commits, with the bad-data
// verdict of every unit in the count's high bits.  The result comes in `res`
// when the committer is the result side, else from the result slot.  In
// early-exit mode the rows after the decision are not all read: the result
// side commits at once, and only the rows the decision used were checked.
__device__ __noinline__ void commit_sequence(const SampleArgs& a, int b, bool rows_bad, bool have, uint4 res) {
  const int lane = threadIdx.x & 31;
  const int K = a.K;
  if (!have) res = wait_result(a.result + b, a.status);
  const bool bad = rows_bad || res.x == kResultBad;
  int32_t* out = a.out_tokens + (size_t)b * (K + 1);
  const int32_t* x = a.tokens + (size_t)b * K;
  if (bad) {
    for (int j = lane; j <= K; j += 32) out[j] = -1;
    if (lane == 0) {
      a.out_n[b] = -1;
      atomicOr(a.status, kStatusBadData);
      if (a.out_resid) a.out_resid[b] = NAN;
      if (a.out_khint) a.out_khint[b] = -1;
      if (a.out_hmean) a.out_hmean[b] = NAN;
    }
  } else {
    const int n = (int)res.x;
    const int token = res.y == kResultBad ? -1 : (int)res.y;
    for (int j = lane; j <= K; j += 32) out[j] = j < n ? __ldg(x + j) : (j == n ? token : -1);
    if (lane == 0) {
      a.out_n[b] = n;
      if (a.out_resid) a.out_resid[b] = __uint_as_float(res.z);
    }
    if (a.out_khint) commit_khint(a, b, n);
  }
  __syncwarp();
}

// The result side's arrival: the result slot has been stored (lane 0) before.
__device__ __forceinline__ void commit_result(const SampleArgs& a, int b, uint4 res) {
  const int lane = threadIdx.x & 31;
  if (a.early_exit) {
    commit_sequence(a, b, false, true, res);
    return;
  }
  int old = 0;
  if (lane == 0) old = atom_add_relaxed(a.seqticket + b, 1) + 1;  // arrivals before this one
  old = __shfl_sync(0xffffffffu, old, 0);
  if ((old & (kUnitBad - 1)) == a.K + 1) commit_sequence(a, b, old >= kUnitBad, true, res);
}

// Decision of sequence b at n (one warp): the tail constants of row n, the
// decision queue entry, and for a bad position the result-side commit arrival.
// (mT, sT, mD, sD, verdict) are those of position n when `have` holds (the
// caller resolved it), else they are read from the workspace.
__device__ __noinline__ void decide_sequence(const SampleArgs& a, int b, int n, bool have, uint2 stT,
                                             uint2 stD, int verdict) {
  const int lane = threadIdx.x & 31;
  const int K = a.K, R = a.R;
  const int qpos = reserve_decision(a, lane);
  if (n > K) {  // K > 31: every position resolved; n = the first verdict that is not an accept
    n = K;
    for (int i0 = 0; i0 < K; i0 += 32) {
      const int i = i0 + lane;
      const int v = i < K ? wait_s32(a.verdict + (size_t)b * (K + 1) + i, a.status) : kVerdictAccept;
      const unsigned bal = __ballot_sync(0xffffffffu, v != kVerdictAccept);
      if (bal) {
        n = i0 + __ffs(bal) - 1;
        break;
      }
    }
    have = false;
  }
  if (!have) {
    const float2* rs = a.rowstat + (size_t)b * R;
    stT = wait_u2(rs + n, a.status);
    stD = n < K ? wait_u2(rs + K + 1 + n, a.status) : make_uint2(0u, 0u);
    verdict = wait_s32(a.verdict + (size_t)b * (K + 1) + n, a.status);
  }
  if (a.early_exit && lane == 0) st_relaxed_s32(a.decided + b, n);  // later slices of b may skip
  SeqInfo si;
  si.b = b;
  si.n = n;
  if (verdict == kVerdictBad) {
    si.mode = kModeBad;
    si.mT = si.mD = si.lam_hi = si.lam_lo = si.sT = 0.f;
  } else {
    si.mT = __uint_as_float(stT.x);
    si.sT = __uint_as_float(stT.y);
    if (n < K) {
      si.mode = kModeResidual;
      si.mD = __uint_as_float(stD.x);
      // log2(sT / sD) as a float pair (fp32 pairs: a double log2 costs about
      // a microsecond of latency here)
      const float2 lt = log2_pair(si.sT), ld = log2_pair(__uint_as_float(stD.y));
      const float2 lam = pair_add(lt, make_float2(-ld.x, -ld.y));
      si.lam_hi = lam.x;
      si.lam_lo = lam.y;
    } else {
      si.mode = kModeBonus;
      si.mD = 0.f;
      si.lam_hi = si.lam_lo = 0.f;
    }
  }
  if (lane == 0) publish_decision(a, qpos, si);
  if (si.mode == kModeBad) {  // no token will be drawn: the result side arrives now
    const uint4 res = make_uint4(kResultBad, kResultBad, 0x7fc00000u, 0u);
    if (lane == 0) st_relaxed_v4(a.result + b, res.x, res.y, res.z, res.w);
    commit_result(a, b, res);
  }
  __syncwarp();
}

__device__ __forceinline__ bool row_ok(uint2 w) {
  const float m = __uint_as_float(w.x), sum = __uint_as_float(w.y);
  return sum > 0.f && sum < INFINITY && m < INFINITY && m > neg_inf();
}

// Merge (in slice order: lane-strided, then the fixed warp merge) the slice
// partials of row r of sequence b from the values already loaded for slice c
// = lane, lane + 32, ...; every lane ends with the row's (m, s) (and t).
template <bool ENT>
__device__ __forceinline__ void merge_row(const SampleArgs& a, int b, int r, float& m, float& s, float& t) {
  const int lane = threadIdx.x & 31;
  const int C = a.CS;
  const float2* pp = a.part + ((size_t)b * a.R + r) * C;
  m = neg_inf();
  s = 0.f;
  t = 0.f;
  for (int c = lane; c < C; c += 32) {
    const uint2 w = wait_u2(pp + c, a.status);
    if constexpr (ENT) {
      const float tc = wait_f32(a.part_t + ((size_t)b * a.R + r) * C + c, a.status);
      mst_merge(m, s, t, __uint_as_float(w.x), __uint_as_float(w.y), tc, a.c_hi);
    } else {
      ms_merge(m, s, __uint_as_float(w.x), __uint_as_float(w.y), a.c_hi);
    }
  }
  if constexpr (ENT) {
    warp_mst(m, s, t, a.c_hi);
  } else {
    warp_ms(m, s, a.c_hi);
  }
}

// Row r's merged statistics into the workspace and the optional outputs (lane 0).
template <bool ENT>
__device__ __forceinline__ void store_row(const SampleArgs& a, int b, int r, float m, float s, float t) {
  const size_t k = (size_t)b * a.R + r;
  st_relaxed_u2(a.rowstat + k, __float_as_uint(m), __float_as_uint(s));
  if (a.out_row_stats) {
    a.out_row_stats[k * 2 + 0] = (float)((double)m * a.inv_tau);
    a.out_row_stats[k * 2 + 1] = s;
  }
  // nats: ln s - ln 2 * t / s (NaN for a row without mass or with NaN)
  if constexpr (ENT) {
    const float h = (float)(log((double)s) - 0.69314718055994530942 * (double)t / (double)s);
    if (a.out_entropy) a.out_entropy[k] = h;
    // the target rows' entropies for the committing warp (a NaN never takes
    // the marker's bit pattern)
    if (a.out_khint && r <= a.K)
      st_relaxed_f32(a.hrow + (size_t)b * (a.K + 1) + r, __float_as_uint(h) == kMarker ? NAN : h);
  }
}

// Unit finisher (one warp): position i of sequence b.
template <class E, bool ENT>
__device__ __noinline__ void unit_finisher(const SampleArgs& a, int b, int i) {
  const int lane = threadIdx.x & 31;
  const int K = a.K, R = a.R;
  const bool pair = i < K;
  const int rT = i, rD = K + 1 + i;
  // the drafted token and the logits at it (written by the slices holding it)
  const int xi = pair ? __ldg(a.tokens + (size_t)b * K + i) : 0;
  float zT = pair ? ld_relaxed_f32(a.zx + (size_t)b * R + rT) : 0.f;
  float zD = pair ? ld_relaxed_f32(a.zx + (size_t)b * R + rD) : 0.f;
  float mT, sT, tT, mD = 0.f, sD = 0.f, tD = 0.f;
  merge_row<ENT>(a, b, rT, mT, sT, tT);
  if (pair) merge_row<ENT>(a, b, rD, mD, sD, tD);
  const uint2 stT = make_uint2(__float_as_uint(mT), __float_as_uint(sT));
  const uint2 stD = make_uint2(__float_as_uint(mD), __float_as_uint(sD));
  if (lane == 0) {
    store_row<ENT>(a, b, rT, mT, sT, tT);
    if (pair) store_row<ENT>(a, b, rD, mD, sD, tD);
  }
  bool bad = !row_ok(stT);
  if (pair) bad = bad || !row_ok(stD) || xi < 0 || xi >= a.V;
  int verdict = bad ? kVerdictBad : kVerdictAccept;
  if (pair && !bad) {
    // a valid token always has a slice that records the logits at it
    if (__float_as_uint(zT) == kMarker) zT = wait_f32(a.zx + (size_t)b * R + rT, a.status);
    if (__float_as_uint(zD) == kMarker) zD = wait_f32(a.zx + (size_t)b * R + rD, a.status);
    bool accept = true;  // q(x) = 0 <= p(x)
    if (zD != neg_inf())
      accept = accept_draw(zT, mT, zD, mD, sT, sD, a.c_hi, a.c_lo,
                           uniform_draw(a.seed, (uint64_t)b, (uint64_t)i, 0));
    verdict = accept ? kVerdictAccept : kVerdictReject;
    if (a.out_pq && lane == 0) {  // the stats export (not the verify path): fp64 from exact differences
      const double lp = ((double)zT - (double)mT) * a.c64;
      const double lq = ((double)zD - (double)mD) * a.c64;
      a.out_pq[((size_t)b * K + i) * 2 + 0] = (float)(exp2(lp) / (double)sT);
      a.out_pq[((size_t)b * K + i) * 2 + 1] = (float)(exp2(lq) / (double)sD);
    }
  }
  // the verdict slot, the resolution and the sequence's unit count, issued
  // together from lane 0
  int n = -1, units = 0;
  if (lane == 0) {
    st_relaxed_s32(a.verdict + (size_t)b * (K + 1) + i, verdict);
    n = resolve_position(a, b, i, verdict);
    if (!a.early_exit) units = atom_add_relaxed(a.seqticket + b, bad ? kUnitBad + 1 : 1) + 1;
  }
  n = __shfl_sync(0xffffffffu, n, 0);
  units = __shfl_sync(0xffffffffu, units, 0);
  if (n >= 0) decide_sequence(a, b, n, n == i, stT, stD, verdict);
  // (the count starts at -1: `units` is the number of earlier arrivals, with
  // kUnitBad added once per unit that had bad data; K + 1 earlier arrivals
  // means every other unit and the result are in)
  if ((units & (kUnitBad - 1)) == K + 1 && !a.early_exit)
    commit_sequence(a, b, units >= kUnitBad || bad, false, make_uint4(0u, 0u, 0u, 0u));
  __syncwarp();
}

// ---------------------------------------------------------------------------
// tail work.  Piece q of a chunk is warp step q: the 32 x VEC elements
// starting at v0 + q * 32 * VEC; its mass is the butterfly sum over lanes of
// each lane's sequential sum of its VEC weights.
// ---------------------------------------------------------------------------

// One warp: the pieces of tail slice s of the tail row(s) into the workspace
// and the slice's mass, the fp32 sum of its pieces in order (every lane).
// RING (the vector path): the loads run kTailStages - 1 warp steps ahead of
// the arithmetic through a per-warp ring in shared memory (16-byte cp.async
// per lane and row), so that a warp keeps three steps of both rows in flight
// without holding them in registers.  With one step in flight a tail warp
// moved its bytes at half the rate of a statistics warp (its loads wait on a
// loaded memory system for about a microsecond), and the tail items of the
// sequences decided together held the grid for tens of microseconds.  The
// scalar path double-buffers in registers.
constexpr int kTailStages = 4;

template <class E, int VEC, bool RING>
__device__ float tail_slice_mass(const SampleArgs& a, int b, int s, const SeqInfo& si) {
  using S = typename E::storage;
  constexpr int STEPW = 32 * VEC;
  const int lane = threadIdx.x & 31;
  const S* rowT = target_row<E>(a, b, si.n);
  const S* rowD = si.mode == kModeResidual ? draft_row<E>(a, b, si.n) : rowT;
  const TailConsts k = tail_consts(a, si);
  const int v0 = s * a.TL, v1 = min(a.V, v0 + a.TL);
  const int nsteps = v1 > v0 ? (v1 - v0 + STEPW - 1) / STEPW : 0;
  float* gp = a.pieces + ((size_t)b * a.TC + s) * a.P;
  float total = 0.f;
  const int e0 = v0 + lane * VEC;
  if constexpr (VEC > 1) {
    if constexpr (RING) {
    // [warp][stage][row][lane]: 8 x 4 x 2 x 32 x 16 B = 32 KB per CTA
    __shared__ uint4 ring[kWarps][kTailStages][2][32];
    uint4(*my)[2][32] = ring[threadIdx.x >> 5];
    if (lane == 0 && v1 > v0) {
      prefetch_l2(rowT + v0, (unsigned)((v1 - v0) * sizeof(S)));
      if (k.residual) prefetch_l2(rowD + v0, (unsigned)((v1 - v0) * sizeof(S)));
    }
    // group q holds step q's copies (an empty group past the end keeps the
    // count uniform); elements past v1 fill whole vectors (V * esz % 16 == 0)
    auto issue = [&](int q) {
      const int e = e0 + q * STEPW;
      if (q < nsteps && e < v1) {
        cp_async16(&my[q % kTailStages][0][lane], rowT + e);
        if (k.residual) cp_async16(&my[q % kTailStages][1][lane], rowD + e);
      }
      cp_async_commit();
    };
#pragma unroll
    for (int q = 0; q < kTailStages - 1; ++q) issue(q);
    for (int q = 0; q < nsteps; ++q) {
      issue(q + kTailStages - 1);  // refills the stage step q - 1 used
      cp_async_wait<kTailStages - 1>();  // step q's group has landed
      const int e = e0 + q * STEPW;
      Raw<E, VEC> t, d;
      if (e < v1) {
        t.w = ld_shared16(&my[q % kTailStages][0][lane]);
        d.w = k.residual ? ld_shared16(&my[q % kTailStages][1][lane]) : t.w;
      } else {
        t.w = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
        d.w = t.w;
      }
      const float ps = warp_sum(lane_mass<E, VEC>(t, d, k));
      if (lane == 0) st_relaxed_f32(gp + q, ps);
      total += ps;
    }
    cp_async_wait<0>();
    return total;
    }
    if (lane == 0 && v1 > v0) {
      prefetch_l2(rowT + v0, (unsigned)((v1 - v0) * sizeof(S)));
      if (k.residual) prefetch_l2(rowD + v0, (unsigned)((v1 - v0) * sizeof(S)));
    }
  }
  {
    Raw<E, VEC> t0{}, d0{}, t1{}, d1{};
    int e = e0;
    if (nsteps > 0) {
      t0 = load_raw<E, VEC>(rowT, e, v1);
      d0 = k.residual ? load_raw<E, VEC>(rowD, e, v1) : t0;
    }
    for (int q = 0; q < nsteps; q += 2, e += 2 * STEPW) {
      const bool has1 = q + 1 < nsteps;
      if (has1) {
        t1 = load_raw<E, VEC>(rowT, e + STEPW, v1);
        d1 = k.residual ? load_raw<E, VEC>(rowD, e + STEPW, v1) : t1;
      }
      float ps = warp_sum(lane_mass<E, VEC>(t0, d0, k));
      if (lane == 0) st_relaxed_f32(gp + q, ps);
      total += ps;
      if (has1) {
        if (q + 2 < nsteps) {
          t0 = load_raw<E, VEC>(rowT, e + 2 * STEPW, v1);
          d0 = k.residual ? load_raw<E, VEC>(rowD, e + 2 * STEPW, v1) : t0;
        }
        ps = warp_sum(lane_mass<E, VEC>(t1, d1, k));
        if (lane == 0) st_relaxed_f32(gp + q + 1, ps);
        total += ps;
      }
    }
  }
  return total;
}

// ---------------------------------------------------------------------------
// select finisher (one warp): inverse CDF over the tail slices' masses
// ---------------------------------------------------------------------------

template <class E, int VEC, bool RING>
__device__ __noinline__ void select_finisher(const SampleArgs& a, SeqInfo si) {
  using S = typename E::storage;
  constexpr int STEPW = 32 * VEC;
  const int lane = threadIdx.x & 31;
  const int b = si.b, n = si.n;
  const int C = a.TC;  // tail slices of the row, in vocabulary order
  float* ts = a.tailsum + (size_t)b * C;
  const double w = uniform_draw(a.seed, (uint64_t)b, (uint64_t)n, 1);
  // Z: the slice masses, lane-strided, four per lane per round of loads, then a
  // fixed-order butterfly
  double z = 0.0;
  for (int c0 = 0; c0 < C; c0 += 128) {
    float v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int t = c0 + 32 * q + lane;
      v[q] = t < C ? ld_relaxed_f32(ts + t) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int t = c0 + 32 * q + lane;
      if (t < C && __float_as_uint(v[q]) == kMarker) v[q] = wait_f32(ts + t, a.status);
      z += (double)v[q];
    }
  }
  double Z = warp_sum_f64(z);
  // Z == 0 after a rejection can only come from rounding (p(x_n) < q(x_n)
  // forces a positive residual); then the draw falls back to p_n itself, and
  // this warp recomputes every piece in bonus mode with the same arithmetic.
  if (si.mode == kModeResidual && !(Z > 0.0)) {
    si.mode = kModeBonus;
    z = 0.0;
    for (int t = 0; t < C; ++t) {
      const float tot = tail_slice_mass<E, VEC, RING>(a, b, t, si);
      if (lane == 0) st_relaxed_f32(ts + t, tot);
      if (lane == (t & 31)) z += (double)tot;
    }
    __syncwarp();
    Z = warp_sum_f64(z);
  }
  const double theta = w * Z;

  // Slice, then piece, then lane, then element holding the crossing.  Only
  // positions with positive mass are ever chosen, so the emitted token always
  // carries weight (and lies below V).
  // (every slice mass has been seen above, so plain relaxed reloads return it)
  double acc = 0.0;
  const int tsel =
      warp_cdf_search(C, theta, 0.0, [&](int t) { return (double)ld_relaxed_f32(ts + t); }, &acc);
  if (tsel < 0) {  // no slice with mass: only an expired wait can cause this
    const uint4 res = make_uint4((uint32_t)n, kResultBad, __float_as_uint(__fdiv_rn((float)Z, si.sT)), 0u);
    if (lane == 0) {
      atomicOr(a.status, kStatusTimeout);
      st_relaxed_v4(a.result + b, res.x, res.y, res.z, res.w);
    }
    commit_result(a, b, res);
    return;
  }
  const int v0 = tsel * a.TL, v1 = min(a.V, v0 + a.TL);
  const int np = (v1 - v0 + STEPW - 1) / STEPW;
  const float* gp = a.pieces + ((size_t)b * C + tsel) * a.P;
  double acc2 = acc;
  const int psel = warp_cdf_search(
      np, theta, acc, [&](int q) { return (double)wait_f32(gp + q, a.status); }, &acc2);
  if (psel < 0) {  // pieces inconsistent with their slice mass (expired wait)
    const uint4 res = make_uint4((uint32_t)n, kResultBad, __float_as_uint(__fdiv_rn((float)Z, si.sT)), 0u);
    if (lane == 0) {
      atomicOr(a.status, kStatusTimeout);
      st_relaxed_v4(a.result + b, res.x, res.y, res.z, res.w);
    }
    commit_result(a, b, res);
    return;
  }

  // rescan the 32 x VEC elements of the piece with the same arithmetic
  const int base = v0 + psel * STEPW + lane * VEC;
  const TailConsts k = tail_consts(a, si);
  const S* rowT = target_row<E>(a, b, n);
  const S* rowD = k.residual ? draft_row<E>(a, b, n) : rowT;
  float wv[VEC];
  const Raw<E, VEC> zt = load_raw<E, VEC>(rowT, base, v1);
  const Raw<E, VEC> zd = k.residual ? load_raw<E, VEC>(rowD, base, v1) : zt;
  lane_weights<E, VEC>(zt, zd, k, wv);
  float ls = 0.f;
#pragma unroll
  for (int q = 0; q < VEC; ++q) ls = __fadd_rn(ls, wv[q]);
  // exclusive prefix of the lane sums in fp64
  double incl = (double)ls;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const double o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  const double excl = incl - (double)ls;
  const unsigned has = __ballot_sync(0xffffffffu, ls > 0.f);
  const unsigned cb = __ballot_sync(0xffffffffu, ls > 0.f && acc2 + excl + (double)ls > theta);
  const int L = cb ? __ffs(cb) - 1 : (has ? 31 - __clz(has) : 0);
  int token = -1;
  if (lane == L) {
    float part = 0.f;
    int pick = -1, lastpos = -1;
#pragma unroll
    for (int q = 0; q < VEC; ++q) {
      part = __fadd_rn(part, wv[q]);
      if (wv[q] > 0.f) {
        lastpos = q;
        if (pick < 0 && acc2 + excl + (double)part > theta) pick = q;
      }
    }
    if (pick < 0) pick = lastpos;
    token = pick >= 0 ? base + pick : -1;
  }
  token = __shfl_sync(0xffffffffu, token, L);
  const uint4 res = make_uint4((uint32_t)n, token >= 0 ? (uint32_t)token : kResultBad,
                               __float_as_uint(__fdiv_rn((float)Z, si.sT)), 0u);
  if (lane == 0) st_relaxed_v4(a.result + b, res.x, res.y, res.z, res.w);
  commit_result(a, b, res);
}

// Stream order.  Claim index f is first mapped to a position-major index:
// the NA slices of the front positions (the row pairs of positions below
// the front count, every sequence) are spread through the stream, FA of every
// FQ claims, and the rest of the position-major order fills the other claims
// and the end of the stream.  Decisions (which mostly come from the front
// positions) then arrive at a steady rate instead of in one burst, so their
// tail work interleaves with the statistics stream, while the end of the
// stream holds later positions, which gate few decisions.
__device__ __forceinline__ int stream_to_pm(const SampleArgs& a, int f) {
  const int blk = fdiv(f, a.div_fq), r = f - blk * a.FQ;
  const int before = blk * a.FA;  // front slices in earlier blocks (before the cap)
  if (r < a.FA && before + r < a.NA) return before + r;
  return a.NA + f - min(a.NA, before + min(r, a.FA));
}

// Flat statistics slice f, position-major: the slices of position 0 of every
// sequence come first (for each sequence its target row, then its draft
// row), then position 1, and so on; position K (the bonus rows) comes last.
// Every sequence is then decided early in the stream (after its first
// rejection's pair), and the rows streamed at the end gate few decisions.
struct SliceId {
  int b, i, r, s;
};
__device__ __forceinline__ SliceId decode_slice(const SampleArgs& a, int f) {
  SliceId id;
  int h = 0;
  if (f < a.FP) {
    id.i = fdiv(f, a.div_pos);
    const int rem = f - id.i * a.B * 2 * a.CS;
    id.b = fdiv(rem, a.div_pair);
    const int r2 = rem - id.b * 2 * a.CS;
    h = r2 >= a.CS ? 1 : 0;
    id.s = r2 - h * a.CS;
  } else {
    id.i = a.K;
    const int rem = f - a.FP;
    id.b = fdiv(rem, a.div_cs);
    id.s = rem - id.b * a.CS;
  }
  id.r = h ? a.K + 1 + id.i : id.i;
  return id;
}

// ---------------------------------------------------------------------------
// statistics unit (one warp)
// ---------------------------------------------------------------------------
// Statistics slice s of row r (position i) of sequence b: the row's (m, s)
// over the slice, then the ticket of unit (b, i).  Returns the ticket's old
// value (lane 0).  Kept out of line so that the stream loop has the register
// file to itself.
template <class E, int VEC, bool ENT>
__device__ __noinline__ int stats_slice(const SampleArgs& a, int b, int i, int r, int s) {
  using S = typename E::storage;
  constexpr int BATCH = 32 * VEC * kUnroll;
  const int lane = threadIdx.x & 31;
  const S* row = r <= a.K ? target_row<E>(a, b, r) : draft_row<E>(a, b, r - a.K - 1);
  const int v0 = s * a.SL, v1 = min(a.V, v0 + a.SL);
  // the drafted token scored by this row (target rows 0..K-1 and every draft
  // row); its load overlaps the stream, and the slice holding it records the
  // logit there for the unit finisher
  const int ti = r < a.K ? r : (r > a.K ? r - a.K - 1 : -1);
  const uint32_t xt = ld_relaxed_if(lane == 0 && ti >= 0, a.tokens + (size_t)b * a.K + ti, kMarker);
  const float cc = a.c_hi;
  float m = neg_inf();
  float2 acc = make_float2(0.f, 0.f), tacc = make_float2(0.f, 0.f);
  // two register buffers: the next batch is in flight while one is reduced
  const int nb = v1 > v0 ? (v1 - v0 + BATCH - 1) / BATCH : 0;
  int e = v0 + lane * VEC;
  Raw<E, VEC> z0[kUnroll], z1[kUnroll];
  if constexpr (VEC > 1) {
    if (lane == 0 && v1 > v0) {
      const unsigned bytes = (unsigned)((v1 - v0) * sizeof(S));
      if (i < a.l2_keep)
        prefetch_l2_pol(row + v0, bytes, l2_policy_evict_last());
      else
        prefetch_l2(row + v0, bytes);
    }
  }
  if (nb > 0) load_batch<E, VEC>(z0, row, e, v1);
  for (int bt = 0; bt < nb; bt += 2, e += 2 * BATCH) {
    if (bt + 1 < nb) load_batch<E, VEC>(z1, row, e + BATCH, v1);
    stats_batch<E, VEC, ENT>(z0, m, acc, tacc, cc);
    if (bt + 1 < nb) {
      if (bt + 2 < nb) load_batch<E, VEC>(z0, row, e + 2 * BATCH, v1);
      stats_batch<E, VEC, ENT>(z1, m, acc, tacc, cc);
    }
  }
  float sum = acc.x + acc.y;
  float tsum = 0.f;
  // the fused exponents' common offset out (see exp_fma_err)
  if constexpr (ENT) tsum = exp_fma_fix(m, cc) * __fmaf_rn(-exp_fma_err(m, cc), sum, tacc.x + tacc.y);
  sum *= exp_fma_fix(m, cc);
  if constexpr (ENT) {
    warp_mst(m, sum, tsum, cc);
  } else {
    warp_ms(m, sum, cc);
  }
  int old = 0;
  if (lane == 0) {
    if constexpr (ENT) st_relaxed_f32(a.part_t + ((size_t)b * a.R + r) * a.CS + s, tsum);
    st_relaxed_u2(a.part + ((size_t)b * a.R + r) * a.CS + s, __float_as_uint(m), __float_as_uint(sum));
    old = ticket_take(&a.unitticket[((size_t)b * (a.K + 1) + i) * kTicketStride]);
    const int xi = (int)xt;
    if (ti >= 0 && xi >= v0 && xi < v1) st_relaxed_f32(a.zx + (size_t)b * a.R + r, E::load1(row + xi));
  }
  return old;
}

// Tail slice s of a decided sequence: the slice's pieces and mass, then the
// sequence's tail ticket; the last ticket runs the select finisher.
template <class E, int VEC, bool RING>
__device__ __noinline__ void tail_slice(const SampleArgs& a, const SeqInfo& si, int s) {
  const int lane = threadIdx.x & 31;
  if (si.mode == kModeBad) return;  // no draw: the decision made the result-side commit arrival
  const int b = si.b;
  const float tot = tail_slice_mass<E, VEC, RING>(a, b, s, si);
  int old = 0;
  if (lane == 0) {
    // pieces and mass are marker-validated by the reader: no ordering needed
    st_relaxed_f32(a.tailsum + (size_t)b * a.TC + s, tot);
    old = ticket_take(&a.tailticket[b]);
  }
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old == a.TC - 1) select_finisher<E, VEC, RING>(a, si);
}

// The next counter after ctr (cyclically) that this warp has not seen run dry.
__device__ __forceinline__ int next_live_counter(int ctr, unsigned dead) {
  for (int k = 1; k <= kSlices; ++k) {
    const int c = (ctr + k) & (kSlices - 1);
    if (!((dead >> c) & 1u)) return c;
  }
  return ctr;
}

// Scheduling.  Statistics slices come from eight claim counters: the k-th
// claim on counter c is flat slice f = k * kSlices + c, where claims
// 0 .. grid-1 of every counter are the warps' static first claims and the
// counters hand out the rest.  The next claim is issued before the current
// slice is processed, so the atomic's latency hides behind the stream.  Tail slices of the first TTo / TC queue positions
// are owned, not claimed: tail item j (queue position j / TC, tail slice
// j % TC) belongs to global warp j % W, where warp slot w of CTA c is global
// warp w * grid + c and W = 8 * grid.  A warp takes its items in order and
// polls the queue entry of its next item with a relaxed load issued before
// each statistics slice; a published item is taken before the next
// statistics slice.  Only when a warp has no statistics slice left does it
// wait (bounded) for its next entry.  The tail items of the last queue
// positions -- the latest decisions, which come near the end of the stream
// -- are claimed in order by warps that have nothing else left, so that no
// late tail waits for a busy owner.
//
// Progress: statistics slices and the finishers they trigger wait only for
// stores that other warps have already issued (their tickets were counted); a
// warp holding a claimed statistics slice never waits, and a warp waits for a
// queue entry only when it has no statistics work left; every sequence is
// decided once the statistics slices of its positions up to the first
// rejection are done.  Every statistics slice is claimed by a CTA that is
// already running: the first claims are numbered by the order in which CTAs
// start (a per-launch ticket), not by their index, and the rest come from the
// counters.  So every queue entry is eventually written and every wait ends,
// whatever part of the grid is resident at a time (another kernel may hold
// some SMs until after this launch's first CTAs finish).
template <class E, int VEC, bool ENT>
__global__ void __launch_bounds__(kThreads, kMinBlocks) sample_kernel(const __grid_constant__ SampleArgs a) {
  const int lane = threadIdx.x & 31;
  const int w = slice_of_warp();
  const int TT = a.B * a.TC;                       // tail items in all
  const int TO = a.TTo;                            // owned tail items: the first TTo
  const int W = kSlices * (int)gridDim.x;          // warps in the grid
  // this CTA's start order in the launch (its first claims and owned tail
  // items follow it), one ticket for the whole CTA
  __shared__ int cta_order;
  if (threadIdx.x == 0) cta_order = ticket_take(a.ctaticket);
  __syncthreads();
  const int tk = cta_order;
  int t = w * (int)gridDim.x + tk;                 // this warp's next owned tail item
  if (t >= TO) t = TT;
  // Statistics claims rotate over the eight counters (warp slot w starts at
  // counter w), so every warp draws equally from every counter and the
  // counters advance together.  A claim past a counter's end marks that
  // counter dead for this warp; the warp leaves the statistics work only when
  // it has seen all eight dead, so no slice is ever left unclaimed.  A claimed
  // slice is processed before a tail item that became ready (other warps'
  // decisions may wait on it); the claim after it is then deferred until the
  // tail item is done.
  // The first claim of every warp comes with its CTA's ticket (claim index tk
  // on counter w), so the first slices start streaming after one round trip
  // per CTA; claims made through the counters are offset by the grid size.
  const int k0 = (int)gridDim.x;
  unsigned dead = 0;
  int ctr = w;
  int f = tk * kSlices + ctr;
  bool held = true;  // f is the result of a claim on counter ctr
  uint32_t seen = poll_decision(a, lane == 0 && t < TO, fdiv(t, a.div_tc));
  for (;;) {
    const bool tail_ready = t < TO && word_set(bcast((int)seen));
    if (held && f >= a.F) {  // the claim came back past the counter's end
      dead |= 1u << ctr;
      held = false;
    }
    if (held) {
      int nctr = ctr, next = 0;
      // Near the end of the statistics stream a claim made ahead would sit
      // behind this slice while idle warps could start it at once, so the
      // last slices are claimed only when a warp is free.
      const bool ahead = !tail_ready && f < a.F - a.claim_tail;
      if (!ahead) held = false;
      if (ahead) {
        nctr = next_live_counter(ctr, dead);
        next = claim_from(a.counter, nctr, lane);
      }
      if (!tail_ready) seen = poll_decision(a, lane == 0 && t < TO, fdiv(t, a.div_tc));
      const SliceId id = decode_slice(a, stream_to_pm(a, f));
      // early exit: a row after a decided sequence's first rejection (or its
      // bonus row after a rejection) cannot change the result; it is not read
      bool skip = false;
      if (a.early_exit && id.i > 0) {
        const int dn = (int)ld_relaxed_if(lane == 0, a.decided + id.b, kMarker);
        skip = bcast(dn) >= 0 && bcast(dn) < id.i;
      }
      if (!skip) {
        const int old = __shfl_sync(0xffffffffu, stats_slice<E, VEC, ENT>(a, id.b, id.i, id.r, id.s), 0);
        if (old == unit_slices(a, id.i) - 1) unit_finisher<E, ENT>(a, id.b, id.i);
      }
      if (ahead) {
        f = (bcast(next) + k0) * kSlices + nctr;
        ctr = nctr;
      }
      continue;
    }
    if (tail_ready) {
      const int pos = fdiv(t, a.div_tc);
      const SeqInfo si = read_decision(a, pos);
      tail_slice<E, VEC, (VEC > 1)>(a, si, t - pos * a.TC);
      t += W;
      if (t >= TO) t = TT;
      seen = poll_decision(a, lane == 0 && t < TO, fdiv(t, a.div_tc));
      continue;
    }
    if (dead != 0xffu) {  // nothing held: claim from the next live counter
      ctr = next_live_counter(ctr, dead);
      f = (bcast(claim_from(a.counter, ctr, lane)) + k0) * kSlices + ctr;
      held = true;
      continue;
    }
    if (t >= TT) {
      // No statistics work and no owned tail item left: take the tail items
      // of the latest decisions (queue positions from TTo / TC on) in claim
      // order, so that they run at once on warps that are free instead of
      // waiting for owners that may still be streaming.
      const int j = TO + bcast(ticket_take_if(lane == 0, a.dclaim));
      if (j >= TT) break;
      uint32_t dseen = kMarker;
      if (lane == 0) dseen = wait_decision(a, fdiv(j, a.div_tc));
      if (!word_set(bcast((int)dseen))) break;
      const int pos = fdiv(j, a.div_tc);
      const SeqInfo si = read_decision(a, pos);
      tail_slice<E, VEC, (VEC > 1)>(a, si, j - pos * a.TC);
      continue;
    }
    // no statistics work left: wait for this warp's next owned decision
    if (lane == 0) seen = wait_decision(a, fdiv(t, a.div_tc));
    if (!word_set(bcast((int)seen))) break;
  }
}

// ---------------------------------------------------------------------------
// host side helpers
// ---------------------------------------------------------------------------
static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace: [counters, tickets, resolution words, queue count (all start at
// all-ones)][marker-filled result slots: part, rowstat, tailsum, queue,
// pieces, zx, verdict, result, and part_t and hrow when the entropy is
// asked for]; one 0xff fill initialises both parts.
static void sample_layout(int B, int K, int CS, int TC, int P, bool ent, size_t* off) {
  const int R = 2 * K + 1;
  size_t o = 0;
  off[0] = o; o += kCounterBytes;                                            // counter
  off[1] = o; o += align_up((size_t)B * (K + 1) * kTicketStride * 4, 16);   // unitticket
  off[2] = o; o += align_up((size_t)B * 4, 16);                             // seqticket
  off[3] = o; o += align_up((size_t)B * 4, 16);                             // tailticket
  off[4] = o; o += 128;                                                      // qcount
  off[22] = o; o += 128;                                                     // dclaim
  off[23] = o; o += 128;                                                     // ctaticket
  off[15] = o; o += align_up((size_t)B * 4, 16);                            // posticket
  off[17] = o; o += align_up((size_t)B * 8, 16);                            // resword
  o = align_up(o, 256);
  off[5] = o;                                                                // end of counter region
  off[6] = o; o += align_up((size_t)B * R * CS * sizeof(float2), 256);      // part
  off[7] = o; o += align_up((size_t)B * R * sizeof(float2), 256);           // rowstat
  off[8] = o; o += align_up((size_t)B * TC * sizeof(float), 256);           // tailsum
  off[10] = o; o += align_up((size_t)B * sizeof(SeqInfo), 256);             // queue
  off[11] = o; o += align_up((size_t)B * TC * P * sizeof(float), 256);      // pieces
  off[13] = o; o += align_up((size_t)B * R * sizeof(float), 256);           // zx
  off[18] = o; o += align_up((size_t)B * (K + 1) * 4, 256);                 // verdict
  off[20] = o; o += align_up((size_t)B * sizeof(uint4), 256);               // result
  off[21] = o; o += align_up((size_t)B * 4, 256);                           // decided
  off[14] = o; if (ent) o += align_up((size_t)B * R * CS * sizeof(float), 256);  // part_t
  off[16] = o; if (ent) o += align_up((size_t)B * (K + 1) * sizeof(float), 256);  // hrow
  off[9] = o;                                                                // end of marker region
  off[12] = o;
}

WsLayout sample_workspace(int B, int K, int CS, int TC, int P, bool ent) {
  size_t off[24];
  sample_layout(B, K, CS, TC, P, ent, off);
  WsLayout l;
  l.total = off[12];
  l.zero_bytes = 0;  // counters and tickets start at -1: one 0xff fill covers everything
  l.marker_off = 0;
  l.marker_bytes = off[9];
  return l;
}

void sample_bind_workspace(SampleArgs& a, void* ws) {
  size_t off[24];
  const bool ent = a.out_entropy != nullptr || a.out_khint != nullptr;
  sample_layout(a.B, a.K, a.CS, a.TC, a.P, ent, off);
  char* p = (char*)ws;
  a.counter = (unsigned long long*)(p + off[0]);
  a.unitticket = (int*)(p + off[1]);
  a.seqticket = (int*)(p + off[2]);
  a.tailticket = (int*)(p + off[3]);
  a.qcount = (int*)(p + off[4]);
  a.dclaim = (int*)(p + off[22]);
  a.ctaticket = (int*)(p + off[23]);
  a.posticket = (int*)(p + off[15]);
  a.resword = (unsigned long long*)(p + off[17]);
  a.part = (float2*)(p + off[6]);
  a.rowstat = (float2*)(p + off[7]);
  a.tailsum = (float*)(p + off[8]);
  a.queue = (SeqInfo*)(p + off[10]);
  a.pieces = (float*)(p + off[11]);
  a.zx = (float*)(p + off[13]);
  a.verdict = (int*)(p + off[18]);
  a.result = (uint4*)(p + off[20]);
  a.decided = (int*)(p + off[21]);
  a.part_t = ent ? (float*)(p + off[14]) : nullptr;
  a.hrow = a.out_khint ? (float*)(p + off[16]) : nullptr;
}

template <class E, int VEC>
static cudaError_t launch_sample_t(const SampleArgs& a, int grid, cudaStream_t s) {
  if (a.out_entropy || a.out_khint)
    sample_kernel<E, VEC, true><<<grid, kThreads, 0, s>>>(a);
  else
    sample_kernel<E, VEC, false><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_sample(const SampleArgs& a, bool bf16, bool vec, int grid, cudaStream_t s) {
  if (bf16) return vec ? launch_sample_t<BF16, 8>(a, grid, s) : launch_sample_t<BF16, 1>(a, grid, s);
  return vec ? launch_sample_t<F32, 4>(a, grid, s) : launch_sample_t<F32, 1>(a, grid, s);
}

template <class E, int VEC>
static int blocks_sample_t() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, sample_kernel<E, VEC, false>, kThreads, 0) !=
      cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

int sample_blocks_per_sm(bool bf16, bool vec) {
  if (bf16) return vec ? blocks_sample_t<BF16, 8>() : blocks_sample_t<BF16, 1>();
  return vec ? blocks_sample_t<F32, 4>() : blocks_sample_t<F32, 1>();
}

cudaError_t sample_set_spin_limit(unsigned n) { return set_spin_limit_here(n); }

// Test probe of the bounded waits (one thread).  Helper k waits once on a
// slot that nothing writes (marker-filled, status word st[k]) and once on a
// slot already written (st[kProbeWaits + k]).  flags[0] bit k: the first wait
// ran out and flagged it; flags[1] bit k: the second one did (never expected).
constexpr int kProbeWaits = 7;
__global__ void wait_probe_kernel(uint32_t* slots, unsigned* st, uint32_t* flags) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  for (int half = 0; half < 2; ++half) {
    uint32_t* sl = slots + half * 16;  // 16 words: one queue entry and its neighbours
    unsigned* s = st + half * kProbeWaits;
    (void)wait_u2(sl, s + 0);
    (void)wait_s32((const int*)sl, s + 1);
    (void)wait_f32((const float*)sl, s + 2);
    (void)wait_f32_acquire((const float*)sl, s + 3);
    (void)wait_result(sl, s + 4);
    SampleArgs a = {};
    a.queue = (SeqInfo*)sl;
    a.status = s + 5;
    const SeqInfo si = read_decision(a, 0);
    if (si.mode != kModeBad && half == 0) atomicOr(s + 5, 4u);  // expired, yet taken as a decision
    a.status = s + 6;
    (void)wait_decision(a, 0);
  }
  uint32_t f0 = 0, f1 = 0;
  for (int k = 0; k < kProbeWaits; ++k) {
    if (st[k] == kStatusTimeout) f0 |= 1u << k;
    if (st[kProbeWaits + k] != 0) f1 |= 1u << k;
  }
  flags[0] = f0;
  flags[1] = f1;
}

cudaError_t sample_wait_probe(uint32_t* flags_host) {
  uint32_t* buf = nullptr;  // [32 slot words][2 x kProbeWaits status words][2 flags]
  cudaError_t e = cudaMalloc(&buf, (32 + 2 * kProbeWaits + 2) * sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  e = cudaMemset(buf, 0xff, 16 * sizeof(uint32_t));  // unwritten: every word the marker
  if (e == cudaSuccess) e = cudaMemset(buf + 16, 0, (16 + 2 * kProbeWaits + 2) * sizeof(uint32_t));
  if (e == cudaSuccess) {
    wait_probe_kernel<<<1, 32>>>(buf, buf + 32, buf + 32 + 2 * kProbeWaits);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess)
    e = cudaMemcpy(flags_host, buf + 32 + 2 * kProbeWaits, 2 * sizeof(uint32_t), cudaMemcpyDeviceToHost);
  const cudaError_t e2 = cudaFree(buf);
  return e != cudaSuccess ? e : e2;
}

}  // namespace sv
