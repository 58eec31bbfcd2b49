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
//     reduced to one (m, s) pair in the workspace.  The warp that takes a
//     sequence's last statistics ticket merges the slice pairs, runs steps
//     2-4 in fp64 and appends the sequence's decision to the decision queue.
//   * tail slice = SL elements of the tail row (pair) of a decided sequence:
//     the mass of every warp step ("piece") of the replacement / bonus
//     distribution.  Tail items are owned by fixed warps; a warp polls its
//     next item's queue entry while it streams statistics slices and takes
//     the item as soon as the entry is there, so no warp ever waits for a decision while
//     statistics work is left, and the re-read rows are still in L2.  The warp
//     that takes the last tail ticket finds the CDF crossing from the slice
//     and piece masses and rescans one piece.
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
// decision queue.  The statistics finisher of a sequence takes the next queue
// position and writes its SeqInfo there with two relaxed 16-byte stores; a
// reader validates each field against kMarker (a NaN no field ever holds).
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

// The whole entry, once its first word has been seen; the other fields were
// stored at the same moment, so the bounded wait is at most a few round trips.
__device__ __noinline__ SeqInfo read_decision(const SampleArgs& a, int pos) {
  const uint32_t* e = (const uint32_t*)(a.queue + pos);
  uint4 x = ld_relaxed_v4(e), y = ld_relaxed_v4(e + 4);
  unsigned it = 0;
  while (!(word_set(x.x) && word_set(x.y) && word_set(x.z) && word_set(x.w) && word_set(y.x) &&
           word_set(y.y) && word_set(y.z) && word_set(y.w)) &&
         ++it < kSpinLimit) {
    __nanosleep(64);
    x = ld_relaxed_v4(e);
    y = ld_relaxed_v4(e + 4);
  }
  SeqInfo si;
  if (it >= kSpinLimit) {
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
// Inputs of the statistics finisher for one chunk of 32 positions (lane i:
// position i0 + i): target row i's and draft row i's (m, s), the drafted token
// and the logits at it.  One round of independent relaxed loads; slots still
// holding the marker are waited for by the finisher.
// ---------------------------------------------------------------------------
struct FinIn {
  uint2 st, sd;
  int xi;
  float zT, zD;
};

__device__ __forceinline__ FinIn load_fin_inputs(const SampleArgs& a, int b, int i0) {
  const int K = a.K, R = a.R;
  const int i = i0 + (threadIdx.x & 31);
  const bool hasT = i <= K, hasD = i < K;
  const float2* rs = a.rowstat + (size_t)b * R;
  const float* zx = a.zx + (size_t)b * R;
  FinIn in;
  in.st = hasT ? ld_relaxed_u2(rs + i) : make_uint2(0u, 0u);
  in.sd = hasD ? ld_relaxed_u2(rs + K + 1 + i) : make_uint2(0u, 0u);
  in.xi = hasD ? __ldg(a.tokens + (size_t)b * K + i) : 0;
  in.zT = hasD ? ld_relaxed_f32(zx + i) : 0.f;
  in.zD = hasD ? ld_relaxed_f32(zx + K + 1 + i) : 0.f;
  return in;
}

// ---------------------------------------------------------------------------
// row finisher (one warp): merges the slice partials of row r in slice order
// (lane-strided, then the fixed warp merge) into rowstat; the last row of a
// sequence then runs the statistics finisher.
// ---------------------------------------------------------------------------
template <class E>
__device__ __noinline__ void stats_finisher(const SampleArgs& a, int b, FinIn pre);

// The sequence ticket is taken with a predicated atomic, and the finisher's
// inputs for positions 0..31 are loaded while it is in flight, so the last
// row goes on to the finisher without another round trip.
template <class E, bool ENT>
__device__ __noinline__ void row_finisher(const SampleArgs& a, int b, int r) {
  const int lane = threadIdx.x & 31;
  const int C = a.CS;
  const float2* pp = a.part + ((size_t)b * a.R + r) * C;
  float m = neg_inf(), s = 0.f, t = 0.f;
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
    // nats: ln s - ln 2 * t / s (NaN for a row without mass or with NaN)
    if (lane == 0)
      a.out_entropy[(size_t)b * a.R + r] =
          (float)(log((double)s) - 0.69314718055994530942 * (double)t / (double)s);
  } else {
    warp_ms(m, s, a.c_hi);
  }
  if (lane == 0) st_relaxed_u2(a.rowstat + (size_t)b * a.R + r, __float_as_uint(m), __float_as_uint(s));
  int old = ticket_take_if(lane == 0, &a.seqticket[b]);
  const FinIn pre = load_fin_inputs(a, b, 0);
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old == a.R - 1) stats_finisher<E>(a, b, pre);
}

// ---------------------------------------------------------------------------
// statistics finisher (one warp): steps 2-4 for sequence b
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool row_ok(uint2 w) {
  const float m = __uint_as_float(w.x), sum = __uint_as_float(w.y);
  return sum > 0.f && sum < INFINITY && m < INFINITY && m > neg_inf();
}
__device__ __forceinline__ uint2 shfl_u2(uint2 v, int src) {
  return make_uint2(__shfl_sync(0xffffffffu, v.x, src), __shfl_sync(0xffffffffu, v.y, src));
}

// Position i of a chunk is lane i: target row i, draft row i, the drafted
// token x_i and the two logits at x_i (recorded by the statistics slices that
// hold them).  Target row K rides along as position K.  Every chunk issues one
// round of independent loads; the decision is published before the output
// tokens are written, and its queue position is taken first so that the
// atomic's round trip overlaps the loads.
template <class E>
__device__ __noinline__ void stats_finisher(const SampleArgs& a, int b, FinIn pre) {
  const int R = a.R, K = a.K;
  const int lane = threadIdx.x & 31;
  const float2* rs = a.rowstat + (size_t)b * R;
  const float* zx = a.zx + (size_t)b * R;
  const int32_t* x = a.tokens + (size_t)b * K;
  const int qpos = reserve_decision(a, lane);
  bool bad = false;
  int n = K;
  uint2 stn = make_uint2(0u, 0u), sdn = make_uint2(0u, 0u);
  for (int i0 = 0; i0 <= K; i0 += 32) {
    const int i = i0 + lane;
    const bool hasT = i <= K, hasD = i < K;
    const FinIn in = i0 == 0 ? pre : load_fin_inputs(a, b, i0);
    uint2 st = in.st, sd = in.sd;
    const int xi = in.xi;
    float zT = in.zT, zD = in.zD;
    if (hasT && st.x == kMarker) st = wait_u2(rs + i, a.status);
    if (hasD && sd.x == kMarker) sd = wait_u2(rs + K + 1 + i, a.status);
    if (a.out_row_stats) {
      if (hasT) {
        a.out_row_stats[((size_t)b * R + i) * 2 + 0] = (float)((double)__uint_as_float(st.x) * a.inv_tau);
        a.out_row_stats[((size_t)b * R + i) * 2 + 1] = __uint_as_float(st.y);
      }
      if (hasD) {
        a.out_row_stats[((size_t)b * R + K + 1 + i) * 2 + 0] =
            (float)((double)__uint_as_float(sd.x) * a.inv_tau);
        a.out_row_stats[((size_t)b * R + K + 1 + i) * 2 + 1] = __uint_as_float(sd.y);
      }
    }
    bool ok = !hasT || row_ok(st);
    if (hasD) ok = ok && row_ok(sd) && xi >= 0 && xi < a.V;
    bad |= !ok;
    bool reject = false;
    if (hasD && ok) {
      // the slice holding x_i writes these; a valid token always has one
      if (__float_as_uint(zT) == kMarker) zT = wait_f32(zx + i, a.status);
      if (__float_as_uint(zD) == kMarker) zD = wait_f32(zx + K + 1 + i, a.status);
      const double mT = __uint_as_float(st.x), sT = __uint_as_float(st.y);
      const double mD = __uint_as_float(sd.x), sD = __uint_as_float(sd.y);
      // log2 of the unnormalised probabilities, from exact differences
      const double lp = ((double)zT - mT) * a.c64;
      const double lq = ((double)zD - mD) * a.c64;
      const double u = uniform_draw(a.seed, (uint64_t)b, (uint64_t)i, 0);
      bool accept;
      if (zD == neg_inf()) {
        accept = true;  // q(x) = 0 <= p(x)
      } else {
        const double ratio = exp2(lp - lq) * (sD / sT);  // p(x) / q(x)
        accept = u < ratio;
      }
      reject = !accept;
      if (a.out_pq) {
        a.out_pq[((size_t)b * K + i) * 2 + 0] = (float)(exp2(lp) / sT);
        a.out_pq[((size_t)b * K + i) * 2 + 1] = (float)(exp2(lq) / sD);
      }
    }
    const unsigned bal = __ballot_sync(0xffffffffu, reject);
    if (n == K && bal) {
      const int L = __ffs(bal) - 1;
      n = i0 + L;
      stn = shfl_u2(st, L);
      sdn = shfl_u2(sd, L);
    } else if (n == K && K - i0 < 32) {  // the chunk holding position K, nothing rejected
      stn = shfl_u2(st, K - i0);
    }
  }
  bad = __any_sync(0xffffffffu, bad);

  SeqInfo si;
  si.b = b;
  if (bad) {
    si.n = 0;
    si.mode = kModeBad;
    si.mT = si.mD = si.lam_hi = si.lam_lo = si.sT = 0.f;
  } else {
    si.n = n;
    si.mT = __uint_as_float(stn.x);
    si.sT = __uint_as_float(stn.y);
    if (n < K) {
      si.mode = kModeResidual;
      si.mD = __uint_as_float(sdn.x);
      const double lam = log2((double)si.sT) - log2((double)__uint_as_float(sdn.y));
      si.lam_hi = (float)lam;
      si.lam_lo = (float)(lam - (double)si.lam_hi);
    } else {
      si.mode = kModeBonus;
      si.mD = 0.f;
      si.lam_hi = si.lam_lo = 0.f;
    }
  }
  if (lane == 0) publish_decision(a, qpos, si);

  int32_t* out = a.out_tokens + (size_t)b * (K + 1);
  if (bad) {
    for (int j = lane; j <= K; j += 32) out[j] = -1;
    if (lane == 0) {
      a.out_n[b] = -1;
      atomicOr(a.status, kStatusBadData);
      if (a.out_resid) a.out_resid[b] = NAN;
    }
  } else {
    for (int j = lane; j <= K; j += 32) {
      if (j < n) out[j] = __ldg(x + j);
      else if (j > n) out[j] = -1;
    }
    if (lane == 0) a.out_n[b] = n;
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// tail work.  Piece q of a chunk is warp step q: the 32 x VEC elements
// starting at v0 + q * 32 * VEC; its mass is the butterfly sum over lanes of
// each lane's sequential sum of its VEC weights.
// ---------------------------------------------------------------------------

// One warp: the pieces of tail slice s of the tail row(s) into the workspace
// and the slice's mass, the fp32 sum of its pieces in order (every lane).
// The loads of the next warp step are issued before the current step's
// arithmetic (two register buffers).
template <class E, int VEC>
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
  if constexpr (VEC > 1) {
    if (lane == 0 && v1 > v0) {
      prefetch_l2(rowT + v0, (unsigned)((v1 - v0) * sizeof(S)));
      if (k.residual) prefetch_l2(rowD + v0, (unsigned)((v1 - v0) * sizeof(S)));
    }
  }
  float total = 0.f;
  int e = v0 + lane * VEC;
  Raw<E, VEC> t0{}, d0{}, t1{}, d1{};
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
  return total;
}

// ---------------------------------------------------------------------------
// select finisher (one warp): inverse CDF over the tail slices' masses
// ---------------------------------------------------------------------------

// First position i < count with positive mass whose running sum (from `run`
// on, in index order) exceeds theta; when rounding leaves theta past every
// running sum, the last position with mass.  Values are read 128 at a time
// (four per lane, one round of loads), the running sum is a warp prefix in
// fp64 over each group of 32.  Returns -1 when no value is positive; *before
// gets the running sum just before the chosen position.
template <class LOAD>
__device__ __forceinline__ int warp_cdf_search(int count, double theta, double run, LOAD load,
                                               double* before) {
  const int lane = threadIdx.x & 31;
  int last = -1;
  double last_before = 0.0;
  for (int b0 = 0; b0 < count; b0 += 128) {
    double vals[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = b0 + 32 * q + lane;
      vals[q] = i < count ? load(i) : 0.0;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int c0 = b0 + 32 * q;
      if (c0 >= count) break;
      const double v = vals[q];
      const bool pos = v > 0.0;
      double incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const double o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      double excl = __shfl_up_sync(0xffffffffu, incl, 1);
      if (lane == 0) excl = 0.0;
      const unsigned hit = __ballot_sync(0xffffffffu, pos && run + incl > theta);
      const unsigned has = __ballot_sync(0xffffffffu, pos);
      if (hit) {
        const int L = __ffs(hit) - 1;
        *before = __shfl_sync(0xffffffffu, run + excl, L);
        return c0 + L;
      }
      if (has) {
        const int L = 31 - __clz(has);
        last = c0 + L;
        last_before = __shfl_sync(0xffffffffu, run + excl, L);
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  *before = last_before;
  return last;
}

template <class E, int VEC>
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
      const float tot = tail_slice_mass<E, VEC>(a, b, t, si);
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
    if (lane == 0) {
      a.out_tokens[(size_t)b * (a.K + 1) + n] = -1;
      atomicOr(a.status, kStatusTimeout);
    }
    __syncwarp();
    return;
  }
  const int v0 = tsel * a.TL, v1 = min(a.V, v0 + a.TL);
  const int np = (v1 - v0 + STEPW - 1) / STEPW;
  const float* gp = a.pieces + ((size_t)b * C + tsel) * a.P;
  double acc2 = acc;
  const int psel = warp_cdf_search(
      np, theta, acc, [&](int q) { return (double)wait_f32(gp + q, a.status); }, &acc2);
  if (psel < 0) {  // pieces inconsistent with their slice mass (expired wait)
    if (lane == 0) {
      a.out_tokens[(size_t)b * (a.K + 1) + n] = -1;
      atomicOr(a.status, kStatusTimeout);
    }
    __syncwarp();
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
  if (lane == 0) {
    a.out_tokens[(size_t)b * (a.K + 1) + n] = token;
    if (a.out_resid) a.out_resid[b] = (float)(Z / (double)si.sT);
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// statistics unit (one warp)
// ---------------------------------------------------------------------------
// Statistics slice s of row r of sequence b: the row's (m, s) over the slice,
// then the row's ticket.  Returns the ticket's old value (lane 0).  Kept out
// of line so that the stream loop has the register file to itself.
template <class E, int VEC, bool ENT>
__device__ __noinline__ int stats_slice(const SampleArgs& a, int b, int r, int s) {
  using S = typename E::storage;
  constexpr int BATCH = 32 * VEC * kUnroll;
  const int lane = threadIdx.x & 31;
  const S* row = r <= a.K ? target_row<E>(a, b, r) : draft_row<E>(a, b, r - a.K - 1);
  const int v0 = s * a.SL, v1 = min(a.V, v0 + a.SL);
  // the drafted token scored by this row (target rows 0..K-1 and every draft
  // row); its load overlaps the stream, and the slice holding it records the
  // logit there for the statistics finisher
  const int ti = r < a.K ? r : (r > a.K ? r - a.K - 1 : -1);
  const uint32_t xt = ld_relaxed_if(lane == 0 && ti >= 0, a.tokens + (size_t)b * a.K + ti, kMarker);
  const float cc = a.c_hi;
  float m = neg_inf();
  f2_t acc = f2(0.f, 0.f), tacc = f2(0.f, 0.f);
  // two register buffers: the next batch is in flight while one is reduced
  const int nb = v1 > v0 ? (v1 - v0 + BATCH - 1) / BATCH : 0;
  int e = v0 + lane * VEC;
  Raw<E, VEC> z0[kUnroll], z1[kUnroll];
  if constexpr (VEC > 1) {
    if (lane == 0 && v1 > v0) prefetch_l2(row + v0, (unsigned)((v1 - v0) * sizeof(S)));
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
  float sum = f2lo(acc) + f2hi(acc);
  float tsum = 0.f;
  if constexpr (ENT) {
    tsum = f2lo(tacc) + f2hi(tacc);
    warp_mst(m, sum, tsum, cc);
  } else {
    warp_ms(m, sum, cc);
  }
  int old = 0;
  if (lane == 0) {
    if constexpr (ENT) st_relaxed_f32(a.part_t + ((size_t)b * a.R + r) * a.CS + s, tsum);
    st_relaxed_u2(a.part + ((size_t)b * a.R + r) * a.CS + s, __float_as_uint(m), __float_as_uint(sum));
    old = ticket_take(&a.rowticket[((size_t)b * a.R + r) * kTicketStride]);
    const int xi = (int)xt;
    if (ti >= 0 && xi >= v0 && xi < v1) st_relaxed_f32(a.zx + (size_t)b * a.R + r, E::load1(row + xi));
  }
  return old;
}

// Tail slice s of a decided sequence: the slice's pieces and mass, then the
// sequence's tail ticket; the last ticket runs the select finisher.
template <class E, int VEC>
__device__ __noinline__ void tail_slice(const SampleArgs& a, const SeqInfo& si, int s) {
  const int lane = threadIdx.x & 31;
  if (si.mode == kModeBad) return;  // outputs already written by the statistics finisher
  const int b = si.b;
  const float tot = tail_slice_mass<E, VEC>(a, b, s, si);
  int old = 0;
  if (lane == 0) {
    // pieces and mass are marker-validated by the reader: no ordering needed
    st_relaxed_f32(a.tailsum + (size_t)b * a.TC + s, tot);
    old = ticket_take(&a.tailticket[b]);
  }
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old == a.TC - 1) select_finisher<E, VEC>(a, si);
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
// claim on counter c is flat slice f = k * kSlices + c.  The next claim
// is issued before the current slice is processed, so the atomic's latency
// hides behind the stream.  Tail slices are owned, not claimed: tail item j
// (queue position j / TC, tail slice j % TC) belongs to global warp j % W,
// where warp slot w of CTA c is global warp w * grid + c and W = 8 * grid.  A
// warp takes its items in order and polls the queue entry of its next item
// with a relaxed load issued before each statistics slice; a published item
// is taken before the next statistics slice.  Only when a warp has no
// statistics slice left does it wait (bounded) for its next entry.
//
// Progress: statistics slices and the finishers they trigger wait only for
// stores that other warps have already issued (their tickets were counted), a
// warp holding a claimed statistics slice never waits, and every sequence is
// decided once its statistics slices are done.  So every queue entry is
// eventually written and every wait ends, whatever part of the grid is
// resident.
template <class E, int VEC, bool ENT>
__global__ void __launch_bounds__(kThreads, kMinBlocks) sample_kernel(const __grid_constant__ SampleArgs a) {
  const int lane = threadIdx.x & 31;
  const int w = slice_of_warp();
  const int per_seq = a.R * a.CS;
  const int TT = a.B * a.TC;                       // tail items in all
  const int W = kSlices * (int)gridDim.x;          // warps in the grid
  int t = w * (int)gridDim.x + (int)blockIdx.x;    // this warp's next tail item
  // Statistics claims rotate over the eight counters (warp slot w starts at
  // counter w), so every warp draws equally from every counter and the
  // counters advance together: a sequence's slices, spread over all eight,
  // are then processed close together in time.  A claim past a counter's end
  // marks that counter dead for this warp; the warp leaves the statistics
  // work only when it has seen all eight dead, so no slice is ever left
  // unclaimed.  A claimed slice is processed before a tail item that became
  // ready (other warps' decisions may wait on it); the claim after it is then
  // deferred until the tail item is done.
  unsigned dead = 0;
  int ctr = w;
  int f = bcast(claim_from(a.counter, ctr, lane)) * kSlices + ctr;
  bool held = true;  // f is the result of a claim on counter ctr
  uint32_t seen = poll_decision(a, lane == 0 && t < TT, fdiv(t, a.div_tc));
  for (;;) {
    const bool tail_ready = t < TT && word_set(bcast((int)seen));
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
      if (!tail_ready) seen = poll_decision(a, lane == 0 && t < TT, fdiv(t, a.div_tc));
      const int b = fdiv(f, a.div_seq), rs = f - b * per_seq, r = fdiv(rs, a.div_cs), s = rs - r * a.CS;
      const int old = __shfl_sync(0xffffffffu, stats_slice<E, VEC, ENT>(a, b, r, s), 0);
      if (old == a.CS - 1) row_finisher<E, ENT>(a, b, r);
      if (ahead) {
        f = bcast(next) * kSlices + nctr;
        ctr = nctr;
      }
      continue;
    }
    if (tail_ready) {
      const int pos = fdiv(t, a.div_tc);
      const SeqInfo si = read_decision(a, pos);
      tail_slice<E, VEC>(a, si, t - pos * a.TC);
      t += W;
      seen = poll_decision(a, lane == 0 && t < TT, fdiv(t, a.div_tc));
      continue;
    }
    if (dead != 0xffu) {  // nothing held: claim from the next live counter
      ctr = next_live_counter(ctr, dead);
      f = bcast(claim_from(a.counter, ctr, lane)) * kSlices + ctr;
      held = true;
      continue;
    }
    if (t >= TT) break;
    // no statistics work left: wait for this warp's next decision
    if (lane == 0) {
      unsigned it = 0, nap = 64;
      seen = poll_decision(a, true, fdiv(t, a.div_tc));
      while (!word_set(seen) && ++it < kSpinLimit) {
        __nanosleep(nap);
        if (nap < 1024) nap <<= 1;
        seen = poll_decision(a, true, fdiv(t, a.div_tc));
      }
      if (!word_set(seen)) atomicOr(a.status, kStatusTimeout);
    }
    if (!word_set(bcast((int)seen))) break;
  }
}

// ---------------------------------------------------------------------------
// host side helpers
// ---------------------------------------------------------------------------
static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace: [counters, tickets, queue count (all start at -1)][marker-filled
// result slots: part, rowstat, tailsum, queue, pieces, zx, and part_t when the
// entropy is asked for]; one 0xff fill initialises both parts.
static void sample_layout(int B, int R, int CS, int TC, int P, bool ent, size_t* off) {
  size_t o = 0;
  off[0] = o; o += kCounterBytes;                                          // counter
  off[1] = o; o += align_up((size_t)B * R * kTicketStride * 4, 16);       // rowticket
  off[2] = o; o += align_up((size_t)B * 4, 16);                           // seqticket
  off[3] = o; o += align_up((size_t)B * 4, 16);                           // tailticket
  off[4] = o; o += 16;                                                     // qcount
  o = align_up(o, 256);
  off[5] = o;                                                              // end of zero region
  off[6] = o; o += align_up((size_t)B * R * CS * sizeof(float2), 256);    // part
  off[7] = o; o += align_up((size_t)B * R * sizeof(float2), 256);         // rowstat
  off[8] = o; o += align_up((size_t)B * TC * sizeof(float), 256);         // tailsum
  off[10] = o; o += align_up((size_t)B * sizeof(SeqInfo), 256);           // queue
  off[11] = o; o += align_up((size_t)B * TC * P * sizeof(float), 256);    // pieces
  off[13] = o; o += align_up((size_t)B * R * sizeof(float), 256);         // zx
  off[14] = o; if (ent) o += align_up((size_t)B * R * CS * sizeof(float), 256);  // part_t
  off[9] = o;                                                              // end of marker region
  off[12] = o;
}

WsLayout sample_workspace(int B, int K, int CS, int TC, int P, bool ent) {
  size_t off[15];
  sample_layout(B, 2 * K + 1, CS, TC, P, ent, off);
  WsLayout l;
  l.total = off[12];
  l.zero_bytes = 0;  // counters and tickets start at -1: one 0xff fill covers everything
  l.marker_off = 0;
  l.marker_bytes = off[9];
  return l;
}

void sample_bind_workspace(SampleArgs& a, void* ws) {
  size_t off[15];
  sample_layout(a.B, a.R, a.CS, a.TC, a.P, a.out_entropy != nullptr, off);
  char* p = (char*)ws;
  a.counter = (unsigned long long*)(p + off[0]);
  a.rowticket = (int*)(p + off[1]);
  a.seqticket = (int*)(p + off[2]);
  a.tailticket = (int*)(p + off[3]);
  a.qcount = (int*)(p + off[4]);
  a.part = (float2*)(p + off[6]);
  a.rowstat = (float2*)(p + off[7]);
  a.tailsum = (float*)(p + off[8]);
  a.queue = (SeqInfo*)(p + off[10]);
  a.pieces = (float*)(p + off[11]);
  a.zx = (float*)(p + off[13]);
  a.part_t = a.out_entropy ? (float*)(p + off[14]) : nullptr;
}

template <class E, int VEC>
static cudaError_t launch_sample_t(const SampleArgs& a, int grid, cudaStream_t s) {
  if (a.out_entropy)
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

}  // namespace sv
