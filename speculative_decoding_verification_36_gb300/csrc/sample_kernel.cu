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
//     2-4 in fp64 and publishes the sequence's decision.
//   * tail slice = SL elements of the tail row (pair): after the decision is
//     published (a bounded wait) it writes the mass of every warp step
//     ("piece") of the replacement / bonus distribution.  Tail units are
//     queued `delta` sequences after the statistics units, so the re-read rows
//     are still in L2.  The warp that takes the last tail ticket finds the CDF
//     crossing from the slice and piece masses and rescans one piece.
// Every reduction runs in a fixed order, so results are run-to-run identical.
#include "sv_common.cuh"
#include "sv_kernels.h"

#include <math.h>

namespace sv {

struct UnitRef {
  int kind;  // 0 statistics, 1 tail
  int b;
  int idx;
};

// Unit index -> (kind, sequence, index within the sequence); 32-bit arithmetic
// (the host keeps the unit count below 2^31).
__device__ __forceinline__ UnitRef decode_unit(const UnitMap& m, int p) {
  const int A = m.A, T = m.T, AT = m.A + m.T;
  const int n1 = m.delta < m.B ? m.delta : m.B;         // statistics-only blocks
  const int n2 = m.B - m.delta > 0 ? m.B - m.delta : 0;  // statistics + tail blocks
  UnitRef u;
  if (p < n1 * A) {
    u.kind = 0;
    u.b = p / A;
    u.idx = p - u.b * A;
    return u;
  }
  p -= n1 * A;
  if (p < n2 * AT) {
    const int blk = p / AT, o = p - blk * AT;
    if (o < A) {
      u.kind = 0;
      u.b = m.delta + blk;
      u.idx = o;
    } else {
      u.kind = 1;
      u.b = blk;
      u.idx = o - A;
    }
    return u;
  }
  p -= n2 * AT;
  u.kind = 1;
  u.b = n2 + p / T;
  u.idx = p - (p / T) * T;
  return u;
}

// ---------------------------------------------------------------------------
// Replacement / bonus weights.  Both are scaled by the target row's sum sT so
// that no division is needed: the inverse CDF only sees ratios.
//   bonus:     w(v) = 2^{(zT - mT) c}                        = sT * p(v)
//   residual:  w(v) = 2^{(zT - mT) c} * (1 - 2^{-delta})     = sT * max(0, p(v) - q(v))
//              delta = (dT - dD) c - log2(sT / sD)          (> 0 iff p(v) > q(v))
// The form 2^{aT}(1 - 2^{-delta}) has no cancellation (see one_minus_exp2_neg).
// Explicit round-to-nearest operations (no contraction) keep the arithmetic
// identical in the tail units and in the final rescan.
// ---------------------------------------------------------------------------
struct TailConsts {
  float mT, mD, c_hi, c_lo, lam_hi, lam_lo;
  int residual;
};

// 1 - 2^{-d} for d > 0 without cancellation.  For d < 1.4, with y = d ln 2:
// 1 - e^{-y} = 2 sinh(y/2) e^{-y/2}; sinh(x) = x (1 + x^2/6 + x^4/120 + x^6/5040)
// (x <= 0.49, the first omitted term is below 1e-8 relative) and e^{-y/2} from
// ex2.  For d >= 1.4 the direct 1 - 2^{-d} (>= 0.62) loses nothing.
__device__ __forceinline__ float one_minus_exp2_neg(float d) {
  const float eh = ex2(__fmul_rn(d, -0.5f));  // 2^{-d/2}
  if (d >= 1.4f) return __fsub_rn(1.f, __fmul_rn(eh, eh));
  const float x = __fmul_rn(d, 0.346573590279972655f);  // (d ln 2) / 2
  const float xx = __fmul_rn(x, x);
  float p = __fmaf_rn(xx, 1.f / 5040.f, 1.f / 120.f);
  p = __fmaf_rn(xx, p, 1.f / 6.f);
  p = __fmaf_rn(xx, p, 1.f);
  return __fmul_rn(__fmul_rn(__fmul_rn(x, p), eh), 2.f);
}

__device__ __forceinline__ float tail_weight(float zT, float zD, const TailConsts& k) {
  const float dT = __fsub_rn(zT, k.mT);
  const float eT = ex2(__fmul_rn(dT, k.c_hi));
  if (!k.residual) return eT;
  const float dD = __fsub_rn(zD, k.mD);
  const float D = __fsub_rn(dT, dD);
  const float delta = __fadd_rn(__fmaf_rn(D, k.c_hi, -k.lam_hi), __fmaf_rn(D, k.c_lo, -k.lam_lo));
  if (!(delta > 0.f)) return 0.f;
  return __fmul_rn(eT, one_minus_exp2_neg(delta));
}

// The same weights for an element pair with packed f32x2 arithmetic: every
// operation rounds exactly as the scalar version above, so pieces and the
// final rescan agree bit for bit.
__device__ __forceinline__ f2_t tail_weight2(f2_t zT, f2_t zD, const TailConsts& k) {
  const f2_t dT = f2sub(zT, f2(k.mT, k.mT));
  const f2_t aT = f2mul(dT, f2(k.c_hi, k.c_hi));
  const float eT0 = ex2(f2lo(aT)), eT1 = ex2(f2hi(aT));
  if (!k.residual) return f2(eT0, eT1);
  const f2_t dD = f2sub(zD, f2(k.mD, k.mD));
  const f2_t D = f2sub(dT, dD);
  const f2_t delta = f2add(f2fma(D, f2(k.c_hi, k.c_hi), f2(-k.lam_hi, -k.lam_hi)),
                           f2fma(D, f2(k.c_lo, k.c_lo), f2(-k.lam_lo, -k.lam_lo)));
  const float d0 = f2lo(delta), d1 = f2hi(delta);
  const float w0 = d0 > 0.f ? __fmul_rn(eT0, one_minus_exp2_neg(d0)) : 0.f;
  const float w1 = d1 > 0.f ? __fmul_rn(eT1, one_minus_exp2_neg(d1)) : 0.f;
  return f2(w0, w1);
}

// The VEC weights of one lane's vector, in element order.
template <class E, int VEC>
__device__ __forceinline__ void lane_weights(const Raw<E, VEC>& zt, const Raw<E, VEC>& zd,
                                             const TailConsts& k, float (&w)[VEC]) {
  if constexpr (VEC == 1) {
    w[0] = tail_weight(elem(zt, 0), elem(zd, 0), k);
  } else {
#pragma unroll
    for (int p = 0; p < VEC / 2; ++p) {
      const f2_t wp = tail_weight2(elem_pair<E, VEC>(zt, p), elem_pair<E, VEC>(zd, p), k);
      w[2 * p] = f2lo(wp);
      w[2 * p + 1] = f2hi(wp);
    }
  }
}

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

__device__ __forceinline__ SeqInfo load_info(const SampleArgs& a, int b) {
  const SeqInfo* g = a.info + b;
  SeqInfo si;
  si.n = __ldcg(&g->n);
  si.mode = __ldcg(&g->mode);
  si.mT = __ldcg(&g->mT);
  si.mD = __ldcg(&g->mD);
  si.lam_hi = __ldcg(&g->lam_hi);
  si.lam_lo = __ldcg(&g->lam_lo);
  si.sT = __ldcg(&g->sT);
  si.pad = 0;
  return si;
}

// ---------------------------------------------------------------------------
// row finisher (one warp): merges the slice partials of row r in slice order
// (lane-strided, then the fixed warp merge) into rowstat; the last row of a
// sequence then runs the statistics finisher.
// ---------------------------------------------------------------------------
template <class E>
__device__ __noinline__ void stats_finisher(const SampleArgs& a, int b);

template <class E>
__device__ __noinline__ void row_finisher(const SampleArgs& a, int b, int r) {
  const int lane = threadIdx.x & 31;
  const int C = a.CU * kSlices;
  const float2* pp = a.part + ((size_t)b * a.R + r) * C;
  float m = neg_inf(), s = 0.f;
  for (int c = lane; c < C; c += 32) {
    const uint2 w = wait_u2(pp + c, a.status);
    ms_merge(m, s, __uint_as_float(w.x), __uint_as_float(w.y), a.c_hi);
  }
  warp_ms(m, s, a.c_hi);
  int old = 0;
  if (lane == 0) {
    st_relaxed_u2(a.rowstat + (size_t)b * a.R + r, __float_as_uint(m), __float_as_uint(s));
    old = atom_add_relaxed(&a.seqticket[b], 1);
  }
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old == a.R - 1) stats_finisher<E>(a, b);
}

// ---------------------------------------------------------------------------
// statistics finisher (one warp): steps 2-4 for sequence b
// ---------------------------------------------------------------------------
template <class E>
__device__ __noinline__ void stats_finisher(const SampleArgs& a, int b) {
  const int R = a.R, K = a.K;
  const int lane = threadIdx.x & 31;
  const float2* rs = a.rowstat + (size_t)b * R;
  for (int r = lane; r < R; r += 32) {
    const uint2 w = wait_u2(rs + r, a.status);  // the row finisher's (m, s)
    if (a.out_row_stats) {
      a.out_row_stats[((size_t)b * R + r) * 2 + 0] = (float)((double)__uint_as_float(w.x) * a.inv_tau);
      a.out_row_stats[((size_t)b * R + r) * 2 + 1] = __uint_as_float(w.y);
    }
  }
  __syncwarp();
  const int32_t* x = a.tokens + (size_t)b * K;
  bool bad = false;
  for (int r = lane; r < R; r += 32) {
    const float2 v = __ldcg(rs + r);
    bad |= !(v.y > 0.f) || !(v.y < INFINITY) || !(v.x < INFINITY) || !(v.x > neg_inf());
  }
  for (int i = lane; i < K; i += 32) bad |= x[i] < 0 || x[i] >= a.V;
  bad = __any_sync(0xffffffffu, bad);

  int n = K;
  if (!bad) {
    for (int i0 = 0; i0 < K; i0 += 32) {
      const int i = i0 + lane;
      bool reject = false;
      if (i < K) {
        const int xi = x[i];
        const float zT = E::load1(target_row<E>(a, b, i) + xi);
        const float zD = E::load1(draft_row<E>(a, b, i) + xi);
        const float2 st = __ldcg(rs + i), sd = __ldcg(rs + K + 1 + i);
        const double mT = st.x, sT = st.y, mD = sd.x, sD = sd.y;
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
      if (bal && n == K) n = i0 + __ffs(bal) - 1;
    }
  }

  int32_t* out = a.out_tokens + (size_t)b * (K + 1);
  SeqInfo si;
  si.pad = 0;
  if (bad) {
    for (int j = lane; j <= K; j += 32) out[j] = -1;
    si.n = -1;
    si.mode = kModeBad;
    si.mT = si.mD = si.lam_hi = si.lam_lo = si.sT = 0.f;
    if (lane == 0) {
      a.out_n[b] = -1;
      atomicOr(a.status, kStatusBadData);
      if (a.out_resid) a.out_resid[b] = NAN;
    }
  } else {
    for (int j = lane; j <= K; j += 32) {
      if (j < n) out[j] = x[j];
      else if (j > n) out[j] = -1;
    }
    const float2 st = __ldcg(rs + n);
    si.n = n;
    si.mT = st.x;
    si.sT = st.y;
    if (n < K) {
      const float2 sd = __ldcg(rs + K + 1 + n);
      si.mode = kModeResidual;
      si.mD = sd.x;
      const double lam = log2((double)st.y) - log2((double)sd.y);
      si.lam_hi = (float)lam;
      si.lam_lo = (float)(lam - (double)si.lam_hi);
    } else {
      si.mode = kModeBonus;
      si.mD = 0.f;
      si.lam_hi = si.lam_lo = 0.f;
    }
    if (lane == 0) a.out_n[b] = n;
  }
  if (lane == 0) {
    a.info[b] = si;
    __threadfence();
    st_release(&a.ready[b], 1);
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// tail work.  Piece q of a chunk is warp step q: the 32 x VEC elements
// starting at v0 + q * 32 * VEC; its mass is the butterfly sum over lanes of
// each lane's sequential sum of its VEC weights.
// ---------------------------------------------------------------------------
template <class E, int VEC>
__device__ __forceinline__ float lane_mass(const Raw<E, VEC>& zt, const Raw<E, VEC>& zd,
                                           const TailConsts& k) {
  float w[VEC];
  lane_weights<E, VEC>(zt, zd, k, w);
  float ls = 0.f;
#pragma unroll
  for (int q = 0; q < VEC; ++q) ls = __fadd_rn(ls, w[q]);
  return ls;
}

// One warp: the pieces of slice s of the tail row(s) into the workspace and
// the slice's fp64 mass (sequential over pieces; returned in every lane).
template <class E, int VEC>
__device__ double tail_slice_mass(const SampleArgs& a, int b, int s, const SeqInfo& si) {
  using S = typename E::storage;
  constexpr int STEPW = 32 * VEC;
  const int lane = threadIdx.x & 31;
  const S* rowT = target_row<E>(a, b, si.n);
  const S* rowD = si.mode == kModeResidual ? draft_row<E>(a, b, si.n) : rowT;
  const TailConsts k = tail_consts(a, si);
  const int v0 = s * a.SL, v1 = min(a.V, v0 + a.SL);
  const int nsteps = v1 > v0 ? (v1 - v0 + STEPW - 1) / STEPW : 0;
  float* gp = a.pieces + ((size_t)b * a.CU * kSlices + s) * a.P;
  if constexpr (VEC > 1) {
    if (lane == 0 && v1 > v0) {
      prefetch_l2(rowT + v0, (unsigned)((v1 - v0) * sizeof(S)));
      if (k.residual) prefetch_l2(rowD + v0, (unsigned)((v1 - v0) * sizeof(S)));
    }
  }
  double total = 0.0;
  int e = v0 + lane * VEC;
  for (int st = 0; st < nsteps; st += kUnroll, e += STEPW * kUnroll) {
    Raw<E, VEC> zt[kUnroll], zd[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      zt[u] = load_raw<E, VEC>(rowT, e + u * STEPW, v1);
      zd[u] = k.residual ? load_raw<E, VEC>(rowD, e + u * STEPW, v1) : zt[u];
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (st + u < nsteps) {
        const float ps = warp_sum(lane_mass<E, VEC>(zt[u], zd[u], k));
        if (lane == 0) gp[st + u] = ps;
        total += (double)ps;
      }
    }
  }
  return total;
}

// ---------------------------------------------------------------------------
// select finisher (one warp): inverse CDF over the tail units' masses
// ---------------------------------------------------------------------------
template <class E, int VEC>
__device__ __noinline__ void select_finisher(const SampleArgs& a, int b) {
  using S = typename E::storage;
  constexpr int STEPW = 32 * VEC;
  const int lane = threadIdx.x & 31;
  if (!ld_acquire(&a.ready[b])) return;
  SeqInfo si = load_info(a, b);
  if (si.mode == kModeBad) return;
  const int C = a.CU * kSlices;  // tail slices of the row, in vocabulary order
  double* ts = a.tailsum + (size_t)b * C;
  double Z = 0.0;
  for (int t = 0; t < C; ++t) Z += wait_f64_acquire(ts + t, a.status);
  // Z == 0 after a rejection can only come from rounding (p(x_n) < q(x_n)
  // forces a positive residual); then the draw falls back to p_n itself, and
  // this warp recomputes every piece in bonus mode with the same arithmetic.
  if (si.mode == kModeResidual && !(Z > 0.0)) {
    si.mode = kModeBonus;
    for (int t = 0; t < C; ++t) {
      const double tot = tail_slice_mass<E, VEC>(a, b, t, si);
      if (lane == 0) ts[t] = tot;
    }
    __threadfence();
    __syncwarp();
    Z = 0.0;
    for (int t = 0; t < C; ++t) Z += __ldcg(ts + t);
  }
  const int n = si.n;
  const double theta = uniform_draw(a.seed, (uint64_t)b, (uint64_t)n, 1) * Z;

  // Slice, then piece, then lane, then element holding the crossing, each by
  // a sequential fp64 prefix.  Only positions with positive mass are ever
  // chosen, so the emitted token always carries weight (and lies below V);
  // when rounding leaves theta past every partial sum, the last position with
  // mass is taken.
  double acc = 0.0;
  int tsel = -1, tlast = -1;
  double acc_last = 0.0;
  for (int t = 0; t < C; ++t) {
    const double v = __ldcg(ts + t);
    if (!(v > 0.0)) continue;
    if (acc + v > theta) {
      tsel = t;
      break;
    }
    tlast = t;
    acc_last = acc;
    acc += v;
  }
  if (tsel < 0) {
    tsel = tlast;
    acc = acc_last;
  }
  if (tsel < 0) {  // no slice with mass: only an expired wait can cause this
    if (lane == 0) {
      a.out_tokens[(size_t)b * (a.K + 1) + n] = -1;
      atomicOr(a.status, kStatusTimeout);
    }
    __syncwarp();
    return;
  }
  const int v0 = tsel * a.SL, v1 = min(a.V, v0 + a.SL);
  const int np = (v1 - v0 + STEPW - 1) / STEPW;
  const float* gp = a.pieces + ((size_t)b * C + tsel) * a.P;
  int psel = -1, plast = -1;
  double acc2 = acc, acc2_last = acc;
  for (int q = 0; q < np; ++q) {
    const double v = (double)__ldcg(gp + q);
    if (!(v > 0.0)) continue;
    if (acc2 + v > theta) {
      psel = q;
      break;
    }
    plast = q;
    acc2_last = acc2;
    acc2 += v;
  }
  if (psel < 0) {
    psel = plast;
    acc2 = acc2_last;
  }
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
template <class E, int VEC>
__device__ __forceinline__ void load_batch(Raw<E, VEC> (&z)[kUnroll], const typename E::storage* row,
                                           int e, int v1) {
  constexpr int STEPW = 32 * VEC;
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) z[u] = load_raw<E, VEC>(row, e + u * STEPW, v1);
}

// One batch into the lane's running (m, s): the batch max first, one rescale
// if it rose, then 2^{(z - m) c} summed with packed pair arithmetic.
template <class E, int VEC>
__device__ __forceinline__ void stats_batch(const Raw<E, VEC> (&z)[kUnroll], float& m, f2_t& acc,
                                            float cc) {
  const float bm = batch_max<E, VEC>(z);
  if (bm > m) {
    const float f = ex2((m - bm) * cc);
    acc = f2mul(acc, f2(f, f));
    m = bm;
  }
  const float base = (m == neg_inf()) ? 0.f : m;
  if constexpr (VEC == 1) {
    float lo = f2lo(acc);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) lo += ex2((z[u].f - base) * cc);
    acc = f2(lo, f2hi(acc));
  } else {
    // The MUFU unit takes the first kMufuPairs element pairs of the batch and
    // the FMA pipe (exp2_poly2) the rest, so that neither unit limits the pass.
    constexpr int kPairs = kUnroll * VEC / 2;
    constexpr int kMufuPairs = kPairs - kPairs / 2;
    const f2_t b2 = f2(base, base), c2 = f2(cc, cc);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
#pragma unroll
      for (int p = 0; p < VEC / 2; ++p) {
        if (u * (VEC / 2) + p < kMufuPairs)
          f2_exp_acc(acc, elem_pair<E, VEC>(z[u], p), b2, c2);
        else
          f2_exp_acc_poly(acc, elem_pair<E, VEC>(z[u], p), b2, c2);
      }
  }
}

// Slice w of statistics unit idx of sequence b: one row's (m, s) over the
// slice, then the row's ticket.  Returns the ticket's old value (lane 0).
template <class E, int VEC>
__device__ int stats_slice(const SampleArgs& a, int b, int idx, int w) {
  using S = typename E::storage;
  constexpr int BATCH = 32 * VEC * kUnroll;
  const int lane = threadIdx.x & 31;
  const int r = idx / a.CU, uc = idx - (idx / a.CU) * a.CU;
  const int s = uc * kSlices + w;
  const S* row = r <= a.K ? target_row<E>(a, b, r) : draft_row<E>(a, b, r - a.K - 1);
  const int v0 = s * a.SL, v1 = min(a.V, v0 + a.SL);
  const float cc = a.c_hi;
  float m = neg_inf();
  f2_t acc = f2(0.f, 0.f);
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
    stats_batch<E, VEC>(z0, m, acc, cc);
    if (bt + 1 < nb) {
      if (bt + 2 < nb) load_batch<E, VEC>(z0, row, e + 2 * BATCH, v1);
      stats_batch<E, VEC>(z1, m, acc, cc);
    }
  }
  float sum = f2lo(acc) + f2hi(acc);
  warp_ms(m, sum, cc);
  int old = 0;
  if (lane == 0) {
    st_relaxed_u2(a.part + ((size_t)b * a.R + r) * (a.CU * kSlices) + s, __float_as_uint(m),
                  __float_as_uint(sum));
    old = atom_add_relaxed(&a.rowticket[((size_t)b * a.R + r) * kTicketStride], 1);
  }
  return old;
}

// Slice w of tail unit uc of sequence b: wait for the decision (bounded),
// claim the next unit, then the slice's pieces and the sequence's ticket.
template <class E, int VEC>
__device__ int tail_slice(const SampleArgs& a, int b, int uc, int w, int& next) {
  const int lane = threadIdx.x & 31;
  int st = 0;
  next = 0;
  if (lane == 0) {
    st = ld_acquire(&a.ready[b]);
    unsigned it = 0;
    while (st == 0 && ++it < kSpinLimit) {
      __nanosleep(128);
      st = ld_acquire(&a.ready[b]);
    }
    if (st == 0) atomicOr(a.status, kStatusTimeout);
    // nothing below waits, so this claim cannot hold up another warp
    next = (int)atomicAdd(a.counter + w * kCounterStride, 1ull);
  }
  st = __shfl_sync(0xffffffffu, st, 0);
  const int s = uc * kSlices + w;
  double tot = 0.0;
  if (st) {
    const SeqInfo si = load_info(a, b);
    if (si.mode != kModeBad) tot = tail_slice_mass<E, VEC>(a, b, s, si);
  }
  int old = 0;
  if (lane == 0) {
    // release: the pieces stored by this lane are visible to whoever sees the mass
    st_release_f64(a.tailsum + (size_t)b * a.CU * kSlices + s, tot);
    old = atom_add_relaxed(&a.tailticket[b], 1);
  }
  return old;
}

// Units are only ever claimed by a warp that is already running, and each
// counter hands them out in increasing order.  A tail slice waits only on the
// statistics slices of its sequence, which belong to units with smaller
// indices on every counter; a warp never holds another claim while it waits,
// and it settles its own tickets before taking new work.  So every slice a
// wait depends on is being processed by a running warp, and every wait ends,
// even when other work keeps part of the grid from being resident.
template <class E, int VEC>
__global__ void __launch_bounds__(kThreads, kMinBlocks) sample_kernel(const __grid_constant__ SampleArgs a) {
  const int lane = threadIdx.x & 31;
  const int w = slice_of_warp();
  const int row_last = a.CU * kSlices - 1, tail_last = a.map.T * kSlices - 1;
  int unit = bcast(claim_unit(a.counter, lane));
  while (unit < a.map.total) {
    const UnitRef u = decode_unit(a.map, unit);
    int next = 0;
    if (u.kind == 0) {
      next = claim_unit(a.counter, lane);
      const int old = __shfl_sync(0xffffffffu, stats_slice<E, VEC>(a, u.b, u.idx, w), 0);
      if (old == row_last) row_finisher<E>(a, u.b, u.idx / a.CU);
    } else {
      const int old = __shfl_sync(0xffffffffu, tail_slice<E, VEC>(a, u.b, u.idx, w, next), 0);
      if (old == tail_last) select_finisher<E, VEC>(a, u.b);
    }
    unit = bcast(next);
  }
}

// ---------------------------------------------------------------------------
// host side helpers
// ---------------------------------------------------------------------------
static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace: [zero-filled: counters, tickets, ready][marker-filled: part,
// rowstat, tailsum][info, pieces].
static void sample_layout(int B, int R, int CU, int P, size_t* off) {
  const size_t C = (size_t)CU * kSlices;
  size_t o = 0;
  off[0] = o; o += kCounterBytes;                                          // counter
  off[1] = o; o += align_up((size_t)B * R * kTicketStride * 4, 16);       // rowticket
  off[2] = o; o += align_up((size_t)B * 4, 16);                           // seqticket
  off[3] = o; o += align_up((size_t)B * 4, 16);                           // tailticket
  off[4] = o; o += align_up((size_t)B * 4, 16);                           // ready
  o = align_up(o, 256);
  off[5] = o;                                                              // end of zero region
  off[6] = o; o += align_up((size_t)B * R * C * sizeof(float2), 256);     // part
  off[7] = o; o += align_up((size_t)B * R * sizeof(float2), 256);         // rowstat
  off[8] = o; o += align_up((size_t)B * C * sizeof(double), 256);         // tailsum
  off[9] = o;                                                              // end of marker region
  off[10] = o; o += align_up((size_t)B * sizeof(SeqInfo), 256);           // info
  off[11] = o; o += align_up((size_t)B * C * P * sizeof(float), 256);     // pieces
  off[12] = o;
}

WsLayout sample_workspace(int B, int K, int CU, int P) {
  size_t off[13];
  sample_layout(B, 2 * K + 1, CU, P, off);
  WsLayout l;
  l.total = off[12];
  l.zero_bytes = off[5];
  l.marker_off = off[6];
  l.marker_bytes = off[9] - off[6];
  return l;
}

void sample_bind_workspace(SampleArgs& a, void* ws) {
  size_t off[13];
  sample_layout(a.B, a.R, a.CU, a.P, off);
  char* p = (char*)ws;
  a.counter = (unsigned long long*)(p + off[0]);
  a.rowticket = (int*)(p + off[1]);
  a.seqticket = (int*)(p + off[2]);
  a.tailticket = (int*)(p + off[3]);
  a.ready = (int*)(p + off[4]);
  a.part = (float2*)(p + off[6]);
  a.rowstat = (float2*)(p + off[7]);
  a.tailsum = (double*)(p + off[8]);
  a.info = (SeqInfo*)(p + off[10]);
  a.pieces = (float*)(p + off[11]);
}

template <class E, int VEC>
static cudaError_t launch_sample_t(const SampleArgs& a, int grid, cudaStream_t s) {
  sample_kernel<E, VEC><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_sample(const SampleArgs& a, bool bf16, bool vec, int grid, cudaStream_t s) {
  if (bf16) return vec ? launch_sample_t<BF16, 8>(a, grid, s) : launch_sample_t<BF16, 1>(a, grid, s);
  return vec ? launch_sample_t<F32, 4>(a, grid, s) : launch_sample_t<F32, 1>(a, grid, s);
}

template <class E, int VEC>
static int blocks_sample_t() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, sample_kernel<E, VEC>, kThreads, 0) != cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

int sample_blocks_per_sm(bool bf16, bool vec) {
  if (bf16) return vec ? blocks_sample_t<BF16, 8>() : blocks_sample_t<BF16, 1>();
  return vec ? blocks_sample_t<F32, 4>() : blocks_sample_t<F32, 1>();
}

}  // namespace sv
