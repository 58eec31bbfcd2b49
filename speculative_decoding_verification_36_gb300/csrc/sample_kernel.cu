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
// Work decomposition (one persistent grid, kThreads threads per CTA):
//   * statistics unit  = one chunk of CH elements of one row: an online
//     (max, sum of exp2) pass with 16-byte streaming loads, reduced to one
//     (m, s) pair per chunk in the workspace.  The CTA that finishes a
//     sequence's last statistics unit (atomic ticket) merges the chunk pairs,
//     runs steps 2-4 in fp64 and publishes the sequence's decision.
//   * tail unit        = one chunk of the tail row (pair); it waits (bounded)
//     for the decision, then writes per-piece masses of the replacement /
//     bonus distribution.  Tail units are queued `delta` sequences after the
//     statistics units, so the re-read row is still in L2.  The CTA that
//     finishes the last tail unit locates the CDF crossing from the chunk and
//     piece masses and rescans a single 32-lane piece.
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

__device__ __forceinline__ UnitRef decode_unit(const UnitMap& m, long long p) {
  const long long A = m.A, T = m.T, AT = m.A + m.T;
  const long long n1 = m.delta < m.B ? m.delta : m.B;         // statistics-only blocks
  const long long n2 = m.B - m.delta > 0 ? m.B - m.delta : 0;  // statistics + tail blocks
  UnitRef u;
  if (p < n1 * A) {
    u.kind = 0;
    u.b = (int)(p / A);
    u.idx = (int)(p % A);
    return u;
  }
  p -= n1 * A;
  if (p < n2 * AT) {
    const long long blk = p / AT, o = p % AT;
    if (o < A) {
      u.kind = 0;
      u.b = (int)(m.delta + blk);
      u.idx = (int)o;
    } else {
      u.kind = 1;
      u.b = (int)blk;
      u.idx = (int)(o - A);
    }
    return u;
  }
  p -= n2 * AT;
  u.kind = 1;
  u.b = (int)(n2 + p / T);
  u.idx = (int)(p % T);
  return u;
}

// ---------------------------------------------------------------------------
// Replacement / bonus weights.  Both are scaled by the target row's sum sT so
// that no division is needed: the inverse CDF only sees ratios.
//   bonus:     w(v) = 2^{(zT - mT) c}                        = sT * p(v)
//   residual:  w(v) = 2^{(zT - mT) c} * (1 - 2^{-delta})     = sT * max(0, p(v) - q(v))
//              delta = (dT - dD) c - log2(sT / sD)          (> 0 iff p(v) > q(v))
// The form 2^{aT}(1 - 2^{-delta}) has no cancellation: 1 - 2^{-delta} is taken
// from its Taylor series for delta < 1.  The explicit _rn intrinsics keep the
// arithmetic identical in the tail units and in the final rescan.
// ---------------------------------------------------------------------------
struct TailConsts {
  float mT, mD, c_hi, c_lo, lam_hi, lam_lo;
  int residual;
};

// 1 - 2^{-d} for d > 0.  For d < 1: y = d ln 2 and
// 1 - e^{-y} = y (1 - y/2 (1 - y/3 (1 - ... (1 - y/11)))), the alternating
// Taylor series cut after y^11/11! (next term below 4e-10 of the result).
__device__ __forceinline__ float one_minus_exp2_neg(float d) {
  if (d >= 1.f) return __fsub_rn(1.f, ex2(-d));
  const float y = __fmul_rn(d, 0.693147180559945309f);
  float acc = 1.f;
  acc = __fmaf_rn(-y * (1.f / 11.f), acc, 1.f);
  acc = __fmaf_rn(-y * (1.f / 10.f), acc, 1.f);
  acc = __fmaf_rn(-y * (1.f / 9.f), acc, 1.f);
  acc = __fmaf_rn(-y * (1.f / 8.f), acc, 1.f);
  acc = __fmaf_rn(-y * (1.f / 7.f), acc, 1.f);
  acc = __fmaf_rn(-y * (1.f / 6.f), acc, 1.f);
  acc = __fmaf_rn(-y * (1.f / 5.f), acc, 1.f);
  acc = __fmaf_rn(-y * (1.f / 4.f), acc, 1.f);
  acc = __fmaf_rn(-y * (1.f / 3.f), acc, 1.f);
  acc = __fmaf_rn(-y * (1.f / 2.f), acc, 1.f);
  return __fmul_rn(y, acc);
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

template <class E>
__device__ __forceinline__ const typename E::storage* target_row(const SampleArgs& a, int b, int r) {
  return (const typename E::storage*)a.target + ((size_t)b * (a.K + 1) + r) * (size_t)a.V;
}
template <class E>
__device__ __forceinline__ const typename E::storage* draft_row(const SampleArgs& a, int b, int r) {
  return (const typename E::storage*)a.draft + ((size_t)b * a.K + r) * (size_t)a.V;
}

struct SampleSmem {
  long long next;
  int flag;
  int state;
  float wm[kWarps];
  float ws[kWarps];
  float rowm[2 * kMaxK + 1];
  float rows[2 * kMaxK + 1];
  float piece[512];
  SeqInfo info;
};

// ---------------------------------------------------------------------------
// statistics finisher: steps 2-4 for sequence b
// ---------------------------------------------------------------------------
template <class E>
__device__ __noinline__ void stats_finisher(const SampleArgs& a, int b, SampleSmem& sm) {
  const int R = a.R, C = a.C, K = a.K;
  for (int r = threadIdx.x; r < R; r += kThreads) {
    const float2* pp = a.part + ((size_t)b * R + r) * C;
    float m = neg_inf(), s = 0.f;
    for (int c = 0; c < C; ++c) {
      const float2 v = __ldcg(pp + c);
      ms_merge(m, s, v.x, v.y, a.c_hi);
    }
    sm.rowm[r] = m;
    sm.rows[r] = s;
    if (a.out_row_stats) {
      a.out_row_stats[((size_t)b * R + r) * 2 + 0] = (float)((double)m * a.inv_tau);
      a.out_row_stats[((size_t)b * R + r) * 2 + 1] = s;
    }
  }
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const int32_t* x = a.tokens + (size_t)b * K;
  bool bad = false;
  for (int r = lane; r < R; r += 32) {
    const float s = sm.rows[r];
    bad |= !(s > 0.f) || !(s < INFINITY) || !(sm.rowm[r] < INFINITY);
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
        const double mT = sm.rowm[i], sT = sm.rows[i];
        const double mD = sm.rowm[K + 1 + i], sD = sm.rows[K + 1 + i];
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
    si.n = n;
    si.mT = sm.rowm[n];
    si.sT = sm.rows[n];
    if (n < K) {
      si.mode = kModeResidual;
      si.mD = sm.rowm[K + 1 + n];
      const double lam = log2((double)sm.rows[n]) - log2((double)sm.rows[K + 1 + n]);
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
}

// ---------------------------------------------------------------------------
// tail work: per-piece masses of one chunk of the tail row
// ---------------------------------------------------------------------------
template <class E, int VEC>
__device__ void tail_compute(const SampleArgs& a, int b, int t, const SeqInfo& si, SampleSmem& sm) {
  using S = typename E::storage;
  constexpr int STEP = kThreads * VEC;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = si.n;
  const S* rowT = target_row<E>(a, b, n);
  const S* rowD = si.mode == kModeResidual ? draft_row<E>(a, b, n) : rowT;
  TailConsts k;
  k.mT = si.mT;
  k.mD = si.mD;
  k.c_hi = a.c_hi;
  k.c_lo = a.c_lo;
  k.lam_hi = si.lam_hi;
  k.lam_lo = si.lam_lo;
  k.residual = si.mode == kModeResidual;
  const int v0 = t * a.CH, v1 = min(a.V, v0 + a.CH);
  // piece (step, warp) = the 32 * VEC elements a warp covers in one step
  const int nsteps = (v1 - v0 + STEP - 1) / STEP;
  int e = v0 + threadIdx.x * VEC;
  for (int st = 0; st < nsteps; st += kTailUnroll, e += STEP * kTailUnroll) {
    Raw<E, VEC> zt[kTailUnroll], zd[kTailUnroll];
#pragma unroll
    for (int u = 0; u < kTailUnroll; ++u) {
      zt[u] = load_raw<E, VEC>(rowT, e + u * STEP, v1);
      zd[u] = k.residual ? load_raw<E, VEC>(rowD, e + u * STEP, v1) : zt[u];
    }
#pragma unroll
    for (int u = 0; u < kTailUnroll; ++u) {
      float ls = 0.f;
#pragma unroll
      for (int q = 0; q < VEC; ++q)
        ls = __fadd_rn(ls, tail_weight(elem(zt[u], q), elem(zd[u], q), k));
      const float ps = warp_sum(ls);
      if (lane == 0 && st + u < nsteps) sm.piece[(st + u) * kWarps + warp] = ps;
    }
  }
  __syncthreads();
  const int np = nsteps * kWarps;
  float* gp = a.pieces + ((size_t)b * a.C + t) * a.P;
  for (int q = threadIdx.x; q < np; q += kThreads) gp[q] = sm.piece[q];
  if (threadIdx.x == 0) {
    double tot = 0.0;
    for (int q = 0; q < np; ++q) tot += (double)sm.piece[q];
    a.tailsum[(size_t)b * a.C + t] = tot;
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// select finisher: inverse CDF over the tail units' masses
// ---------------------------------------------------------------------------
template <class E, int VEC>
__device__ __noinline__ void select_finisher(const SampleArgs& a, int b, SampleSmem& sm) {
  using S = typename E::storage;
  constexpr int STEP = kThreads * VEC;
  if (threadIdx.x == 0) {
    sm.state = ld_acquire(&a.ready[b]);
    if (sm.state) {
      const SeqInfo* g = a.info + b;
      sm.info.n = __ldcg(&g->n);
      sm.info.mode = __ldcg(&g->mode);
      sm.info.mT = __ldcg(&g->mT);
      sm.info.mD = __ldcg(&g->mD);
      sm.info.lam_hi = __ldcg(&g->lam_hi);
      sm.info.lam_lo = __ldcg(&g->lam_lo);
      sm.info.sT = __ldcg(&g->sT);
    }
  }
  __syncthreads();
  if (!sm.state || sm.info.mode == kModeBad) return;
  SeqInfo si = sm.info;
  const int C = a.C;
  const double* ts = a.tailsum + (size_t)b * C;
  // Z == 0 after a rejection can only come from rounding (p(x_n) < q(x_n)
  // forces a positive residual); then the draw falls back to p_n itself.
  double Z = 0.0;
  for (int t = 0; t < C; ++t) Z += __ldcg(ts + t);
  if (si.mode == kModeResidual && !(Z > 0.0)) {
    si.mode = kModeBonus;
    for (int t = 0; t < C; ++t) tail_compute<E, VEC>(a, b, t, si, sm);
    Z = 0.0;
    for (int t = 0; t < C; ++t) Z += __ldcg(ts + t);
  }
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const int n = si.n;
  const double theta = uniform_draw(a.seed, (uint64_t)b, (uint64_t)n, 1) * Z;

  // Chunk, then piece, then lane, then element holding the crossing, each by
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
  const int v0 = tsel * a.CH, v1 = min(a.V, v0 + a.CH);
  const int np = (v1 - v0 + STEP - 1) / STEP * kWarps;
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

  // rescan the 32 x VEC elements of the piece with the same arithmetic
  const int step = psel / kWarps, w = psel % kWarps;
  const int base = v0 + step * STEP + w * 32 * VEC + lane * VEC;
  TailConsts k;
  k.mT = si.mT;
  k.mD = si.mD;
  k.c_hi = a.c_hi;
  k.c_lo = a.c_lo;
  k.lam_hi = si.lam_hi;
  k.lam_lo = si.lam_lo;
  k.residual = si.mode == kModeResidual;
  const S* rowT = target_row<E>(a, b, n);
  const S* rowD = k.residual ? draft_row<E>(a, b, n) : rowT;
  float wv[VEC];
  const Raw<E, VEC> zt = load_raw<E, VEC>(rowT, base, v1);
  const Raw<E, VEC> zd = k.residual ? load_raw<E, VEC>(rowD, base, v1) : zt;
  float ls = 0.f;
#pragma unroll
  for (int q = 0; q < VEC; ++q) {
    wv[q] = tail_weight(elem(zt, q), elem(zd, q), k);
    ls = __fadd_rn(ls, wv[q]);
  }
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
}

// ---------------------------------------------------------------------------
// the two unit kinds
// ---------------------------------------------------------------------------
template <class E, int VEC>
__device__ void stats_unit(const SampleArgs& a, int b, int idx, SampleSmem& sm) {
  using S = typename E::storage;
  constexpr int STEP = kThreads * VEC;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = idx / a.C, c = idx - (idx / a.C) * a.C;
  const S* row = r <= a.K ? target_row<E>(a, b, r) : draft_row<E>(a, b, r - a.K - 1);
  const int v0 = c * a.CH, v1 = min(a.V, v0 + a.CH);
  const float cc = a.c_hi;
  float m = neg_inf();
  float s4[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) s4[u] = 0.f;
  const int nbatch = (v1 - v0 + STEP * kUnroll - 1) / (STEP * kUnroll);
  int e = v0 + threadIdx.x * VEC;
  for (int bt = 0; bt < nbatch; ++bt, e += STEP * kUnroll) {
    Raw<E, VEC> z[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) z[u] = load_raw<E, VEC>(row, e + u * STEP, v1);
    float bm = neg_inf();
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
#pragma unroll
      for (int q = 0; q < VEC; ++q) bm = fmaxf(bm, elem(z[u], q));
    if (bm > m) {
      const float f = ex2((m - bm) * cc);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) s4[u] *= f;
      m = bm;
    }
    const float base = (m == neg_inf()) ? 0.f : m;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
#pragma unroll
      for (int q = 0; q < VEC; ++q) s4[u] += ex2((elem(z[u], q) - base) * cc);
  }
  float s = (s4[0] + s4[1]) + (s4[2] + s4[3]);
  warp_ms(m, s, cc);
  if (lane == 0) {
    sm.wm[warp] = m;
    sm.ws[warp] = s;
  }
  __syncthreads();
  if (warp == 0) {
    m = lane < kWarps ? sm.wm[lane] : neg_inf();
    s = lane < kWarps ? sm.ws[lane] : 0.f;
    warp_ms(m, s, cc);
    if (lane == 0) {
      a.part[((size_t)b * a.R + r) * a.C + c] = make_float2(m, s);
      __threadfence();
      const int done = atomicAdd(&a.ticket1[b], 1);
      sm.flag = done == a.map.A - 1;
    }
  }
  __syncthreads();
  if (sm.flag) {
    __threadfence();
    stats_finisher<E>(a, b, sm);
  }
}

template <class E, int VEC>
__device__ void tail_unit(const SampleArgs& a, int b, int t, SampleSmem& sm) {
  if (threadIdx.x == 0) {
    int st = ld_acquire(&a.ready[b]);
    unsigned it = 0;
    while (st == 0 && ++it < kSpinLimit) {
      __nanosleep(128);
      st = ld_acquire(&a.ready[b]);
    }
    if (st == 0) atomicOr(a.status, kStatusTimeout);
    sm.state = st;
    if (st) {
      const SeqInfo* g = a.info + b;
      sm.info.n = __ldcg(&g->n);
      sm.info.mode = __ldcg(&g->mode);
      sm.info.mT = __ldcg(&g->mT);
      sm.info.mD = __ldcg(&g->mD);
      sm.info.lam_hi = __ldcg(&g->lam_hi);
      sm.info.lam_lo = __ldcg(&g->lam_lo);
      sm.info.sT = __ldcg(&g->sT);
    }
  }
  __syncthreads();
  if (sm.state && sm.info.mode != kModeBad) {
    const SeqInfo si = sm.info;
    tail_compute<E, VEC>(a, b, t, si, sm);
  }
  if (threadIdx.x == 0) {
    __threadfence();
    const int done = atomicAdd(&a.ticket2[b], 1);
    sm.flag = done == a.map.T - 1;
  }
  __syncthreads();
  if (sm.flag) {
    __threadfence();
    select_finisher<E, VEC>(a, b, sm);
  }
}

// Units are only ever claimed from the global counter by a CTA that is already
// running, and claims are handed out in increasing order.  A tail unit waits
// only on statistics units with smaller indices, which are therefore held by
// running CTAs (or finished), so every wait ends even when other work keeps
// part of the grid from being resident.
template <class E, int VEC>
__global__ void __launch_bounds__(kThreads, 2) sample_kernel(const SampleArgs a) {
  __shared__ SampleSmem sm;
  if (threadIdx.x == 0) sm.next = (long long)atomicAdd((unsigned long long*)a.counter, 1ull);
  __syncthreads();
  long long unit = sm.next;
  __syncthreads();
  while (unit < a.map.total) {
    if (threadIdx.x == 0)
      sm.next = (long long)atomicAdd((unsigned long long*)a.counter, 1ull);
    const UnitRef u = decode_unit(a.map, unit);
    if (u.kind == 0)
      stats_unit<E, VEC>(a, u.b, u.idx, sm);
    else
      tail_unit<E, VEC>(a, u.b, u.idx, sm);
    __syncthreads();
    unit = sm.next;
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// host side helpers
// ---------------------------------------------------------------------------
static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t sample_workspace_bytes(int B, int K, int C, int P, size_t* counter_bytes) {
  const int R = 2 * K + 1;
  size_t off = 0;
  off += 16;                          // counter (64-bit) + pad
  off += align_up((size_t)B * 4, 16);  // ticket1
  off += align_up((size_t)B * 4, 16);  // ticket2
  off += align_up((size_t)B * 4, 16);  // ready
  if (counter_bytes) *counter_bytes = off;
  off = align_up(off, 256);
  off += align_up((size_t)B * R * C * sizeof(float2), 256);
  off += align_up((size_t)B * sizeof(SeqInfo), 256);
  off += align_up((size_t)B * C * sizeof(double), 256);
  off += align_up((size_t)B * C * P * sizeof(float), 256);
  return off;
}

void sample_bind_workspace(SampleArgs& a, void* ws) {
  char* p = (char*)ws;
  const int B = a.B, R = a.R, C = a.C;
  a.counter = (int*)p;
  p += 16;
  a.ticket1 = (int*)p;
  p += align_up((size_t)B * 4, 16);
  a.ticket2 = (int*)p;
  p += align_up((size_t)B * 4, 16);
  a.ready = (int*)p;
  p += align_up((size_t)B * 4, 16);
  p = (char*)ws + align_up((size_t)(p - (char*)ws), 256);
  a.part = (float2*)p;
  p += align_up((size_t)B * R * C * sizeof(float2), 256);
  a.info = (SeqInfo*)p;
  p += align_up((size_t)B * sizeof(SeqInfo), 256);
  a.tailsum = (double*)p;
  p += align_up((size_t)B * C * sizeof(double), 256);
  a.pieces = (float*)p;
}

int sample_pieces_per_unit(int CH, bool bf16, bool vec) {
  const int step = kThreads * (vec ? (bf16 ? 8 : 4) : 1);
  return (CH + step - 1) / step * kWarps;
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
