// tree_sample_kernel.cu -- stochastic (temperature > 0) verification of a token
// tree per sequence.
//
// [P4] "Speculative Decoding in Production: How Small Draft Models & Medusa
// Heads Deliver 2x-3x LLM Speedups Without Accuracy Loss", sec. 4 (a tree of
// candidate continuations verified in one target pass, the longest accepted
// path kept), with the acceptance rule and residual of [P1] "Speculative
// Decoding & Draft Model Topologies ...", sec. 2, applied node by node: the
// children of the current node u are tried in index order against the current
// target distribution P (initially softmax of target row u), each accepted with
// probability min(1, P(x) / Q(x)), Q = softmax of draft row u (the distribution
// the children were drawn from); a rejected child replaces P by
// norm(max(0, P - Q)).  When no child is accepted (or u is a leaf) one token is
// drawn from the current P by inverse CDF.
//
// Residuals in closed form.  Write rho(v) = P0(v) / Q(v) = 2^delta(v) for the
// row's own distributions.  After k rejections the current distribution is
// P_k(v) = Q(v) max(0, rho(v) - A_k) / B_k with A_0 = 0, B_0 = 1,
// A_k = A_{k-1} + B_{k-1} and B_k = sum_v P0(v) (1 - 2^{-(delta(v) - L_k)})_+,
// L_k = log2 A_k (induction on max(0, P_{k-1} - Q) = Q max(0, rho - A_k) /
// B_{k-1}).  Since Q rho = P0 and A_k 2^{-L_k} = 1, the weight of v is
// P0(v) (1 - 2^{-(delta(v) - L_k)}): the chain's cancellation-free residual
// weight with the threshold moved by L_k.  So each rejection costs one pass
// over the row pair for B_k, no distribution is ever stored, and the
// acceptance ratio of a child x is P_k(x) / Q(x) = max(0, rho(x) - A_k) / B_k,
// evaluated in fp64 (for the first child, k = 0, the ratio 2^delta comes
// from ex2: see exp2_neg).
//
// Two kernels: row statistics (m, s) of every target and draft row (a flat
// list of slices over all sequences, each warp taking every W-th slice, the
// row's last slice merging the row), then the walk: one thread-block cluster
// of C CTAs per sequence (C chosen so that all clusters are resident at once),
// each pass over a row pair split into one contiguous chunk per warp of the
// cluster, the warp masses exchanged through distributed shared memory.
#include "sv_common.cuh"
#include "sv_kernels.h"

#include <cooperative_groups.h>
#include <math.h>
#include <string.h>

namespace cg = cooperative_groups;

namespace sv {

template <class E>
__device__ __forceinline__ const typename E::storage* tree_row(const TreeSampleArgs& a, int b, int rr) {
  // rr in [0, N] target rows, [N + 1, 2N + 1] draft rows
  const int N1 = a.N + 1;
  const typename E::storage* base = (const typename E::storage*)(rr < N1 ? a.target : a.draft);
  return base + ((size_t)b * N1 + (size_t)(rr < N1 ? rr : rr - N1)) * (size_t)a.V;
}

// ---------------------------------------------------------------------------
// row statistics
// ---------------------------------------------------------------------------
template <class E, int VEC>
__global__ void __launch_bounds__(kThreads, kMinBlocks) tree_stats_kernel(const __grid_constant__ TreeSampleArgs a) {
  using S = typename E::storage;
  constexpr int BATCH = 32 * VEC * kUnroll;
  const int lane = threadIdx.x & 31;
  const long long W = (long long)gridDim.x * kWarps;
  // the walk launch may become resident as this grid's CTAs retire
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (long long f = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5); f < a.F; f += W) {
    const long long row_id = f / a.CS;
    const int s = (int)(f - row_id * a.CS);
    const int b = (int)(row_id / a.RR), rr = (int)(row_id - (long long)b * a.RR);
    const S* row = tree_row<E>(a, b, rr);
    const int v0 = s * a.SL, v1 = min(a.V, v0 + a.SL);
    const float cc = a.c_hi;
    float m = neg_inf();
    float2 acc = make_float2(0.f, 0.f), tacc = make_float2(0.f, 0.f);
    const int nb = v1 > v0 ? (v1 - v0 + BATCH - 1) / BATCH : 0;
    int e = v0 + lane * VEC;
    Raw<E, VEC> z0[kUnroll], z1[kUnroll];
    if constexpr (VEC > 1) {
      if (lane == 0 && v1 > v0) prefetch_l2(row + v0, (unsigned)((v1 - v0) * sizeof(S)));
    }
    if (nb > 0) load_batch<E, VEC>(z0, row, e, v1);
    for (int bt = 0; bt < nb; bt += 2, e += 2 * BATCH) {
      if (bt + 1 < nb) load_batch<E, VEC>(z1, row, e + BATCH, v1);
      stats_batch<E, VEC, false>(z0, m, acc, tacc, cc);
      if (bt + 1 < nb) {
        if (bt + 2 < nb) load_batch<E, VEC>(z0, row, e + 2 * BATCH, v1);
        stats_batch<E, VEC, false>(z1, m, acc, tacc, cc);
      }
    }
    float sum = (acc.x + acc.y) * exp_fma_fix(m, cc);  // the fused exponents' common factor out
    warp_ms(m, sum, cc);
    float2* pp = a.part + (size_t)row_id * a.CS;
    int old = 0;
    if (lane == 0) {
      st_relaxed_u2(pp + s, __float_as_uint(m), __float_as_uint(sum));
      old = ticket_take(&a.rowticket[(size_t)row_id * kTicketStride]);
    }
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old == a.CS - 1) {  // the row's last slice: merge the row in slice order
      float mm = neg_inf(), ss = 0.f;
      for (int c = lane; c < a.CS; c += 32) {
        const uint2 w = wait_u2(pp + c, a.status);
        ms_merge(mm, ss, __uint_as_float(w.x), __uint_as_float(w.y), cc);
      }
      warp_ms(mm, ss, cc);
      if (lane == 0) st_relaxed_u2(a.rowstat + row_id, __float_as_uint(mm), __float_as_uint(ss));
    }
  }
}

// ---------------------------------------------------------------------------
// the walk
// ---------------------------------------------------------------------------
constexpr int kWalkWarps = kWalkThreads / 32;
constexpr int kWalkSteps = 128;  // step sums kept per warp for the final search
constexpr int kWalkU = 4;        // warp steps per load group
constexpr int kMaxWalkCluster = 16;  // CTAs per sequence at most (a non-portable cluster size)

// Mass of one warp's chunk [v0, v1) of the current weights (in lane 0): the
// fp64 sum, in step order, of the fp32 step sums (each the butterfly sum of
// the lanes' element-order sums).  Step sums 0 .. kWalkSteps-1 are also left in `steps`
// for chunk_select.  Loads run kWalkU steps ahead of the arithmetic.
template <class E, int VEC>
__device__ double chunk_mass(const typename E::storage* rowT, const typename E::storage* rowD, int v0,
                             int v1, const TailConsts& k, float* steps) {
  constexpr int STEPW = 32 * VEC;
  constexpr int U = kWalkU;
  const int lane = threadIdx.x & 31;
  const int nsteps = v1 > v0 ? (v1 - v0 + STEPW - 1) / STEPW : 0;
  const int e0 = v0 + lane * VEC;
  double total = 0.0;
  Raw<E, VEC> t0[U], d0[U], t1[U], d1[U];
  // positions past v1 load as -inf (weight 0) without touching memory
  auto load_group = [&](Raw<E, VEC>(&t)[U], Raw<E, VEC>(&d)[U], int q0) {
#pragma unroll
    for (int i = 0; i < U; ++i) {
      const int e = e0 + (q0 + i) * STEPW;
      t[i] = load_raw<E, VEC>(rowT, e, v1);
      d[i] = k.residual ? load_raw<E, VEC>(rowD, e, v1) : t[i];
    }
  };
  auto sum_group = [&](const Raw<E, VEC>(&t)[U], const Raw<E, VEC>(&d)[U], int q0) {
#pragma unroll
    for (int i = 0; i < U; ++i) {
      if (q0 + i < nsteps) {
        const float sq = warp_sum(lane_mass<E, VEC>(t[i], d[i], k));
        if (lane == 0) total += (double)sq;  // fp64 in one lane: the result is lane 0's
        if (lane == 0 && q0 + i < kWalkSteps) steps[q0 + i] = sq;
      }
    }
  };
  if (nsteps > 0) load_group(t0, d0, 0);
  for (int q = 0; q < nsteps; q += 2 * U) {
    const bool has1 = q + U < nsteps;
    if (has1) load_group(t1, d1, q + U);
    sum_group(t0, d0, q);
    if (has1) {
      if (q + 2 * U < nsteps) load_group(t0, d0, q + 2 * U);
      sum_group(t1, d1, q + U);
    }
  }
  return total;
}

// One warp step at `base`: the position where the running sum, starting at
// `before`, first passes theta (crossed = true), else the step's last
// position with positive weight (-1 if none).  *step_sum gets the step's
// butterfly sum.
template <class E, int VEC>
__device__ int step_select(const typename E::storage* rowT, const typename E::storage* rowD, int base, int v1,
                           const TailConsts& k, double theta, double before, bool& crossed, float* step_sum) {
  const int lane = threadIdx.x & 31;
  const int e = base + lane * VEC;
  const Raw<E, VEC> zt = load_raw<E, VEC>(rowT, e, v1);
  const Raw<E, VEC> zd = k.residual ? load_raw<E, VEC>(rowD, e, v1) : zt;
  float wv[VEC];
  lane_weights<E, VEC>(zt, zd, k, wv);
  float ls = 0.f;
#pragma unroll
  for (int q = 0; q < VEC; ++q) ls = __fadd_rn(ls, wv[q]);
  *step_sum = warp_sum(ls);
  // exclusive prefix of the lane sums in fp64
  double incl = (double)ls;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const double o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  const double excl = incl - (double)ls;
  const unsigned cb = __ballot_sync(0xffffffffu, ls > 0.f && before + excl + (double)ls > theta);
  const unsigned has = __ballot_sync(0xffffffffu, ls > 0.f);
  crossed = cb != 0u;
  if (!cb && !has) return -1;
  const int L = cb ? __ffs(cb) - 1 : 31 - __clz(has);
  int tok = -1;
  if (lane == L) {
    float part = 0.f;
    int pick = -1, lastpos = -1;
#pragma unroll
    for (int q = 0; q < VEC; ++q) {
      part = __fadd_rn(part, wv[q]);
      if (wv[q] > 0.f) {
        lastpos = q;
        if (cb && pick < 0 && before + excl + (double)part > theta) pick = q;
      }
    }
    if (pick < 0) pick = lastpos;
    tok = e + pick;
  }
  return __shfl_sync(0xffffffffu, tok, L);
}

// The token holding the CDF crossing inside a warp's chunk, the running sum
// starting at `before`: the step is found from the stored step sums (32 at a
// time), then searched position by position; steps past kWalkSteps are
// searched one at a time.  Only positions with positive weight are chosen;
// when rounding leaves theta past every running sum the chunk's last such
// position is taken.
template <class E, int VEC>
__device__ int chunk_select(const typename E::storage* rowT, const typename E::storage* rowD, int v0, int v1,
                            const TailConsts& k, double theta, double before, const float* steps) {
  constexpr int STEPW = 32 * VEC;
  const int lane = threadIdx.x & 31;
  const int nsteps = v1 > v0 ? (v1 - v0 + STEPW - 1) / STEPW : 0;
  const int nst = min(nsteps, kWalkSteps);
  double run = before;
  int lastq = -1;
  double last_before = 0.0;
  bool crossed = false;
  float ps = 0.f;
  for (int base = 0; base < nst; base += 32) {
    const int q = base + lane;
    const float sq = q < nst ? steps[q] : 0.f;
    double incl = (double)sq;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const double o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    double excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = 0.0;
    const unsigned cb = __ballot_sync(0xffffffffu, sq > 0.f && run + incl > theta);
    const unsigned has = __ballot_sync(0xffffffffu, sq > 0.f);
    if (cb) {
      const int L = __ffs(cb) - 1;
      const double bq = run + __shfl_sync(0xffffffffu, excl, L);
      return step_select<E, VEC>(rowT, rowD, v0 + (base + L) * STEPW, v1, k, theta, bq, crossed, &ps);
    }
    if (has) {
      const int L = 31 - __clz(has);
      lastq = base + L;
      last_before = run + __shfl_sync(0xffffffffu, excl, L);
    }
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  int last_tok = -1;
  for (int q = nst; q < nsteps; ++q) {
    const int tok = step_select<E, VEC>(rowT, rowD, v0 + q * STEPW, v1, k, theta, run, crossed, &ps);
    if (crossed) return tok;
    if (tok >= 0) last_tok = tok;
    run += (double)ps;
  }
  if (last_tok >= 0) return last_tok;
  if (lastq >= 0)
    return step_select<E, VEC>(rowT, rowD, v0 + lastq * STEPW, v1, k, theta, last_before, crossed, &ps);
  return -1;
}

// log2 of a double x >= 1 from its float split x = hi + lo: log2(hi) as a
// float pair, plus lo / (hi ln 2) (error about 1e-11).  A double log2 costs
// about a microsecond of latency on this GPU, on the walk's serial path.
__device__ __forceinline__ double log2_split(double x) {
  const float hi = (float)x;
  const float lo = (float)(x - (double)hi);
  const float2 l = log2_pair(hi);
  return (double)l.x + ((double)l.y + (double)__fdiv_rn(lo, hi) * 1.4426950408889634074);
}

// 2^d for d < 0 from the ex2 instruction on the fractional part: relative
// error below 3e-7.  An acceptance decision u < 2^d taken with it can differ
// from the exact one only for |u - 2^d| below 3e-7, inside the 1e-6
// boundary band of the parity accounting.
__device__ __forceinline__ double exp2_neg(double d) {
  if (d < -160.0) return 0.0;
  const double n = floor(d);
  return ldexp((double)ex2((float)(d - n)), (int)n);
}

struct WalkShared {
  // residual state of the current node (thread 0 keeps it; fp64 stays in thread 0)
  double A, B, L, lam, sT;
  float mT, mD;        // row maxima of the current node's target and draft rows
  float lam_hi, lam_lo;  // log2(sT / sD) + L of the next pass, as a float pair
  int residual;        // the next pass weighs the residual (1) or P itself (0)
  int k;               // rejections at the current node
  int u;               // current node (-1: the root)
  int len;             // path entries written
  int decision;        // 1: accept the child under test
  int current;         // the last pass's masses are those of the current distribution
  int pick;            // warp of the cluster whose chunk holds the final draw (-1: none here)
  int tok_out;         // rank 0 only: the drawn token, written by the picking CTA
  double pick_before;
  double theta;
};

// One cluster of a.C CTAs per sequence.  Every CTA runs the same control
// flow: after each pass over the row pair every CTA pushes its fp64 mass into
// the shared memory of all CTAs of the cluster, so after the cluster barrier
// every CTA holds the same per-CTA masses, forms the same sums in the same
// order and takes the same decisions; rank 0 alone writes the outputs.  All
// fp64 arithmetic runs in one thread (or one lane per warp): the fp64 rate of
// the part is a small fraction of its fp32 rate.
template <class E, int VEC>
__global__ void __launch_bounds__(kWalkThreads, 1) tree_walk_kernel(const __grid_constant__ TreeSampleArgs a) {
  using S = typename E::storage;
  constexpr int NW = kWalkWarps;
  __shared__ WalkShared sh;
  __shared__ int s_par[kMaxTreeNodes];
  __shared__ int s_tok[kMaxTreeNodes];
  __shared__ float s_zt[kMaxTreeNodes];  // node i's token: its logit in the parent's target row
  __shared__ float s_zd[kMaxTreeNodes];  // ... and in the parent's draft row
  __shared__ double s_u[kMaxTreeNodes];  // node i's acceptance uniform
  __shared__ double s_wm[NW];                 // this CTA's warp masses of the last pass
  __shared__ double s_cta[2][kMaxWalkCluster];  // every CTA's mass, pushed by its owner
  __shared__ float s_steps[NW][kWalkSteps];
  cg::cluster_group cluster = cg::this_cluster();
  const int C = a.C;
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.x / C;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = a.N, N1 = N + 1;
  const float2* rs = a.rowstat + (size_t)b * a.RR;
  int32_t* path = a.out_path + (size_t)b * N1;

  // The launch is programmatically dependent on the statistics launch: until
  // griddepcontrol.wait below only the sequence's inputs are read, so this
  // part overlaps the end of the statistics.
  // Inputs of the sequence and their check (identical in every CTA).
  bool bad = false;
  for (int i = tid; i < N; i += kWalkThreads) {
    const int p = __ldg(a.parents + (size_t)b * N + i), t = __ldg(a.tokens + (size_t)b * N + i);
    s_par[i] = p;
    s_tok[i] = t;
    bad |= p < -1 || p >= i || t < 0 || t >= a.V;
  }
  bad = __syncthreads_or(bad);
  if (!bad) {
    // every node's decision inputs at once, off the walk's serial path
    for (int i = tid; i < N; i += kWalkThreads) {
      const int x = s_tok[i], pr = s_par[i];
      s_zt[i] = E::load1(tree_row<E>(a, b, pr + 1) + x);
      s_zd[i] = E::load1(tree_row<E>(a, b, N1 + pr + 1) + x);
      s_u[i] = uniform_draw(a.seed, (uint64_t)b, (uint64_t)i, 0);
    }
    // the row statistics, written by the statistics launch
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int r = tid; r < a.RR; r += kWalkThreads) {
      const float2 v = __ldcg(rs + r);
      bad |= !(v.y > 0.f) || !(v.y < INFINITY) || !(v.x < INFINITY) || !(v.x > neg_inf());
    }
    bad = __syncthreads_or(bad);
  }
  if (rank == 0)
    for (int j = tid; j <= N; j += kWalkThreads) path[j] = -1;
  if (bad) {  // every CTA of the cluster returns here; no shared memory was shared yet
    if (tid == 0 && rank == 0) {
      a.out_len[b] = -1;
      atomicOr(a.status, kStatusBadData);
    }
    return;
  }
  if (tid == 0) {
    sh.u = -1;
    sh.len = 0;
    sh.tok_out = -1;  // set before the first cluster barrier; the final draw follows one
  }
  __syncthreads();

  const int gw = rank * NW + warp;  // warp index within the cluster
  const int v0 = (int)min((long long)gw * a.chunk, (long long)a.V);
  const int v1 = (int)min((long long)v0 + a.chunk, (long long)a.V);
  int buf = 0;  // s_cta buffer of the next pass
  // One pass with the constants in sh: returns (in thread 0) the cluster's
  // mass, the fp64 sum of the per-CTA masses in rank order, each the fp64 sum
  // of its warp masses in warp order.
  auto pass = [&](const S* rowT, const S* rowD) -> double {
    TailConsts k;
    k.mT = sh.mT;
    k.mD = sh.mD;
    k.c_hi = a.c_hi;
    k.c_lo = a.c_lo;
    k.lam_hi = sh.lam_hi;
    k.lam_lo = sh.lam_lo;
    k.residual = sh.residual;
    const double wm = chunk_mass<E, VEC>(rowT, rowD, v0, v1, k, s_steps[warp]);
    if (lane == 0) s_wm[warp] = wm;
    __syncthreads();
    if (warp == 0) {
      double cs = 0.0;
      if (lane == 0)
        for (int j = 0; j < NW; ++j) cs += s_wm[j];
      cs = __shfl_sync(0xffffffffu, cs, 0);
      if (lane < C) *cluster.map_shared_rank(&s_cta[buf][rank], lane) = cs;
    }
    cluster.sync();
    double sum = 0.0;
    if (tid == 0)
      for (int r = 0; r < C; ++r) sum += s_cta[buf][r];
    buf ^= 1;  // the next pass writes the other buffer while this one may still be read
    return sum;
  };

  for (;;) {
    // the current node: its row pair, statistics and residual state
    const int u = sh.u;
    const int row = u + 1;
    const S* rowT = tree_row<E>(a, b, row);
    const S* rowD = tree_row<E>(a, b, N1 + row);
    if (tid == 0) {
      const float2 st = __ldcg(rs + row), sd = __ldcg(rs + N1 + row);
      sh.mT = st.x;
      sh.mD = sd.x;
      sh.sT = (double)st.y;
      const float2 lt = log2_pair(st.y), ld = log2_pair(sd.y);  // log2(sT / sD) as a float pair
      const float2 lp = pair_add(lt, make_float2(-ld.x, -ld.y));
      sh.lam = (double)lp.x + (double)lp.y;
      sh.k = 0;
      sh.A = 0.0;
      sh.B = 1.0;
      sh.L = 0.0;
      sh.current = 0;
    }
    __syncthreads();
    bool moved = false;
    for (int c = 0; c < N && !moved; ++c) {
      if (s_par[c] != u) continue;
      if (tid == 0) {
        const int x = s_tok[c];
        const float zT = s_zt[c], zD = s_zd[c];
        bool accept;
        if (zD == neg_inf()) {
          accept = true;  // Q(x) = 0
        } else {
          const double delta = (((double)zT - sh.mT) - ((double)zD - sh.mD)) * a.c64 - sh.lam;
          if (sh.k == 0) {  // P_0(x) / Q(x) = 2^delta
            accept = delta >= 0.0 || s_u[c] < exp2_neg(delta);
          } else {  // after a rejection, (rho - A) may cancel: fp64 throughout
            const double rho = exp2(delta);
            const double g = fmax(0.0, rho - sh.A) / sh.B;  // P_k(x) / Q(x)
            accept = g >= 1.0 || s_u[c] < g;
          }
        }
        sh.decision = accept;
        if (accept) {
          if (rank == 0) path[sh.len] = x;
          sh.len += 1;
          sh.u = c;
        } else {
          // constants of the pass for B_{k+1}: threshold moved by L_{k+1} = log2(A_k + B_k)
          const double shifted = sh.lam + log2_split(sh.A + sh.B);
          sh.lam_hi = (float)shifted;
          sh.lam_lo = (float)(shifted - (double)sh.lam_hi);
          sh.residual = 1;
        }
      }
      __syncthreads();
      if (sh.decision) {
        moved = true;
        break;
      }
      // rejected: the next residual's mass, B_{k+1} = sum P0 (1 - 2^{-(delta - L)})_+
      const double sum = pass(rowT, rowD);
      if (tid == 0) {
        const double Bk = sum / sh.sT;  // weights are sT * P0 (...)
        sh.current = Bk > 0.0;
        if (Bk > 0.0) {  // else only rounding emptied the residual: keep P
          const double A1 = sh.A + sh.B;
          sh.L = log2_split(A1);
          sh.A = A1;
          sh.B = Bk;
          sh.k += 1;
        }
      }
      __syncthreads();
    }
    if (moved) continue;

    // no child accepted (or a leaf): one token from the current distribution
    if (!sh.current) {
      if (tid == 0) {
        const double shifted = sh.lam + sh.L;
        sh.lam_hi = (float)shifted;
        sh.lam_lo = (float)(shifted - (double)sh.lam_hi);
        sh.residual = sh.k > 0;
      }
      __syncthreads();
      pass(rowT, rowD);
    }
    const int last = buf ^ 1;  // buffer of the pass that matches the current distribution
    if (tid == 0) {
      double Z = 0.0;
      for (int r = 0; r < C; ++r) Z += s_cta[last][r];
      const double theta = uniform_draw(a.seed, (uint64_t)b, (uint64_t)row, 1) * Z;
      // the CTA, then the warp, whose chunk holds the crossing (positive mass only)
      double run = 0.0, last_before = 0.0;
      int pr = -1, lastr = -1;
      for (int r = 0; r < C; ++r) {
        const double m = s_cta[last][r];
        if (!(m > 0.0)) continue;
        if (run + m > theta) {
          pr = r;
          break;
        }
        lastr = r;
        last_before = run;
        run += m;
      }
      if (pr < 0) {
        pr = lastr;
        run = last_before;
      }
      int pick = -1;
      if (pr == rank) {
        double wrun = run, wlast_before = run;
        int lastw = -1;
        for (int j = 0; j < NW; ++j) {
          const double m = s_wm[j];
          if (!(m > 0.0)) continue;
          if (wrun + m > theta) {
            pick = j;
            break;
          }
          lastw = j;
          wlast_before = wrun;
          wrun += m;
        }
        if (pick < 0) {
          pick = lastw;
          wrun = wlast_before;
        }
        run = wrun;
      }
      sh.pick = pick;
      sh.pick_before = run;
      sh.theta = theta;
    }
    __syncthreads();
    if (warp == sh.pick) {
      TailConsts k;
      k.mT = sh.mT;
      k.mD = sh.mD;
      k.c_hi = a.c_hi;
      k.c_lo = a.c_lo;
      k.lam_hi = sh.lam_hi;
      k.lam_lo = sh.lam_lo;
      k.residual = sh.residual;
      const int tok = chunk_select<E, VEC>(rowT, rowD, v0, v1, k, sh.theta, sh.pick_before, s_steps[warp]);
      if (lane == 0) *cluster.map_shared_rank(&sh.tok_out, 0) = tok;
    }
    cluster.sync();  // the token is in rank 0; no CTA's shared memory is read after this
    if (rank == 0 && tid == 0) {
      const int tok = sh.tok_out;
      if (tok >= 0) {
        path[sh.len] = tok;
        a.out_len[b] = sh.len + 1;
      } else {  // no mass anywhere: only an expired wait in the statistics can do this
        a.out_len[b] = -1;
        atomicOr(a.status, kStatusTimeout);
      }
    }
    return;
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static size_t align_up_t(size_t x, size_t al) { return (x + al - 1) / al * al; }

// [row tickets (start at -1)][marker-filled: part, rowstat]; one 0xff fill.
static void tree_layout(int B, int RR, int CS, size_t* off) {
  const size_t rows = (size_t)B * RR;
  size_t o = 0;
  off[0] = o; o += align_up_t(rows * kTicketStride * 4, 256);            // rowticket
  off[1] = o; o += align_up_t(rows * CS * sizeof(float2), 256);          // part
  off[2] = o; o += align_up_t(rows * sizeof(float2), 256);               // rowstat
  off[3] = o;
}

WsLayout tree_sample_workspace(int B, int RR, int CS) {
  size_t off[4];
  tree_layout(B, RR, CS, off);
  WsLayout l;
  l.total = off[3];
  l.zero_bytes = 0;
  l.marker_off = 0;
  l.marker_bytes = off[3];
  return l;
}

void tree_sample_bind_workspace(TreeSampleArgs& a, void* ws) {
  size_t off[4];
  tree_layout(a.B, a.RR, a.CS, off);
  char* p = (char*)ws;
  a.rowticket = (int*)(p + off[0]);
  a.part = (float2*)(p + off[1]);
  a.rowstat = (float2*)(p + off[2]);
}

template <class E, int VEC>
static cudaError_t launch_tree_sample_t(const TreeSampleArgs& a, int stats_grid, cudaStream_t s) {
  tree_stats_kernel<E, VEC><<<stats_grid, kThreads, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)a.B * (unsigned)a.C);
  cfg.blockDim = dim3(kWalkThreads);
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)a.C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  // programmatic dependent launch: the walk reads its inputs while the
  // statistics finish and waits for them in griddepcontrol.wait
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, tree_walk_kernel<E, VEC>, a);
}

cudaError_t launch_tree_sample(const TreeSampleArgs& a, bool bf16, bool vec, int stats_grid, cudaStream_t s) {
  if (bf16) return vec ? launch_tree_sample_t<BF16, 8>(a, stats_grid, s) : launch_tree_sample_t<BF16, 1>(a, stats_grid, s);
  return vec ? launch_tree_sample_t<F32, 4>(a, stats_grid, s) : launch_tree_sample_t<F32, 1>(a, stats_grid, s);
}

template <class E, int VEC>
static int blocks_tree_stats_t() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, tree_stats_kernel<E, VEC>, kThreads, 0) != cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

// Clusters of C walk CTAs that fit on the device at once (0: none).
template <class E, int VEC>
static int walk_clusters_t(int C) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)C);
  cfg.blockDim = dim3(kWalkThreads);
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (C > 8 &&
      cudaFuncSetAttribute(tree_walk_kernel<E, VEC>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
          cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (cudaOccupancyMaxActiveClusters(&n, tree_walk_kernel<E, VEC>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

int tree_walk_clusters(bool bf16, bool vec, int C) {
  if (bf16) return vec ? walk_clusters_t<BF16, 8>(C) : walk_clusters_t<BF16, 1>(C);
  return vec ? walk_clusters_t<F32, 4>(C) : walk_clusters_t<F32, 1>(C);
}

int tree_stats_blocks_per_sm(bool bf16, bool vec) {
  if (bf16) return vec ? blocks_tree_stats_t<BF16, 8>() : blocks_tree_stats_t<BF16, 1>();
  return vec ? blocks_tree_stats_t<F32, 4>() : blocks_tree_stats_t<F32, 1>();
}

cudaError_t tree_sample_set_spin_limit(unsigned n) { return set_spin_limit_here(n); }

}  // namespace sv
