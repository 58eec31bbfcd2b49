// greedy_kernel.cu -- greedy (temperature 0) chain verification and greedy
// verification of a candidate tree.
//
// Chain ("Speculative Decoding at Scale ..." sequence diagram: accept the
// matching tokens, reject the first mismatch, one bonus token): g_i is the
// argmax of target row i with the lowest id winning ties; n is the first i
// with x_i != g_i (K when all match); the emitted tokens are x_0..x_{n-1}, g_n.
//
// Tree ("Speculative Decoding & Draft Model Topologies ..." sec. 4: all nodes
// verified in one pass under a 2D tree mask, the longest accepted path wins;
// "Speculative Decoding in Production ..." sec. 4: SpecInfer trees of top-2
// candidates): row 0 is the root, row i+1 is node i.  Node i is accepted when
// its parent is accepted (the root always is) and its token equals the argmax
// of its parent's row.  Output: the tokens of the deepest accepted node's path
// (lowest node index on ties), the bonus argmax of that node's row, and the
// N x N ancestor-or-self bitmask of the tree.
//
// Both use the sliced-unit loop of the sampling kernel without tail units: a
// slice of one row is reduced to (max, lowest argmax, NaN seen); the warp
// taking a sequence's last ticket merges the slices in order and writes that
// sequence's outputs.
//
// Early exit ("Speculative Decoding for LLM Inference ..." section "The
// draft-and-verify loop": what follows the first rejection is discarded):
// rows are streamed by position (chain) or node index (tree), and a row that
// cannot change the result -- a position after a decided sequence's first
// mismatch, a node already known to be rejected -- is skipped.  Row finishers
// resolve positions / nodes as their rows complete, and the warp whose
// resolution settles the sequence writes its outputs.
#include "sv_common.cuh"
#include "sv_kernels.h"

#include <limits.h>

namespace sv {

template <class E>
__device__ __forceinline__ const typename E::storage* grow(const GreedyArgs& a, int b, int r) {
  return (const typename E::storage*)a.target + ((size_t)b * a.R + r) * (size_t)a.V;
}

__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Batch maximum that propagates NaN (a NaN anywhere makes the result NaN).
template <class E, int VEC>
__device__ __forceinline__ float batch_max_nan(const Raw<E, VEC> (&z)[kUnroll]) {
  if constexpr (VEC == 8) {
    uint32_t mw = bf16x2_max_nan(bf16x2_max_nan(z[0].w.x, z[0].w.y), bf16x2_max_nan(z[0].w.z, z[0].w.w));
#pragma unroll
    for (int u = 1; u < kUnroll; ++u)
      mw = bf16x2_max_nan(mw, bf16x2_max_nan(bf16x2_max_nan(z[u].w.x, z[u].w.y),
                                             bf16x2_max_nan(z[u].w.z, z[u].w.w)));
    const float lo = bf16_lo(mw), hi = bf16_hi(mw);
    return (lo != lo || hi != hi) ? lo + hi : fmaxf(lo, hi);
  } else {
    float bm = neg_inf();
    bool nan = false;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
#pragma unroll
      for (int q = 0; q < VEC; ++q) {
        const float x = elem(z[u], q);
        bm = fmaxf(bm, x);
        nan |= x != x;
      }
    return nan ? __int_as_float(0x7fc00000) : bm;
  }
}

template <class E, int VEC>
__device__ __forceinline__ void argmax_batch(const Raw<E, VEC> (&z)[kUnroll], int e, float& best, int& bi,
                                             bool& nan) {
  constexpr int STEPW = 32 * VEC;
  const float bm = batch_max_nan<E, VEC>(z);
  if (bm != bm) {
    nan = true;
  } else if (bm > best) {
    int found = INT_MAX;
#pragma unroll
    for (int u = kUnroll - 1; u >= 0; --u)
#pragma unroll
      for (int q = VEC - 1; q >= 0; --q)
        if (elem(z[u], q) == bm) found = e + u * STEPW + q;
    best = bm;
    bi = found;
  }
}

template <class E, int VEC>
__device__ __forceinline__ void gload_batch(Raw<E, VEC> (&z)[kUnroll], const typename E::storage* row, int e,
                                            int v1) {
  constexpr int STEPW = 32 * VEC;
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) z[u] = load_raw<E, VEC>(row, e + u * STEPW, v1);
}

// Slice w of unit idx of sequence b (one warp): (max, lowest argmax, NaN
// seen) into the workspace as one 64-bit word, then the row's ticket; returns
// the atomic's old value (lane 0).
template <class E, int VEC>
__device__ int argmax_slice(const GreedyArgs& a, int b, int idx, int w) {
  using S = typename E::storage;
  constexpr int BATCH = 32 * VEC * kUnroll;
  const int lane = threadIdx.x & 31;
  const int r = idx / a.CU, uc = idx - (idx / a.CU) * a.CU;
  const int s = uc * kSlices + w;
  const S* row = grow<E>(a, b, r);
  const int v0 = s * a.SL, v1 = min(a.V, v0 + a.SL);
  float best = neg_inf();
  int bi = INT_MAX;
  bool nan = false;
  const int nb = v1 > v0 ? (v1 - v0 + BATCH - 1) / BATCH : 0;
  int e = v0 + lane * VEC;
  Raw<E, VEC> z0[kUnroll], z1[kUnroll];
  if constexpr (VEC > 1) {
    if (lane == 0 && v1 > v0) prefetch_l2(row + v0, (unsigned)((v1 - v0) * sizeof(S)));
  }
  if (nb > 0) gload_batch<E, VEC>(z0, row, e, v1);
  for (int bt = 0; bt < nb; bt += 2, e += 2 * BATCH) {
    if (bt + 1 < nb) gload_batch<E, VEC>(z1, row, e + BATCH, v1);
    argmax_batch<E, VEC>(z0, e, best, bi, nan);
    if (bt + 1 < nb) {
      if (bt + 2 < nb) gload_batch<E, VEC>(z0, row, e + 2 * BATCH, v1);
      argmax_batch<E, VEC>(z1, e + BATCH, best, bi, nan);
    }
  }
  warp_am(best, bi);
  const bool anynan = __any_sync(0xffffffffu, nan);
  int old = 0;
  if (lane == 0) {
    const size_t o = ((size_t)b * a.R + r) * (a.CU * kSlices) + s;
    st_relaxed_u2(a.part + o, __float_as_uint(best), (uint32_t)bi | (anynan ? 0x80000000u : 0u));
    old = ticket_take(&a.rowticket[((size_t)b * a.R + r) * kTicketStride]);
  }
  return old;
}

// Row finisher (one warp): merges the slice results of row r (lowest index
// wins ties, so the merge order does not matter) into g[b][r] (-2 for an
// unusable row: NaN, +inf, all -inf); returns true in the lane-uniform sense
// when this was the sequence's last row.
__device__ __noinline__ bool row_argmax_finisher(const GreedyArgs& a, int b, int r) {
  const int lane = threadIdx.x & 31;
  const int C = a.CU * kSlices;
  const uint2* pp = a.part + ((size_t)b * a.R + r) * C;
  float v = neg_inf();
  int i = INT_MAX;
  bool nan = false;
  for (int c = lane; c < C; c += 32) {
    const uint2 w = wait_u2(pp + c, a.status);
    am_merge(v, i, __uint_as_float(w.x), (int)(w.y & 0x7fffffffu));
    nan |= (w.y >> 31) != 0;
  }
  warp_am(v, i);
  nan = __any_sync(0xffffffffu, nan);
  const int gv = (nan || !(v > neg_inf()) || !(v < INFINITY) || i == INT_MAX) ? -2 : i;
  int old = 0;
  if (lane == 0) {
    st_relaxed_s32(a.g + (size_t)b * a.R + r, gv);
    old = ticket_take(&a.seqticket[b]);
  }
  old = __shfl_sync(0xffffffffu, old, 0);
  return old == a.R - 1;
}

// Early-exit row finisher (one warp): the argmax of row r of sequence b, the
// verdict of position r (bad row or token, match, mismatch), its resolution
// and, when that resolution decides the sequence, the sequence's outputs.
// Only what the result uses is checked, in position order: a bad row or token
// after the first mismatch is never read.
__device__ __noinline__ void ee_row_finisher(const GreedyArgs& a, int b, int r) {
  const int lane = threadIdx.x & 31;
  const int K = a.K;
  const int C = a.CU * kSlices;
  const uint2* pp = a.part + ((size_t)b * a.R + r) * C;
  float v = neg_inf();
  int i = INT_MAX;
  bool nan = false;
  for (int c = lane; c < C; c += 32) {
    const uint2 w = wait_u2(pp + c, a.status);
    am_merge(v, i, __uint_as_float(w.x), (int)(w.y & 0x7fffffffu));
    nan |= (w.y >> 31) != 0;
  }
  warp_am(v, i);
  nan = __any_sync(0xffffffffu, nan);
  const int gv = (nan || !(v > neg_inf()) || !(v < INFINITY) || i == INT_MAX) ? -2 : i;
  int verdict = gv < 0 ? kVerdictBad : kVerdictAccept;
  if (r < K && verdict == kVerdictAccept) {
    const int x = __ldg(a.tokens + (size_t)b * K + r);
    verdict = (x < 0 || x >= a.V) ? kVerdictBad : (x == gv ? kVerdictAccept : kVerdictReject);
  }
  int n = -1;
  if (lane == 0) {
    st_relaxed_s32(a.g + (size_t)b * a.R + r, gv);
    st_relaxed_s32(a.verdict + (size_t)b * a.R + r, verdict);
    unsigned long long bits = 1ull << r;
    if (verdict != kVerdictAccept && r < K) bits |= 1ull << (32 + r);
    const unsigned long long old_set = ~atomicAnd(a.resword + b, ~bits);
    const int was = decided_n(old_set, K), now = decided_n(old_set | bits, K);
    if (was < 0 && now >= 0) {
      n = now;
      st_relaxed_s32(a.decided + b, n);  // later rows of b may skip
    }
  }
  n = __shfl_sync(0xffffffffu, n, 0);
  if (n < 0) return;
  // decided at n: positions 0..n-1 matched; position n mismatched, was bad,
  // or is the bonus row
  const int vn = n == r ? verdict : wait_s32(a.verdict + (size_t)b * a.R + n, a.status);
  const bool bad = vn == kVerdictBad;
  const int gn = bad ? -1 : (n == r ? gv : wait_s32(a.g + (size_t)b * a.R + n, a.status));
  const int32_t* x = a.tokens + (size_t)b * K;
  int32_t* out = a.out_tokens + (size_t)b * (K + 1);
  for (int j = lane; j <= K; j += 32) out[j] = bad ? -1 : (j < n ? __ldg(x + j) : (j == n ? gn : -1));
  if (lane == 0) {
    a.out_n[b] = bad ? -1 : n;
    if (bad) atomicOr(a.status, kStatusBadData);
  }
  __syncwarp();
}

// The finished argmax of row r (waits for the row finisher's store).
__device__ __forceinline__ int row_g(const GreedyArgs& a, int b, int r) {
  return wait_s32(a.g + (size_t)b * a.R + r, a.status);
}

// Chain finisher (one warp): acceptance while x_i equals the argmax.
__device__ __noinline__ void chain_finisher(const GreedyArgs& a, int b) {
  const int K = a.K;
  const int lane = threadIdx.x & 31;
  const int* g = a.g + (size_t)b * (K + 1);
  for (int r = lane; r <= K; r += 32) {
    const int v = row_g(a, b, r);
    if (a.out_row_argmax) a.out_row_argmax[(size_t)b * (K + 1) + r] = v < 0 ? -1 : v;
  }
  __syncwarp();
  const int32_t* x = a.tokens + (size_t)b * K;
  bool bad = false;
  for (int r = lane; r <= K; r += 32) bad |= __ldcg(g + r) < 0;
  for (int i = lane; i < K; i += 32) bad |= x[i] < 0 || x[i] >= a.V;
  bad = __any_sync(0xffffffffu, bad);
  int n = K;
  for (int i0 = 0; i0 < K && !bad; i0 += 32) {
    const int i = i0 + lane;
    const unsigned mis = __ballot_sync(0xffffffffu, i < K && x[i] != __ldcg(g + min(i, K)));
    if (mis) {
      n = i0 + __ffs(mis) - 1;
      break;
    }
  }
  const int gn = bad ? -1 : __ldcg(g + n);
  int32_t* out = a.out_tokens + (size_t)b * (K + 1);
  for (int j = lane; j <= K; j += 32) out[j] = bad ? -1 : (j < n ? x[j] : (j == n ? gn : -1));
  if (lane == 0) {
    a.out_n[b] = bad ? -1 : n;
    if (bad) atomicOr(a.status, kStatusBadData);
  }
  __syncwarp();
}

// Tree finisher (one warp): argmax of every row, acceptance of every node,
// the deepest accepted path, the bonus token and the ancestor-or-self bitmask.
//
// Nodes are resolved 32 at a time (lane = node), in index order.  Parents
// precede children, so a node's parent is either the root, a node of an
// earlier chunk (its results are already in the workspace) or a node of the
// same chunk.  Within a chunk, pointer jumping over the in-chunk parent links
// (five shuffle rounds) combines acceptance (AND), depth (sum) and the
// ancestor bits of the chunk's own mask column; everything above the chunk
// comes from the topmost in-chunk ancestor's outside parent.  Ancestors have
// smaller indices than their descendants, so mask columns to the right of a
// node's chunk are zero.
__device__ __noinline__ void tree_finisher(const GreedyArgs& a, int b) {
  const int N = a.K;
  const int W = (N + 31) >> 5;
  const int lane = threadIdx.x & 31;
  const int32_t* tok = a.tokens + (size_t)b * N;
  const int32_t* par = a.parents + (size_t)b * N;
  const int* g = a.g + (size_t)b * (N + 1);
  int* depth = a.depth + (size_t)b * (N + 1);
  int* acc = a.acc + (size_t)b * (N + 1);
  bool bad = false;
  for (int r = lane; r <= N; r += 32) {
    const int v = row_g(a, b, r);
    bad |= v < 0;
    if (a.out_row_argmax) a.out_row_argmax[(size_t)b * (N + 1) + r] = v < 0 ? -1 : v;
  }
  for (int i = lane; i < N; i += 32) bad |= par[i] < -1 || par[i] >= i || tok[i] < 0 || tok[i] >= a.V;
  bad = __any_sync(0xffffffffu, bad);
  __syncwarp();
  int32_t* path = a.out_tokens + (size_t)b * (N + 1);
  uint32_t* mask = a.out_mask + (size_t)b * N * W;
  if (bad) {
    for (int j = lane; j <= N; j += 32) path[j] = -1;
    for (int j = lane; j < N * W; j += 32) mask[j] = 0u;
    if (lane == 0) {
      a.out_n[b] = -1;
      atomicOr(a.status, kStatusBadData);
    }
    __syncwarp();
    return;
  }
  int best_d = 0, best_i = -1;  // the root: depth 0
  for (int c = 0; c < W; ++c) {
    const int i0 = 32 * c, i = i0 + lane;
    const bool valid = i < N;
    const int p = valid ? __ldg(par + i) : -1;
    const int t = valid ? __ldg(tok + i) : -1;
    const bool inside = valid && p >= i0;  // parent in this chunk
    // outside parent (or the root): its acceptance and depth are final
    const int gp = valid ? __ldcg(g + p + 1) : -1;
    int ok = valid && t == gp;
    int d = 1;
    if (valid && !inside && p >= 0) {
      ok = ok && __ldcg(acc + p);
      d += __ldcg(depth + p);
    }
    int link = inside ? p - i0 : -1;
    int top = lane;
    uint32_t colbits = valid ? 1u << lane : 0u;  // ancestor-or-self bits in column c
#pragma unroll
    for (int step = 0; step < 5; ++step) {
      const int src = link >= 0 ? link : lane;
      const int ok_s = __shfl_sync(0xffffffffu, ok, src);
      const int d_s = __shfl_sync(0xffffffffu, d, src);
      const int link_s = __shfl_sync(0xffffffffu, link, src);
      const int top_s = __shfl_sync(0xffffffffu, top, src);
      const uint32_t bits_s = __shfl_sync(0xffffffffu, colbits, src);
      if (link >= 0) {
        ok = ok && ok_s;
        d += d_s;
        colbits |= bits_s;
        top = top_s;
        link = link_s;
      }
    }
    // the outside parent of the topmost in-chunk ancestor
    const int ext = __shfl_sync(0xffffffffu, p, top);
    if (valid) {
      st_relaxed_s32(acc + i, ok);
      st_relaxed_s32(depth + i, d);
      uint32_t* row = mask + (size_t)i * W;
      for (int w = 0; w < c; ++w) row[w] = ext >= 0 ? __ldcg(mask + (size_t)ext * W + w) : 0u;
      row[c] = colbits;
      for (int w = c + 1; w < W; ++w) row[w] = 0u;
    }
    // deepest accepted node, lowest index on ties
    int kd = valid && ok ? d : 0, ki = valid && ok ? i : INT_MAX;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const int od = __shfl_xor_sync(0xffffffffu, kd, off);
      const int oi = __shfl_xor_sync(0xffffffffu, ki, off);
      if (od > kd || (od == kd && oi < ki)) {
        kd = od;
        ki = oi;
      }
    }
    if (kd > best_d) {
      best_d = kd;
      best_i = ki;
    }
    __threadfence();  // this chunk's acc, depth and mask rows before the next chunk reads them
    __syncwarp();
  }
  // path tokens: every ancestor-or-self j of the best node sits at depth[j] - 1
  if (best_i >= 0) {
    const uint32_t* brow = mask + (size_t)best_i * W;
    for (int j = lane; j <= best_i; j += 32) {
      if ((__ldcg(brow + (j >> 5)) >> (j & 31)) & 1u) path[__ldcg(depth + j) - 1] = __ldg(tok + j);
    }
  }
  if (lane == 0) {
    path[best_d] = __ldcg(g + best_i + 1);
    a.out_n[b] = best_d + 1;
  }
  for (int j = best_d + 1 + lane; j <= N; j += 32) path[j] = -1;
  __syncwarp();
}

// Row argmax of row r (one warp): -2 for an unusable row (NaN, +inf, no
// finite maximum).
__device__ __forceinline__ int merged_row_argmax(const GreedyArgs& a, int b, int r) {
  const int lane = threadIdx.x & 31;
  const int C = a.CU * kSlices;
  const uint2* pp = a.part + ((size_t)b * a.R + r) * C;
  float v = neg_inf();
  int i = INT_MAX;
  bool nan = false;
  for (int c = lane; c < C; c += 32) {
    const uint2 w = wait_u2(pp + c, a.status);
    am_merge(v, i, __uint_as_float(w.x), (int)(w.y & 0x7fffffffu));
    nan |= (w.y >> 31) != 0;
  }
  warp_am(v, i);
  nan = __any_sync(0xffffffffu, nan);
  return (nan || !(v > neg_inf()) || !(v < INFINITY) || i == INT_MAX) ? -2 : i;
}

__device__ __noinline__ void ee_tree_update(const GreedyArgs& a, int b, unsigned long long rd);

// Tree early exit, row finisher (one warp): the row's argmax, then the
// sequence's update with this row done.
__device__ __noinline__ void ee_tree_row_finisher(const GreedyArgs& a, int b, int r) {
  const int lane = threadIdx.x & 31;
  const int gv = merged_row_argmax(a, b, r);
  unsigned long long rd = 0;
  if (lane == 0) {
    st_relaxed_s32(a.g + (size_t)b * a.R + r, gv);
    rd = ~atomicAnd(a.resword + b, ~(1ull << r)) | (1ull << r);
  }
  rd = __shfl_sync(0xffffffffu, rd, 0);
  ee_tree_update(a, b, rd);
}

// Tree early exit (one warp, N <= 32: lane j is node j).  Called by the
// finisher of a row of sequence b with `rd`, the sequence's rows known to be
// done (bit r: row r, row 0 the root's).  From the argmax of every done row it
// derives, for every node, whether it is known accepted (every link of its
// root path matches: node == argmax of the parent's row) or known rejected
// (some link is known not to match); unknown links are those whose parent
// row is not done.  The rejected nodes are published for the skip check.  Once
// every node is resolved and the rows of the root and of every accepted node
// are done, one warp (the first to get there) writes the outputs; the rows
// under rejected nodes are never needed.  Bad data is checked on what is used:
// every parent index, the root's row, the rows of accepted nodes and the
// tokens of nodes whose parent is accepted.
__device__ __noinline__ void ee_tree_update(const GreedyArgs& a, int b, unsigned long long rd) {
  const int N = a.K;
  const int lane = threadIdx.x & 31;
  const bool valid = lane < N;
  const int32_t* tok = a.tokens + (size_t)b * N;
  const int32_t* par = a.parents + (size_t)b * N;
  const int* g = a.g + (size_t)b * a.R;
  const int p = valid ? __ldg(par + lane) : -1;
  const int t = valid ? __ldg(tok + lane) : -1;
  const bool bad_par = valid && (p < -1 || p >= lane);
  const int prow = bad_par ? 0 : p + 1;
  const bool pdone = valid && !bad_par && ((rd >> prow) & 1ull);
  const int gp = pdone ? wait_s32(g + prow, a.status) : -3;
  // the link into this node: known match, known mismatch, or unknown
  bool acc = pdone && gp >= 0 && t == gp;
  bool rej = pdone && !acc;
  int link = (valid && !bad_par) ? p : -1;  // parent lane (-1: the root)
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int src = link >= 0 ? link : lane;
    const bool acc_s = __shfl_sync(0xffffffffu, acc, src);
    const bool rej_s = __shfl_sync(0xffffffffu, rej, src);
    const int link_s = __shfl_sync(0xffffffffu, link, src);
    if (link >= 0) {
      acc = acc && acc_s;
      rej = rej || rej_s;
      link = link_s;
    }
  }
  const unsigned full = N == 32 ? 0xffffffffu : ((1u << N) - 1u);
  const unsigned A = __ballot_sync(0xffffffffu, valid && acc) & full;
  const unsigned Rm = __ballot_sync(0xffffffffu, valid && rej) & full;
  if (lane == 0 && Rm) atomicAnd(a.rejc + b, ~Rm);
  if (__any_sync(0xffffffffu, bad_par)) {
    // the mask needs every parent: the sequence is bad whatever its rows say
  } else {
    if ((A | Rm) != full) return;                                  // not resolved yet
    if (!(rd & 1ull) || (((unsigned)(rd >> 1) & A) != A)) return;  // used rows still being read
  }
  int claim = 0;
  if (lane == 0) claim = atomicCAS(a.decided + b, (int)kMarker, 1) == (int)kMarker ? 1 : 0;
  if (!__shfl_sync(0xffffffffu, claim, 0)) return;
  // the sequence's outputs (this warp alone)
  const int W = (N + 31) >> 5;  // 1
  int32_t* path = a.out_tokens + (size_t)b * (N + 1);
  uint32_t* mask = a.out_mask + (size_t)b * N * W;
  bool bad = __any_sync(0xffffffffu, bad_par);
  if (!bad) {
    const int g0 = wait_s32(g, a.status);
    const bool pacc = valid && (p < 0 || ((A >> p) & 1u));
    const bool tok_bad = pacc && (t < 0 || t >= a.V);
    const bool row_bad = valid && ((A >> lane) & 1u) && wait_s32(g + lane + 1, a.status) < 0;
    bad = g0 < 0 || __any_sync(0xffffffffu, tok_bad || row_bad);
  }
  if (bad) {
    for (int j = lane; j <= N; j += 32) path[j] = -1;
    for (int j = lane; j < N * W; j += 32) mask[j] = 0u;
    if (lane == 0) {
      a.out_n[b] = -1;
      atomicOr(a.status, kStatusBadData);
    }
    __syncwarp();
    return;
  }
  // depth and ancestor-or-self bits by pointer jumping over the parent links
  int d = valid ? 1 : 0;
  uint32_t bits = valid ? 1u << lane : 0u;
  link = valid ? p : -1;
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int src = link >= 0 ? link : lane;
    const int d_s = __shfl_sync(0xffffffffu, d, src);
    const uint32_t bits_s = __shfl_sync(0xffffffffu, bits, src);
    const int link_s = __shfl_sync(0xffffffffu, link, src);
    if (link >= 0) {
      d += d_s;
      bits |= bits_s;
      link = link_s;
    }
  }
  if (valid) mask[lane] = bits;
  // the deepest accepted node, lowest index on ties (the root: depth 0)
  int kd = valid && ((A >> lane) & 1u) ? d : 0, ki = kd ? lane : INT_MAX;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const int od = __shfl_xor_sync(0xffffffffu, kd, off);
    const int oi = __shfl_xor_sync(0xffffffffu, ki, off);
    if (od > kd || (od == kd && oi < ki)) {
      kd = od;
      ki = oi;
    }
  }
  const int best = kd ? ki : -1;
  const uint32_t bbits = best >= 0 ? __shfl_sync(0xffffffffu, bits, best) : 0u;
  if (valid && ((bbits >> lane) & 1u)) path[d - 1] = t;
  for (int j = kd + 1 + lane; j <= N; j += 32) path[j] = -1;
  if (lane == 0) {
    path[kd] = wait_s32(g + best + 1, a.status);
    a.out_n[b] = kd + 1;
  }
  __syncwarp();
}

// Independent warps claim units in increasing order from their counters.
// The warp taking a row's last ticket merges the row; the one merging a
// sequence's last row runs its finisher.  The only waits are for stores that
// are already issued (slots leaving the marker state).
//
// Early exit (EE, chain only): units are taken by position (row 0 of every
// sequence, then row 1, ...), each row's finisher resolves its position, and
// a unit of row r of a sequence already decided at n < r is skipped.
template <class E, int VEC, bool TREE, bool EE>
__global__ void __launch_bounds__(kThreads, kMinBlocks) argmax_kernel(const __grid_constant__ GreedyArgs a) {
  const int lane = threadIdx.x & 31;
  const int w = slice_of_warp();
  const int last = a.CU * kSlices - 1;  // the last slice of a row
  int unit = bcast(claim_unit(a.counter, lane));
  while (unit < a.map.total) {
    const int next = claim_unit(a.counter, lane);
    int b, idx;
    bool skip = false;
    if constexpr (EE) {
      const int per_pos = a.B * a.CU;
      const int r = unit / per_pos, rem = unit - r * per_pos;
      b = rem / a.CU;
      idx = r * a.CU + (rem - b * a.CU);
      if (r > 0) {
        if constexpr (TREE) {
          // the row of node r - 1: skipped once the node is known rejected
          const unsigned rej = ~(unsigned)bcast((int)ld_relaxed_if(lane == 0, a.rejc + b, 0xffffffffu));
          skip = (rej >> (r - 1)) & 1u;
        } else {
          const int dn = bcast((int)ld_relaxed_if(lane == 0, a.decided + b, kMarker));
          skip = dn >= 0 && dn < r;
        }
      }
    } else {
      b = unit / a.map.A;
      idx = unit - b * a.map.A;
    }
    if (!skip) {
      const int old = __shfl_sync(0xffffffffu, argmax_slice<E, VEC>(a, b, idx, w), 0);
      if (old == last) {
        if constexpr (EE && TREE) {
          ee_tree_row_finisher(a, b, idx / a.CU);
        } else if constexpr (EE) {
          ee_row_finisher(a, b, idx / a.CU);
        } else if (row_argmax_finisher(a, b, idx / a.CU)) {
          if (TREE)
            tree_finisher(a, b);
          else
            chain_finisher(a, b);
        }
      }
    }
    unit = bcast(next);
  }
}

// ---------------------------------------------------------------------------
// host side helpers
// ---------------------------------------------------------------------------
static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace: [counters, tickets (start at -1), resolution words (all-ones:
// empty)][marker-filled: part, g, decided, verdict, rejc][depth, acc]; one
// 0xff fill initialises the first two parts.
static void greedy_layout(int B, int R, int CU, size_t* off) {
  const size_t C = (size_t)CU * kSlices;
  size_t o = 0;
  off[0] = o; o += kCounterBytes;                                     // counter
  off[1] = o; o += align_up((size_t)B * R * kTicketStride * 4, 16);  // rowticket
  off[2] = o; o += align_up((size_t)B * 4, 16);                      // seqticket
  off[10] = o; o += align_up((size_t)B * 8, 16);                     // resword
  o = align_up(o, 256);
  off[3] = o;                                                         // end of zero region
  off[4] = o; o += align_up((size_t)B * R * C * sizeof(uint2), 256);  // part
  off[5] = o; o += align_up((size_t)B * R * 4, 256);                  // g
  off[11] = o; o += align_up((size_t)B * 4, 256);                     // decided
  off[12] = o; o += align_up((size_t)B * R * 4, 256);                 // verdict
  off[13] = o; o += align_up((size_t)B * 4, 256);                     // rejc
  off[6] = o;                                                         // end of marker region
  off[7] = o; o += align_up((size_t)B * R * 4, 256);                  // depth
  off[8] = o; o += align_up((size_t)B * R * 4, 256);                  // acc
  off[9] = o;
}

WsLayout greedy_workspace(int B, int R, int CU) {
  size_t off[14];
  greedy_layout(B, R, CU, off);
  WsLayout l;
  l.total = off[9];
  l.zero_bytes = 0;  // counters and tickets start at -1: one 0xff fill covers everything
  l.marker_off = 0;
  l.marker_bytes = off[6];
  return l;
}

void greedy_bind_workspace(GreedyArgs& a, void* ws) {
  size_t off[14];
  greedy_layout(a.B, a.R, a.CU, off);
  char* p = (char*)ws;
  a.counter = (unsigned long long*)(p + off[0]);
  a.rowticket = (int*)(p + off[1]);
  a.seqticket = (int*)(p + off[2]);
  a.part = (uint2*)(p + off[4]);
  a.g = (int*)(p + off[5]);
  a.depth = (int*)(p + off[7]);
  a.acc = (int*)(p + off[8]);
  a.resword = (unsigned long long*)(p + off[10]);
  a.decided = (int*)(p + off[11]);
  a.verdict = (int*)(p + off[12]);
  a.rejc = (unsigned*)(p + off[13]);
}

template <class E, int VEC, bool TREE>
static cudaError_t launch_t(const GreedyArgs& a, int grid, cudaStream_t s) {
  if (a.early_exit)
    argmax_kernel<E, VEC, TREE, true><<<grid, kThreads, 0, s>>>(a);
  else
    argmax_kernel<E, VEC, TREE, false><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_greedy(const GreedyArgs& a, bool bf16, bool vec, int grid, cudaStream_t s) {
  if (bf16) return vec ? launch_t<BF16, 8, false>(a, grid, s) : launch_t<BF16, 1, false>(a, grid, s);
  return vec ? launch_t<F32, 4, false>(a, grid, s) : launch_t<F32, 1, false>(a, grid, s);
}
cudaError_t launch_tree(const GreedyArgs& a, bool bf16, bool vec, int grid, cudaStream_t s) {
  if (bf16) return vec ? launch_t<BF16, 8, true>(a, grid, s) : launch_t<BF16, 1, true>(a, grid, s);
  return vec ? launch_t<F32, 4, true>(a, grid, s) : launch_t<F32, 1, true>(a, grid, s);
}

template <class K>
static int occ(K kernel) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, 0) != cudaSuccess) return 1;
  return n > 0 ? n : 1;
}

int greedy_blocks_per_sm(bool bf16, bool vec) {
  if (bf16) return vec ? occ(argmax_kernel<BF16, 8, false, false>) : occ(argmax_kernel<BF16, 1, false, false>);
  return vec ? occ(argmax_kernel<F32, 4, false, false>) : occ(argmax_kernel<F32, 1, false, false>);
}
int tree_blocks_per_sm(bool bf16, bool vec) {
  if (bf16) return vec ? occ(argmax_kernel<BF16, 8, true, false>) : occ(argmax_kernel<BF16, 1, true, false>);
  return vec ? occ(argmax_kernel<F32, 4, true, false>) : occ(argmax_kernel<F32, 1, true, false>);
}

cudaError_t greedy_set_spin_limit(unsigned n) { return set_spin_limit_here(n); }

}  // namespace sv
