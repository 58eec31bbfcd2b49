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
// Both use the persistent unit loop of the sampling kernel without tail
// units: a unit is one chunk of one row reduced to (max, lowest argmax, NaN
// seen); the CTA finishing a sequence's last unit (atomic ticket) merges the
// chunks in order and writes that sequence's outputs.
#include "sv_common.cuh"
#include "sv_kernels.h"

#include <limits.h>

namespace sv {

struct ArgmaxSmem {
  long long next;
  int flag;
  float wv[kWarps];
  int wi[kWarps];
};

struct TreeSmem {
  ArgmaxSmem base;
  int g[kMaxTreeNodes + 1];
  int depth[kMaxTreeNodes];
  unsigned char acc[kMaxTreeNodes];
  int best;
};

template <class E>
__device__ __forceinline__ const typename E::storage* grow(const GreedyArgs& a, int b, int r) {
  return (const typename E::storage*)a.target + ((size_t)b * a.R + r) * (size_t)a.V;
}

// One chunk of one row: returns true in every thread of the CTA that finished
// the sequence's last unit.
template <class E, int VEC>
__device__ bool argmax_unit(const GreedyArgs& a, int b, int idx, ArgmaxSmem& sm) {
  using S = typename E::storage;
  constexpr int STEP = kThreads * VEC;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = idx / a.C, c = idx - (idx / a.C) * a.C;
  const S* row = grow<E>(a, b, r);
  const int v0 = c * a.CH, v1 = min(a.V, v0 + a.CH);
  float best = neg_inf();
  int bi = INT_MAX;
  bool nan = false;
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
      for (int q = 0; q < VEC; ++q) {
        const float x = elem(z[u], q);
        bm = fmaxf(bm, x);
        nan |= x != x;
      }
    if (bm > best) {
      int found = INT_MAX;
#pragma unroll
      for (int u = kUnroll - 1; u >= 0; --u)
#pragma unroll
        for (int q = VEC - 1; q >= 0; --q)
          if (elem(z[u], q) == bm) found = e + u * STEP + q;
      best = bm;
      bi = found;
    }
  }
  warp_am(best, bi);
  if (lane == 0) {
    sm.wv[warp] = best;
    sm.wi[warp] = bi;
  }
  const int any_nan = __syncthreads_or(nan);
  if (warp == 0) {
    best = lane < kWarps ? sm.wv[lane] : neg_inf();
    bi = lane < kWarps ? sm.wi[lane] : INT_MAX;
    warp_am(best, bi);
    if (lane == 0) {
      const size_t o = ((size_t)b * a.R + r) * a.C + c;
      a.part_v[o] = best;
      a.part_i[o] = bi;
      a.part_nan[o] = any_nan;
      __threadfence();
      const int done = atomicAdd(&a.ticket1[b], 1);
      sm.flag = done == a.map.A - 1;
    }
  }
  __syncthreads();
  if (sm.flag) __threadfence();
  return sm.flag != 0;
}

// Merge the chunk results of row r (chunk order, lowest index on ties).
// Returns the argmax, or -1 when the row is unusable (NaN, +inf, all -inf).
__device__ __forceinline__ int merged_argmax(const GreedyArgs& a, int b, int r) {
  const size_t o = ((size_t)b * a.R + r) * a.C;
  float v = neg_inf();
  int i = INT_MAX;
  int nan = 0;
  for (int c = 0; c < a.C; ++c) {
    am_merge(v, i, __ldcg(a.part_v + o + c), __ldcg(a.part_i + o + c));
    nan |= __ldcg(a.part_nan + o + c);
  }
  if (nan || !(v > neg_inf()) || !(v < INFINITY) || i == INT_MAX) return -1;
  return i;
}

template <class E, int VEC>
__global__ void __launch_bounds__(kThreads) greedy_kernel(const GreedyArgs a) {
  __shared__ ArgmaxSmem sm;
  __shared__ int g[kMaxK + 1];
  if (threadIdx.x == 0) sm.next = (long long)atomicAdd((unsigned long long*)a.counter, 1ull);
  __syncthreads();
  long long unit = sm.next;
  __syncthreads();
  while (unit < a.map.total) {
    if (threadIdx.x == 0) sm.next = (long long)atomicAdd((unsigned long long*)a.counter, 1ull);
    const int b = (int)(unit / a.map.A), idx = (int)(unit % a.map.A);
    if (argmax_unit<E, VEC>(a, b, idx, sm)) {
      const int K = a.K;
      for (int r = threadIdx.x; r <= K; r += kThreads) {
        g[r] = merged_argmax(a, b, r);
        if (a.out_row_argmax) a.out_row_argmax[(size_t)b * (K + 1) + r] = g[r];
      }
      __syncthreads();
      if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int32_t* x = a.tokens + (size_t)b * K;
        bool bad = false;
        for (int r = lane; r <= K; r += 32) bad |= g[r] < 0;
        for (int i = lane; i < K; i += 32) bad |= x[i] < 0 || x[i] >= a.V;
        bad = __any_sync(0xffffffffu, bad);
        int n = K;
        for (int i0 = 0; i0 < K && !bad; i0 += 32) {
          const int i = i0 + lane;
          const unsigned mis = __ballot_sync(0xffffffffu, i < K && x[i] != g[i]);
          if (mis) {
            n = i0 + __ffs(mis) - 1;
            break;
          }
        }
        int32_t* out = a.out_tokens + (size_t)b * (K + 1);
        for (int j = lane; j <= K; j += 32)
          out[j] = bad ? -1 : (j < n ? x[j] : (j == n ? g[n] : -1));
        if (lane == 0) {
          a.out_n[b] = bad ? -1 : n;
          if (bad) atomicOr(a.status, kStatusBadData);
        }
      }
    }
    __syncthreads();
    unit = sm.next;
    __syncthreads();
  }
}

template <class E, int VEC>
__global__ void __launch_bounds__(kThreads) tree_kernel(const GreedyArgs a) {
  __shared__ TreeSmem ts;
  ArgmaxSmem& sm = ts.base;
  if (threadIdx.x == 0) sm.next = (long long)atomicAdd((unsigned long long*)a.counter, 1ull);
  __syncthreads();
  long long unit = sm.next;
  __syncthreads();
  const int N = a.K;
  const int W = (N + 31) >> 5;
  while (unit < a.map.total) {
    if (threadIdx.x == 0) sm.next = (long long)atomicAdd((unsigned long long*)a.counter, 1ull);
    const int b = (int)(unit / a.map.A), idx = (int)(unit % a.map.A);
    if (argmax_unit<E, VEC>(a, b, idx, sm)) {
      const int32_t* tok = a.tokens + (size_t)b * N;
      const int32_t* par = a.parents + (size_t)b * N;
      int bad = 0;
      for (int r = threadIdx.x; r <= N; r += kThreads) {
        ts.g[r] = merged_argmax(a, b, r);
        bad |= ts.g[r] < 0;
        if (a.out_row_argmax) a.out_row_argmax[(size_t)b * (N + 1) + r] = ts.g[r];
      }
      for (int i = threadIdx.x; i < N; i += kThreads)
        bad |= par[i] < -1 || par[i] >= i || tok[i] < 0 || tok[i] >= a.V;
      bad = __syncthreads_or(bad);
      int32_t* path = a.out_tokens + (size_t)b * (N + 1);
      uint32_t* mask = a.out_mask + (size_t)b * N * W;
      if (bad) {
        for (int j = threadIdx.x; j <= N; j += kThreads) path[j] = -1;
        for (int j = threadIdx.x; j < N * W; j += kThreads) mask[j] = 0u;
        if (threadIdx.x == 0) {
          a.out_n[b] = -1;
          atomicOr(a.status, kStatusBadData);
        }
      } else {
        if (threadIdx.x == 0) {
          // parents precede children, so one pass in node order settles acceptance
          int best = -1, bd = 0;
          for (int i = 0; i < N; ++i) {
            const int p = par[i];
            const bool ok = (p < 0 || ts.acc[p]) && tok[i] == ts.g[p + 1];
            ts.acc[i] = ok;
            ts.depth[i] = p < 0 ? 1 : ts.depth[p] + 1;
            if (ok && ts.depth[i] > bd) {
              bd = ts.depth[i];
              best = i;
            }
          }
          int pos = bd - 1;
          for (int node = best; node >= 0; node = par[node]) path[pos--] = tok[node];
          path[bd] = ts.g[best + 1];
          a.out_n[b] = bd + 1;
          ts.best = bd;
        }
        __syncthreads();
        for (int j = ts.best + 1 + threadIdx.x; j <= N; j += kThreads) path[j] = -1;
        // ancestor-or-self bitmask, one word column per thread, node order
        for (int w = threadIdx.x; w < W; w += kThreads) {
          for (int i = 0; i < N; ++i) {
            const int p = par[i];
            uint32_t word = p >= 0 ? mask[(size_t)p * W + w] : 0u;
            if ((i >> 5) == w) word |= 1u << (i & 31);
            mask[(size_t)i * W + w] = word;
          }
        }
      }
    }
    __syncthreads();
    unit = sm.next;
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// host side helpers
// ---------------------------------------------------------------------------
static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t greedy_workspace_bytes(int B, int R, int C, size_t* counter_bytes) {
  size_t off = 16 + align_up((size_t)B * 4, 16);
  if (counter_bytes) *counter_bytes = off;
  off = align_up(off, 256);
  const size_t n = (size_t)B * R * C;
  off += align_up(n * 4, 256) * 3;
  return off;
}

void greedy_bind_workspace(GreedyArgs& a, void* ws) {
  char* p = (char*)ws;
  a.counter = (int*)p;
  p += 16;
  a.ticket1 = (int*)p;
  p += align_up((size_t)a.B * 4, 16);
  p = (char*)ws + align_up((size_t)(p - (char*)ws), 256);
  const size_t n = (size_t)a.B * a.R * a.C;
  a.part_v = (float*)p;
  p += align_up(n * 4, 256);
  a.part_i = (int*)p;
  p += align_up(n * 4, 256);
  a.part_nan = (int*)p;
}

template <class E, int VEC>
static cudaError_t launch_greedy_t(const GreedyArgs& a, int grid, cudaStream_t s) {
  greedy_kernel<E, VEC><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}
template <class E, int VEC>
static cudaError_t launch_tree_t(const GreedyArgs& a, int grid, cudaStream_t s) {
  tree_kernel<E, VEC><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_greedy(const GreedyArgs& a, bool bf16, bool vec, int grid, cudaStream_t s) {
  if (bf16) return vec ? launch_greedy_t<BF16, 8>(a, grid, s) : launch_greedy_t<BF16, 1>(a, grid, s);
  return vec ? launch_greedy_t<F32, 4>(a, grid, s) : launch_greedy_t<F32, 1>(a, grid, s);
}
cudaError_t launch_tree(const GreedyArgs& a, bool bf16, bool vec, int grid, cudaStream_t s) {
  if (bf16) return vec ? launch_tree_t<BF16, 8>(a, grid, s) : launch_tree_t<BF16, 1>(a, grid, s);
  return vec ? launch_tree_t<F32, 4>(a, grid, s) : launch_tree_t<F32, 1>(a, grid, s);
}

template <class K>
static int occ(K kernel) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, 0) != cudaSuccess) return 1;
  return n > 0 ? n : 1;
}

int greedy_blocks_per_sm(bool bf16, bool vec) {
  if (bf16) return vec ? occ(greedy_kernel<BF16, 8>) : occ(greedy_kernel<BF16, 1>);
  return vec ? occ(greedy_kernel<F32, 4>) : occ(greedy_kernel<F32, 1>);
}
int tree_blocks_per_sm(bool bf16, bool vec) {
  if (bf16) return vec ? occ(tree_kernel<BF16, 8>) : occ(tree_kernel<BF16, 1>);
  return vec ? occ(tree_kernel<F32, 4>) : occ(tree_kernel<F32, 1>);
}

}  // namespace sv
