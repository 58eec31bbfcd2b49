// acceptance_kernel.cu -- batched acceptance statistics over verify outputs.
//
// [P2] "Speculative Decoding for LLM Inference: How Draft-and-Verify
// Accelerates Token Generation", section "How much speedup to expect": the
// per-position acceptance rate alpha and the expected number of tokens per
// draft-and-verify iteration, here measured over a batch of outputs.
//
// hist[j] counts the sequences with n_accepted == j (j = 0..K); hist[K+1]
// counts the rest (bad sequences, n = -1, and anything outside [0, K]).
// alpha[i] = #(n > i) / #(n >= i); mean_tokens = mean of n + 1.  All counts
// are exact integers, so the results do not depend on the order of the atomics.
#include "sv_kernels.h"

#include <math.h>

namespace sv {

// Per-CTA histogram in shared memory (warp-aggregated increments), then one
// 64-bit atomic per bin.
__global__ void __launch_bounds__(256) acceptance_hist_kernel(const int32_t* __restrict__ n, int B, int K,
                                                              unsigned long long* hist) {
  extern __shared__ unsigned sh_hist[];
  const int bins = K + 2;
  for (int i = threadIdx.x; i < bins; i += blockDim.x) sh_hist[i] = 0u;
  __syncthreads();
  // lanes holding the same bin add once, through their lowest lane
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long end = ((long long)B + 31) / 32 * 32;  // whole warps stay converged
  for (long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x; b < end; b += stride) {
    int bin = -1;
    if (b < B) {
      const int v = __ldg(n + b);
      bin = (v >= 0 && v <= K) ? v : K + 1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, bin);
    if (bin >= 0 && (threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&sh_hist[bin], (unsigned)__popc(peers));
  }
  __syncthreads();
  for (int i = threadIdx.x; i < bins; i += blockDim.x) {
    const unsigned c = sh_hist[i];
    if (c) atomicAdd(hist + i, (unsigned long long)c);
  }
}

// alpha and mean tokens from the finished histogram (one thread: K + 2 bins).
__global__ void acceptance_finish_kernel(const unsigned long long* hist, int K, double* alpha,
                                         double* mean_tokens) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  unsigned long long reached = 0;  // #(n >= i), built from the top down
  unsigned long long count = 0;
  double total = 0.0;
  for (int j = K; j >= 0; --j) {
    const unsigned long long h = hist[j];
    count += h;
    total += (double)h * (double)(j + 1);
    if (alpha && j < K) {
      // here `reached` still holds #(n > j); adding h gives #(n >= j)
      const unsigned long long accepted = reached;
      reached += h;
      alpha[j] = reached ? (double)accepted / (double)reached : (double)NAN;
    } else {
      reached += h;
    }
  }
  if (mean_tokens) *mean_tokens = count ? total / (double)count : (double)NAN;
}

cudaError_t launch_acceptance(const int32_t* n, int B, int K, unsigned long long* hist, double* alpha,
                              double* mean_tokens, int sms, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(hist, 0, sizeof(unsigned long long) * (size_t)(K + 2), s);
  if (e != cudaSuccess) return e;
  if (B > 0) {
    // eight CTAs per SM keep enough loads in flight to stream n_accepted; the
    // flush is one 64-bit atomic per CTA and bin
    long long blocks = ((long long)B + 255) / 256;
    const long long cap = (long long)sms * 8;
    if (blocks > cap) blocks = cap;
    acceptance_hist_kernel<<<(int)blocks, 256, sizeof(unsigned) * (size_t)(K + 2), s>>>(n, B, K, hist);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (alpha || mean_tokens) {
    acceptance_finish_kernel<<<1, 32, 0, s>>>(hist, K, alpha, mean_tokens);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace sv
