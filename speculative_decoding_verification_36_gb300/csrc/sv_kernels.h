// sv_kernels.h -- parameter blocks and launchers shared by the C-ABI layer
// (api.cu) and the kernel translation units.  Internal to the library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

constexpr int kThreads = 512;             // threads per CTA for every kernel
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;                // 16-byte vectors in flight per thread (statistics, argmax)
constexpr int kTailUnroll = 2;            // vectors in flight per row in the tail units
constexpr int kMaxSteps = 32;             // steps (kThreads vectors) per chunk: pieces <= 512
constexpr int kMaxK = 255;                // rows per sequence stay <= 2*255+1 < kThreads
constexpr int kMaxTreeNodes = 1024;

// Per-sequence decision left by the statistics finisher for the tail units.
struct SeqInfo {
  int n;         // accepted count; the tail row is target row n (and draft row n)
  int mode;      // kModeResidual, kModeBonus, kModeBad
  float mT;      // max raw logit of target row n
  float mD;      // max raw logit of draft row n (residual mode)
  float lam_hi;  // log2(sT / sD) as a float pair
  float lam_lo;
  float sT;      // sum_v exp2((z - mT) * c) of target row n
  int pad;
};
constexpr int kModeResidual = 0;
constexpr int kModeBonus = 1;
constexpr int kModeBad = 2;

// Work units are chunks of rows.  A persistent grid claims them in a global
// order in which each sequence's statistics units come first and its tail
// units (the residual / bonus row, split the same way) follow `delta`
// sequences later, so that the re-read of the tail row hits L2.
struct UnitMap {
  int B;
  int A;      // statistics units per sequence (rows * chunks)
  int T;      // tail units per sequence (0 for the greedy kernels)
  int delta;  // slack, in sequences, between statistics and tail units
  long long total;
};

struct SampleArgs {
  const void* target;
  const void* draft;
  const int32_t* tokens;
  int B, K, V;
  int R;   // rows per sequence = 2K+1
  int CH;  // chunk length in elements (multiple of 8)
  int C;   // chunks per row
  int P;   // piece slots per tail unit
  UnitMap map;
  float c_hi, c_lo;  // log2(e)/temperature as a float pair
  double c64;        // the same in double
  double inv_tau;    // 1 / temperature
  uint64_t seed;
  int32_t* out_tokens;
  int32_t* out_n;
  float* out_row_stats;  // optional [B, R, 2]: max(z)/tau, sum exp(z/tau - max)
  float* out_pq;         // optional [B, K, 2]: p_i(x_i), q_i(x_i)
  float* out_resid;      // optional [B]: mass of the replacement distribution
  // workspace
  int* counter;   // [1] 64-bit count of claimed units
  int* ticket1;   // [B] finished statistics units
  int* ticket2;   // [B] finished tail units
  int* ready;     // [B] 0 until the statistics finisher published SeqInfo
  float2* part;   // [B, R, C] per-chunk (m, s)
  SeqInfo* info;  // [B]
  double* tailsum;  // [B, C] per tail-unit mass
  float* pieces;    // [B, C, P] per-piece mass
  unsigned* status;
};

struct GreedyArgs {
  const void* target;
  const int32_t* tokens;     // chain: [B, K]; tree: [B, N]
  const int32_t* parents;    // tree only: [B, N]
  int B, K, V;               // chain: K drafts; tree: K = N nodes
  int R;                     // rows per sequence: K+1 (chain) or N+1 (tree)
  int CH, C;
  UnitMap map;
  int32_t* out_tokens;       // chain [B, K+1]; tree out_path [B, N+1]
  int32_t* out_n;            // chain [B];     tree out_len  [B]
  uint32_t* out_mask;        // tree [B, N, ceil(N/32)]
  int32_t* out_row_argmax;   // optional [B, R]
  int* counter;
  int* ticket1;
  float* part_v;             // [B, R, C] chunk max
  int* part_i;               // [B, R, C] chunk argmax (lowest index)
  int* part_nan;             // [B, R, C] chunk saw a NaN
  unsigned* status;
};

// Workspace bytes for each kernel (the counters come first and are zeroed by
// the caller before every launch; `counter_bytes` reports how many).
size_t sample_workspace_bytes(int B, int K, int C, int P, size_t* counter_bytes);
size_t greedy_workspace_bytes(int B, int R, int C, size_t* counter_bytes);

// Bind workspace pointers into the argument blocks.
void sample_bind_workspace(SampleArgs& a, void* ws);
void greedy_bind_workspace(GreedyArgs& a, void* ws);

// Launchers: `grid` CTAs of kThreads threads, persistent.  `vec` selects the
// 16-byte vector path (rows 16-byte aligned) or the scalar path.
cudaError_t launch_sample(const SampleArgs& a, bool bf16, bool vec, int grid, cudaStream_t s);
cudaError_t launch_greedy(const GreedyArgs& a, bool bf16, bool vec, int grid, cudaStream_t s);
cudaError_t launch_tree(const GreedyArgs& a, bool bf16, bool vec, int grid, cudaStream_t s);

// Resident CTAs per SM for each kernel (occupancy calculator).
int sample_blocks_per_sm(bool bf16, bool vec);
int greedy_blocks_per_sm(bool bf16, bool vec);
int tree_blocks_per_sm(bool bf16, bool vec);

// Piece slots per tail unit for a chunk of CH elements.
int sample_pieces_per_unit(int CH, bool bf16, bool vec);

}  // namespace sv
