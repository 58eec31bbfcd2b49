// sv_kernels.h -- parameter blocks and launchers shared by the C-ABI layer
// (api.cu) and the kernel translation units.  Internal to the library.
//
// Work decomposition (all three kernels): a persistent grid of independent
// warps.  A row is cut into slices of SL elements.  Slices are numbered flat
// (the argmax kernels: sequence-major; the sampling kernel: by draft
// position) and slice f is handed out by claim counter f % kSlices, so each
// counter sees one eighth of the claims and every counter has the same amount
// of work.  A slice is reduced to one partial result in the workspace; the
// warp that takes the last ticket of a row (argmax kernels) or of a
// position's row pair (sampling kernel) runs the finisher.  There are no
// CTA-wide barriers: a warp that finishes a row or a sequence stalls only
// itself.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

constexpr int kThreads = 256;  // 8 independent warps per CTA
constexpr int kWarps = kThreads / 32;
constexpr int kSlices = kWarps;  // claim counters (and warp slots) per CTA
static_assert((kSlices & (kSlices - 1)) == 0, "counter rotation masks with kSlices - 1");
constexpr int kCounterStride = 16;  // claim counters 128 bytes apart
constexpr int kTicketStride = 8;    // per-row tickets 32 bytes apart (no same-address pile-up)
constexpr int kMinBlocks = 4;  // resident CTAs per SM the register budget allows (64 regs)
constexpr int kUnroll = 2;     // 16-byte vectors per lane per load batch; two batches in flight
constexpr int kMaxK = 255;
constexpr int kMaskMaxK = 31;  // resolution words hold positions 0..31 (K <= 31)
constexpr int kMaxTreeNodes = 1024;
constexpr unsigned kSpinLimit = 1u << 22;  // bounded waits: about 0.5 s with 128 ns naps

// Division by a per-launch constant d >= 1 for dividends below 2^31, as one
// widening multiply and a shift (Granlund and Montgomery, "Division by
// invariant integers using multiplication", PLDI 1994, theorem 4.2 with N = 31:
// l = ceil(log2 d), m = floor(2^(31+l) / d) + 1 < 2^32, q = (n m) >> (31 + l)).
struct FastDiv {
  uint32_t m;
  int shift;
};
inline FastDiv make_fastdiv(uint32_t d) {
  int l = 0;
  while ((1ull << l) < d) ++l;
  FastDiv f;
  f.m = (uint32_t)((1ull << (31 + l)) / d + 1);
  f.shift = 31 + l;
  return f;
}

// Per-sequence decision, published by the sequence's decider as one 32-byte
// entry of the decision queue.  Entries start filled with kMarker words and
// every field is written once with a value that is never kMarker (n >= 0, and
// the floats are finite), so a reader knows a field has arrived from its value
// alone: no fence or acquire is needed on the hot path.
struct SeqInfo {
  int b;         // sequence
  int n;         // accepted count (0 for a bad sequence); the tail row is row n
  int mode;      // kModeResidual, kModeBonus, kModeBad
  float mT;      // max raw logit of target row n
  float mD;      // max raw logit of draft row n (residual mode)
  float lam_hi;  // log2(sT / sD) as a float pair
  float lam_lo;
  float sT;      // sum_v exp2((z - mT) * c) of target row n
};
constexpr int kModeResidual = 0;
constexpr int kModeBonus = 1;
constexpr int kModeBad = 2;

// Statistics units are numbered sequence-major: unit u is index u % A of
// sequence u / A on every counter.
struct UnitMap {
  int A;      // statistics units per sequence (rows * CU)
  int total;  // statistics units per counter: B * A
};

struct SampleArgs {
  const void* target;
  const void* draft;
  const int32_t* tokens;
  int B, K, V;
  int R;   // rows per sequence = 2K+1
  int SL;  // statistics slice length in elements (a whole number of load batches)
  int CS;  // statistics slices per row = ceil(V / SL)
  int TL;  // tail slice length in elements (a whole number of warp steps)
  int TC;  // tail slices per row = ceil(V / TL)
  int P;   // pieces (warp steps) per tail slice
  int F;   // statistics slices in all: B * R * CS
  int FP;  // slices of positions 0..K-1 (row pairs), which come first: K * B * 2 * CS
  int NA;  // slices of the front positions (spread through the stream)
  int FA, FQ;  // FA front slices in every block of FQ claims
  FastDiv div_fq;
  int claim_tail;  // within this many slices of the end, claims are not made ahead
  int l2_keep;     // rows of positions < l2_keep are prefetched into L2 with evict_last
  int early_exit;  // read only the rows the result depends on (positions 0..n, row K if n = K)
  int TTo;         // owned tail items (the first TTo); the rest are claimed by free warps
  FastDiv div_pos, div_pair, div_cs, div_tc;  // division by B * 2 * CS, 2 * CS, CS and TC
  float c_hi, c_lo;  // log2(e)/temperature as a float pair
  double c64;        // the same in double
  double inv_tau;    // 1 / temperature
  uint64_t seed;
  int32_t* out_tokens;
  int32_t* out_n;
  float* out_row_stats;  // optional [B, R, 2]: max(z)/tau, sum exp(z/tau - max)
  float* out_pq;         // optional [B, K, 2]: p_i(x_i), q_i(x_i)
  float* out_resid;      // optional [B]: mass of the replacement distribution
  float* out_entropy;    // optional [B, R]: entropy (nats) of each row's softmax
  // optional suggested next draft length: K moved one step up when the mean
  // entropy of target rows 0..n is below h_lo, down when above h_hi, then
  // clamped to [k_min, k_max]; -1 for a bad sequence
  int32_t* out_khint;    // [B]
  float* out_hmean;      // optional [B]: that mean entropy (nats)
  double h_lo, h_hi;
  int k_min, k_max;
  // workspace, filled with all-ones bytes before the launch: the counters and
  // tickets (counter, unitticket, seqticket, posticket, tailticket, qcount,
  // dclaim, ctaticket) then start at -1, the resolution words at the empty
  // set (stored complemented), and the result slots (part, rowstat, zx,
  // verdict, result, tailsum, queue, pieces) hold the kMarker "not yet
  // written" pattern.
  unsigned long long* counter;  // kSlices claim counters, kCounterStride apart
  int* unitticket;  // [B, K+1] (kTicketStride apart) finished slices of a position unit
  int* seqticket;   // [B] commit count: finished units (+ 0x10000 per unit with bad data) and the result
  int* posticket;   // [B] resolved positions (K > 31 only)
  unsigned long long* resword;  // [B] resolved / rejected positions, complemented (K <= 31)
  int* verdict;     // [B, K+1] accept / reject / bad of each position
  uint4* result;    // [B] (n, token, residual mass bits, 0) for the commit
  int* decided;     // [B] n once the sequence is decided (early exit), kMarker before
  int* tailticket;  // [B] finished tail slices
  int* qcount;      // decision-queue positions taken so far
  int* dclaim;      // tail items of the last queue positions claimed so far
  int* ctaticket;   // CTAs started so far (each CTA's first claims follow its ticket)
  float2* part;     // [B, R, CS] per-slice (m, s)
  float2* rowstat;  // [B, R] merged (m, s) of each row
  float* zx;        // [B, R] logit at the drafted token, written by the slice holding it
  float* part_t;    // [B, R, CS] per-slice entropy accumulator (with out_entropy or out_khint)
  float* hrow;      // [B, K+1] entropy of each target row (only with out_khint)
  float* tailsum;   // [B, TC] per tail-slice mass
  SeqInfo* queue;   // [B] decisions in the order they were made
  float* pieces;    // [B, TC, P] per-piece mass
  unsigned* status;
};

struct GreedyArgs {
  const void* target;
  const int32_t* tokens;   // chain: [B, K]; tree: [B, N]
  const int32_t* parents;  // tree only: [B, N]
  int B, K, V;             // chain: K drafts; tree: K = N nodes
  int R;                   // rows per sequence: K+1 (chain) or N+1 (tree)
  int SL, CS, CU;          // slice length, slices per row, units per row
  UnitMap map;
  int32_t* out_tokens;      // chain [B, K+1]; tree out_path [B, N+1]
  int32_t* out_n;           // chain [B];     tree out_len  [B]
  uint32_t* out_mask;       // tree [B, N, ceil(N/32)]
  int32_t* out_row_argmax;  // optional [B, R]
  // workspace, filled with all-ones bytes before the launch: counter,
  // rowticket and seqticket start at -1; part and g hold the "not yet
  // written" marker.
  unsigned long long* counter;  // kSlices claim counters, kCounterStride apart
  int* rowticket;  // [B, R] (kTicketStride apart) finished slices of a row
  int* seqticket;  // [B] finished rows of a sequence
  uint2* part;     // [B, R, CU * kSlices] slice (max bits, argmax | NaN-seen << 31)
  int* g;          // [B, R] row argmax, -2 for an unusable row
  int* depth;     // [B, R] tree finisher scratch
  int* acc;       // [B, R] tree finisher scratch
  // early exit (chain, 1 <= K <= 31): rows streamed by position; the row
  // finisher resolves its position and the resolution that decides the
  // sequence writes its outputs; rows after a decided sequence's n are skipped
  int early_exit;
  unsigned long long* resword;  // [B] resolution words, stored complemented (all-ones: empty);
                                // tree: bit r set when row r is done
  int* decided;                 // [B] n once decided (marker before); tree: the output writer's claim
  int* verdict;                 // [B, R] position verdicts (marker before)
  unsigned* rejc;               // [B] tree: complement of the rejected-node mask (all-ones: none)
  unsigned* status;
};
constexpr int kTreeEarlyExitMaxN = 32;  // tree early exit: one warp holds a sequence's nodes

// Workspace layout of each kernel: `total` bytes; [0, zero_bytes) must be
// zero-filled (neither kernel uses one) and [marker_off, marker_off +
// marker_bytes) filled with 0xff
// bytes before every launch.
struct WsLayout {
  size_t total, zero_bytes, marker_off, marker_bytes;
};
WsLayout sample_workspace(int B, int K, int CS, int TC, int P, bool ent);
WsLayout greedy_workspace(int B, int R, int CU);

// Stochastic tree verification (tree_sample_kernel.cu).  Rows per sequence:
// target rows 0..N (row 0 the root, row i+1 node i), then draft rows 0..N.
struct TreeSampleArgs {
  const void* target;
  const void* draft;
  const int32_t* tokens;   // [B, N]
  const int32_t* parents;  // [B, N]
  int B, N, V;
  int RR;   // rows per sequence, both models: 2 (N + 1)
  int SL;   // statistics slice length in elements
  int CS;   // statistics slices per row
  long long F;  // statistics slices in all: B * RR * CS
  int C;        // CTAs (one cluster) per sequence in the walk: 1, 2, 4, 8 or 16
  int chunk;    // elements per warp of the cluster in the walk passes (whole warp steps)
  float c_hi, c_lo;  // log2(e) / temperature as a float pair
  double c64;
  uint64_t seed;
  int32_t* out_path;  // [B, N+1]
  int32_t* out_len;   // [B]
  // workspace, filled with all-ones bytes: row tickets start at -1, part and
  // rowstat hold the "not yet written" marker
  int* rowticket;    // [B * RR] (kTicketStride apart)
  float2* part;      // [B * RR, CS] per-slice (m, s)
  float2* rowstat;   // [B * RR] merged (m, s)
  unsigned* status;
};
constexpr int kWalkThreads = 512;  // threads per walk CTA (a cluster of C per sequence)
WsLayout tree_sample_workspace(int B, int RR, int CS);
void tree_sample_bind_workspace(TreeSampleArgs& a, void* ws);
cudaError_t launch_tree_sample(const TreeSampleArgs& a, bool bf16, bool vec, int stats_grid, cudaStream_t s);
int tree_stats_blocks_per_sm(bool bf16, bool vec);
int tree_walk_clusters(bool bf16, bool vec, int C);


// Bind workspace pointers into the argument blocks.
void sample_bind_workspace(SampleArgs& a, void* ws);
void greedy_bind_workspace(GreedyArgs& a, void* ws);

// Launchers: `grid` CTAs of kThreads threads, persistent.  `vec` selects the
// 16-byte vector path (rows 16-byte aligned) or the scalar path.
cudaError_t launch_sample(const SampleArgs& a, bool bf16, bool vec, int grid, cudaStream_t s);
cudaError_t launch_greedy(const GreedyArgs& a, bool bf16, bool vec, int grid, cudaStream_t s);
cudaError_t launch_tree(const GreedyArgs& a, bool bf16, bool vec, int grid, cudaStream_t s);

// N-gram (prompt-lookup) drafting (ngram_kernel.cu).  A persistent scan grid
// claims (sequence, chunk) entries from a counter and stores each chunk's best
// end in the entry's slot; a second launch (programmatic stream serialisation)
// reduces each sequence's slots and writes the drafts.
// Workspace (zeroed): slot [B * chunks], counter.
constexpr int kNgramMaxN = 32;  // longest n-gram matched
struct NgramArgs {
  const int32_t* tokens;   // [B, stride] histories
  long long stride;        // row stride and the largest valid length
  const int32_t* lengths;  // [B]
  int B, n_min, n_max, K;
  int chunks;              // entries per sequence: ceil(stride / chunk)
  int vec;                 // every row starts on a 16-byte boundary (bulk copies)
  int32_t* drafts;         // [B, K]
  int32_t* n_drafts;       // [B]
  int32_t* match_len;      // [B]
  unsigned long long* slot;  // [B, chunks] best (m << 32) | e of each chunk, 0 = none
  int* counter;              // entries claimed so far
  unsigned* status;
};
int ngram_chunk();
int ngram_blocks_per_sm();  // scan CTAs resident per SM (0: the launch cannot be configured)
cudaError_t ngram_set_spin_limit(unsigned n);
cudaError_t launch_ngram(const NgramArgs& a, int grid, cudaStream_t s);

// Acceptance statistics: zeroes hist[0..K+1], counts n_accepted into it and,
// when alpha / mean_tokens are given, derives them (acceptance_kernel.cu).
cudaError_t launch_acceptance(const int32_t* n, int B, int K, unsigned long long* hist, double* alpha,
                              double* mean_tokens, int sms, cudaStream_t s);

// Resident CTAs per SM for each kernel (occupancy calculator).
int sample_blocks_per_sm(bool bf16, bool vec);
int greedy_blocks_per_sm(bool bf16, bool vec);
int tree_blocks_per_sm(bool bf16, bool vec);

// Elements per warp step (32 lanes x one vector) and per load batch.
inline int step_elems(bool bf16, bool vec) { return 32 * (vec ? (bf16 ? 8 : 4) : 1); }
inline int batch_elems(bool bf16, bool vec) { return step_elems(bf16, vec) * kUnroll; }

// Bytes of the claim-counter block at the start of each workspace.
constexpr size_t kCounterBytes = (size_t)kSlices * kCounterStride * 8;

// The bit pattern of a slot that has not been written yet.
constexpr unsigned kMarker = 0xffffffffu;

// The bounded-wait limit of each kernel translation unit on the current device
// (spec_test_spin_limit).
cudaError_t sample_set_spin_limit(unsigned n);
// Runs every bounded-wait helper on an unwritten and a written slot (test
// hook; synchronous).  flags_host[0]: bits of the helpers that ran out on the
// unwritten slot; flags_host[1]: bits of those that flagged a written one.
cudaError_t sample_wait_probe(uint32_t* flags_host);
cudaError_t greedy_set_spin_limit(unsigned n);
cudaError_t tree_sample_set_spin_limit(unsigned n);

}  // namespace sv
