// api.cu -- the C ABI of libspecverify.so (declared in include/specverify.h).
//
// Host-side argument checks, per-device state (SM count, occupancy, the
// stream-ordered scratch pool, the device status word), the choice of chunk
// length and grid, and the launches.  No verify arithmetic happens here.
#include "specverify.h"
#include "sv_kernels.h"

#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <stdlib.h>

#include <atomic>
#include <mutex>

// Sticky per-device status word (SPEC_FLAG_* bits), read and cleared by
// spec_get_status.
__device__ unsigned g_spec_status;

// Scratch of spec_verify_bf16_static_scratch.  Some callers cannot let the
// library allocate device memory on their behalf:
//   * a serving process that reserved nearly all of HBM up front (for its KV
//     cache) leaves the library's pool no room to grow, and a failed pool
//     allocation in the middle of a decode step is not recoverable there;
//   * latency-critical loops must not enter the allocator, whose locks and
//     pool growth add jitter to an otherwise fixed-cost step;
//   * devices or virtualised set-ups without stream-ordered memory pools
//     (cudaDevAttrMemoryPoolsSupported == 0) cannot serve
//     cudaMallocFromPoolAsync at all.
// For them the library carries one fixed scratch buffer per device in its
// own image: this file-scope array, created when the module is loaded.  Its
// address is looked up once per device with cudaGetSymbolAddress.
constexpr size_t kStaticScratchBytes = SPEC_STATIC_SCRATCH_BYTES;
__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace {

struct DeviceState {
  bool init = false;
  int sms = 0;
  cudaMemPool_t pool = nullptr;  // created by the first call that allocates
  void* static_scratch = nullptr;  // looked up by the first static-scratch call
  cudaStream_t side = nullptr;     // scratch is allocated and filled here, off the caller's stream
  cudaEvent_t side_done = nullptr;
  unsigned* status = nullptr;
  int occ_sample[2][2] = {{0, 0}, {0, 0}};  // [bf16][vec]
  int occ_greedy[2][2] = {{0, 0}, {0, 0}};
  int occ_tree[2][2] = {{0, 0}, {0, 0}};
  int occ_tree_stats[2][2] = {{0, 0}, {0, 0}};
  int walk_clusters[2][2][5] = {};  // [bf16][vec][log2 C]: walk clusters resident at once
  int occ_ngram = 0;                // n-gram scan CTAs per SM
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
thread_local char g_cuda_msg[256] = "no CUDA error recorded";

int cuda_fail(cudaError_t e, const char* where) {
  snprintf(g_cuda_msg, sizeof g_cuda_msg, "%s: %s (%s)", where, cudaGetErrorString(e),
           cudaGetErrorName(e));
  return SPEC_ERR_CUDA;
}

int get_device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice, "device index");
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.init) {
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    e = cudaGetSymbolAddress((void**)&d.status, g_spec_status);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
    for (int bf = 0; bf < 2; ++bf)
      for (int v = 0; v < 2; ++v) {
        d.occ_sample[bf][v] = sv::sample_blocks_per_sm(bf, v);
        d.occ_greedy[bf][v] = sv::greedy_blocks_per_sm(bf, v);
        d.occ_tree[bf][v] = sv::tree_blocks_per_sm(bf, v);
        d.occ_tree_stats[bf][v] = sv::tree_stats_blocks_per_sm(bf, v);
        for (int c = 0; c < 5; ++c) d.walk_clusters[bf][v][c] = sv::tree_walk_clusters(bf, v, 1 << c);
      }
    d.occ_ngram = sv::ngram_blocks_per_sm();
    d.init = true;
  }
  *out = &d;
  return SPEC_OK;
}

// The library's stream-ordered pool on the current device, created on first
// use.
int ensure_pool(DeviceState* d) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (d->pool) return SPEC_OK;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  cudaMemPoolProps props;
  memset(&props, 0, sizeof props);
  props.allocType = cudaMemAllocationTypePinned;
  props.location.type = cudaMemLocationTypeDevice;
  props.location.id = dev;
  cudaMemPool_t pool = nullptr;
  e = cudaMemPoolCreate(&pool, &props);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemPoolCreate");
  uint64_t keep = UINT64_MAX;  // keep freed scratch in the pool between calls
  e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
  // an allocation never waits for the stream that freed a block: the pool
  // hands out another block instead, so a call's scratch can be prepared
  // while the previous call's kernel still runs
  int no_wait = 0;
  if (e == cudaSuccess) e = cudaMemPoolSetAttribute(pool, cudaMemPoolReuseAllowInternalDependencies, &no_wait);
  if (e != cudaSuccess) {
    cudaMemPoolDestroy(pool);
    return cuda_fail(e, "cudaMemPoolSetAttribute");
  }
  d->pool = pool;
  return SPEC_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Launch parameters of the persistent kernels, measured on GB300 with the c3
// workload (the measurements are in the design notes):
constexpr int kSliceBytes = 16384;        // statistics slice of the sampling kernel (full read)
constexpr int kSliceBytesEarlyExit = 12288;  // ... with early exit, and of the stochastic tree's statistics
constexpr int kSmallSliceBytes = 8192;    // ... for a batch with fewer than ~6 slices per warp
constexpr int kTinySliceBytes = 4096;     // ... for one whose 8 KB slices would leave warps without one
constexpr int kTailBytes = 6144;          // bytes of each of the two rows in a tail item
constexpr int kSmallTailBytes = 2048;     // ... for a small batch
constexpr int kArgmaxSliceBytes = 8192;   // slice of the greedy and tree kernels
constexpr int kClaimTail = 1;             // final statistics slices not claimed ahead
constexpr int kFrontPositions = 1;        // draft positions whose row pairs are spread through the stream
constexpr int kFrontSpanPercent = 60;     // ... over this percent of it (position 0 decides most sequences)
constexpr int kL2KeepPositions = 1;       // positions whose rows are prefetched into L2 with evict_last
constexpr int kLateTailPercent = 6;       // latest decisions whose tail items free warps claim
constexpr int kLateTailPercentEarlyExit = 25;

// Slice length: a whole number of warp load batches (32 lanes x kUnroll
// vectors) covering about `bytes`; a row shorter than one slice is one slice.
void choose_slices(int V, int vec_elems, size_t esz, int bytes, int* SL, int* CS, int* CU) {
  const long long batch = 32LL * vec_elems * sv::kUnroll;
  long long k = ((long long)bytes / (long long)esz + batch - 1) / batch;
  if (k < 1) k = 1;
  long long sl = k * batch;
  if (sl >= V) sl = ((long long)V + 7) / 8 * 8;
  *SL = (int)sl;
  *CS = (int)((V + sl - 1) / sl);
  *CU = (*CS + sv::kSlices - 1) / sv::kSlices;
}

// Each counter's units are shared by one warp of every CTA, so a grid of
// `total_units` CTAs already gives every unit its own warp.
int grid_for(int total_units, int capacity) {
  if (total_units < 1) total_units = 1;
  return total_units < capacity ? total_units : capacity;
}

// Element offsets are 64-bit; unit indices and per-row positions are 32-bit.
bool sizes_ok(int B, int rows, int V) {
  const double total = (double)B * (double)rows * (double)V;
  const double units = (double)B * (double)(rows + 1) * ((double)V / 1024.0 + 1.0);
  return V <= 0x7fff0000 && total < 4.0e18 && units < 2.0e9;
}

// Scratch from the library's pool with the zero region and the "not yet
// written" marker region initialised.  Outside stream capture the allocation
// and fills run on the device's side stream and the caller's stream waits for
// them through an event: they do not depend on the caller's earlier work, so
// they can run while the previous kernel drains, and the caller's stream sees
// one launch per call instead of a fill, a gap and a launch.  (The caller's
// stream returns the scratch with cudaFreeAsync after the kernel.)
// Scratch allocations still to be failed on purpose (spec_test_fail_allocations).
std::atomic<int> g_fail_allocs{0};

int run_scratch(DeviceState* d, const sv::WsLayout& l, cudaStream_t stream, void** ws) {
  const int rc = ensure_pool(d);
  if (rc) return rc;
  for (int k = g_fail_allocs.load(); k > 0; k = g_fail_allocs.load())
    if (g_fail_allocs.compare_exchange_weak(k, k - 1))
      return cuda_fail(cudaErrorMemoryAllocation, "cudaMallocFromPoolAsync (failed on request)");
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  if (cap == cudaStreamCaptureStatusNone) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!d->side) {
      e = cudaStreamCreateWithFlags(&d->side, cudaStreamNonBlocking);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d->side_done, cudaEventDisableTiming);
      if (e != cudaSuccess) return cuda_fail(e, "side stream");
    }
    e = cudaMallocFromPoolAsync(ws, l.total, d->pool, d->side);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMallocFromPoolAsync");
    if (l.zero_bytes) e = cudaMemsetAsync(*ws, 0, l.zero_bytes, d->side);
    if (e == cudaSuccess && l.marker_bytes)
      e = cudaMemsetAsync((char*)*ws + l.marker_off, 0xff, l.marker_bytes, d->side);
    if (e == cudaSuccess) e = cudaEventRecord(d->side_done, d->side);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, d->side_done, 0);
    if (e != cudaSuccess) {
      cudaFreeAsync(*ws, d->side);
      return cuda_fail(e, "scratch preparation");
    }
    return SPEC_OK;
  }
  e = cudaMallocFromPoolAsync(ws, l.total, d->pool, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMallocFromPoolAsync");
  if (l.zero_bytes) e = cudaMemsetAsync(*ws, 0, l.zero_bytes, stream);
  if (e == cudaSuccess && l.marker_bytes)
    e = cudaMemsetAsync((char*)*ws + l.marker_off, 0xff, l.marker_bytes, stream);
  if (e != cudaSuccess) {
    cudaFreeAsync(*ws, stream);
    return cuda_fail(e, "cudaMemsetAsync");
  }
  return SPEC_OK;
}

// The static scratch buffer, with the same two regions initialised on the
// stream (cudaMemsetAsync only; nothing is allocated).  A layout larger than
// the buffer is refused before anything is launched.
int static_scratch(DeviceState* d, const sv::WsLayout& l, cudaStream_t stream, void** ws) {
  if (l.total > kStaticScratchBytes) return SPEC_ERR_SCRATCH;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!d->static_scratch) {
      const cudaError_t e = cudaGetSymbolAddress(&d->static_scratch, g_static_scratch);
      if (e != cudaSuccess) {
        d->static_scratch = nullptr;
        return cuda_fail(e, "cudaGetSymbolAddress");
      }
    }
  }
  *ws = d->static_scratch;
  cudaError_t e = cudaSuccess;
  if (l.zero_bytes) e = cudaMemsetAsync(*ws, 0, l.zero_bytes, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync((char*)*ws + l.marker_off, 0xff, l.marker_bytes, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  return SPEC_OK;
}

// Scratch for one call: stream-ordered from the pool (returned after the
// launch), or the static buffer.
int get_scratch(DeviceState* d, bool use_static, const sv::WsLayout& l, cudaStream_t stream,
                void** ws) {
  return use_static ? static_scratch(d, l, stream, ws) : run_scratch(d, l, stream, ws);
}
cudaError_t put_scratch(bool use_static, void* ws, cudaStream_t stream) {
  return use_static ? cudaSuccess : cudaFreeAsync(ws, stream);
}

// Greedy chain (tree == false) or tree (tree == true) verification.
int argmax_impl(bool tree, bool bf16, const void* target, const int32_t* tokens,
                const int32_t* parents, int B, int K, int V, int32_t* out_tokens, int32_t* out_n,
                uint32_t* out_mask, int32_t* out_row_argmax, cudaStream_t stream,
                bool use_static = false, bool early_exit = false) {
  DeviceState* d = nullptr;
  int rc = get_device_state(&d);
  if (rc) return rc;
  const size_t esz = bf16 ? 2 : 4;
  const bool vec = aligned16(target) && ((size_t)V * esz) % 16 == 0;
  const int capacity = d->sms * (tree ? d->occ_tree[bf16][vec] : d->occ_greedy[bf16][vec]);
  sv::GreedyArgs a;
  memset(&a, 0, sizeof a);
  a.target = target;
  a.tokens = tokens;
  a.parents = parents;
  a.B = B;
  a.K = K;
  a.V = V;
  a.R = K + 1;
  choose_slices(V, vec ? (bf16 ? 8 : 4) : 1, esz, kArgmaxSliceBytes, &a.SL, &a.CS, &a.CU);
  a.map.A = a.R * a.CU;
  if ((long long)B * a.map.A >= INT_MAX) return SPEC_ERR_SHAPE;  // slices are indexed with int
  a.map.total = B * a.map.A;
  a.out_tokens = out_tokens;
  a.out_n = out_n;
  a.out_mask = out_mask;
  a.out_row_argmax = out_row_argmax;
  // early exit: the chain's resolution word holds positions 0..31; a tree's
  // nodes are resolved by one warp (N <= 32)
  a.early_exit = (early_exit && !out_row_argmax &&
                  (tree ? (K >= 1 && K <= sv::kTreeEarlyExitMaxN) : (K >= 1 && K <= sv::kMaskMaxK)))
                     ? 1 : 0;
  a.status = d->status;
  void* ws = nullptr;
  rc = get_scratch(d, use_static, sv::greedy_workspace(B, a.R, a.CU), stream, &ws);
  if (rc) return rc;
  sv::greedy_bind_workspace(a, ws);
  const int grid = grid_for(a.map.total, capacity);
  cudaError_t e = tree ? sv::launch_tree(a, bf16, vec, grid, stream)
                       : sv::launch_greedy(a, bf16, vec, grid, stream);
  cudaError_t e2 = put_scratch(use_static, ws, stream);
  if (e != cudaSuccess) return cuda_fail(e, tree ? "tree verify launch" : "greedy verify launch");
  if (e2 != cudaSuccess) return cuda_fail(e2, "cudaFreeAsync");
  return SPEC_OK;
}

int greedy_impl(bool bf16, const void* target, const int32_t* tokens, int B, int K, int V,
                int32_t* out_tokens, int32_t* out_n, int32_t* out_row_argmax, cudaStream_t stream,
                bool use_static = false, bool early_exit = false) {
  if (!target || !out_tokens || !out_n || (K > 0 && !tokens)) return SPEC_ERR_NULL;
  if (B < 0 || K < 0 || K > sv::kMaxK || V < 1 || !sizes_ok(B, K + 1, V)) return SPEC_ERR_SHAPE;
  if (B == 0) return SPEC_OK;
  return argmax_impl(false, bf16, target, tokens, nullptr, B, K, V, out_tokens, out_n, nullptr,
                     out_row_argmax, stream, use_static, early_exit);
}

// The draft-length suggestion's parameters and outputs (spec_verify_khint_*).
struct KHint {
  double h_lo, h_hi;
  int k_min, k_max;
  int32_t* out_k;
  float* out_hmean;
};

int verify_impl(bool bf16, const void* target, const void* draft, const int32_t* tokens, int B,
                int K, int V, float temperature, uint64_t seed, int32_t* out_tokens, int32_t* out_n,
                float* out_row_stats, float* out_pq, float* out_resid, float* out_entropy,
                cudaStream_t stream,
                bool use_static = false, bool early_exit = false, const KHint* kh = nullptr) {
  if (!(temperature >= 0.f) || (temperature > 0.f && temperature < 1e-30f))
    return SPEC_ERR_TEMPERATURE;
  if (temperature == 0.f)
    return greedy_impl(bf16, target, tokens, B, K, V, out_tokens, out_n, nullptr, stream,
                       use_static, early_exit);
  if (!target || !out_tokens || !out_n || (K > 0 && (!tokens || !draft))) return SPEC_ERR_NULL;
  if (B < 0 || K < 0 || K > sv::kMaxK || V < 1 || !sizes_ok(B, 2 * K + 1, V)) return SPEC_ERR_SHAPE;
  if (B == 0) return SPEC_OK;
  DeviceState* d = nullptr;
  int rc = get_device_state(&d);
  if (rc) return rc;
  const size_t esz = bf16 ? 2 : 4;
  const bool vec = aligned16(target) && (K == 0 || aligned16(draft)) && ((size_t)V * esz) % 16 == 0;
  const int capacity = d->sms * d->occ_sample[bf16][vec];
  sv::SampleArgs a;
  memset(&a, 0, sizeof a);
  a.target = target;
  a.draft = draft;
  a.tokens = tokens;
  a.B = B;
  a.K = K;
  a.V = V;
  a.R = 2 * K + 1;
  const int vec_elems = vec ? (bf16 ? 8 : 4) : 1;
  int CU = 0;
  // A batch too small to give every warp of the grid about six 12 KB
  // statistics slices streams 8 KB slices and lets free warps take all of its
  // tail items (c2: 68 us instead of 75 us per call).  Larger batches stream
  // 16 KB slices, or 12 KB with early exit (c3: 252 instead of 256 us with
  // the full read; the early exit is 4 us slower with 16 KB).
  choose_slices(V, vec_elems, esz, kSliceBytesEarlyExit, &a.SL, &a.CS, &CU);
  const bool small = (long long)B * a.R * a.CS < 6LL * capacity * sv::kWarps;
  if (small) {
    choose_slices(V, vec_elems, esz, kSmallSliceBytes, &a.SL, &a.CS, &CU);
    // fewer 8 KB slices than warps (c1: 144 of 4864): 4 KB slices, each in
    // fewer dependent load rounds (c1 -0.7 us; 1 KB slices were slower)
    if ((long long)B * a.R * a.CS < (long long)capacity * sv::kWarps)
      choose_slices(V, vec_elems, esz, kTinySliceBytes, &a.SL, &a.CS, &CU);
  } else if (!early_exit)
    choose_slices(V, vec_elems, esz, kSliceBytes, &a.SL, &a.CS, &CU);
  // tail slices: whole warp steps, kSmallTailBytes per row for a small batch
  // (c2: 2 KB, -0.7 us against 4 KB), else kTailBytes (c3: 6 KB, against 8
  // or 12 KB)
  const int step = 32 * vec_elems;
  const long long tl_elems = (long long)(small ? kSmallTailBytes : kTailBytes) / (long long)esz;
  a.P = (int)((tl_elems + step - 1) / step);
  if (a.P < 1) a.P = 1;
  a.TL = a.P * step;
  a.TC = (int)(((long long)V + a.TL - 1) / a.TL);
  // the kernel indexes slices, tail items and pieces with int: sizes_ok
  // assumes at least 1024 elements per slice, checked here for the slices
  // actually chosen
  if ((long long)B * a.R * a.CS >= INT_MAX || (long long)B * a.TC * a.P >= INT_MAX) return SPEC_ERR_SHAPE;
  a.F = B * a.R * a.CS;
  a.FP = K * B * 2 * a.CS;
  a.div_pos = sv::make_fastdiv((uint32_t)(B * 2 * a.CS));
  a.div_pair = sv::make_fastdiv((uint32_t)(2 * a.CS));
  a.div_cs = sv::make_fastdiv((uint32_t)a.CS);
  a.div_tc = sv::make_fastdiv((uint32_t)a.TC);
  // Stream order: the front positions' slices are spread over the first
  // `front_span` percent of the stream (100 or more, or a span shorter than
  // their own share: position-major order).
  {
    // early exit keeps plain position-major order: a sequence's later rows
    // then come after its decision, so they can be skipped
    // (and a small batch, whose stream is short: its position-0 decisions
    // come earlier in plain position-major order, c2 -1 us)
    const int fp = (early_exit || small) ? 0 : (kFrontPositions > K ? K : kFrontPositions);
    a.NA = fp * B * 2 * a.CS;
    a.FQ = 64;
    const double span = (double)kFrontSpanPercent / 100.0 * (double)a.F;
    int fa = a.FQ;
    if (a.NA > 0 && span > (double)a.NA) fa = (int)ceil((double)a.FQ * (double)a.NA / span);
    a.FA = fa < 1 ? 1 : (fa > a.FQ ? a.FQ : fa);
    // every front slice must land inside the stream: the claim index of the
    // last one, ((NA-1) / FA) * FQ + (NA-1) % FA, below F (FA = FQ always is)
    while (a.NA > 0 && a.FA < a.FQ &&
           (long long)((a.NA - 1) / a.FA) * a.FQ + (a.NA - 1) % a.FA >= (long long)a.F)
      ++a.FA;
    a.div_fq = sv::make_fastdiv((uint32_t)a.FQ);
  }
  const int grid = grid_for((a.F + sv::kSlices - 1) / sv::kSlices, capacity);
  a.claim_tail = kClaimTail;
  a.l2_keep = kL2KeepPositions;
  a.early_exit = early_exit ? 1 : 0;
  // the tail items of the last late_tails percent of queue positions (the
  // latest decisions) go to whichever warps are free
  // (measured on c3: 6 % with the full read, 25 % with early exit, where
  // most of the grid is free once the first position has been streamed)
  {
    const int want = small ? 100 : (early_exit ? kLateTailPercentEarlyExit : kLateTailPercent);
    const int pct = want > 100 ? 100 : want;
    int late = (int)(((long long)B * pct + 99) / 100);
    if (late > B) late = B;
    a.TTo = (B - late) * a.TC;
  }
  const double c = 1.4426950408889634074 / (double)temperature;  // log2(e) / tau
  a.c64 = c;
  a.c_hi = (float)c;
  a.c_lo = (float)(c - (double)a.c_hi);
  a.inv_tau = 1.0 / (double)temperature;
  a.seed = seed;
  a.out_tokens = out_tokens;
  a.out_n = out_n;
  a.out_row_stats = out_row_stats;
  a.out_pq = out_pq;
  a.out_resid = out_resid;
  a.out_entropy = out_entropy;
  if (kh) {
    a.out_khint = kh->out_k;
    a.out_hmean = kh->out_hmean;
    a.h_lo = kh->h_lo;
    a.h_hi = kh->h_hi;
    a.k_min = kh->k_min;
    a.k_max = kh->k_max;
  }
  a.status = d->status;
  void* ws = nullptr;
  rc = get_scratch(d, use_static, sv::sample_workspace(B, K, a.CS, a.TC, a.P, out_entropy != nullptr || kh != nullptr),
                   stream, &ws);
  if (rc) return rc;
  sv::sample_bind_workspace(a, ws);
  cudaError_t e = sv::launch_sample(a, bf16, vec, grid, stream);
  cudaError_t e2 = put_scratch(use_static, ws, stream);
  if (e != cudaSuccess) return cuda_fail(e, "sampling verify launch");
  if (e2 != cudaSuccess) return cuda_fail(e2, "cudaFreeAsync");
  return SPEC_OK;
}

int tree_impl(bool bf16, const void* target, const int32_t* tree_tokens, const int32_t* parents,
              int B, int N, int V, int32_t* out_path, int32_t* out_len, uint32_t* out_mask,
              cudaStream_t stream, bool early_exit = false) {
  if (!target || !out_path || !out_len || (N > 0 && (!tree_tokens || !parents || !out_mask)))
    return SPEC_ERR_NULL;
  if (B < 0 || N < 0 || N > sv::kMaxTreeNodes || V < 1 || !sizes_ok(B, N + 1, V))
    return SPEC_ERR_SHAPE;
  if (B == 0) return SPEC_OK;
  return argmax_impl(true, bf16, target, tree_tokens, parents, B, N, V, out_path, out_len, out_mask,
                     nullptr, stream, false, early_exit);
}

// Stochastic tree verification: row statistics of all 2 (N + 1) rows of every
// sequence, then one CTA per sequence walks its tree.
int tree_sample_impl(bool bf16, const void* target, const void* draft, const int32_t* tree_tokens,
                     const int32_t* parents, int B, int N, int V, float temperature, uint64_t seed,
                     int32_t* out_path, int32_t* out_len, cudaStream_t stream) {
  if (!(temperature >= 1e-30f)) return SPEC_ERR_TEMPERATURE;
  if (!target || !draft || !out_path || !out_len || (N > 0 && (!tree_tokens || !parents)))
    return SPEC_ERR_NULL;
  if (B < 0 || N < 0 || N > sv::kMaxTreeNodes || V < 1 || !sizes_ok(B, 2 * (N + 1), V))
    return SPEC_ERR_SHAPE;
  if (B == 0) return SPEC_OK;
  DeviceState* d = nullptr;
  int rc = get_device_state(&d);
  if (rc) return rc;
  const size_t esz = bf16 ? 2 : 4;
  const bool vec = aligned16(target) && aligned16(draft) && ((size_t)V * esz) % 16 == 0;
  const int vec_elems = vec ? (bf16 ? 8 : 4) : 1;
  sv::TreeSampleArgs a;
  memset(&a, 0, sizeof a);
  a.target = target;
  a.draft = draft;
  a.tokens = tree_tokens;
  a.parents = parents;
  a.B = B;
  a.N = N;
  a.V = V;
  a.RR = 2 * (N + 1);
  int CU = 0;
  choose_slices(V, vec_elems, esz, kSliceBytesEarlyExit, &a.SL, &a.CS, &CU);
  a.F = (long long)B * a.RR * a.CS;
  // walk: the widest cluster (16, 8, 4, 2 CTAs) for which every sequence's
  // cluster is resident at once, else one CTA per sequence; each pass gives
  // every warp of the cluster one contiguous run of whole warp steps
  a.C = 1;
  for (int c = 4; c >= 1; --c)
    if (B <= d->walk_clusters[bf16][vec][c]) {
      a.C = 1 << c;
      break;
    }
  const long long step = 32LL * vec_elems;
  const long long warps = (long long)a.C * (sv::kWalkThreads / 32);
  const long long per_warp = ((long long)V + warps - 1) / warps;
  a.chunk = (int)((per_warp + step - 1) / step * step);
  const double c = 1.4426950408889634074 / (double)temperature;  // log2(e) / tau
  a.c64 = c;
  a.c_hi = (float)c;
  a.c_lo = (float)(c - (double)a.c_hi);
  a.seed = seed;
  a.out_path = out_path;
  a.out_len = out_len;
  a.status = d->status;
  void* ws = nullptr;
  rc = get_scratch(d, false, sv::tree_sample_workspace(B, a.RR, a.CS), stream, &ws);
  if (rc) return rc;
  sv::tree_sample_bind_workspace(a, ws);
  const long long capacity = (long long)d->sms * d->occ_tree_stats[bf16][vec];
  const long long want = (a.F + sv::kWarps - 1) / sv::kWarps;  // one slice per warp
  const int stats_grid = (int)(want < capacity ? want : capacity);
  cudaError_t e = sv::launch_tree_sample(a, bf16, vec, stats_grid, stream);
  cudaError_t e2 = put_scratch(false, ws, stream);
  if (e != cudaSuccess) return cuda_fail(e, "tree sampling verify launch");
  if (e2 != cudaSuccess) return cuda_fail(e2, "cudaFreeAsync");
  return SPEC_OK;
}

}  // namespace

extern "C" {

int spec_verify_f32(const float* target_logits, const float* draft_logits,
                    const int32_t* draft_tokens, int B, int K, int V, float temperature,
                    uint64_t seed, int32_t* out_tokens, int32_t* out_n_accepted,
                    cudaStream_t stream) {
  return verify_impl(false, target_logits, draft_logits, draft_tokens, B, K, V, temperature, seed,
                     out_tokens, out_n_accepted, nullptr, nullptr, nullptr, nullptr, stream);
}

int spec_verify_bf16(const uint16_t* target_logits, const uint16_t* draft_logits,
                     const int32_t* draft_tokens, int B, int K, int V, float temperature,
                     uint64_t seed, int32_t* out_tokens, int32_t* out_n_accepted,
                     cudaStream_t stream) {
  return verify_impl(true, target_logits, draft_logits, draft_tokens, B, K, V, temperature, seed,
                     out_tokens, out_n_accepted, nullptr, nullptr, nullptr, nullptr, stream);
}

int spec_verify_early_exit_f32(const float* target_logits, const float* draft_logits,
                               const int32_t* draft_tokens, int B, int K, int V, float temperature,
                               uint64_t seed, int32_t* out_tokens, int32_t* out_n_accepted,
                               cudaStream_t stream) {
  return verify_impl(false, target_logits, draft_logits, draft_tokens, B, K, V, temperature, seed,
                     out_tokens, out_n_accepted, nullptr, nullptr, nullptr, nullptr, stream, false, true);
}

int spec_verify_early_exit_bf16(const uint16_t* target_logits, const uint16_t* draft_logits,
                                const int32_t* draft_tokens, int B, int K, int V, float temperature,
                                uint64_t seed, int32_t* out_tokens, int32_t* out_n_accepted,
                                cudaStream_t stream) {
  return verify_impl(true, target_logits, draft_logits, draft_tokens, B, K, V, temperature, seed,
                     out_tokens, out_n_accepted, nullptr, nullptr, nullptr, nullptr, stream, false, true);
}

int spec_verify_bf16_static_scratch(const uint16_t* target_logits, const uint16_t* draft_logits,
                                    const int32_t* draft_tokens, int B, int K, int V,
                                    float temperature, uint64_t seed, int32_t* out_tokens,
                                    int32_t* out_n_accepted, cudaStream_t stream) {
  return verify_impl(true, target_logits, draft_logits, draft_tokens, B, K, V, temperature, seed,
                     out_tokens, out_n_accepted, nullptr, nullptr, nullptr, nullptr, stream, true);
}

int spec_verify_stats_f32(const float* target_logits, const float* draft_logits,
                          const int32_t* draft_tokens, int B, int K, int V, float temperature,
                          uint64_t seed, int32_t* out_tokens, int32_t* out_n_accepted,
                          float* out_row_stats, float* out_pq, float* out_resid_mass,
                          float* out_row_entropy, cudaStream_t stream) {
  return verify_impl(false, target_logits, draft_logits, draft_tokens, B, K, V, temperature, seed,
                     out_tokens, out_n_accepted, out_row_stats, out_pq, out_resid_mass,
                     out_row_entropy, stream);
}

static int khint_impl(bool bf16, const void* target, const void* draft, const int32_t* tokens, int B,
                      int K, int V, float temperature, uint64_t seed, double h_lo, double h_hi,
                      int k_min, int k_max, int32_t* out_tokens, int32_t* out_n, int32_t* out_k,
                      float* out_hmean, cudaStream_t stream) {
  if (!(temperature > 0.f)) return SPEC_ERR_TEMPERATURE;  // the entropies need tau > 0
  if (!out_k) return SPEC_ERR_NULL;
  if (k_min < 0 || k_max > sv::kMaxK || k_min > k_max || !(h_lo <= h_hi)) return SPEC_ERR_HINT;
  const KHint kh = {h_lo, h_hi, k_min, k_max, out_k, out_hmean};
  return verify_impl(bf16, target, draft, tokens, B, K, V, temperature, seed, out_tokens, out_n,
                     nullptr, nullptr, nullptr, nullptr, stream, false, false, &kh);
}

int spec_verify_khint_f32(const float* target_logits, const float* draft_logits,
                          const int32_t* draft_tokens, int B, int K, int V, float temperature,
                          uint64_t seed, double h_lo, double h_hi, int k_min, int k_max,
                          int32_t* out_tokens, int32_t* out_n_accepted, int32_t* out_k_next,
                          float* out_mean_entropy, cudaStream_t stream) {
  return khint_impl(false, target_logits, draft_logits, draft_tokens, B, K, V, temperature, seed, h_lo,
                    h_hi, k_min, k_max, out_tokens, out_n_accepted, out_k_next, out_mean_entropy, stream);
}

int spec_verify_khint_bf16(const uint16_t* target_logits, const uint16_t* draft_logits,
                           const int32_t* draft_tokens, int B, int K, int V, float temperature,
                           uint64_t seed, double h_lo, double h_hi, int k_min, int k_max,
                           int32_t* out_tokens, int32_t* out_n_accepted, int32_t* out_k_next,
                           float* out_mean_entropy, cudaStream_t stream) {
  return khint_impl(true, target_logits, draft_logits, draft_tokens, B, K, V, temperature, seed, h_lo,
                    h_hi, k_min, k_max, out_tokens, out_n_accepted, out_k_next, out_mean_entropy, stream);
}

int spec_verify_stats_bf16(const uint16_t* target_logits, const uint16_t* draft_logits,
                           const int32_t* draft_tokens, int B, int K, int V, float temperature,
                           uint64_t seed, int32_t* out_tokens, int32_t* out_n_accepted,
                           float* out_row_stats, float* out_pq, float* out_resid_mass,
                           float* out_row_entropy, cudaStream_t stream) {
  return verify_impl(true, target_logits, draft_logits, draft_tokens, B, K, V, temperature, seed,
                     out_tokens, out_n_accepted, out_row_stats, out_pq, out_resid_mass,
                     out_row_entropy, stream);
}

int spec_verify_greedy_argmax_f32(const float* target_logits, const int32_t* draft_tokens, int B,
                                  int K, int V, int32_t* out_tokens, int32_t* out_n_accepted,
                                  int32_t* out_row_argmax, cudaStream_t stream) {
  return greedy_impl(false, target_logits, draft_tokens, B, K, V, out_tokens, out_n_accepted,
                     out_row_argmax, stream);
}

int spec_verify_greedy_argmax_bf16(const uint16_t* target_logits, const int32_t* draft_tokens,
                                   int B, int K, int V, int32_t* out_tokens,
                                   int32_t* out_n_accepted, int32_t* out_row_argmax,
                                   cudaStream_t stream) {
  return greedy_impl(true, target_logits, draft_tokens, B, K, V, out_tokens, out_n_accepted,
                     out_row_argmax, stream);
}

int spec_tree_verify_greedy_f32(const float* target_logits, const int32_t* tree_tokens,
                                const int32_t* parent_idx, int B, int N, int V, int32_t* out_path,
                                int32_t* out_len, uint32_t* out_mask, cudaStream_t stream) {
  return tree_impl(false, target_logits, tree_tokens, parent_idx, B, N, V, out_path, out_len,
                   out_mask, stream);
}

int spec_tree_verify_greedy_bf16(const uint16_t* target_logits, const int32_t* tree_tokens,
                                 const int32_t* parent_idx, int B, int N, int V,
                                 int32_t* out_path, int32_t* out_len, uint32_t* out_mask,
                                 cudaStream_t stream) {
  return tree_impl(true, target_logits, tree_tokens, parent_idx, B, N, V, out_path, out_len,
                   out_mask, stream);
}

int spec_tree_verify_greedy_early_exit_f32(const float* target_logits, const int32_t* tree_tokens,
                                           const int32_t* parent_idx, int B, int N, int V,
                                           int32_t* out_path, int32_t* out_len, uint32_t* out_mask,
                                           cudaStream_t stream) {
  return tree_impl(false, target_logits, tree_tokens, parent_idx, B, N, V, out_path, out_len,
                   out_mask, stream, true);
}

int spec_tree_verify_greedy_early_exit_bf16(const uint16_t* target_logits, const int32_t* tree_tokens,
                                            const int32_t* parent_idx, int B, int N, int V,
                                            int32_t* out_path, int32_t* out_len, uint32_t* out_mask,
                                            cudaStream_t stream) {
  return tree_impl(true, target_logits, tree_tokens, parent_idx, B, N, V, out_path, out_len,
                   out_mask, stream, true);
}

int spec_tree_verify_sampling_f32(const float* target_logits, const float* draft_logits,
                                  const int32_t* tree_tokens, const int32_t* parent_idx, int B, int N,
                                  int V, float temperature, uint64_t seed, int32_t* out_path,
                                  int32_t* out_len, cudaStream_t stream) {
  return tree_sample_impl(false, target_logits, draft_logits, tree_tokens, parent_idx, B, N, V,
                          temperature, seed, out_path, out_len, stream);
}

int spec_tree_verify_sampling_bf16(const uint16_t* target_logits, const uint16_t* draft_logits,
                                   const int32_t* tree_tokens, const int32_t* parent_idx, int B,
                                   int N, int V, float temperature, uint64_t seed, int32_t* out_path,
                                   int32_t* out_len, cudaStream_t stream) {
  return tree_sample_impl(true, target_logits, draft_logits, tree_tokens, parent_idx, B, N, V,
                          temperature, seed, out_path, out_len, stream);
}

int spec_acceptance_stats(const int32_t* n_accepted, int B, int K, uint64_t* out_hist,
                          double* out_alpha, double* out_mean_tokens, cudaStream_t stream) {
  if (!out_hist || (B > 0 && !n_accepted)) return SPEC_ERR_NULL;
  if (B < 0 || K < 0 || K > sv::kMaxTreeNodes) return SPEC_ERR_SHAPE;
  DeviceState* d = nullptr;
  const int rc = get_device_state(&d);
  if (rc) return rc;
  const cudaError_t e = sv::launch_acceptance(n_accepted, B, K, (unsigned long long*)out_hist,
                                              K > 0 ? out_alpha : nullptr, out_mean_tokens, d->sms,
                                              stream);
  if (e != cudaSuccess) return cuda_fail(e, "acceptance statistics launch");
  return SPEC_OK;
}

int spec_ngram_draft(const int32_t* tokens, const int32_t* lengths, int B, int stride, int n_min, int n_max,
                     int K, int32_t* out_drafts, int32_t* out_n_drafts, int32_t* out_match_len,
                     cudaStream_t stream) {
  if (B < 0 || stride < 1 || stride > (1 << 30) || n_min < 1 || n_max < n_min || n_max > sv::kNgramMaxN ||
      K < 0 || K > 4096)
    return SPEC_ERR_SHAPE;
  if (B == 0) return SPEC_OK;
  if (!tokens || !lengths || !out_n_drafts || (K > 0 && !out_drafts)) return SPEC_ERR_NULL;
  const long long chunks = ((long long)stride + sv::ngram_chunk() - 1) / sv::ngram_chunk();
  // entries are 32-bit; the claim counter overshoots the total by two claims per CTA
  if ((long long)B * chunks >= (1LL << 31) - (1LL << 20)) return SPEC_ERR_SHAPE;
  DeviceState* d = nullptr;
  int rc = get_device_state(&d);
  if (rc) return rc;
  if (d->occ_ngram < 1) return cuda_fail(cudaErrorInvalidConfiguration, "n-gram scan shared memory");
  sv::NgramArgs a;
  memset(&a, 0, sizeof a);
  a.tokens = tokens;
  a.stride = stride;
  a.lengths = lengths;
  a.B = B;
  a.n_min = n_min;
  a.n_max = n_max;
  a.K = K;
  a.chunks = (int)chunks;
  a.vec = aligned16(tokens) && stride % 4 == 0;
  a.drafts = out_drafts;
  a.n_drafts = out_n_drafts;
  a.status = d->status;
  // match_len is optional: without it the kernel writes into scratch
  const long long entries = (long long)B * chunks;
  sv::WsLayout l;
  const size_t slots = ((size_t)entries * 8 + 255) / 256 * 256;
  const size_t counter = 256;
  l.total = slots + counter + (out_match_len ? 0 : ((size_t)B * 4 + 255) / 256 * 256);
  l.zero_bytes = slots + counter;  // no chunk's best end yet; the counter at 0
  l.marker_off = 0;
  l.marker_bytes = 0;
  void* ws = nullptr;
  rc = get_scratch(d, false, l, stream, &ws);
  if (rc) return rc;
  a.slot = (unsigned long long*)ws;
  a.counter = (int*)((char*)ws + slots);
  a.match_len = out_match_len ? out_match_len : (int32_t*)((char*)ws + slots + counter);
  const long long capacity = (long long)d->sms * d->occ_ngram;
  const int grid = (int)(entries < capacity ? entries : capacity);
  cudaError_t e = sv::launch_ngram(a, grid, stream);
  cudaError_t e2 = put_scratch(false, ws, stream);
  if (e != cudaSuccess) return cuda_fail(e, "n-gram drafting launch");
  if (e2 != cudaSuccess) return cuda_fail(e2, "cudaFreeAsync");
  return SPEC_OK;
}

int spec_test_fail_allocations(int n) { return g_fail_allocs.exchange(n < 0 ? 0 : n); }

int spec_test_spin_limit(uint32_t iterations) {
  DeviceState* d = nullptr;
  const int rc = get_device_state(&d);
  if (rc) return rc;
  const unsigned n = iterations ? iterations : sv::kSpinLimit;
  cudaError_t e = cudaDeviceSynchronize();  // no launch in flight sees a changed limit
  if (e == cudaSuccess) e = sv::sample_set_spin_limit(n);
  if (e == cudaSuccess) e = sv::greedy_set_spin_limit(n);
  if (e == cudaSuccess) e = sv::tree_sample_set_spin_limit(n);
  if (e == cudaSuccess) e = sv::ngram_set_spin_limit(n);
  if (e != cudaSuccess) return cuda_fail(e, "spin limit");
  return SPEC_OK;
}

int spec_test_wait_probe(uint32_t* out_flags) {
  if (!out_flags) return SPEC_ERR_NULL;
  DeviceState* d = nullptr;
  const int rc = get_device_state(&d);
  if (rc) return rc;
  const cudaError_t e = sv::sample_wait_probe(out_flags);
  if (e != cudaSuccess) return cuda_fail(e, "wait probe");
  return SPEC_OK;
}

int spec_get_status(cudaStream_t stream, uint32_t* flags_out) {
  DeviceState* d = nullptr;
  int rc = get_device_state(&d);
  if (rc) return rc;
  unsigned v = 0;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  e = cudaMemcpyAsync(&v, d->status, sizeof v, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(d->status, 0, sizeof v, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "status word");
  if (flags_out) *flags_out = v;
  return SPEC_OK;
}

const char* spec_status_string(int code) {
  switch (code) {
    case SPEC_OK:
      return "ok";
    case SPEC_ERR_NULL:
      return "a required pointer is NULL";
    case SPEC_ERR_SHAPE:
      return "bad shape: B < 0, K outside [0, 255], N outside [0, 1024], V < 1, or size overflow";
    case SPEC_ERR_TEMPERATURE:
      return "bad temperature: NaN, negative, or in (0, 1e-30)";
    case SPEC_ERR_CUDA:
      return g_cuda_msg;
    case SPEC_ERR_HINT:
      return "bad draft-length parameters: need 0 <= k_min <= k_max <= 255 and h_lo <= h_hi (no NaN)";
    case SPEC_ERR_SCRATCH:
      return "the problem needs more scratch than the static buffer holds "
             "(SPEC_STATIC_SCRATCH_BYTES)";
    default:
      return "unknown status code";
  }
}

}  // extern "C"
