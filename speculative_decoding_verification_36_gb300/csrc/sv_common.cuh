// sv_common.cuh -- device building blocks shared by the verify kernels.
//
// Layout conventions (all row-major, contiguous):
//   target logits  [B, K+1, V]   row i scores draft position i, row K is the bonus row
//   draft logits   [B, K,   V]
//   tree target    [B, N+1, V]   row 0 is the root, row i+1 belongs to node i
// Logits are fp32 or bf16 (stored as raw 16-bit words and widened exactly).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sv_kernels.h"

namespace sv {


// The limit in force for every bounded wait of this translation unit's
// kernels (one copy per translation unit and device).  spec_test_spin_limit
// lowers it so that a test can make waits run out on purpose.  It is read
// with a volatile load, and only once a wait has found its slot unset: no
// device code writes it, and the host changes it between launches.
static __device__ unsigned g_spin_limit = kSpinLimit;
__device__ __forceinline__ unsigned spin_limit() { return *(const volatile unsigned*)&g_spin_limit; }
// Host side: set this translation unit's copy on the current device.
static inline cudaError_t set_spin_limit_here(unsigned n) {
  return cudaMemcpyToSymbol(g_spin_limit, &n, sizeof n);
}

// status bits OR-ed into the library's device status word
constexpr unsigned kStatusBadData = 1u;  // NaN / +inf logit, empty row, bad token or parent
constexpr unsigned kStatusTimeout = 2u;  // a bounded wait ran out (should never happen)

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// 2^x with the MUFU unit (ex2.approx, denormal results flushed to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// packed fp32 pairs (f32x2 arithmetic: two IEEE operations per instruction)
// ---------------------------------------------------------------------------
typedef unsigned long long f2_t;
__device__ __forceinline__ f2_t f2(float lo, float hi) {
  f2_t r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float f2lo(f2_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f2hi(f2_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ f2_t f2sub(f2_t a, f2_t b) {
  f2_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2_t f2mul(f2_t a, f2_t b) {
  f2_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2_t f2fma(f2_t a, f2_t b, f2_t c) {
  f2_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ f2_t f2add(f2_t a, f2_t b) {
  f2_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// 2^{(z - base) * c} for both halves, accumulated into acc (per-element IEEE
// rounding identical to the scalar sequence sub, mul, ex2, add).
__device__ __forceinline__ void f2_exp_acc(f2_t& acc, f2_t z, f2_t base, f2_t c) {
  const f2_t t = f2mul(f2sub(z, base), c);
  acc = f2add(acc, f2(ex2(f2lo(t)), ex2(f2hi(t))));
}

// The same with the entropy accumulator tacc += 2^t t (t <= 0: exponents are
// taken relative to the running maximum).  t is clamped at -126 for the
// product, so masked (-inf) elements and underflowed terms add 0, not NaN.
__device__ __forceinline__ void f2_exp_acc_ent(f2_t& acc, f2_t& tacc, f2_t z, f2_t base, f2_t c) {
  const f2_t t = f2mul(f2sub(z, base), c);
  const f2_t e = f2(ex2(f2lo(t)), ex2(f2hi(t)));
  acc = f2add(acc, e);
  tacc = f2fma(e, f2(fmaxf(f2lo(t), -126.f), fmaxf(f2hi(t), -126.f)), tacc);
}

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// 16-byte streaming load that does not allocate in L1 (the data is read once
// per unit; the one re-read comes from L2).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Element storage types.  kVec = elements per 16-byte vector on the aligned
// path; the scalar path (rows not 16-byte aligned) loads one element at a time.
struct F32 {
  using storage = float;
  static constexpr int kVec = 4;
  static constexpr uint32_t kNegInfWord = 0xff800000u;
  __device__ static float load1(const storage* p) { return __ldg(p); }
};
struct BF16 {
  using storage = uint16_t;
  static constexpr int kVec = 8;
  static constexpr uint32_t kNegInfWord = 0xff80ff80u;  // two bf16 -inf
  __device__ static float load1(const storage* p) {
    return __uint_as_float(((uint32_t)__ldg(p)) << 16);
  }
};

// VEC elements kept in their storage form (16 bytes on the vector path) and
// widened to fp32 when used.
template <class E, int VEC>
struct Raw {
  uint4 w;
};
template <class E>
struct Raw<E, 1> {
  float f;
};

// Load VEC consecutive elements starting at element e of row.  Elements at or
// beyond `end` read as -inf (they never win a max and add 0 to a sum).
template <class E, int VEC>
__device__ __forceinline__ Raw<E, VEC> load_raw(const typename E::storage* row, int e, int end) {
  Raw<E, VEC> r;
  if constexpr (VEC == 1) {
    r.f = e < end ? E::load1(row + e) : neg_inf();
  } else {
    if (e < end)
      r.w = ld_stream16(row + e);
    else
      r.w = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
  }
  return r;
}

__device__ __forceinline__ uint32_t word_of(const uint4& w, int i) {
  return i == 0 ? w.x : (i == 1 ? w.y : (i == 2 ? w.z : w.w));
}

// Element q of a loaded vector, as fp32 (exact widening).
template <class E, int VEC>
__device__ __forceinline__ float elem(const Raw<E, VEC>& r, int q) {
  if constexpr (VEC == 1) {
    return r.f;
  } else if constexpr (VEC == 8) {
    const uint32_t w = word_of(r.w, q >> 1);
    return (q & 1) ? bf16_hi(w) : bf16_lo(w);
  } else {
    return __uint_as_float(word_of(r.w, q));
  }
}

// Elements 2p and 2p+1 of a loaded vector as a packed pair.
template <class E, int VEC>
__device__ __forceinline__ f2_t elem_pair(const Raw<E, VEC>& r, int p) {
  if constexpr (VEC == 8) {
    const uint32_t w = word_of(r.w, p);
    return f2(bf16_lo(w), bf16_hi(w));
  } else {
    return f2(__uint_as_float(word_of(r.w, 2 * p)), __uint_as_float(word_of(r.w, 2 * p + 1)));
  }
}

// The same pair as a float2 (register pair).
template <class E, int VEC>
__device__ __forceinline__ float2 elem_pair2(const Raw<E, VEC>& r, int p) {
  if constexpr (VEC == 8) {
    const uint32_t w = word_of(r.w, p);
    return make_float2(bf16_lo(w), bf16_hi(w));
  } else {
    return make_float2(__uint_as_float(word_of(r.w, 2 * p)), __uint_as_float(word_of(r.w, 2 * p + 1)));
  }
}

// Maximum over a batch of kUnroll loaded vectors (NaN never wins: max ignores
// a NaN operand).
template <class E, int VEC>
__device__ __forceinline__ float batch_max(const Raw<E, VEC> (&z)[kUnroll]) {
  if constexpr (VEC == 8) {
    uint32_t mw = bf16x2_max(bf16x2_max(z[0].w.x, z[0].w.y), bf16x2_max(z[0].w.z, z[0].w.w));
#pragma unroll
    for (int u = 1; u < kUnroll; ++u)
      mw = bf16x2_max(mw, bf16x2_max(bf16x2_max(z[u].w.x, z[u].w.y), bf16x2_max(z[u].w.z, z[u].w.w)));
    return fmaxf(bf16_lo(mw), bf16_hi(mw));
  } else {
    float bm = neg_inf();
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
#pragma unroll
      for (int q = 0; q < VEC; ++q) bm = fmaxf(bm, elem(z[u], q));
    return bm;
  }
}

// Bulk L2 prefetch (TMA engine) of a contiguous byte range: one instruction
// starts streaming a whole slice into L2 while the warp works, so the warp's
// own loads mostly wait on L2 rather than DRAM.  Start and size must be
// multiples of 16 bytes (the vector path guarantees both).
__device__ __forceinline__ void prefetch_l2(const void* p, unsigned bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// The same with an L2 eviction-priority policy (createpolicy).  The default
// bulk prefetch inserts lines that L2 gives up quickly; rows that will be
// read a second time are prefetched with evict_last instead.
__device__ __forceinline__ void prefetch_l2_pol(const void* p, unsigned bytes, uint64_t pol) {
  asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(p), "r"(bytes), "l"(pol)
               : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Asynchronous 16-byte copies global -> shared (no register staging), grouped
// per thread: a thread waits only for its own groups, and every lane reads
// back only what it copied itself, so no barrier is needed.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned d = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 ld_shared16(const void* smem) {
  uint4 r;
  const unsigned a = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(a) : "memory");
  return r;
}

// Coherent loads / stores / atomics on workspace values shared between warps.
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int atom_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Relaxed (unordered, cheap) 64-bit stores / loads and atomics for per-slice
// results.  A reader learns that a slot is complete from its content: slots are
// pre-filled with the kMarker pattern (a NaN no result ever takes).
__device__ __forceinline__ void st_relaxed_u2(void* p, uint32_t x, uint32_t y) {
  asm volatile("st.relaxed.gpu.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ uint2 ld_relaxed_u2(const void* p) {
  uint2 v;
  asm volatile("ld.relaxed.gpu.global.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_v4(void* p, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.relaxed.gpu.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(x), "r"(y), "r"(z), "r"(w)
               : "memory");
}
__device__ __forceinline__ uint4 ld_relaxed_v4(const void* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_f32(float* p, float v) {
  asm volatile("st.relaxed.gpu.global.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}
__device__ __forceinline__ float ld_relaxed_f32(const float* p) {
  float v;
  asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_s32(int* p, int v) {
  asm volatile("st.relaxed.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_relaxed_s32(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_f32(float* p, float v) {
  asm volatile("st.release.gpu.global.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}
__device__ __forceinline__ float ld_acquire_f32(const float* p) {
  float v;
  asm volatile("ld.acquire.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ int atom_add_relaxed(int* p, int v) {
  int old;
  asm volatile("atom.relaxed.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
// A ticket on a counter that starts at -1: the number of earlier takers.
__device__ __forceinline__ int ticket_take(int* p) { return atom_add_relaxed(p, 1) + 1; }

// Bounded waits for a slot to leave the marker state.  A ticket count says
// every writer has issued its store; the store itself may land a moment later.
__device__ __forceinline__ uint2 wait_u2(const void* p, unsigned* status) {
  uint2 v = ld_relaxed_u2(p);
  unsigned it = 0;
  while (v.x == kMarker && ++it < spin_limit()) {
    __nanosleep(64);
    v = ld_relaxed_u2(p);
  }
  if (v.x == kMarker) atomicOr(status, kStatusTimeout);
  return v;
}
__device__ __forceinline__ int wait_s32(const int* p, unsigned* status) {
  int v = ld_relaxed_s32(p);
  unsigned it = 0;
  while (v == (int)kMarker && ++it < spin_limit()) {
    __nanosleep(64);
    v = ld_relaxed_s32(p);
  }
  if (v == (int)kMarker) atomicOr(status, kStatusTimeout);
  return v;
}
__device__ __forceinline__ float wait_f32(const float* p, unsigned* status) {
  float v = ld_relaxed_f32(p);
  unsigned it = 0;
  while (__float_as_uint(v) == kMarker && ++it < spin_limit()) {
    __nanosleep(64);
    v = ld_relaxed_f32(p);
  }
  if (__float_as_uint(v) == kMarker) atomicOr(status, kStatusTimeout);
  return v;
}
__device__ __forceinline__ float wait_f32_acquire(const float* p, unsigned* status) {
  float v = ld_acquire_f32(p);
  unsigned it = 0;
  while (__float_as_uint(v) == kMarker && ++it < spin_limit()) {
    __nanosleep(64);
    v = ld_acquire_f32(p);
  }
  if (__float_as_uint(v) == kMarker) atomicOr(status, kStatusTimeout);
  return v;
}

// A 16-byte result slot whose first three words have all been written.
__device__ __forceinline__ uint4 wait_result(const void* p, unsigned* status) {
  uint4 v = ld_relaxed_v4(p);
  unsigned it = 0;
  while ((v.x == kMarker || v.y == kMarker || v.z == kMarker) && ++it < spin_limit()) {
    __nanosleep(64);
    v = ld_relaxed_v4(p);
  }
  if (v.x == kMarker || v.y == kMarker || v.z == kMarker) atomicOr(status, kStatusTimeout);
  return v;
}

// n / d for 0 <= n < 2^31 with d's FastDiv constants.
__device__ __forceinline__ int fdiv(int n, const FastDiv& f) {
  return (int)(((unsigned long long)(unsigned)n * f.m) >> f.shift);
}

// Lane 0 of warp w claims the next unit from counter w.  The atomic is a
// predicated instruction rather than a branch, so nothing reads its result
// register until the value is broadcast: the claim's round trip overlaps
// whatever the warp does in between.
__device__ __forceinline__ int slice_of_warp() { return (threadIdx.x >> 5) % kSlices; }
// Claim counters and tickets start at all-ones (-1), so that one 0xff fill
// initialises the whole workspace; the helpers below return the number of
// earlier increments (the first taker gets 0).
__device__ __forceinline__ int claim_from(unsigned long long* counter, int ctr, int lane) {
  unsigned long long v = ~0ull;
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.eq.s32 p, %1, 0;\n\t"
      "@p atom.relaxed.gpu.global.add.u64 %0, [%2], 1;\n\t}"
      : "+l"(v)
      : "r"(lane), "l"(counter + ctr * kCounterStride)
      : "memory");
  return (int)(v + 1);
}
__device__ __forceinline__ int claim_unit(unsigned long long* counter, int lane) {
  return claim_from(counter, slice_of_warp(), lane);
}
// A ticket taken only where `pred` holds (0 elsewhere), with no wait at the
// issue point.
__device__ __forceinline__ int ticket_take_if(bool pred, int* p) {
  int r = -1;
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "@q atom.relaxed.gpu.global.add.s32 %0, [%2], 1;\n\t}"
      : "+r"(r)
      : "r"((unsigned)pred), "l"(p)
      : "memory");
  return r + 1;
}
// The same for a relaxed 32-bit load issued only where `pred` holds; `v` is
// returned unchanged elsewhere.
__device__ __forceinline__ uint32_t ld_relaxed_if(bool pred, const void* p, uint32_t v) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "@q ld.relaxed.gpu.global.u32 %0, [%2];\n\t}"
      : "+r"(v)
      : "r"((unsigned)pred), "l"(p)
      : "memory");
  return v;
}
__device__ __forceinline__ int bcast(int v) { return __shfl_sync(0xffffffffu, v, 0); }

// ---------------------------------------------------------------------------
// Position verdicts and the per-sequence resolution word of the chain
// verifies: a sequence is decided once positions 0..n are resolved with
// 0..n-1 accepted and n rejected (or bad), or 0..K resolved with all K
// accepted.
// ---------------------------------------------------------------------------
constexpr int kVerdictAccept = 0;
constexpr int kVerdictReject = 1;
constexpr int kVerdictBad = 2;

// Decided count n for the set of resolved / rejected positions `set` (bit i:
// position i resolved; bit 32 + i: position i rejected, i < K), or -1 while
// the prefix that fixes n is incomplete.
__device__ __forceinline__ int decided_n(unsigned long long set, int K) {
  const unsigned rej = K > 0 ? (unsigned)(set >> 32) & (0xffffffffu >> (32 - K)) : 0u;
  const int r = rej ? __ffs(rej) - 1 : K;
  const unsigned long long need = (2ull << r) - 1ull;
  return (set & need) == need ? r : -1;
}

// ---------------------------------------------------------------------------
// Online softmax statistics: (m, s) with m the running max of the raw logits
// and s = sum exp2((z - m) * c), c = log2(e) / temperature.  Terms are always
// taken relative to the current max, so the dominant terms carry exponent 0.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ms_merge(float& m, float& s, float m2, float s2, float c) {
  float mn = fmaxf(m, m2);
  float base = (mn == neg_inf()) ? 0.f : mn;
  s = s * ex2((m - base) * c) + s2 * ex2((m2 - base) * c);
  m = mn;
}

// (m, s) over the 32 lanes, every lane ends with the total: the warp max
// first, then each lane's sum rescaled to it once, then a butterfly sum.
__device__ __forceinline__ void warp_ms(float& m, float& s, float c) {
  float mx = m;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  const float base = (mx == neg_inf()) ? 0.f : mx;
  float t = s * ex2((m - base) * c);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
  m = mx;
  s = t;
}

// Entropy statistics (m, s, t) with t = sum 2^d d over the same terms as s,
// d = (z - m) c.  Moving the reference maximum from m to m' shifts every
// exponent by delta = (m - m') c <= 0, and 2^(d + delta) (d + delta) =
// 2^delta (2^d d + delta 2^d), so t' = 2^delta (t + delta s); an empty
// accumulator (m = -inf) has t = 0.  The entropy of the row in nats is then
// ln s - ln 2 * t / s.  s is updated with exactly the expressions of ms_merge
// and warp_ms, so asking for the entropy changes no other result.
__device__ __forceinline__ float t_rescaled(float m, float s, float t, float base, float c) {
  if (m == neg_inf()) return 0.f;
  const float delta = (m - base) * c;
  return ex2(delta) * (t + delta * s);
}
__device__ __forceinline__ void mst_merge(float& m, float& s, float& t, float m2, float s2, float t2, float c) {
  const float mn = fmaxf(m, m2);
  const float base = (mn == neg_inf()) ? 0.f : mn;
  t = t_rescaled(m, s, t, base, c) + t_rescaled(m2, s2, t2, base, c);
  s = s * ex2((m - base) * c) + s2 * ex2((m2 - base) * c);
  m = mn;
}
__device__ __forceinline__ void warp_mst(float& m, float& s, float& t, float c) {
  float mx = m;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  const float base = (mx == neg_inf()) ? 0.f : mx;
  float u = s * ex2((m - base) * c);
  float v = t_rescaled(m, s, t, base, c);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    u += __shfl_xor_sync(0xffffffffu, u, off);
    v += __shfl_xor_sync(0xffffffffu, v, off);
  }
  m = mx;
  s = u;
  t = v;
}

// ---------------------------------------------------------------------------
// Streaming statistics of one row segment: kUnroll 16-byte vectors per lane per
// batch, reduced into the lane's running (m, s) (and the entropy accumulator).
// ---------------------------------------------------------------------------
template <class E, int VEC>
__device__ __forceinline__ void load_batch(Raw<E, VEC> (&z)[kUnroll], const typename E::storage* row,
                                           int e, int v1) {
  constexpr int STEPW = 32 * VEC;
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) z[u] = load_raw<E, VEC>(row, e + u * STEPW, v1);
}

// One batch into the lane's running (m, s): the batch max first, one rescale
// if it rose, then the exponentials, with float2 arithmetic on register pairs.
// Without the entropy accumulator each exponent is one fused multiply-add,
// z c - fl(m c): every term then carries the same factor 2^e with
// e = m c - fl(m c) (the rounding of the product, below 2^-24 |m c|), which
// exp_fma_fix takes out of the lane's sum once, at the end; rescales use the
// same rounded products, so terms added before and after a rescale carry the
// same factor.  With the entropy accumulator the exponent is (z - m) c, whose
// terms the accumulator t = sum 2^d d needs exactly.
template <class E, int VEC, bool ENT>
__device__ __forceinline__ void stats_batch(const Raw<E, VEC> (&z)[kUnroll], float& m, float2& acc,
                                            float2& tacc, float cc) {
  const float bm = batch_max<E, VEC>(z);
  if (bm > m) {
    // the sums are relative to fl(m c), the base of the fused exponents
    const float delta = __fsub_rn(__fmul_rn(m, cc), __fmul_rn(bm, cc));  // -inf when m was -inf
    const float f = ex2(delta);
    if constexpr (ENT) {
      // t' = 2^delta (t + delta s); an empty accumulator stays empty
      tacc = m == neg_inf() ? make_float2(0.f, 0.f)
                            : __fmul2_rn(make_float2(f, f), __ffma2_rn(make_float2(delta, delta), acc, tacc));
    }
    acc = __fmul2_rn(acc, make_float2(f, f));
    m = bm;
  }
  const float base = (m == neg_inf()) ? 0.f : m;
  if constexpr (VEC == 1) {
    const float nmc = -__fmul_rn(base, cc);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const float d = __fmaf_rn(z[u].f, cc, nmc);
      const float e = ex2(d);
      acc.x += e;
      if constexpr (ENT) tacc.x = fmaf(e, fmaxf(d, -126.f), tacc.x);  // 0 * -inf would be NaN
    }
  } else {
    const float2 c2 = make_float2(cc, cc);
    const float2 nmc = make_float2(-__fmul_rn(base, cc), -__fmul_rn(base, cc));
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
#pragma unroll
      for (int p = 0; p < VEC / 2; ++p) {
        const float2 d = __ffma2_rn(elem_pair2<E, VEC>(z[u], p), c2, nmc);
        const float2 e = make_float2(ex2(d.x), ex2(d.y));
        acc = __fadd2_rn(acc, e);
        if constexpr (ENT) tacc = __ffma2_rn(e, make_float2(fmaxf(d.x, -126.f), fmaxf(d.y, -126.f)), tacc);
      }
  }
}

// Error-free sum a + b = hi + lo (Knuth's TwoSum), round-to-nearest steps.
__device__ __forceinline__ float2 two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  return make_float2(s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb)));
}

// Float pairs (hi + lo, |lo| <= ulp(hi) / 2): renormalising sum, product
// (the product's error from one FMA) and sum.
__device__ __forceinline__ float2 fast_two_sum(float a, float b) {  // |a| >= |b|
  const float s = __fadd_rn(a, b);
  return make_float2(s, __fsub_rn(b, __fsub_rn(s, a)));
}
__device__ __forceinline__ float2 pair_mul(float2 a, float2 b) {
  const float p = __fmul_rn(a.x, b.x);
  const float e = __fadd_rn(__fmaf_rn(a.x, b.x, -p), __fadd_rn(__fmul_rn(a.x, b.y), __fmul_rn(a.y, b.x)));
  return fast_two_sum(p, e);
}
__device__ __forceinline__ float2 pair_add(float2 a, float2 b) {
  const float2 s = two_sum(a.x, b.x);
  return fast_two_sum(s.x, __fadd_rn(s.y, __fadd_rn(a.y, b.y)));
}

// log2(x) of a positive normal float as a float pair, within about 2e-11:
// x = 2^e m with m in [sqrt(1/2), sqrt(2)), ln m = 2 atanh(s) with
// s = (m - 1) / (m + 1), |s| < 0.172, atanh(s) = s + s^3/3 + s^5/5 + ...;
// s and s^3/3 are float pairs, s^5/5 + ... (below 3e-5 of s) is fp32.
__device__ __forceinline__ float2 log2_pair(float x) {
  const int bits = __float_as_int(x);
  int e = ((bits >> 23) & 0xff) - 127;
  float m = __int_as_float((bits & 0x007fffff) | 0x3f800000);  // [1, 2)
  if (m > 1.41421356f) {
    m = __fmul_rn(m, 0.5f);
    e += 1;
  }
  const float num = __fsub_rn(m, 1.f);  // exact
  const float2 den = two_sum(m, 1.f);
  const float sh = __fdiv_rn(num, den.x);
  const float rem = __fmaf_rn(-sh, den.x, num);  // exact remainder
  const float2 sv = fast_two_sum(sh, __fdiv_rn(__fmaf_rn(-sh, den.y, rem), den.x));
  const float t = __fmul_rn(sv.x, sv.x);
  float q = 1.f / 15.f;  // Q(t) = 1/5 + t/7 + t^2/9 + t^3/11 + t^4/13 + t^5/15
  q = __fmaf_rn(q, t, 1.f / 13.f);
  q = __fmaf_rn(q, t, 1.f / 11.f);
  q = __fmaf_rn(q, t, 1.f / 9.f);
  q = __fmaf_rn(q, t, 1.f / 7.f);
  q = __fmaf_rn(q, t, 1.f / 5.f);
  const float2 s3 = pair_mul(pair_mul(sv, sv), sv);
  const float2 s33 = pair_mul(s3, make_float2(0.333333343f, -9.93410776e-9f));  // 1/3 as a pair
  const float tail = __fmul_rn(__fmul_rn(s3.x, t), q);                          // s^5 Q(s^2)
  const float2 at = pair_add(pair_add(sv, s33), make_float2(tail, 0.f));
  const float2 l2m = pair_mul(make_float2(__fmul_rn(at.x, 2.f), __fmul_rn(at.y, 2.f)),
                              make_float2(1.44269502f, 1.92596303e-8f));  // 1/ln 2 as a pair
  return pair_add(make_float2((float)e, 0.f), l2m);
}

// The acceptance test u < p(x) / q(x) for a drafted token with q(x) > 0:
// p(x) / q(x) = 2^{((zT - mT) - (zD - mD)) c} sD / sT.  The exponent comes
// from error-free differences and c = c_hi + c_lo (about 45 bits), 2^f from
// the ex2 instruction (relative error below 2^-21) and sD / sT from one
// correctly rounded division, so alpha is within about 4e-7 (relative) of
// the exact ratio.  A decision can then differ from the exact one only when
// |u - min(1, alpha)| is below 4e-7, inside the 1e-6 band the boundary
// accounting allows; q == p gives alpha == 1 exactly.  fp32 instead of fp64:
// on this GPU a double exp2 and division on the decision path cost over a
// microsecond per call.
__device__ __forceinline__ bool accept_draw(float zT, float mT, float zD, float mD, float sT, float sD,
                                            float c_hi, float c_lo, double u) {
  if (zT == neg_inf()) return false;  // p(x) = 0 < u
  const float2 dT = two_sum(zT, -mT), dD = two_sum(zD, -mD);
  const float2 E = two_sum(dT.x, -dD.x);
  const float El = __fadd_rn(E.y, __fsub_rn(dT.y, dD.y));
  const float xh = __fmul_rn(E.x, c_hi);
  const float xl = __fadd_rn(__fmaf_rn(E.x, c_hi, -xh), __fmaf_rn(E.x, c_lo, __fmul_rn(El, c_hi)));
  // row sums lie in [1, V]: sD / sT is within [2^-31, 2^31]
  if (xh > 160.f) return true;
  if (xh < -160.f) return false;
  const float n = floorf(xh);
  const float g = __fmul_rn(ex2(__fsub_rn(xh, n)), __fmaf_rn(xl, 0.69314718055994530942f, 1.f));
  return u < (double)ldexpf(__fmul_rn(g, __fdiv_rn(sD, sT)), (int)n);
}

// e = m c - fl(m c): stats_batch's fused exponents d_f = z c - fl(m c) exceed
// the exact (z - m) c by e, so a lane's sums relative to fl(m c) relate to
// the exact ones as s = 2^{-e} s_f and t = sum d 2^d = 2^{-e} (t_f - e s_f).
// |e| < 2^-24 |m c|: the first-order factor 1 - e ln 2 is exact to far below
// fp32.
__device__ __forceinline__ float exp_fma_err(float m, float cc) {
  const float base = (m == neg_inf()) ? 0.f : m;
  return __fmaf_rn(base, cc, -__fmul_rn(base, cc));
}
__device__ __forceinline__ float exp_fma_fix(float m, float cc) {
  return __fmaf_rn(-exp_fma_err(m, cc), 0.69314718055994530942f, 1.f);
}

// ---------------------------------------------------------------------------
// Replacement / bonus weights.  Both are scaled by the target row's sum sT so
// that no division is needed: the inverse CDF only sees ratios.
//   bonus:     w(v) = 2^{(zT - mT) c}                        = sT * p(v)
//   residual:  w(v) = 2^{(zT - mT) c} * (1 - 2^{-delta})     = sT * max(0, p(v) - q(v))
//              delta = (dT - dD) c - log2(sT / sD)          (> 0 iff p(v) > q(v))
// The form 2^{aT}(1 - 2^{-delta}) has no cancellation (see resid_factor).
// Explicit round-to-nearest operations (no contraction) keep the arithmetic
// identical in the tail units and in the final rescan.
// ---------------------------------------------------------------------------
struct TailConsts {
  float mT, mD, c_hi, c_lo, lam_hi, lam_lo;
  int residual;
};

// max(0, 1 - 2^{-d}) without cancellation and without branches.  With
// eh = 2^{-d/2} (ex2) and x = d ln2 / 2:
//   d >= 1.4:  1 - eh^2                                   (>= 0.62, nothing cancels)
//   d <  1.4:  1 - e^{-2x} = 2 sinh(x) e^{-x} = x (2 + x^2/3 + x^4/60 + x^6/2520) eh
// (|x| < 0.49 there, so the first omitted term is below 1e-8 relative).  For
// d <= 0 the second form is <= 0 and the clamp returns 0.  Both forms are
// evaluated and one is selected, so the packed version below can share every
// instruction between the two elements of a pair.
__device__ __forceinline__ float resid_factor(float d) {
  const float eh = ex2(__fmul_rn(d, -0.5f));
  const float A = __fsub_rn(1.f, __fmul_rn(eh, eh));
  const float x = __fmul_rn(d, 0.346573590279972655f);
  const float xx = __fmul_rn(x, x);
  float p = __fmaf_rn(xx, 1.f / 2520.f, 1.f / 60.f);
  p = __fmaf_rn(xx, p, 1.f / 3.f);
  p = __fmaf_rn(xx, p, 2.f);
  const float Bv = __fmul_rn(__fmul_rn(x, p), eh);
  return fmaxf(d >= 1.4f ? A : Bv, 0.f);
}

// resid_factor on both elements of a pair, with every operation rounding as
// in the scalar version (bit-identical results); float2 arithmetic on register
// pairs.
__device__ __forceinline__ float2 resid_factor2(float2 d) {
  const float2 hd = __fmul2_rn(d, make_float2(-0.5f, -0.5f));
  const float2 eh = make_float2(ex2(hd.x), ex2(hd.y));
  const float2 A = __fadd2_rn(make_float2(1.f, 1.f), __fmul2_rn(make_float2(-1.f, -1.f), __fmul2_rn(eh, eh)));
  const float2 x = __fmul2_rn(d, make_float2(0.346573590279972655f, 0.346573590279972655f));
  const float2 xx = __fmul2_rn(x, x);
  float2 p = __ffma2_rn(xx, make_float2(1.f / 2520.f, 1.f / 2520.f), make_float2(1.f / 60.f, 1.f / 60.f));
  p = __ffma2_rn(xx, p, make_float2(1.f / 3.f, 1.f / 3.f));
  p = __ffma2_rn(xx, p, make_float2(2.f, 2.f));
  const float2 Bv = __fmul2_rn(__fmul2_rn(x, p), eh);
  return make_float2(fmaxf(d.x >= 1.4f ? A.x : Bv.x, 0.f), fmaxf(d.y >= 1.4f ? A.y : Bv.y, 0.f));
}

__device__ __forceinline__ float tail_weight(float zT, float zD, const TailConsts& k) {
  const float dT = __fsub_rn(zT, k.mT);
  const float eT = ex2(__fmul_rn(dT, k.c_hi));
  if (!k.residual) return eT;
  const float dD = __fsub_rn(zD, k.mD);
  const float D = __fsub_rn(dT, dD);
  const float delta = __fadd_rn(__fmaf_rn(D, k.c_hi, -k.lam_hi), __fmaf_rn(D, k.c_lo, -k.lam_lo));
  return __fmul_rn(eT, resid_factor(delta));
}

// The same weights for an element pair with float2 arithmetic on register
// pairs: every operation rounds exactly as the scalar version above.
__device__ __forceinline__ float2 tail_weight2(float2 zT, float2 zD, const TailConsts& k) {
  const float2 dT = __fadd2_rn(zT, make_float2(-k.mT, -k.mT));
  const float2 aT = __fmul2_rn(dT, make_float2(k.c_hi, k.c_hi));
  const float2 eT = make_float2(ex2(aT.x), ex2(aT.y));
  if (!k.residual) return eT;
  const float2 dD = __fadd2_rn(zD, make_float2(-k.mD, -k.mD));
  const float2 D = __fadd2_rn(dT, __fmul2_rn(dD, make_float2(-1.f, -1.f)));
  const float2 delta = __fadd2_rn(__ffma2_rn(D, make_float2(k.c_hi, k.c_hi), make_float2(-k.lam_hi, -k.lam_hi)),
                                  __ffma2_rn(D, make_float2(k.c_lo, k.c_lo), make_float2(-k.lam_lo, -k.lam_lo)));
  return __fmul2_rn(eT, resid_factor2(delta));
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
      const float2 wp = tail_weight2(elem_pair2<E, VEC>(zt, p), elem_pair2<E, VEC>(zd, p), k);
      w[2 * p] = wp.x;
      w[2 * p + 1] = wp.y;
    }
  }
}

// Sum, in element order, of one lane's VEC weights.
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

// Argmax with the lowest index winning ties.
__device__ __forceinline__ void am_merge(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}
__device__ __forceinline__ void warp_am(float& v, int& i) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float v2 = __shfl_xor_sync(0xffffffffu, v, off);
    int i2 = __shfl_xor_sync(0xffffffffu, i, off);
    am_merge(v, i, v2, i2);
  }
}

// Butterfly sums: every lane adds the same two operands at every stage, so all
// lanes end with the same, run-to-run identical value.
__device__ __forceinline__ double warp_sum_f64(double x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// ---------------------------------------------------------------------------
// Inverse-CDF search over a run of masses (one warp)
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

// ---------------------------------------------------------------------------
// Philox-4x64-10 (Salmon et al., "Parallel Random Numbers: As Easy as 1, 2,
// 3", SC'11): ten rounds of two 64x64->128 multiplies with the key bumped by
// the two Weyl increments between rounds.  The verify step keys it with
// (seed, "SPECVERI") and counts with (sequence, position, stream, 0).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t philox_first_word(uint64_t seed, uint64_t seq, uint64_t pos,
                                                      uint64_t stream) {
  uint64_t c0 = seq, c1 = pos, c2 = stream, c3 = 0;
  uint64_t k0 = seed, k1 = 0x5350454356455249ull;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t a0 = 0xD2E7470EE14C6C93ull * c0;  // low halves
    const uint64_t a1 = 0xCA5A826395121157ull * c2;
    const uint64_t h0 = __umul64hi(0xD2E7470EE14C6C93ull, c0);
    const uint64_t h1 = __umul64hi(0xCA5A826395121157ull, c2);
    const uint64_t n0 = h1 ^ c1 ^ k0;
    const uint64_t n2 = h0 ^ c3 ^ k1;
    c0 = n0;
    c1 = a1;
    c2 = n2;
    c3 = a0;
    k0 += 0x9E3779B97F4A7C15ull;
    k1 += 0xBB67AE8584CAA73Bull;
  }
  return c0;
}

// u = (2 * (r >> 12) + 1) * 2^-53: an odd multiple of 2^-53 strictly inside
// (0, 1), exact in fp64 (the top 52 bits of r: a token of probability p is
// drawn with probability p to within 2^-52).
__device__ __forceinline__ double uniform_draw(uint64_t seed, uint64_t seq, uint64_t pos,
                                               uint64_t stream) {
  uint64_t r = philox_first_word(seed, seq, pos, stream);
  return (double)(2 * (r >> 12) + 1) * 0x1.0p-53;
}

}  // namespace sv
