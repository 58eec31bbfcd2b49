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

constexpr unsigned kSpinLimit = 1u << 22; // bounded waits: about 0.5 s with 128 ns naps

// status bits OR-ed into the library's device status word
constexpr unsigned kStatusBadData = 1u;   // NaN / +inf logit, empty row, bad token or parent
constexpr unsigned kStatusTimeout = 2u;   // a bounded wait ran out (should never happen)

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// 2^x with the MUFU unit (ex2.approx, denormal results flushed to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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
// widened to fp32 when used; this halves the registers a bf16 batch needs.
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

// Coherent (L1-bypassing) loads of workspace values written by other CTAs.
__device__ __forceinline__ float2 ldcg_f2(const float2* p) { return __ldcg(p); }
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
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

// Butterfly merge of (m, s) across the 32 lanes; every lane ends with the total.
__device__ __forceinline__ void warp_ms(float& m, float& s, float c) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    float s2 = __shfl_xor_sync(0xffffffffu, s, off);
    ms_merge(m, s, m2, s2, c);
  }
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

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
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

// u = (2 * (r >> 41) + 1) * 2^-24: an odd multiple of 2^-24 strictly inside (0, 1),
// exact in fp32 and fp64.
__device__ __forceinline__ double uniform_draw(uint64_t seed, uint64_t seq, uint64_t pos,
                                               uint64_t stream) {
  uint64_t r = philox_first_word(seed, seq, pos, stream);
  return (double)(2 * (r >> 41) + 1) * 0x1.0p-24;
}

}  // namespace sv
