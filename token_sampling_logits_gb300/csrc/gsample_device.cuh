// Device building blocks of the gsample kernels (sm_103a).
//
// Philox4x32-10 follows Salmon, Moraes, Dror and Shaw, "Parallel Random
// Numbers: As Easy as 1, 2, 3" (SC'11), section 3. The Gumbel transform and the
// argmax follow "Softmax-free GPU sampling: Gumbel-max categorical sampling
// kernel" (lablup/mlxcel issue #900), Background: score = logits/T + g with
// g = -log(-log u), one index-carrying max per row.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace gsample {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

// Per-row cross-CTA merge state (16 bytes). `key` holds the best packed
// (score, index) seen so far; `ticket` counts CTAs that finished the row. The
// last CTA of a row writes the result and zeroes both, so a workspace is left
// clean after every launch.
struct WsRow {
  unsigned long long key;
  unsigned int ticket;
  unsigned int reserved;
};
static_assert(sizeof(WsRow) == 16, "workspace row is 16 bytes");

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon et al. 2011): two 32x32->64 multiplies per round with
// the paper's 4x32 multipliers, a Weyl-sequence key schedule (golden ratio and
// sqrt(3)-1 in 32-bit fixed point), ten rounds.
// ---------------------------------------------------------------------------
constexpr uint32_t kPhiloxM0 = 0xD2511F53u;
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const unsigned long long p0 = (unsigned long long)kPhiloxM0 * c.x;
    const unsigned long long p1 = (unsigned long long)kPhiloxM1 * c.z;
    c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k0, (uint32_t)p1,
                   (uint32_t)(p0 >> 32) ^ c.w ^ k1, (uint32_t)p0);
    k0 += kPhiloxW0;  // bumping after the last round is harmless
    k1 += kPhiloxW1;
  }
  return c;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int w) {
  return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}

// ---------------------------------------------------------------------------
// Uniform and Gumbel. u = ((r >> 9) + 0.5) * 2^-23 = (2k + 1) * 2^-24 with
// k = r >> 9: it is formed exactly as (1 + k*2^-23) - (1 - 2^-24), both terms
// within a factor of two of each other, so the subtraction is exact.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float uniform_open(uint32_t r) {
  return __uint_as_float(0x3F800000u | (r >> 9)) - __uint_as_float(0x3F7FFFFFu);
}

// g = -log(-log u). u is exact and logf is accurate to an ulp over its whole
// range, so -logf(u) keeps full relative precision even next to u = 1.
__device__ __forceinline__ float gumbel_of_word(uint32_t r) {
  return -logf(-logf(uniform_open(r)));
}

// Upper bound on g(r) from integer/bit operations only. With v = 1 - u (also
// exact, the same construction on ~r): -log u >= v, so g <= -ln v; and writing
// v = 2^e (1 + f), -log2 v = -e - log2(1 + f) <= -e - f, which is
// (bits(1.0f) - bits(v)) / 2^23. Hence g <= (bits(1) - bits(v)) * ln2 / 2^23.
__device__ __forceinline__ float gumbel_bound_of_word(uint32_t r) {
  const float v = uniform_open(~r);
  const uint32_t d = 0x3F800000u - __float_as_uint(v);
  return __uint2float_rn(d) * (0.69314718f / 8388608.0f);
}

// Largest binary32 Gumbel value the kernels can produce is 16.6355 (at
// u = 1 - 2^-24); pruning uses a slightly larger constant.
constexpr float kGumbelMax = 16.64f;

// ---------------------------------------------------------------------------
// Packed ordered keys: high word = an order-preserving image of the binary32
// score, low word = 0xFFFFFFFF - index, so an unsigned 64-bit max picks the
// largest score and, among equal scores, the smallest index. 0 means "empty"
// (no real score maps to 0).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ordered_bits(float s) {
  if (s == 0.0f) s = 0.0f;  // -0 and +0 compare equal, so give them one key
  const uint32_t b = __float_as_uint(s);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float score_of_key(unsigned long long key) {
  if (key == 0ull) return -INFINITY;
  const uint32_t o = (uint32_t)(key >> 32);
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

__device__ __forceinline__ unsigned long long pack_key(float s, int32_t idx) {
  return ((unsigned long long)ordered_bits(s) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}

__device__ __forceinline__ int64_t index_of_key(unsigned long long key) {
  return key == 0ull ? -1 : (int64_t)(0xFFFFFFFFu - (uint32_t)key);
}

// (s, i) is better than (bs, bi): larger score, or equal score and lower index.
// -inf is never a candidate.
__device__ __forceinline__ void take_better(float s, int32_t i, float& bs, int32_t& bi) {
  if (s > -INFINITY && (s > bs || (s == bs && i < bi))) {
    bs = s;
    bi = i;
  }
}

__device__ __forceinline__ void warp_argmax(float& s, int32_t& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float os = __shfl_xor_sync(0xFFFFFFFFu, s, o);
    const int32_t oi = __shfl_xor_sync(0xFFFFFFFFu, i, o);
    if (os > s || (os == s && oi < i)) {
      s = os;
      i = oi;
    }
  }
}

// ---------------------------------------------------------------------------
// Exact pruning. Given L, the exact score of some element of the row, an element
// whose score cannot reach L cannot be the row's argmax. For x < thr_x the
// binary32 score fl(fl(x/T) + g) < L holds for every g <= kGumbelMax: the margin
// 1e-3 * (1 + |L|) dwarfs the few-ulp rounding of the threshold arithmetic. The
// second test uses the per-element bound on g once the Philox word is known;
// its extra 0.01 covers the binary32 error of g itself (a few 1e-6).
// ---------------------------------------------------------------------------
struct Prune {
  float thr_x;  // skip x < thr_x (NaN never passes)
  float lm;     // skip when x * (1/T) + bound(g) < lm
  bool use_bound;
};

__device__ __forceinline__ Prune make_prune(float L, float T) {
  Prune p;
  if (L == INFINITY) {  // only +inf logits can still win
    p.thr_x = INFINITY;
    p.lm = -INFINITY;
    p.use_bound = false;
  } else if (!(L > -INFINITY) || !(T >= 1e-20f && T <= 1e20f)) {
    p.thr_x = -INFINITY;  // nothing known yet, or an extreme temperature: no pruning
    p.lm = -INFINITY;
    p.use_bound = false;
  } else {
    const float margin = 1e-3f * (1.0f + fabsf(L));
    p.thr_x = (L - kGumbelMax - margin) * T;
    p.lm = L - margin - 0.01f;
    p.use_bound = true;
  }
  return p;
}

// ---------------------------------------------------------------------------
// Loads. Logit rows are read exactly once, so the 128-bit loads go through the
// non-coherent path, skip L1 allocation and carry an L2 evict-first policy.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* ptr, uint64_t pol) {
  uint4 v;
  asm volatile(
      "ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(ptr), "l"(pol));
  return v;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

__device__ __forceinline__ float f16_bits_to_f32(uint32_t h) {
  return __half2float(__ushort_as_half((unsigned short)h));
}

}  // namespace gsample
