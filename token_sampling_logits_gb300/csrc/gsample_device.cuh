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

// Per-row merge state (16 bytes). `key` holds the best packed (score, index)
// merged so far; `ticket` counts the units of the row already finished (the
// sampler) or the CTAs that finished it (the HLG kernel); `hint` holds the
// order-preserving bits of the best score any warp has published for pruning.
// Whoever completes a row writes its result and zeroes all three, so a
// workspace is left clean after every launch.
struct WsRow {
  unsigned long long key;
  unsigned int ticket;
  unsigned int hint;
};
static_assert(sizeof(WsRow) == 16, "workspace row is 16 bytes");

// Programmatic dependent launch. Every kernel of the library is launched with
// programmatic stream serialization, so its CTAs may be scheduled while the
// previous kernel of the stream drains. Each kernel first waits for that
// kernel to complete and its memory to be visible (griddepcontrol.wait),
// before touching global memory, then lets the next kernel of the stream be
// scheduled early in turn. A kernel that follows on the same stream with the
// same launch attribute must likewise wait before reading the indices.
__device__ __forceinline__ void pdl_wait_then_release() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

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

// The blocks of one row share counter words 1..3 (row, lo32(offset),
// hi32(offset)) and the key, so in the first two rounds one of the two
// multiplies does not depend on the group index: it is done once per row.
//   round 0: (h0, l0) = M0 * g          ->  (u1, L1, h0 ^ u2, l0)
//   round 1: (h1, l1) = M1 * (h0 ^ u2)  ->  (h1 ^ u3, l1, l0 ^ u4, w2)
// with (H1, L1) = M1 * off0, u1 = H1 ^ row ^ k0, u2 = off1 ^ k1,
// u3 = L1 ^ (k0 + W0), (H0, w2) = M0 * u1, u4 = H0 ^ (k1 + W1).
// Rounds 2..9 then run as usual. The result equals philox4x32_10 on
// (g, row, off0, off1).
struct PhiloxRow {
  uint32_t k0, k1, u2, u3, u4, w2;
};

__device__ __forceinline__ PhiloxRow philox_row(uint32_t row, uint32_t off0, uint32_t off1,
                                                uint32_t k0, uint32_t k1) {
  const unsigned long long p1 = (unsigned long long)kPhiloxM1 * off0;
  const uint32_t u1 = (uint32_t)(p1 >> 32) ^ row ^ k0;
  const unsigned long long p0 = (unsigned long long)kPhiloxM0 * u1;
  PhiloxRow r;
  r.k0 = k0;
  r.k1 = k1;
  r.u2 = off1 ^ k1;
  r.u3 = (uint32_t)p1 ^ (k0 + kPhiloxW0);
  r.u4 = (uint32_t)(p0 >> 32) ^ (k1 + kPhiloxW1);
  r.w2 = (uint32_t)p0;
  return r;
}

// N blocks of a row (groups g[0..N-1]), interleaved round by round.
template <int N>
__device__ __forceinline__ void philox_row_xn(const uint32_t (&g)[N], const PhiloxRow& pr,
                                              uint4 (&out)[N]) {
  uint4 c[N];
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const unsigned long long a = (unsigned long long)kPhiloxM0 * g[j];
    const uint32_t z = (uint32_t)(a >> 32) ^ pr.u2;
    const unsigned long long b = (unsigned long long)kPhiloxM1 * z;
    c[j] = make_uint4((uint32_t)(b >> 32) ^ pr.u3, (uint32_t)b, (uint32_t)a ^ pr.u4, pr.w2);
  }
  uint32_t k0 = pr.k0 + 2u * kPhiloxW0, k1 = pr.k1 + 2u * kPhiloxW1;
#pragma unroll
  for (int round = 2; round < 10; ++round) {
#pragma unroll
    for (int j = 0; j < N; ++j) {
      const unsigned long long p0 = (unsigned long long)kPhiloxM0 * c[j].x;
      const unsigned long long p1 = (unsigned long long)kPhiloxM1 * c[j].z;
      c[j] = make_uint4((uint32_t)(p1 >> 32) ^ c[j].y ^ k0, (uint32_t)p1,
                        (uint32_t)(p0 >> 32) ^ c[j].w ^ k1, (uint32_t)p0);
    }
    k0 += kPhiloxW0;
    k1 += kPhiloxW1;
  }
#pragma unroll
  for (int j = 0; j < N; ++j) out[j] = c[j];
}

__device__ __forceinline__ void philox_row_x4(const uint32_t (&g)[4], const PhiloxRow& pr,
                                              uint4 (&out)[4]) {
  philox_row_xn<4>(g, pr, out);
}

__device__ __forceinline__ uint4 philox_row_1(uint32_t g, const PhiloxRow& pr) {
  const unsigned long long a = (unsigned long long)kPhiloxM0 * g;
  const uint32_t z = (uint32_t)(a >> 32) ^ pr.u2;
  const unsigned long long b = (unsigned long long)kPhiloxM1 * z;
  uint4 c = make_uint4((uint32_t)(b >> 32) ^ pr.u3, (uint32_t)b, (uint32_t)a ^ pr.u4, pr.w2);
  uint32_t k0 = pr.k0 + 2u * kPhiloxW0, k1 = pr.k1 + 2u * kPhiloxW1;
#pragma unroll
  for (int round = 2; round < 10; ++round) {
    const unsigned long long p0 = (unsigned long long)kPhiloxM0 * c.x;
    const unsigned long long p1 = (unsigned long long)kPhiloxM1 * c.z;
    c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k0, (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ k1,
                   (uint32_t)p0);
    k0 += kPhiloxW0;
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

// The bound on g that the pruning relies on: -log u >= 1 - u = v, hence
// g = -log(-log u) <= -log v (v is formed exactly, like u, from ~r).
__device__ __forceinline__ float gumbel_bound_of_word(uint32_t r) {
  return -logf(uniform_open(~r));
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

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = w > v ? w : v;
  }
  return v;
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

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Once the Philox word w of an element is known: can x/T + g(w) still reach L?
// Because -log u >= 1 - u = v, g = -log(-log u) <= -log v, so reaching L needs
// v <= exp(x/T - L). The pruning margins are folded into lm; the test is
// evaluated as v <= 2^(x*a + c) with a = log2(e)/T and c = -lm*log2(e). The
// approximate exponential errs by about 1e-7 relative, far inside the e^0.01
// slack of lm. NaN or -inf logits never pass; +inf always does. Without a finite
// L (use_bound false) the caller falls back to x >= thr_x.
struct ReachTest {
  float a, c;
};

__device__ __forceinline__ ReachTest make_reach(const Prune& p, float rT) {
  constexpr float kLog2e = 1.4426950408889634f;
  return ReachTest{rT * kLog2e, -p.lm * kLog2e};
}

__device__ __forceinline__ bool may_reach(float x, uint32_t w, const ReachTest& t) {
  return uniform_open(~w) <= ex2_approx(fmaf(x, t.a, t.c));
}

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
// Exact scores of the sampled path: s = x / T (IEEE division) + g(word).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float exact_score(float x, uint32_t word, float T) {
  return x == INFINITY ? INFINITY : __fdiv_rn(x, T) + gumbel_of_word(word);
}

// Rare path: the element-wise test, then the exact score.
__device__ __forceinline__ void score_group(uint32_t gid, float x0, float x1, float x2, float x3,
                                         uint4 w, Prune pr, ReachTest rt, float T, float* bs_io,
                                         int32_t* bi_io) {
  const float x[4] = {x0, x1, x2, x3};
  float bs = *bs_io;
  int32_t bi = *bi_io;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t wd = word_of(w, t);
    const bool need = pr.use_bound ? may_reach(x[t], wd, rt) : (x[t] >= pr.thr_x);
    if (need) take_better(exact_score(x[t], wd, T), (int32_t)(4 * gid + t), bs, bi);
  }
  *bs_io = bs;
  *bi_io = bi;
}

// The group test as an integer threshold on the group's largest Philox word,
// computed from its largest logit alone, before the block is known (v = 1 - u
// only shrinks as the word grows, so one word covers all four elements).
// may_reach(x, w) is v = (2k+1)*2^-24 <= e with k = 2^23 - 1 - (w >> 9) and
// e = 2^(x*a + c). That holds iff w >= ceil(2^23 - 0.5 - e*2^23) * 512, and
// that threshold is at least 2^32 - 256 - e*2^32. The fma below rounds once,
// by at most 128 at these magnitudes, so truncating 2^32 - 1024 - e*2^32
// (saturated to [0, 2^32 - 1]) never exceeds the exact threshold: every word
// that passes may_reach passes this test, and only words within about 1200 of
// the boundary pass this one alone. The exact pass tests every element again.
// +inf logits give threshold 0 (always pass). So does a NaN group maximum,
// which needs all four logits NaN: such a group then goes through the exact
// pass, which rejects it. Only the dense path meets one: the compacted and
// cluster paths take groups with xm >= thr_x, and a tile whose groups are all
// NaN fails the tile test. Without a finite L the test is x >= thr_x.
__device__ __forceinline__ uint32_t word_threshold(float xm, const Prune& pr, const ReachTest& rt) {
  const float e = pr.use_bound ? ex2_approx(fmaf(xm, rt.a, rt.c))
                               : (xm >= pr.thr_x ? INFINITY : 0.0f);
  uint32_t w;
  asm("cvt.rzi.sat.u32.f32 %0, %1;" : "=r"(w) : "f"(fmaf(-e, 4294967296.0f, 4294966272.0f)));
  return w;
}

__device__ __forceinline__ uint32_t max_word(const uint4& w) {
  return max(max(w.x, w.y), max(w.z, w.w));
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

// ---------------------------------------------------------------------------
// Shared-memory and cp.async primitives, and 16-bit widening (one definition
// for every kernel of the library).
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ float half_to_f32(uint32_t h) {
  return DT == 1 ? bf16_bits_to_f32(h) : f16_bits_to_f32(h);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "l"(pol)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

}  // namespace gsample
