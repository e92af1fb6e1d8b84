// Top-k / top-p sampling on the Gumbel path: the follow-up that "Softmax-free
// GPU sampling: Gumbel-max categorical sampling kernel" (lablup/mlxcel issue
// #900, Background) names as "rejection-based top-k/top-p".
//
// The filter set K of a row is the first r candidates (logits that are neither
// NaN nor -inf) in the order (logit descending, index ascending), r the
// smaller of top_k and the nucleus size (the shortest prefix whose softmax
// mass reaches top_p). The sample is the Gumbel-max over K with the row's
// usual Philox noise: argmax over i in K of x_i / T + g_i.
//
// Rejection. The plain sampler's draw over the whole row is a proposal. When
// it lies in K it is also the argmax over K (the best of a superset that falls
// in the subset), so it stands. filter_row_kernel decides that from one pass
// over the row: the proposal's rank (candidates before it) against top_k, and
// the mass before it against top_p times the row's mass. A rejected proposal
// means K ends before it, so the same pass lists the candidates at or above
// the proposal in shared memory, and the row is resolved from that list: it
// is sorted into the order, K's length comes from top_k and the prefix sums
// of fixed-point masses, then the Gumbel-max over K. Rows whose list
// overflows are flagged in their workspace slot and resolved by
// filter_exact_kernel: K's last element by a radix select over the whole row
// in global memory (counts for top_k, fixed-point masses for top_p).
// Every path gives the same index: the argmax over K of the same scores.
#include <cstdint>

#include "gsample_internal.h"
#include "gsample_slice.cuh"

namespace gsample {
namespace {

using namespace slice;

#ifndef GSAMPLE_FILT_THREADS
#define GSAMPLE_FILT_THREADS 1024
#endif
constexpr int kFiltThreads = GSAMPLE_FILT_THREADS;
constexpr int kFiltWarps = kFiltThreads / 32;
constexpr float kLog2e = 1.4426950408889634f;
// Fixed-point masses of the exact path: e^((x - M) / T) in (0, 1] times 2^40.
// Integer sums are exact and order-free, so the selection is deterministic.

// Unit u of a row through the read-only cache (the exact path reads a row
// several times, so it keeps the default L2 policy); -inf past V.
template <int DT, bool VEC>
__device__ __forceinline__ uint4 unit_cached(const char* row, int32_t u, int32_t V) {
  constexpr int EPU = HCfg<DT, VEC>::kEPU;
  if constexpr (VEC) {
    if ((u + 1) * EPU <= V) return __ldg(reinterpret_cast<const uint4*>(row) + u);
  }
  return load_unit<DT, VEC>(row, u, V, 0ull);  // the padded plain-load path only
}

template <int DT>
__device__ __forceinline__ float elt_at(const char* row, int64_t i) {
  if constexpr (DT == 0) {
    return __ldg(reinterpret_cast<const float*>(row) + i);
  } else {
    return half_to_f32<DT>(__ldg(reinterpret_cast<const unsigned short*>(row) + i));
  }
}

// Every unit of a row, kInFlight of them per thread loaded before any is used,
// so that one CTA keeps enough bytes in flight. f(unit, u, valid) runs for
// every slot; the iteration count is the same for every lane of a warp (warp
// collectives may run inside f), and slots past the row have valid = false.
constexpr int kInFlight = 4;

template <int DT, bool VEC, typename F>
__device__ __forceinline__ void for_units(const char* row, int32_t NU, int32_t V, F&& f) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int32_t ub = warp * 32; ub < NU; ub += kInFlight * kFiltThreads) {
    uint4 r[kInFlight];
#pragma unroll
    for (int j = 0; j < kInFlight; ++j) {
      const int32_t u = ub + lane + j * kFiltThreads;
      r[j] = u < NU ? unit_cached<DT, VEC>(row, u, V) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < kInFlight; ++j) {
      const int32_t u = ub + lane + j * kFiltThreads;
      f(r[j], u, u < NU);
    }
  }
}

__device__ __forceinline__ bool is_candidate(float x) { return x > -INFINITY; }  // NaN: false

struct RowFilter {
  float T, p;
  int32_t k;
  bool k_on, p_on;
};

__device__ __forceinline__ RowFilter row_filter(const FilterParams& fp, int64_t b) {
  RowFilter f;
  f.T = fp.temperature[b];
  f.k = fp.top_k ? fp.top_k[b] : 0;
  f.p = fp.top_p ? fp.top_p[b] : 1.0f;
  f.k_on = f.k >= 1;
  f.p_on = f.p < 1.0f;  // NaN: off
  return f;
}

// Block-wide sums and maxima in a fixed order (warp butterflies, then warp 0
// over the warps' partials), so every launch rounds the same way.
template <typename Tv, typename Op>
__device__ __forceinline__ Tv block_reduce(Tv v, Op op, Tv* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  if (warp == 0) {
    Tv t = scratch[0];
    for (int i = 1; i < kFiltWarps; ++i) t = op(t, scratch[i]);
    if (lane == 0) scratch[0] = t;
  }
  __syncthreads();
  const Tv r = scratch[0];
  __syncthreads();
  return r;
}

struct AddF {
  __device__ float operator()(float a, float b) const { return a + b; }
};
struct AddU {
  __device__ unsigned operator()(unsigned a, unsigned b) const { return a + b; }
};
struct AddU64 {
  __device__ unsigned long long operator()(unsigned long long a, unsigned long long b) const {
    return a + b;
  }
};
struct MaxF {
  __device__ float operator()(float a, float b) const { return fmaxf(a, b); }
};

__device__ __forceinline__ unsigned long long fixed_mass(float x, float M, float a);

// ---------------------------------------------------------------------------
// One CTA per filtered row, one pass over it. It tests the proposal in
// out_idx[b]: its rank among the candidates against top_k, and the mass of
// the candidates before it against top_p times the row's mass (both relative
// to the proposal's own mass; an overflow only rejects). In the same pass it
// lists every candidate whose key is at least the proposal's in shared memory
// (kListCap entries). A rejected proposal means K ends before it, so K lies
// in that list, and the row is resolved from it: the list sorted into the
// order, K's length from top_k and the prefix sums of fixed-point masses
// relative to the row maximum, then the Gumbel-max over K. A row whose list overflowed, or
// whose targets the list cannot reach (a binary32 rejection at the nucleus
// edge), is flagged in its workspace slot for filter_exact_kernel.
// ---------------------------------------------------------------------------
#ifndef GSAMPLE_FILT_LIST
#define GSAMPLE_FILT_LIST 16384
#endif
constexpr int kListCap = GSAMPLE_FILT_LIST;  // entries (key, index) of 8 bytes: 128 KB
static_assert((kListCap & (kListCap - 1)) == 0, "the list is sorted in place: a power of two");

template <int DT, bool VEC>
__global__ void __launch_bounds__(kFiltThreads, 1) filter_row_kernel(const FilterParams fp) {
  pdl_wait_then_release();
  extern __shared__ __align__(16) uint2 s_list[];
  __shared__ float sf[kFiltWarps];
  __shared__ unsigned su[kFiltWarps];
  __shared__ unsigned long long sl[kFiltWarps];
  __shared__ unsigned s_n;
  __shared__ unsigned long long s_best[kFiltWarps];
  const int64_t b = blockIdx.x;
  if (b >= fp.B) return;
  const RowFilter f = row_filter(fp, b);
  if (!(f.T > 0.0f) || !(f.k_on || f.p_on)) return;  // greedy or unfiltered: stands
  const int64_t w = fp.out_idx[b];
  if (w < 0) return;  // no candidate at all
  const char* row = fp.logits + b * fp.ld_bytes;
  const float xw = elt_at<DT>(row, w);
  if (xw == INFINITY) return;  // the first +inf entry heads the order
  constexpr int EPU = HCfg<DT, VEC>::kEPU;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t key_w = ordered_bits(xw);
  const float a = kLog2e / f.T;
  if (threadIdx.x == 0) s_n = 0u;
  __syncthreads();

  unsigned cnt = 0, n = 0;
  float s_low = 0.0f, s_high = 0.0f, mb = 0.0f;
  for_units<DT, VEC>(row, fp.units_per_row, fp.V, [&](const uint4& r, int32_t u, bool valid) {
#pragma unroll
    for (int e = 0; e < EPU; ++e) {
      const float x = valid ? elt<DT, VEC>(r, e) : -INFINITY;
      const bool cand = is_candidate(x);
      const uint32_t key = ordered_bits(x);
      const uint32_t i = (uint32_t)(u * EPU + e);
      const bool high = cand && key >= key_w;
      // list the candidates at or above the proposal (one atomic per warp)
      const unsigned hm = __ballot_sync(0xFFFFFFFFu, high);
      if (hm) {
        unsigned base = 0;
        if (lane == __ffs(hm) - 1) base = atomicAdd(&s_n, (unsigned)__popc(hm));
        base = __shfl_sync(0xFFFFFFFFu, base, __ffs(hm) - 1);
        const unsigned pos = base + __popc(hm & ((1u << lane) - 1u));
        if (high && pos < (unsigned)kListCap) s_list[pos] = make_uint2(key, i);
      }
      if (!cand) continue;
      ++n;
      const bool before = x > xw || (x == xw && i < (uint32_t)w);
      cnt += before ? 1u : 0u;
      if (f.p_on) {
        // the acceptance test sums in binary32; its rounding only matters at
        // the nucleus edge, where the parity rule exempts the row
        const float m = ex2_approx((x - xw) * a);
        if (high) {
          s_high += m;
          mb += before ? m : 0.0f;
        } else {
          s_low += m;
        }
      }
    }
  });
  cnt = block_reduce(cnt, AddU(), su);
  n = block_reduce(n, AddU(), su);
  if (f.p_on) {
    s_low = block_reduce(s_low, AddF(), sf);
    s_high = block_reduce(s_high, AddF(), sf);
    mb = block_reduce(mb, AddF(), sf);
  }
  bool ok = !f.k_on || cnt < (unsigned)f.k;
  if (f.p_on) ok = ok && (f.p <= 0.0f ? cnt == 0u : mb < f.p * (s_low + s_high));
  if (ok) return;  // the proposal is the argmax over K
  const unsigned n_list = s_n;
  if (n_list > (unsigned)kListCap) {
    if (threadIdx.x == 0) fp.ws[b].hint = 1u;  // resolved by filter_exact_kernel
    return;
  }

  // Sort the list into the order K is a prefix of: key descending, index
  // ascending (a bitonic sort of the composite (~key, index), padded to a
  // power of two with entries that sort last).
  int npad = 1;
  while (npad < (int)n_list) npad <<= 1;
  for (int j = (int)n_list + threadIdx.x; j < npad; j += kFiltThreads)
    s_list[j] = make_uint2(0u, 0xFFFFFFFFu);
  __syncthreads();
  for (int kk = 2; kk <= npad; kk <<= 1) {
    for (int jj = kk >> 1; jj > 0; jj >>= 1) {
      for (int i = threadIdx.x; i < npad; i += kFiltThreads) {
        const int l = i ^ jj;
        if (l <= i) continue;
        const uint2 x0 = s_list[i], x1 = s_list[l];
        const unsigned long long c0 = ((unsigned long long)~x0.x << 32) | x0.y;
        const unsigned long long c1 = ((unsigned long long)~x1.x << 32) | x1.y;
        if ((c0 > c1) == ((i & kk) == 0)) {
          s_list[i] = x1;
          s_list[l] = x0;
        }
      }
      __syncthreads();
    }
  }
  const float M = score_of_key((unsigned long long)s_list[0].x << 32 | 1ull);  // row maximum

  // K = the first r listed entries, r = min(r_k, r_p): r_p from the prefix
  // sums of the fixed-point masses (2^-40 units, relative to the maximum).
  unsigned r = f.k_on && (unsigned)f.k < n ? (unsigned)f.k : n;
  if (f.p_on && f.p <= 0.0f) r = 1u;
  if (f.p_on && f.p > 0.0f) {
    const int chunk = ((int)n_list + kFiltThreads - 1) / kFiltThreads;
    const int j0 = threadIdx.x * chunk, j1 = min(j0 + chunk, (int)n_list);
    unsigned long long mine = 0;
    for (int j = j0; j < j1; ++j)
      mine += fixed_mass(score_of_key((unsigned long long)s_list[j].x << 32 | 1ull), M, a);
    // the candidates below the proposal, summed relative to it in binary32
    unsigned long long S = block_reduce(mine, AddU64(), sl);
    S += __float2ull_rn(s_low * exp2f((xw - M) * a) * 1099511627776.0f);
    const unsigned long long target = (unsigned long long)ceil((double)f.p * (double)S);
    unsigned long long incl = mine;  // exclusive scan of the chunks' sums
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) s_best[warp] = incl;
    if (threadIdx.x == 0) s_n = 0xFFFFFFFFu;
    __syncthreads();
    unsigned long long cum = incl - mine;
    for (int i = 0; i < warp; ++i) cum += s_best[i];
    for (int j = j0; j < j1; ++j) {
      const unsigned long long c =
          cum + fixed_mass(score_of_key((unsigned long long)s_list[j].x << 32 | 1ull), M, a);
      if (cum < target && c >= target) s_n = (unsigned)j + 1u;
      cum = c;
    }
    __syncthreads();
    const unsigned r_p = s_n;
    if (r_p == 0xFFFFFFFFu && r > n_list) {
      // K reaches past the proposal after all (a binary32 rejection at the
      // nucleus edge): the global path decides
      if (threadIdx.x == 0) fp.ws[b].hint = 1u;
      return;
    }
    if (r_p < r) r = r_p;
  }
  if (r > n_list) {  // cannot happen after a rejection; decided globally to be safe
    if (threadIdx.x == 0) fp.ws[b].hint = 1u;
    return;
  }

  // The Gumbel-max over K.
  const uint64_t sd = fp.seed[b], of = fp.offset[b];
  const PhiloxRow ph =
      philox_row((uint32_t)b, (uint32_t)of, (uint32_t)(of >> 32), (uint32_t)sd, (uint32_t)(sd >> 32));
  float bs = -INFINITY;
  int32_t bi = INT32_MAX;
  for (int j = threadIdx.x; j < (int)r; j += kFiltThreads) {
    const uint32_t key = s_list[j].x, i = s_list[j].y;
    const float x = score_of_key((unsigned long long)key << 32 | 1ull);
    const uint4 blk = philox_row_1(i >> 2, ph);
    take_better(exact_score(x, word_of(blk, i & 3u), f.T), (int32_t)i, bs, bi);
  }
  warp_argmax(bs, bi);
  if (lane == 0) s_best[warp] = bi != INT32_MAX ? pack_key(bs, bi) : 0ull;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long best = 0ull;
    for (int i = 0; i < kFiltWarps; ++i) best = s_best[i] > best ? s_best[i] : best;
    fp.out_idx[b] = index_of_key(best);
  }
}

// ---------------------------------------------------------------------------
// The exact path for a rejected row: K's last element by radix select, then
// the Gumbel-max over K. One CTA per row; the row is read from L2 after the
// first pass.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long fixed_mass(float x, float M, float a) {
  // e^((x - M) / T) in (0, 1], scaled by 2^40 (exact: a power of two) and
  // converted exactly: the fixed-point value keeps binary32's 24 bits.
  return __float2ull_rn(exp2f((x - M) * a) * 1099511627776.0f);
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kFiltThreads, 1) filter_exact_kernel(const FilterParams fp) {
  pdl_wait_then_release();
  __shared__ unsigned s_cnt[256];
  __shared__ unsigned long long s_mass[256];
  __shared__ float sf[kFiltWarps];
  __shared__ unsigned su[kFiltWarps];
  __shared__ unsigned long long sl[kFiltWarps];
  __shared__ uint32_t s_sel[3];  // the chosen digit and count before it; then the tie bound
  __shared__ unsigned long long s_best[kFiltWarps];
  const int64_t b = blockIdx.x;
  if (b >= fp.B) return;
  if (fp.ws[b].hint == 0u) return;  // the proposal stood
  constexpr int EPU = HCfg<DT, VEC>::kEPU;
  const RowFilter f = row_filter(fp, b);
  const char* row = fp.logits + b * fp.ld_bytes;
  const int32_t NU = fp.units_per_row;
  const int32_t V = fp.V;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // Row maximum and candidate count.
  float M = -INFINITY;
  unsigned n = 0;
  for_units<DT, VEC>(row, NU, V, [&](const uint4& r, int32_t, bool valid) {
    if (!valid) return;
#pragma unroll
    for (int e = 0; e < EPU; ++e) {
      const float x = elt<DT, VEC>(r, e);
      if (is_candidate(x)) {
        M = fmaxf(M, x);
        ++n;
      }
    }
  });
  M = block_reduce(M, MaxF(), sf);
  n = block_reduce(n, AddU(), su);
  const float a = kLog2e / f.T;

  // Targets: the r_k-th candidate, or the first whose cumulative mass reaches
  // top_p * S (in 2^-40 units), whichever comes first.
  unsigned k_target = f.k_on && (unsigned)f.k < n ? (unsigned)f.k : n;
  bool p_on = f.p_on;
  if (p_on && f.p <= 0.0f) {
    k_target = 1;
    p_on = false;
  }
  long long m_target = 0;
  if (p_on) {
    unsigned long long S = 0;
    for_units<DT, VEC>(row, NU, V, [&](const uint4& r, int32_t, bool valid) {
      if (!valid) return;
#pragma unroll
      for (int e = 0; e < EPU; ++e) {
        const float x = elt<DT, VEC>(r, e);
        if (is_candidate(x)) S += fixed_mass(x, M, a);
      }
    });
    S = block_reduce(S, AddU64(), sl);
    m_target = (long long)ceil((double)f.p * (double)S);
  }

  // The proposal was rejected, so K's last element comes before it in the
  // order: only candidates with a key at least the proposal's take part in the
  // selection (few, so the histograms see little contention). Should the
  // check's binary32 test have rejected a proposal that lies in K after all,
  // those candidates cannot reach the targets, and the selection runs again
  // over every candidate.
  uint32_t floor_key = ordered_bits(elt_at<DT>(row, fp.out_idx[b]));
  uint32_t prefix = 0;
  unsigned k_rem = k_target;
  long long m_rem = m_target;
  for (int attempt = 0; attempt < 2; ++attempt) {
    prefix = 0;
    uint32_t pmask = 0;
    k_rem = k_target;
    m_rem = m_target;
    bool reached = true;
    // Radix select on the order-preserving keys, eight bits at a time from
    // the top; larger keys come first.
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = threadIdx.x; i < 256; i += kFiltThreads) {
        s_cnt[i] = 0u;
        s_mass[i] = 0ull;
      }
      __syncthreads();
      for_units<DT, VEC>(row, NU, V, [&](const uint4& r, int32_t, bool valid) {
#pragma unroll
        for (int e = 0; e < EPU; ++e) {
          const float x = valid ? elt<DT, VEC>(r, e) : -INFINITY;
          const uint32_t key = ordered_bits(x);
          const bool in = is_candidate(x) && key >= floor_key && (key & pmask) == prefix;
          const uint32_t d = in ? (key >> shift) & 0xFFu : 0x100u;
          // one atomic per distinct digit of the warp for the counts
          const unsigned peers = __match_any_sync(0xFFFFFFFFu, d);
          if (in && lane == __ffs(peers) - 1) atomicAdd(&s_cnt[d], (unsigned)__popc(peers));
          if (in && p_on) atomicAdd(&s_mass[d], fixed_mass(x, M, a));
        }
      });
      __syncthreads();
      if (threadIdx.x == 0) {
        unsigned c = 0;
        long long m = 0;
        int d = 255;
        for (; d >= 0; --d) {
          if (s_cnt[d] == 0u) continue;
          if (c + s_cnt[d] >= k_rem || (p_on && m + (long long)s_mass[d] >= m_rem)) break;
          c += s_cnt[d];
          m += (long long)s_mass[d];
        }
        s_sel[0] = d < 0 ? 0xFFFFFFFFu : (uint32_t)d;  // none: the targets lie further on
        s_sel[1] = c;
        sl[0] = (unsigned long long)m;
      }
      __syncthreads();
      const uint32_t d = s_sel[0];
      const unsigned c_before = s_sel[1];
      const long long m_before = (long long)sl[0];
      __syncthreads();
      if (d == 0xFFFFFFFFu) {
        reached = false;
        break;
      }
      k_rem -= c_before;
      m_rem -= m_before;
      prefix |= d << shift;
      pmask |= 0xFFu << shift;
    }
    if (reached) break;
    floor_key = 0u;  // every candidate
  }
  const uint32_t key_b = prefix;

  // How many of the entries with key key_b (all of equal mass) K takes, in
  // index order: n_take; then the index of the n_take-th of them.
  unsigned n_take = k_rem;
  if (p_on) {
    const float xb = score_of_key((unsigned long long)key_b << 32 | 1ull);
    const long long eb = (long long)fixed_mass(xb, M, a);
    const unsigned np = m_rem <= 0 ? 1u : (eb > 0 ? (unsigned)((m_rem + eb - 1) / eb) : 0xFFFFFFFFu);
    n_take = np < n_take ? np : n_take;
  }
  if (n_take < 1u) n_take = 1u;
  unsigned ties = 0;
  for_units<DT, VEC>(row, NU, V, [&](const uint4& r, int32_t, bool valid) {
    if (!valid) return;
#pragma unroll
    for (int e = 0; e < EPU; ++e) {
      const float x = elt<DT, VEC>(r, e);
      ties += (is_candidate(x) && ordered_bits(x) == key_b) ? 1u : 0u;
    }
  });
  ties = block_reduce(ties, AddU(), su);
  uint32_t idx_b = 0xFFFFFFFFu;  // all entries with key key_b are in K
  if (n_take < ties) {
    // Rare (several entries share K's last key): the n_take-th of them in
    // index order, each thread counting a contiguous chunk of the row.
    const int32_t chunk = (NU + kFiltThreads - 1) / kFiltThreads;
    const int32_t u0 = threadIdx.x * chunk, u1 = min(u0 + chunk, NU);
    unsigned mine = 0;  // entries with key key_b in this thread's chunk
    for (int32_t u = u0; u < u1; ++u) {
      const uint4 r = unit_cached<DT, VEC>(row, u, V);
#pragma unroll
      for (int e = 0; e < EPU; ++e) {
        const float x = elt<DT, VEC>(r, e);
        mine += (is_candidate(x) && ordered_bits(x) == key_b) ? 1u : 0u;
      }
    }
    unsigned incl = mine;  // exclusive scan: warp scan, then the warps' totals
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) su[warp] = incl;
    __syncthreads();
    unsigned before = incl - mine;
    for (int i = 0; i < warp; ++i) before += su[i];
    if (before < n_take && n_take <= before + mine) {
      unsigned seen = before;
      bool found = false;
      for (int32_t u = u0; u < u1 && !found; ++u) {
        const uint4 r = unit_cached<DT, VEC>(row, u, V);
        for (int e = 0; e < EPU; ++e) {
          const float x = elt<DT, VEC>(r, e);
          if (is_candidate(x) && ordered_bits(x) == key_b && ++seen == n_take) {
            s_sel[2] = (uint32_t)(u * EPU + e);
            found = true;
            break;
          }
        }
      }
    }
    __syncthreads();
    idx_b = s_sel[2];
  }

  // The Gumbel-max over K: a Philox block per group holding a member of K.
  const uint64_t sd = fp.seed[b], of = fp.offset[b];
  const PhiloxRow ph =
      philox_row((uint32_t)b, (uint32_t)of, (uint32_t)(of >> 32), (uint32_t)sd, (uint32_t)(sd >> 32));
  float bs = -INFINITY;
  int32_t bi = INT32_MAX;
  for_units<DT, VEC>(row, NU, V, [&](const uint4& r, int32_t u, bool valid) {
    if (!valid) return;
#pragma unroll
    for (int g = 0; g < EPU / 4; ++g) {
      bool any = false;
      bool in[4];
      float xs[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int e = g * 4 + t;
        xs[t] = elt<DT, VEC>(r, e);
        const uint32_t i = (uint32_t)(u * EPU + e);
        const uint32_t key = ordered_bits(xs[t]);
        in[t] = is_candidate(xs[t]) && (key > key_b || (key == key_b && i <= idx_b));
        any |= in[t];
      }
      if (!any) continue;
      const int32_t i0 = u * EPU + g * 4;
      const uint4 blk = philox_row_1((uint32_t)i0 >> 2, ph);
#pragma unroll
      for (int t = 0; t < 4; ++t)
        if (in[t]) take_better(exact_score(xs[t], word_of(blk, t), f.T), i0 + t, bs, bi);
    }
  });
  warp_argmax(bs, bi);
  if (lane == 0) s_best[warp] = bi != INT32_MAX ? pack_key(bs, bi) : 0ull;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long best = 0ull;
    for (int i = 0; i < kFiltWarps; ++i) best = s_best[i] > best ? s_best[i] : best;
    fp.out_idx[b] = index_of_key(best);
    fp.ws[b].hint = 0u;  // the workspace is left clean
  }
}

template <int DT, bool VEC>
void* check_fn() {
  return reinterpret_cast<void*>(&filter_row_kernel<DT, VEC>);
}
template <int DT, bool VEC>
void* exact_fn() {
  return reinterpret_cast<void*>(&filter_exact_kernel<DT, VEC>);
}

void* pick(int dtype, bool vec, bool exact) {
  switch (dtype * 2 + (vec ? 1 : 0)) {
    case 0: return exact ? exact_fn<0, false>() : check_fn<0, false>();
    case 1: return exact ? exact_fn<0, true>() : check_fn<0, true>();
    case 2: return exact ? exact_fn<1, false>() : check_fn<1, false>();
    case 3: return exact ? exact_fn<1, true>() : check_fn<1, true>();
    case 4: return exact ? exact_fn<2, false>() : check_fn<2, false>();
    default: return exact ? exact_fn<2, true>() : check_fn<2, true>();
  }
}

cudaError_t launch_one(const FilterParams& p, int dtype, bool vec, bool exact,
                       cudaStream_t stream) {
  void* args[] = {const_cast<FilterParams*>(&p)};
  void* fn = pick(dtype, vec, exact);
  const size_t smem = exact ? 0 : (size_t)kListCap * sizeof(uint2);
  if (smem && cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
                  cudaSuccess)
    return cudaGetLastError();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.B);
  cfg.blockDim = dim3(kFiltThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

cudaError_t launch_filter(const FilterParams& p, int dtype, bool vec, cudaStream_t stream) {
  cudaError_t e = launch_one(p, dtype, vec, false, stream);
  if (e != cudaSuccess) return e;
  return launch_one(p, dtype, vec, true, stream);
}

}  // namespace gsample
