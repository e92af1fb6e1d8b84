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
// in the subset), so it stands. A rejected proposal means K ends before it, so
// K's last element is found among the candidates at or above the proposal.
//
// Layout: one thread-block cluster per filtered row, each CTA holding its
// slice of the row in shared memory (requested at once with cp.async), so
// every phase after the first reads shared memory only:
//   1. the test: the proposal's rank (candidates before it) against top_k and
//      the binary32 mass before it against top_p times the row's mass; the
//      CTAs' partial sums meet over distributed shared memory in rank order,
//      so every CTA takes the same decision. Units holding a logit at or
//      above the proposal are marked on the way.
//   2. a rejected row: K's last key by a radix select over the order-preserving
//      keys of the marked units, eight bits per level (two levels decide a
//      bf16 key, three an f16 key, four an f32 key), with counts for top_k
//      and 2^-E fixed-point masses relative to the row maximum for top_p;
//      every CTA sums the cluster's digit histograms (integers: exact in any
//      order) and picks the same digit.
//   3. the entries equal to K's last key that K takes, in index order: the
//      slices are consecutive index ranges, so each CTA knows from the
//      cluster's per-CTA tie counts how many of its own it takes.
//   4. the Gumbel-max over K's members in the slice, merged over the cluster;
//      rank 0 writes out_idx.
// The only waits are hardware CTA and cluster barriers, and the result does
// not depend on the order of any atomic.
#include <cooperative_groups.h>

#include <climits>
#include <cstdint>

#include "gsample_internal.h"
#include "gsample_slice.cuh"

namespace cg = cooperative_groups;

namespace gsample {
namespace {

using namespace slice;

constexpr int kFiltThreads = 256;  // one thread per digit of a radix level
constexpr int kFiltWarps = kFiltThreads / 32;
constexpr int kMaxCluster = 16;
constexpr int kLocalCap = 512;  // entries of a CTA's list of candidates at or above the proposal
constexpr size_t kFiltSmemLimit = 200 * 1024;
constexpr float kLog2e = 1.4426950408889634f;

// Unit u of a row from global memory through the read-only cache (the path
// for slices too large for shared memory re-reads them in every phase).
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

__device__ __forceinline__ bool is_candidate(float x) { return x > -INFINITY; }  // NaN: false

// The row's filter. top_p <= 0 keeps only the first element, which is top_k = 1.
struct RowFilter {
  float T, p;
  int32_t k;
  bool k_on, p_on;
};

__device__ __forceinline__ RowFilter row_filter(const FilterParams& fp, int64_t b) {
  RowFilter f;
  f.T = __ldg(fp.temperature + b);
  f.k = fp.top_k ? __ldg(fp.top_k + b) : 0;
  f.p = fp.top_p ? __ldg(fp.top_p + b) : 1.0f;
  f.k_on = f.k >= 1;
  f.p_on = f.p < 1.0f;  // NaN: off
  if (f.p_on && f.p <= 0.0f) {
    f.k = 1;
    f.k_on = true;
    f.p_on = false;
  }
  return f;
}

// e^((x - M) / T) in (0, 1] in units of 2^-E (scale = 2^E, exact in binary32),
// converted exactly: the fixed-point value keeps binary32's 24 bits. Integer
// sums of these are exact and independent of order.
__device__ __forceinline__ unsigned long long fixed_mass(float x, float M, float a, float scale) {
  return __float2ull_rn(exp2f((x - M) * a) * scale);
}

// This CTA's share of the acceptance test, read by every CTA of the cluster.
struct Partial {
  float S;       // binary32 mass of the candidates, relative to the proposal's
  float mb;      // the same for the candidates before the proposal
  float M;       // largest logit
  unsigned cnt;  // candidates before the proposal
  unsigned nl;   // candidates at or above the proposal (the floor set)
};

// Order-preserving keys in the bits the logit's dtype can set: a bf16 logit
// fixes the top 16 bits of its binary32 key and an f16 logit the top 19; the
// others follow the sign (zeros for positive logits, ones for negative ones).
// The radix select runs on ck = key >> kZB relative to the proposal's, so a
// bf16 row whose candidates above the proposal span fewer than 256 bf16
// values needs one level.
template <int DT>
struct KeyBits {
  static constexpr int kZB = DT == 1 ? 16 : (DT == 2 ? 13 : 0);
};

template <int DT>
__device__ __forceinline__ uint32_t key_of_ck(uint32_t ck) {
  constexpr int ZB = KeyBits<DT>::kZB;
  if constexpr (ZB == 0) {
    return ck;
  } else {
    const uint32_t k = ck << ZB;
    return (k & 0x80000000u) ? k : (k | ((1u << ZB) - 1u));
  }
}

__device__ __forceinline__ int bit_length(uint32_t v) { return v ? 32 - __clz(v) : 0; }

// One radix level over values v (relative keys, or inverted indices): the
// bits [s_lo, s_hi) form the digit, the bits from s_hi up must equal those of
// `prefix` (the digits chosen so far).
struct Level {
  int s_hi, s_lo;
  uint32_t prefix;
  __device__ __forceinline__ bool match(uint32_t v) const {
    return s_hi >= 32 || (v >> s_hi) == (prefix >> s_hi);
  }
  __device__ __forceinline__ uint32_t digit(uint32_t v) const {
    return (v >> s_lo) & ((1u << (s_hi - s_lo)) - 1u);
  }
};

// Shared scratch of find_boundary.
struct ScanShared {
  unsigned c[kFiltWarps];
  unsigned long long m[kFiltWarps];
  int sel;
  unsigned exc;
  unsigned long long exm;
};

// Thread t holds the totals (c, m) of digit 255 - t. The first digit from the
// top at which the cumulative count reaches k_rem or the cumulative mass
// reaches m_rem (both at least 1): its count and mass above it go to
// *above_c, *above_m. Returns the digit, or -1 if neither target is reached.
// Called by every thread of the CTA; ends with a barrier.
__device__ __forceinline__ int find_boundary(unsigned c, unsigned long long m, unsigned k_rem,
                                             unsigned long long m_rem, bool p_on, ScanShared& sh,
                                             unsigned* above_c, unsigned long long* above_m) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) sh.sel = kFiltThreads;
  unsigned ic = c;
  unsigned long long im = m;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned tc = __shfl_up_sync(0xFFFFFFFFu, ic, o);
    const unsigned long long tm = __shfl_up_sync(0xFFFFFFFFu, im, o);
    if (lane >= o) {
      ic += tc;
      im += tm;
    }
  }
  if (lane == 31) {
    sh.c[warp] = ic;
    sh.m[warp] = im;
  }
  __syncthreads();
  for (int i = 0; i < warp; ++i) {
    ic += sh.c[i];
    im += sh.m[i];
  }
  const unsigned ec = ic - c;
  const unsigned long long em = im - m;
  if ((ec < k_rem && k_rem <= ic) || (p_on && em < m_rem && m_rem <= im))
    atomicMin(&sh.sel, (int)threadIdx.x);
  __syncthreads();
  const int ts = sh.sel;
  if (ts < kFiltThreads && (int)threadIdx.x == ts) {
    sh.exc = ec;
    sh.exm = em;
  }
  __syncthreads();
  *above_c = sh.exc;
  *above_m = sh.exm;
  __syncthreads();
  return ts < kFiltThreads ? 255 - ts : -1;
}

// Exclusive scan of one value per thread over the CTA (warp scans, then the
// warps' totals in order); *total gets the CTA's sum. Ends with a barrier.
__device__ __forceinline__ unsigned block_exclusive_scan(unsigned v, unsigned* scratch,
                                                         unsigned* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  unsigned before = 0, all = 0;
#pragma unroll
  for (int i = 0; i < kFiltWarps; ++i) {
    before += i < warp ? scratch[i] : 0u;
    all += scratch[i];
  }
  *total = all;
  __syncthreads();
  return before + incl - v;
}

// ---------------------------------------------------------------------------
// One cluster of fp.cluster CTAs per row; CTA `rank` holds units
// [rank * units_per_cta, (rank + 1) * units_per_cta) of the row. The
// proposal in out_idx[b] is tested and, when rejected, replaced by the
// Gumbel-max over K.
// ---------------------------------------------------------------------------
template <int DT, bool VEC, bool RESIDENT>
__global__ void __launch_bounds__(kFiltThreads, 4) filter_cluster_kernel(const FilterParams fp) {
  using C = HCfg<DT, VEC>;
  constexpr int EPU = C::kEPU;
  constexpr int ZB = KeyBits<DT>::kZB;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ Partial s_wp[kFiltWarps];
  __shared__ Partial s_part;  // this CTA's partial, read by the whole cluster
  __shared__ Partial s_tot;   // the row's totals
  __shared__ unsigned s_hc[2][256];            // digit counts of a level (two buffers)
  __shared__ unsigned long long s_hm[2][256];  // digit masses of a level
  __shared__ ScanShared s_scan;
  __shared__ unsigned s_sc[kFiltWarps];
  __shared__ uint2 s_list[kLocalCap];   // this slice's candidates at or above the proposal
  __shared__ unsigned s_ln;             // their number (may exceed kLocalCap)
  __shared__ unsigned s_lists[2];       // the cluster's: total, largest
  __shared__ unsigned s_loff[kMaxCluster + 1];  // offsets of the CTAs' lists in rank 0's gather
  __shared__ unsigned s_tie[2];         // entries equal to K's last key before this slice, in it
  __shared__ int32_t s_idx;
  __shared__ unsigned s_tcnt;           // entries on K's last key, gathered for one warp
  __shared__ uint32_t s_tidx[32];
  __shared__ unsigned long long s_best[kFiltWarps];
  __shared__ unsigned long long s_key;  // this CTA's best (score, index) key, read by rank 0

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int nrank = fp.cluster;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t b = blockIdx.x / nrank;
  // Every CTA of a cluster reads the same row, filter and proposal, so the
  // early exits below are taken by the whole cluster or by none of it.
  const RowFilter f = row_filter(fp, b);
  if (!(f.T > 0.0f) || !(f.k_on || f.p_on)) return;  // greedy or unfiltered: the proposal stands
  const char* row = fp.logits + b * fp.ld_bytes;
  const uint64_t sd = __ldg(fp.seed + b), of = __ldg(fp.offset + b);
  if (threadIdx.x == 0) s_ln = 0u;
  const int32_t u_lo = rank * fp.units_per_cta;
  const int32_t u_hi = min(fp.units_per_row, u_lo + fp.units_per_cta);
  const uint32_t slice = (uint32_t)__cvta_generic_to_shared(smem);

  // The slice, requested at once, before the wait for the proposal: the logits
  // do not depend on the kernel that writes it, so their stream overlaps that
  // kernel's tail. Each thread later reads back only the units it requested
  // (unit u_lo + threadIdx.x + j * kFiltThreads), so its own cp.async wait is
  // all the ordering it needs; no CTA leaves with a copy in flight. This
  // kernel does not release its own dependents early: a successor resident
  // while the filter's later waves still need the SMs would take their room.
  if constexpr (RESIDENT) {
    const uint64_t pol = evict_first_policy();
    for (int32_t u = u_lo + threadIdx.x; u < u_hi; u += kFiltThreads) {
      const uint32_t dst = slice + (uint32_t)(u - u_lo) * 16u;
      if (VEC && (u + 1) * EPU <= fp.V)
        cp_async16(dst, row + (size_t)u * 16, pol);
      else
        sts128(dst, load_unit<DT, VEC>(row, u, fp.V, pol));
    }
    cp_async_commit();
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t w = fp.out_idx[b];
  const float xw = w >= 0 ? elt_at<DT>(row, w) : -INFINITY;
  if constexpr (RESIDENT) cp_async_wait<0>();
  // no candidate at all, or the first +inf entry heads the order: the proposal stands
  if (w < 0 || xw == INFINITY) return;
  __syncthreads();
  auto unit_at = [&](int32_t u) -> uint4 {
    if constexpr (RESIDENT)
      return lds128(slice + (uint32_t)(u - u_lo) * 16u);
    else
      return unit_cached<DT, VEC>(row, u, fp.V);
  };

  // 1. The test. Masses are relative to the proposal's (binary32, e^((x - xw)/T)
  // <= e^19.5 since no logit can outscore the proposal by more than the range
  // of the Gumbel noise); a NaN logit adds nothing. A resident slice also lists
  // its floor set (candidates at or above the proposal) as (key, index), in
  // case the proposal is rejected.
  const float a = kLog2e / f.T;
  // mass(x) = 2^(x*a - xw*a): the one rounding of xw*a scales every mass
  // alike, so it cancels out of the test; a NaN or -inf logit gives 2^-127,
  // flushed to zero.
  const float nxa = -(xw * a);
  auto mass_w = [&](float x) { return ex2_approx(fmaxf(fmaf(x, a, nxa), -127.0f)); };
  unsigned cnt = 0;
  float S = 0.0f, mb = 0.0f, tmax = -INFINITY;
  uint64_t marks = 0;  // bit j: the thread's j-th unit holds a logit >= xw (j >= 64: visited anyway)
  {
    int j = 0;
    for (int32_t u = u_lo + threadIdx.x; u < u_hi; u += kFiltThreads, ++j) {
      const uint4 r = unit_at(u);
      float um = -INFINITY;
#pragma unroll
      for (int e = 0; e < EPU; ++e) {
        const float x = elt<DT, VEC>(r, e);
        um = fmaxf(um, x);
        if (f.p_on) S += mass_w(x);
      }
      tmax = fmaxf(tmax, um);
      if (um >= xw) {
        if (j < 64) marks |= 1ull << j;
#pragma unroll
        for (int e = 0; e < EPU; ++e) {
          const float x = elt<DT, VEC>(r, e);
          const int64_t i = (int64_t)u * EPU + e;
          if (x >= xw) {
            // once the list is full the row cannot take the list path, so
            // a long floor set stops contending for the counter
            if (RESIDENT && *reinterpret_cast<volatile unsigned*>(&s_ln) < (unsigned)kLocalCap) {
              const unsigned pos = atomicAdd(&s_ln, 1u);
              if (pos < (unsigned)kLocalCap) s_list[pos] = make_uint2(ordered_bits(x), (uint32_t)i);
            }
            if (x > xw || i < w) {
              ++cnt;
              if (f.p_on) mb += mass_w(x);
            }
          }
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, o);
    S += __shfl_xor_sync(0xFFFFFFFFu, S, o);
    mb += __shfl_xor_sync(0xFFFFFFFFu, mb, o);
    tmax = fmaxf(tmax, __shfl_xor_sync(0xFFFFFFFFu, tmax, o));
  }
  if (lane == 0) s_wp[warp] = Partial{S, mb, tmax, cnt, 0u};
  __syncthreads();
  if (threadIdx.x == 0) {
    Partial t = s_wp[0];
    for (int i = 1; i < kFiltWarps; ++i) {
      t.S += s_wp[i].S;
      t.mb += s_wp[i].mb;
      t.M = fmaxf(t.M, s_wp[i].M);
      t.cnt += s_wp[i].cnt;
    }
    t.nl = s_ln;
    s_part = t;
  }
  cluster.sync();
  if (warp == 0) {
    // the cluster's partials summed in rank order: every CTA rounds the same way
    Partial o{0.0f, 0.0f, -INFINITY, 0u, 0u};
    if (lane < nrank) o = *cluster.map_shared_rank(&s_part, lane);
    Partial t = o;
    for (int q = 1; q < nrank; ++q) {
      t.S += __shfl_sync(0xFFFFFFFFu, o.S, q);
      t.mb += __shfl_sync(0xFFFFFFFFu, o.mb, q);
      t.M = fmaxf(t.M, __shfl_sync(0xFFFFFFFFu, o.M, q));
      t.cnt += __shfl_sync(0xFFFFFFFFu, o.cnt, q);
    }
    if (lane == 0) s_tot = t;
    // the CTAs' lists: offsets in rank 0's gather, total and largest
    unsigned incl = o.nl, mx = o.nl;
#pragma unroll
    for (int q = 1; q < 32; q <<= 1) {
      const unsigned v = __shfl_up_sync(0xFFFFFFFFu, incl, q);
      if (lane >= q) incl += v;
      mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, q));
    }
    if (lane <= nrank) s_loff[lane] = incl - o.nl;
    if (lane == 31) {
      s_lists[0] = incl;
      s_lists[1] = mx;
    }
  }
  __syncthreads();
  const Partial tot = s_tot;
  bool ok = !f.k_on || tot.cnt < (unsigned)f.k;
  if (f.p_on) ok = ok && tot.mb < f.p * tot.S;
  if (ok) {
    cluster.sync();  // no CTA leaves while another still reads its partial
    return;
  }


  // 2. A rejected proposal: K ends before it, so K's last element is among the
  // floor set (the candidates with a key at least the proposal's, all in the
  // marked units). Targets: top_k entries (k_rem) and the first prefix whose
  // fixed-point mass reaches top_p times the row's (m_rem; the row's mass is
  // the binary32 sum above, rescaled to the row maximum). The select runs on
  // rel = ck(key) - ck(key_w) over the floor set, eight bits a level from the
  // top bit of its span. Should neither target be reached within the floor
  // set (a binary32 rejection at the nucleus edge), K holds the proposal,
  // which then stands.
  const float M = tot.M;
  const float scale = fp.mass_scale;
  const uint32_t key_w = ordered_bits(xw);
  const uint32_t ck_w = key_w >> ZB;
  const int nb = bit_length((ordered_bits(M) >> ZB) - ck_w);
  unsigned k_rem = f.k_on ? (unsigned)f.k : 0xFFFFFFFFu;
  unsigned long long m_rem = ULLONG_MAX;
  if (f.p_on) {
    const double Sf = (double)tot.S * (double)exp2f((xw - M) * a) * (double)scale;
    m_rem = (unsigned long long)ceil((double)f.p * Sf);
    if (m_rem < 1ull) m_rem = 1ull;
  }
  const PhiloxRow ph =
      philox_row((uint32_t)b, (uint32_t)of, (uint32_t)(of >> 32), (uint32_t)sd, (uint32_t)(sd >> 32));
  const unsigned n_all = s_lists[0];
  // A CTA whose count reached kLocalCap may have skipped entries: that row
  // takes the cluster-wide select.
  if (RESIDENT && s_lists[1] < (unsigned)kLocalCap && n_all <= 2u * (unsigned)fp.units_per_cta) {
    // 2a. Rank 0 gathers the cluster's lists into its slice buffer, the other
    // CTAs leave, and rank 0 resolves the row alone.
    uint2* lst = reinterpret_cast<uint2*>(smem);
    if (rank == 0) {
      for (unsigned g0 = 0; g0 < n_all; g0 += 4u * kFiltThreads) {
        uint2 v[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const unsigned g = g0 + (unsigned)(t * kFiltThreads) + threadIdx.x;
          if (g < n_all) {
            int q = 0;
            while (q + 1 < nrank && s_loff[q + 1] <= g) ++q;
            v[t] = cluster.map_shared_rank(s_list, q)[g - s_loff[q]];
          }
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const unsigned g = g0 + (unsigned)(t * kFiltThreads) + threadIdx.x;
          if (g < n_all) lst[g] = v[t];
        }
      }
    }
    cluster.sync();  // rank 0 has read every list
    if (rank != 0) return;

    int hb = 0;
    uint32_t prefix = 0;
    unsigned t_b = 0;  // entries on K's last key
    for (int s_hi = nb;;) {
      const int s_lo = s_hi > 8 ? s_hi - 8 : 0;
      const Level lv{s_hi, s_lo, prefix};
      s_hc[hb][threadIdx.x] = 0u;
      s_hm[hb][threadIdx.x] = 0ull;
      __syncthreads();
      for (unsigned i = threadIdx.x; i < n_all; i += kFiltThreads) {
        const uint32_t key = lst[i].x;
        const uint32_t rel = (key >> ZB) - ck_w;
        if (lv.match(rel)) {
          const uint32_t d = lv.digit(rel);
          atomicAdd(&s_hc[hb][d], 1u);
          if (f.p_on)
            atomicAdd(&s_hm[hb][d], fixed_mass(score_of_key((unsigned long long)key << 32 | 1ull),
                                               M, a, scale));
        }
      }
      __syncthreads();
      unsigned ac;
      unsigned long long am;
      const int d = find_boundary(s_hc[hb][255 - threadIdx.x], s_hm[hb][255 - threadIdx.x], k_rem,
                                  m_rem, f.p_on, s_scan, &ac, &am);
      if (d < 0) return;  // K reaches past the floor set: the proposal stands
      k_rem -= ac;
      m_rem -= am;
      prefix |= (uint32_t)d << s_lo;
      t_b = s_hc[hb][d];
      hb ^= 1;
      if (s_lo == 0) break;
      s_hi = s_lo;
    }
    const uint32_t key_b = key_of_ck<DT>(ck_w + prefix);
    unsigned n_take = k_rem;
    if (f.p_on) {
      const unsigned long long eb =
          fixed_mass(score_of_key((unsigned long long)key_b << 32 | 1ull), M, a, scale);
      const unsigned long long np = eb > 0ull ? (m_rem + eb - 1ull) / eb : ULLONG_MAX;
      if (np < (unsigned long long)n_take) n_take = (unsigned)np;
    }
    if (n_take < 1u) n_take = 1u;
    // K takes the first n_take entries on key_b in index order: the n_take-th
    // largest inverted index, eight bits a level.
    int32_t idx_b = INT32_MAX;
    if (n_take < t_b && t_b <= 32u) {
      // few entries on key_b: one warp ranks their indices
      if (threadIdx.x == 0) {
        s_tcnt = 0u;
        s_idx = INT32_MAX;
      }
      __syncthreads();
      for (unsigned i = threadIdx.x; i < n_all; i += kFiltThreads) {
        if (lst[i].x == key_b) {
          const unsigned pos = atomicAdd(&s_tcnt, 1u);
          if (pos < 32u) s_tidx[pos] = lst[i].y;
        }
      }
      __syncthreads();
      if (warp == 0) {
        const uint32_t v = lane < (int)t_b ? s_tidx[lane] : 0xFFFFFFFFu;
        unsigned r = 0;
        for (unsigned q = 0; q < t_b; ++q) r += s_tidx[q] < v ? 1u : 0u;
        if (lane < (int)t_b && r == n_take - 1u) s_idx = (int32_t)v;
      }
      __syncthreads();
      idx_b = s_idx;
    } else if (n_take < t_b) {
      unsigned kk = n_take;
      uint32_t ip = 0;
      bool found = true;
      for (int s_hi = 32; s_hi > 0; s_hi -= 8) {
        const Level lv{s_hi, s_hi - 8, ip};
        s_hc[hb][threadIdx.x] = 0u;
        __syncthreads();
        for (unsigned i = threadIdx.x; i < n_all; i += kFiltThreads) {
          const uint32_t inv = ~lst[i].y;
          if (lst[i].x == key_b && lv.match(inv)) atomicAdd(&s_hc[hb][lv.digit(inv)], 1u);
        }
        __syncthreads();
        unsigned ac;
        unsigned long long am;
        const int d = find_boundary(s_hc[hb][255 - threadIdx.x], 0ull, kk, ULLONG_MAX, false,
                                    s_scan, &ac, &am);
        hb ^= 1;
        if (d < 0) {  // cannot happen: kk never exceeds the entries left
          found = false;
          break;
        }
        kk -= ac;
        ip |= (uint32_t)d << (s_hi - 8);
      }
      if (found) idx_b = (int32_t)~ip;
    }
    // The Gumbel-max over K's entries of the list.
    float bs = -INFINITY;
    int32_t bi = INT32_MAX;
    for (unsigned i = threadIdx.x; i < n_all; i += kFiltThreads) {
      const uint32_t key = lst[i].x;
      const int32_t idx = (int32_t)lst[i].y;
      if (key > key_b || (key == key_b && idx <= idx_b)) {
        const float x = score_of_key((unsigned long long)key << 32 | 1ull);
        const uint4 blk = philox_row_1((uint32_t)idx >> 2, ph);
        take_better(exact_score(x, word_of(blk, idx & 3), f.T), idx, bs, bi);
      }
    }
    warp_argmax(bs, bi);
    if (lane == 0) s_best[warp] = bi != INT32_MAX ? pack_key(bs, bi) : 0ull;
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned long long best = 0ull;
      for (int i = 0; i < kFiltWarps; ++i) best = s_best[i] > best ? s_best[i] : best;
      if (best) fp.out_idx[b] = index_of_key(best);
    }
    return;
  }

  // 2b. The lists overflowed (or the slices are not resident): every CTA
  // histograms its own floor set, and every CTA sums the cluster's histograms
  // (integers: the same in any order) and picks the same digit.
  int hb = 0, h_last = 0, d_last = 0;
  uint32_t prefix = 0;
  for (int s_hi = nb;;) {
    const int s_lo = s_hi > 8 ? s_hi - 8 : 0;
    const Level lv{s_hi, s_lo, prefix};
    s_hc[hb][threadIdx.x] = 0u;
    s_hm[hb][threadIdx.x] = 0ull;
    __syncthreads();
    {
      int j = 0;
      for (int32_t u = u_lo + threadIdx.x; u < u_hi; u += kFiltThreads, ++j) {
        if (j < 64 && !((marks >> j) & 1ull)) continue;
        const uint4 r = unit_at(u);
#pragma unroll
        for (int e = 0; e < EPU; ++e) {
          const float x = elt<DT, VEC>(r, e);
          const uint32_t key = ordered_bits(x);
          const uint32_t rel = (key >> ZB) - ck_w;
          if (is_candidate(x) && key >= key_w && lv.match(rel)) {
            const uint32_t d = lv.digit(rel);
            atomicAdd(&s_hc[hb][d], 1u);
            if (f.p_on) atomicAdd(&s_hm[hb][d], fixed_mass(x, M, a, scale));
          }
        }
      }
    }
    cluster.sync();
    // thread t: digit 255 - t, summed over the cluster
    const int dg = 255 - (int)threadIdx.x;
    unsigned c = 0;
    unsigned long long m = 0;
#pragma unroll 4
    for (int q = 0; q < nrank; ++q) {
      c += *cluster.map_shared_rank(&s_hc[hb][dg], q);
      if (f.p_on) m += *cluster.map_shared_rank(&s_hm[hb][dg], q);
    }
    unsigned ac;
    unsigned long long am;
    const int d = find_boundary(c, m, k_rem, m_rem, f.p_on, s_scan, &ac, &am);
    if (d < 0) {  // K reaches past the floor set: the proposal stands
      cluster.sync();  // every CTA has read this level's histograms
      return;
    }
    k_rem -= ac;
    m_rem -= am;
    prefix |= (uint32_t)d << s_lo;
    h_last = hb;
    d_last = d;
    hb ^= 1;
    if (s_lo == 0) break;
    s_hi = s_lo;
  }
  const uint32_t key_b = key_of_ck<DT>(ck_w + prefix);

  // 3. The entries on K's last key that K takes (n_take of them, in index
  // order; every one of them has the same mass), and from the cluster's
  // per-CTA counts of such entries (the last level's digit) how many of this
  // slice's: all, none, or the first `take`, found by a scan of the slice.
  unsigned n_take = k_rem;
  if (f.p_on) {
    const unsigned long long eb =
        fixed_mass(score_of_key((unsigned long long)key_b << 32 | 1ull), M, a, scale);
    const unsigned long long np = eb > 0ull ? (m_rem + eb - 1ull) / eb : ULLONG_MAX;
    if (np < (unsigned long long)n_take) n_take = (unsigned)np;
  }
  if (n_take < 1u) n_take = 1u;
  if (warp == 0) {
    const unsigned own = lane < nrank ? *cluster.map_shared_rank(&s_hc[h_last][d_last], lane) : 0u;
    unsigned incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == rank) {
      s_tie[0] = incl - own;
      s_tie[1] = own;
    }
  }
  __syncthreads();
  int32_t idx_bound = -1;  // this slice's entries on key_b with an index up to idx_bound are in K
  {
    const unsigned before = s_tie[0], mine = s_tie[1];
    const unsigned take = n_take <= before ? 0u : min(n_take - before, mine);
    if (take == mine) {
      idx_bound = INT32_MAX;
    } else if (take > 0u) {
      if (threadIdx.x == 0) s_idx = -1;
      unsigned need = take;
      for (int32_t base = u_lo; base < u_hi; base += kFiltThreads) {
        const int32_t u = base + threadIdx.x;
        uint4 r = make_uint4(0u, 0u, 0u, 0u);
        unsigned n = 0;
        if (u < u_hi) {
          r = unit_at(u);
#pragma unroll
          for (int e = 0; e < EPU; ++e) {
            const float x = elt<DT, VEC>(r, e);
            n += (is_candidate(x) && ordered_bits(x) == key_b) ? 1u : 0u;
          }
        }
        unsigned total = 0;
        const unsigned ex = block_exclusive_scan(n, s_sc, &total);
        if (n > 0u && ex < need && need <= ex + n) {
          unsigned seen = ex;
#pragma unroll
          for (int e = 0; e < EPU; ++e) {
            const float x = elt<DT, VEC>(r, e);
            if (is_candidate(x) && ordered_bits(x) == key_b && ++seen == need) {
              s_idx = u * EPU + e;
              break;
            }
          }
        }
        __syncthreads();
        if (need <= total) break;
        need -= total;
      }
      idx_bound = s_idx;
    }
  }

  // 4. The Gumbel-max over K's members in the slice: a Philox block for each
  // group of four holding one (every member lies in a marked unit).
  float bs = -INFINITY;
  int32_t bi = INT32_MAX;
  {
    int j = 0;
    for (int32_t u = u_lo + threadIdx.x; u < u_hi; u += kFiltThreads, ++j) {
      if (j < 64 && !((marks >> j) & 1ull)) continue;
      const uint4 r = unit_at(u);
#pragma unroll
      for (int g = 0; g < EPU / 4; ++g) {
        float xs[4];
        bool in[4];
        bool any = false;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          xs[t] = elt<DT, VEC>(r, g * 4 + t);
          const uint32_t key = ordered_bits(xs[t]);
          const int32_t i = u * EPU + g * 4 + t;
          in[t] = is_candidate(xs[t]) && (key > key_b || (key == key_b && i <= idx_bound));
          any |= in[t];
        }
        if (!any) continue;
        const int32_t i0 = u * EPU + g * 4;
        const uint4 blk = philox_row_1((uint32_t)i0 >> 2, ph);
#pragma unroll
        for (int t = 0; t < 4; ++t)
          if (in[t]) take_better(exact_score(xs[t], word_of(blk, t), f.T), i0 + t, bs, bi);
      }
    }
  }
  warp_argmax(bs, bi);
  if (lane == 0) s_best[warp] = bi != INT32_MAX ? pack_key(bs, bi) : 0ull;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long best = 0ull;
    for (int i = 0; i < kFiltWarps; ++i) best = s_best[i] > best ? s_best[i] : best;
    s_key = best;
  }
  cluster.sync();
  if (rank == 0 && warp == 0) {
    unsigned long long k = lane < nrank ? *cluster.map_shared_rank(&s_key, lane) : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long t = __shfl_xor_sync(0xFFFFFFFFu, k, o);
      k = t > k ? t : k;
    }
    if (lane == 0 && k) fp.out_idx[b] = index_of_key(k);
  }
  cluster.sync();  // every CTA's shared memory stays until rank 0 has read it
}

template <int DT, bool VEC, bool RES>
void* fk() {
  return reinterpret_cast<void*>(&filter_cluster_kernel<DT, VEC, RES>);
}

void* select_filter(int dtype, bool vec, bool resident) {
  switch (dtype * 4 + (vec ? 2 : 0) + (resident ? 1 : 0)) {
    case 0: return fk<0, false, false>();
    case 1: return fk<0, false, true>();
    case 2: return fk<0, true, false>();
    case 3: return fk<0, true, true>();
    case 4: return fk<1, false, false>();
    case 5: return fk<1, false, true>();
    case 6: return fk<1, true, false>();
    case 7: return fk<1, true, true>();
    case 8: return fk<2, false, false>();
    case 9: return fk<2, false, true>();
    case 10: return fk<2, true, false>();
    default: return fk<2, true, true>();
  }
}

}  // namespace

size_t filter_smem_limit() { return kFiltSmemLimit; }

void* filter_kernel_fn(int dtype, bool vec, bool resident, int* threads) {
  *threads = kFiltThreads;
  return select_filter(dtype, vec, resident);
}

// One-time per-device setup of both variants of (dtype, vec): allow clusters
// of up to 16 CTAs and the full shared-memory slice, then report the largest
// cluster the device can co-schedule.
int filter_max_cluster(int dtype, bool vec) {
  for (int res = 0; res < 2; ++res) {
    void* fn = select_filter(dtype, vec, res != 0);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             res ? (int)kFiltSmemLimit : 0) != cudaSuccess)
      return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kMaxCluster);
  cfg.blockDim = dim3(kFiltThreads);
  cfg.dynamicSmemBytes = kFiltSmemLimit;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kMaxCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int size = 0;
  if (cudaOccupancyMaxPotentialClusterSize(&size, select_filter(dtype, vec, true), &cfg) !=
      cudaSuccess)
    return 0;
  return size < kMaxCluster ? size : kMaxCluster;
}

cudaError_t launch_filter(const FilterParams& p, int dtype, bool vec, cudaStream_t stream) {
  const size_t need = (size_t)p.units_per_cta * 16;
  const bool resident = need <= kFiltSmemLimit;
  void* fn = select_filter(dtype, vec, resident);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * p.cluster));
  cfg.blockDim = dim3(kFiltThreads);
  cfg.dynamicSmemBytes = resident ? need : 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = pdl_attribute();
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  void* args[] = {const_cast<FilterParams*>(&p)};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace gsample
