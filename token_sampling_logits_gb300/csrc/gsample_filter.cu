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
// in the subset), so it stands. filter_check_kernel decides that from one
// pass over the row: the proposal's rank (candidates before it) against
// top_k, and the mass before it against top_p times the row's mass. Rows
// whose proposal is rejected are flagged in their workspace slot, and
// filter_exact_kernel resolves them exactly: it finds K's last element by a
// radix select over the logits' order-preserving keys (counts for top_k,
// fixed-point masses for top_p), then takes the Gumbel-max over K. Both give
// the same index: the argmax over K of the same scores.
#include <cstdint>

#include "gsample_internal.h"
#include "gsample_slice.cuh"

namespace gsample {
namespace {

using namespace slice;

constexpr int kFiltThreads = 512;
constexpr int kFiltWarps = kFiltThreads / 32;
constexpr float kLog2e = 1.4426950408889634f;
// Fixed-point masses of the exact path: e^((x - M) / T) in (0, 1] times 2^40.
// Integer sums are exact and order-free, so the selection is deterministic.
constexpr double kMassScale = 1099511627776.0;  // 2^40

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

// ---------------------------------------------------------------------------
// The acceptance test of the proposal in out_idx[b]: its rank among the
// candidates and the softmax mass of the candidates before it (relative to the
// proposal's own, so no row maximum is needed; an overflow only rejects).
// ---------------------------------------------------------------------------
template <int DT, bool VEC>
__global__ void __launch_bounds__(kFiltThreads) filter_check_kernel(const FilterParams fp) {
  pdl_wait_then_release();
  __shared__ float sf[kFiltWarps];
  __shared__ unsigned su[kFiltWarps];
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
  const float a = kLog2e / f.T;
  unsigned cnt = 0;
  float S = 0.0f, MB = 0.0f;
  for (int32_t u = threadIdx.x; u < fp.units_per_row; u += kFiltThreads) {
    const uint4 r = unit_cached<DT, VEC>(row, u, fp.V);
#pragma unroll
    for (int e = 0; e < EPU; ++e) {
      const float x = elt<DT, VEC>(r, e);
      if (!is_candidate(x)) continue;
      const int64_t i = (int64_t)u * EPU + e;
      const bool before = x > xw || (x == xw && i < w);
      cnt += before ? 1u : 0u;
      if (f.p_on) {
        const float m = exp2f((x - xw) * a);
        S += m;
        MB += before ? m : 0.0f;
      }
    }
  }
  cnt = block_reduce(cnt, AddU(), su);
  if (f.p_on) {
    S = block_reduce(S, AddF(), sf);
    MB = block_reduce(MB, AddF(), sf);
  }
  if (threadIdx.x == 0) {
    bool ok = !f.k_on || cnt < (unsigned)f.k;
    if (f.p_on) ok = ok && (f.p <= 0.0f ? cnt == 0u : MB < f.p * S);
    if (!ok) fp.ws[b].hint = 1u;  // rejected: resolved by filter_exact_kernel
  }
}

// ---------------------------------------------------------------------------
// The exact path for a rejected row: K's last element by radix select, then
// the Gumbel-max over K. One CTA per row; the row is read from L2 after the
// first pass.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long fixed_mass(float x, float M, float a) {
  return (unsigned long long)((double)exp2f((x - M) * a) * kMassScale + 0.5);
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kFiltThreads) filter_exact_kernel(const FilterParams fp) {
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

  // Row maximum and candidate count.
  float M = -INFINITY;
  unsigned n = 0;
  for (int32_t u = threadIdx.x; u < NU; u += kFiltThreads) {
    const uint4 r = unit_cached<DT, VEC>(row, u, fp.V);
#pragma unroll
    for (int e = 0; e < EPU; ++e) {
      const float x = elt<DT, VEC>(r, e);
      if (is_candidate(x)) {
        M = fmaxf(M, x);
        ++n;
      }
    }
  }
  M = block_reduce(M, MaxF(), sf);
  n = block_reduce(n, AddU(), su);
  const float a = kLog2e / f.T;

  // Targets: the r_k-th candidate, or the first whose cumulative mass reaches
  // top_p * S (in 2^-40 units), whichever comes first.
  unsigned k_rem = f.k_on && (unsigned)f.k < n ? (unsigned)f.k : n;
  bool p_on = f.p_on;
  if (p_on && f.p <= 0.0f) {
    k_rem = 1;
    p_on = false;
  }
  long long m_rem = 0;
  if (p_on) {
    unsigned long long S = 0;
    for (int32_t u = threadIdx.x; u < NU; u += kFiltThreads) {
      const uint4 r = unit_cached<DT, VEC>(row, u, fp.V);
#pragma unroll
      for (int e = 0; e < EPU; ++e) {
        const float x = elt<DT, VEC>(r, e);
        if (is_candidate(x)) S += fixed_mass(x, M, a);
      }
    }
    S = block_reduce(S, AddU64(), sl);
    m_rem = (long long)ceil((double)f.p * (double)S);
  }

  // Radix select on the order-preserving keys, eight bits at a time from the
  // top; larger keys come first.
  uint32_t prefix = 0, pmask = 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kFiltThreads) {
      s_cnt[i] = 0u;
      s_mass[i] = 0ull;
    }
    __syncthreads();
    for (int32_t u = threadIdx.x; u < NU; u += kFiltThreads) {
      const uint4 r = unit_cached<DT, VEC>(row, u, fp.V);
#pragma unroll
      for (int e = 0; e < EPU; ++e) {
        const float x = elt<DT, VEC>(r, e);
        if (!is_candidate(x)) continue;
        const uint32_t key = ordered_bits(x);
        if ((key & pmask) != prefix) continue;
        const uint32_t d = (key >> shift) & 0xFFu;
        atomicAdd(&s_cnt[d], 1u);
        if (p_on) atomicAdd(&s_mass[d], fixed_mass(x, M, a));
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned c = 0;
      long long m = 0;
      int d = 255, last = -1;
      for (; d >= 0; --d) {
        if (s_cnt[d] == 0u) continue;
        last = d;
        if (c + s_cnt[d] >= k_rem || (p_on && m + (long long)s_mass[d] >= m_rem)) break;
        c += s_cnt[d];
        m += (long long)s_mass[d];
      }
      if (d < 0) d = last < 0 ? 0 : last;  // cannot happen: the targets lie inside the counts
      s_sel[0] = (uint32_t)d;
      s_sel[1] = c;
      sl[0] = (unsigned long long)m;
    }
    __syncthreads();
    const uint32_t d = s_sel[0];
    k_rem -= s_sel[1];
    m_rem -= (long long)sl[0];
    prefix |= d << shift;
    pmask |= 0xFFu << shift;
    __syncthreads();
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
  const int32_t chunk = (NU + kFiltThreads - 1) / kFiltThreads;
  const int32_t u0 = threadIdx.x * chunk, u1 = min(u0 + chunk, NU);
  unsigned mine = 0;
  for (int32_t u = u0; u < u1; ++u) {
    const uint4 r = unit_cached<DT, VEC>(row, u, fp.V);
#pragma unroll
    for (int e = 0; e < EPU; ++e) {
      const float x = elt<DT, VEC>(r, e);
      mine += (is_candidate(x) && ordered_bits(x) == key_b) ? 1u : 0u;
    }
  }
  // Exclusive scan of the threads' counts (warp scan, then the warps' totals).
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) su[warp] = incl;
  __syncthreads();
  unsigned before = incl - mine;
  for (int i = 0; i < warp; ++i) before += su[i];
  if (threadIdx.x == 0) s_sel[2] = 0xFFFFFFFFu;
  __syncthreads();
  if (before < n_take && n_take <= before + mine) {
    unsigned seen = before;
    for (int32_t u = u0; u < u1 && s_sel[2] == 0xFFFFFFFFu; ++u) {
      const uint4 r = unit_cached<DT, VEC>(row, u, fp.V);
      for (int e = 0; e < EPU; ++e) {
        const float x = elt<DT, VEC>(r, e);
        if (is_candidate(x) && ordered_bits(x) == key_b && ++seen == n_take) {
          s_sel[2] = (uint32_t)(u * EPU + e);
          break;
        }
      }
    }
  }
  __syncthreads();
  const uint32_t idx_b = s_sel[2];

  // The Gumbel-max over K: a Philox block per group holding a member of K.
  const uint64_t sd = fp.seed[b], of = fp.offset[b];
  const PhiloxRow ph =
      philox_row((uint32_t)b, (uint32_t)of, (uint32_t)(of >> 32), (uint32_t)sd, (uint32_t)(sd >> 32));
  float bs = -INFINITY;
  int32_t bi = INT32_MAX;
  for (int32_t u = threadIdx.x; u < NU; u += kFiltThreads) {
    const uint4 r = unit_cached<DT, VEC>(row, u, fp.V);
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
  }
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
  return reinterpret_cast<void*>(&filter_check_kernel<DT, VEC>);
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.B);
  cfg.blockDim = dim3(kFiltThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, pick(dtype, vec, exact), args);
}

}  // namespace

cudaError_t launch_filter(const FilterParams& p, int dtype, bool vec, cudaStream_t stream) {
  cudaError_t e = launch_one(p, dtype, vec, false, stream);
  if (e != cudaSuccess) return e;
  return launch_one(p, dtype, vec, true, stream);
}

}  // namespace gsample
