// Categorical baseline sampler: softmax(x / T) drawn by the inverse CDF of one
// uniform per row. This is the path "Softmax-free GPU sampling: Gumbel-max
// categorical sampling kernel" (lablup/mlxcel issue #900) measures Gumbel-max
// against ("Background": a normalisation pass over the vocabulary before the
// categorical draw; "Performance validation": baseline categorical path vs
// Gumbel-max over V x B). It exists to state that comparison as a measured
// ratio on this GPU.
//
// Definition (per row, T > 0): M = the largest finite logit, weights
// e_i = exp((x_i - M) / T) (0 for -inf and NaN), S = sum e_i, t = u * S with u
// the uniform of element 0's Philox word (the Gumbel path's stream and
// mapping), answer = the smallest i whose running sum exceeds t. T <= 0 or NaN
// is greedy; a +inf logit takes all the mass (its lowest index); a row with no
// candidate returns -1.
//
// Layout: one thread-block cluster per row, as for the HLG sampler. Each CTA
// requests its whole slice at once with cp.async into shared memory. Each
// thread owns a contiguous chunk of the slice, so the running sum is a scan:
// thread sums, then a block scan, then a scan over the cluster's CTA totals
// read through distributed shared memory. Every CTA computes the same t and
// finds the CTA, then the thread, whose range holds it; that thread walks its
// chunk. Float sums give the CDF to about 1e-6 of S; the tests check that the
// index returned is the inverse CDF of a target within 1e-5 of S of the exact
// one, and the draws' distribution by chi-square.
#include <cooperative_groups.h>

#include <cstdint>

#include "gsample_internal.h"
#include "gsample_slice.cuh"

namespace cg = cooperative_groups;

namespace gsample {
namespace {

using namespace slice;

constexpr int kCatThreads = 512;
constexpr int kCatWarps = kCatThreads / 32;

// e = 2^((x - M) * log2(e) / T): written with explicit roundings so that the
// thread-sum pass and the final walk compute bit-identical weights.
__device__ __forceinline__ float cat_weight(float x, float M, float k) {
  if (!(x > -INFINITY)) return 0.0f;  // -inf, NaN
  const float d = __fsub_rn(x, M);
  if (d == 0.0f) return 1.0f;
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(__fmul_rn(d, k)));
  return y;
}

struct CatPart {
  float M;      // largest finite logit of the CTA's slice
  int32_t inf;  // lowest +inf index of the slice, or INT32_MAX
};

template <int DT, bool VEC, bool RESIDENT>
__global__ void __launch_bounds__(kCatThreads) categorical_kernel(const RowClusterParams p) {
  using C = HCfg<DT, VEC>;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ CatPart s_part;  // read by the whole cluster
  __shared__ float s_total;   // this CTA's weight sum, read by the whole cluster
  __shared__ unsigned long long s_best;
  __shared__ float s_wf[kCatWarps];
  __shared__ int32_t s_wi[kCatWarps];
  __shared__ unsigned long long s_wk[kCatWarps];
  __shared__ float s_row[3];  // M, target CTA's local target, flags
  __shared__ int32_t s_pick[2];

  pdl_wait_then_release();
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t b = blockIdx.x / p.cluster;
  const int32_t NU = p.units_per_row;
  const int32_t u_lo = rank * p.units_per_cta;
  const int32_t u_hi = min(NU, u_lo + p.units_per_cta);
  const char* row = p.logits + b * p.ld_bytes;
  const uint32_t slice = (uint32_t)__cvta_generic_to_shared(smem);
  const uint64_t pol = evict_first_policy();
  const float T = __ldg(p.temperature + b);
  const bool sampled = T > 0.0f;
  // The row's seed and offset, requested now so that their latency hides
  // behind the slice load.
  const uint64_t sd = sampled ? __ldg(p.seed + b) : 0ull;
  const uint64_t of = sampled ? __ldg(p.offset + b) : 0ull;
  float u_row = 0.0f;

  if constexpr (RESIDENT) {
    for (int32_t u = u_lo + tid; u < u_hi; u += kCatThreads) {
      const uint32_t dst = slice + (uint32_t)(u - u_lo) * 16u;
      if (VEC && (u + 1) * C::kEPU <= p.V)
        cp_async16(dst, row + (size_t)u * 16, pol);
      else
        sts128(dst, load_unit<DT, VEC>(row, u, p.V, pol));
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  // The row's uniform (element 0's word of its Philox stream), needed only by
  // warp 0 after the scans, is drawn while the slice is in flight.
  if (warp == 0 && sampled) {
    const uint4 blk = philox4x32_10(make_uint4(0u, (uint32_t)b, (uint32_t)of, (uint32_t)(of >> 32)),
                                    (uint32_t)sd, (uint32_t)(sd >> 32));
    u_row = uniform_open(blk.x);
  }
  if constexpr (RESIDENT) {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();  // each thread reads units other threads copied
  }
  auto unit_at = [&](int32_t u) -> uint4 {
    if constexpr (RESIDENT)
      return lds128(slice + (uint32_t)(u - u_lo) * 16u);
    else
      return load_unit<DT, VEC>(row, u, p.V, pol);
  };
  // This thread's contiguous chunk of units [c0, c1).
  const int32_t n = max(0, u_hi - u_lo);
  const int32_t per = n / kCatThreads, rem = n % kCatThreads;
  const int32_t c0 = u_lo + tid * per + min(tid, rem);
  const int32_t c1 = c0 + per + (tid < rem ? 1 : 0);

  // Pass A: the thread's largest logit (lowest index), largest finite logit and
  // lowest +inf index.
  float cand_x = -INFINITY, fmax_x = -INFINITY;
  int32_t cand_i = INT32_MAX, inf_i = INT32_MAX;
  for (int32_t u = c0; u < c1; ++u) {
    const uint4 r = unit_at(u);
#pragma unroll
    for (int e = 0; e < C::kEPU; ++e) {
      const float x = elt<DT, VEC>(r, e);
      const int32_t i = u * C::kEPU + e;
      if (x > cand_x) {
        cand_x = x;
        cand_i = i;
      }
      if (x == INFINITY) {
        if (inf_i == INT32_MAX) inf_i = i;
      } else {
        fmax_x = fmaxf(fmax_x, x);
      }
    }
  }

  int64_t answer = -1;
  bool have_answer = false;  // the answer is known to every CTA (rank 0 writes it)
  if (!sampled) {
    // Greedy: CTA best key; rank 0 merges the cluster's keys below.
    float s = cand_x;
    int32_t i = cand_x > -INFINITY ? cand_i : INT32_MAX;
    warp_argmax(s, i);
    if (lane == 0) s_wk[warp] = (i != INT32_MAX && s > -INFINITY) ? pack_key(s, i) : 0ull;
    __syncthreads();
    if (warp == 0) {
      const unsigned long long k = warp_max_u64(lane < kCatWarps ? s_wk[lane] : 0ull);
      if (lane == 0) s_best = k;
    }
    cluster.sync();
    if (rank == 0 && warp == 0) {
      const unsigned long long k =
          warp_max_u64(lane < p.cluster ? *cluster.map_shared_rank(&s_best, lane) : 0ull);
      if (lane == 0) p.out_idx[b] = index_of_key(k);
    }
    cluster.sync();
    return;
  }

  // Row maximum and +inf over the cluster.
  {
    float m = fmax_x;
    int32_t f = inf_i;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      f = min(f, __shfl_xor_sync(0xFFFFFFFFu, f, o));
    }
    if (lane == 0) {
      s_wf[warp] = m;
      s_wi[warp] = f;
    }
    __syncthreads();
    if (warp == 0) {
      m = lane < kCatWarps ? s_wf[lane] : -INFINITY;
      f = lane < kCatWarps ? s_wi[lane] : INT32_MAX;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        f = min(f, __shfl_xor_sync(0xFFFFFFFFu, f, o));
      }
      if (lane == 0) s_part = CatPart{m, f};
    }
  }
  cluster.sync();
  if (warp == 0) {
    CatPart q{-INFINITY, INT32_MAX};
    if (lane < p.cluster) q = *cluster.map_shared_rank(&s_part, lane);
    float m = q.M;
    int32_t f = q.inf;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      f = min(f, __shfl_xor_sync(0xFFFFFFFFu, f, o));
    }
    if (lane == 0) {
      s_row[0] = m;
      s_pick[0] = f;
    }
  }
  __syncthreads();
  const float M = s_row[0];
  if (s_pick[0] != INT32_MAX) {  // a +inf logit takes all the mass
    answer = s_pick[0];
    have_answer = true;
  } else if (!(M > -INFINITY)) {  // nothing can be drawn
    answer = -1;
    have_answer = true;
  }

  float thread_sum = 0.0f, excl = 0.0f;
  const float k = 1.4426950408889634f / T;
  if (!have_answer) {
    // Pass B: thread sums of the weights, then an exclusive block scan.
    for (int32_t u = c0; u < c1; ++u) {
      const uint4 r = unit_at(u);
#pragma unroll
      for (int e = 0; e < C::kEPU; ++e) thread_sum += cat_weight(elt<DT, VEC>(r, e), M, k);
    }
    // Exclusive prefixes are taken from the neighbour's inclusive value, so
    // that a range ends exactly where the next one starts within a warp.
    float incl = thread_sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    float ex_lane = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
    if (lane == 0) ex_lane = 0.0f;
    if (lane == 31) s_wf[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      float wi = lane < kCatWarps ? s_wf[lane] : 0.0f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xFFFFFFFFu, wi, o);
        if (lane >= o) wi += t;
      }
      float ex_warp = __shfl_up_sync(0xFFFFFFFFu, wi, 1);
      if (lane == 0) ex_warp = 0.0f;
      if (lane < kCatWarps) s_wf[lane] = ex_warp;  // exclusive warp offsets
      if (lane == kCatWarps - 1) s_total = wi;
    }
    __syncthreads();
    excl = s_wf[warp] + ex_lane;
  }
  cluster.sync();  // every CTA's total is visible (taken by all CTAs of the row alike)
  if (!have_answer) {
    if (warp == 0) {
      // Scan of the CTA totals; the target t = u * S; the CTA holding it.
      const float tot = lane < p.cluster ? *cluster.map_shared_rank(&s_total, lane) : 0.0f;
      float inc = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += t;
      }
      const float S = __shfl_sync(0xFFFFFFFFu, inc, 31);
      const float t = u_row * S;
      const unsigned hit = __ballot_sync(0xFFFFFFFFu, lane < p.cluster && t < inc);
      const unsigned pos = __ballot_sync(0xFFFFFFFFu, lane < p.cluster && tot > 0.0f);
      const int cstar = hit ? __ffs(hit) - 1 : 31 - __clz(pos);  // else: the last CTA with mass
      float ex = __shfl_up_sync(0xFFFFFFFFu, inc, 1);
      if (lane == 0) ex = 0.0f;
      const float base = __shfl_sync(0xFFFFFFFFu, ex, cstar);
      if (lane == 0) {
        s_pick[1] = cstar;
        s_row[1] = t - base;
      }
    }
  }
  // Done with other CTAs' shared memory; the matching wait is at the exit.
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  __syncthreads();
  if (have_answer) {
    if (rank == 0 && tid == 0) p.out_idx[b] = answer;
  } else if (rank == s_pick[1]) {
    // The thread whose range [excl, excl + sum) holds the local target; if
    // rounding leaves none, the last thread with mass.
    const float tl = s_row[1];
    const bool hold = thread_sum > 0.0f && tl < excl + thread_sum;
    const bool mass = thread_sum > 0.0f;
    const unsigned hw = __ballot_sync(0xFFFFFFFFu, hold), mw = __ballot_sync(0xFFFFFFFFu, mass);
    if (lane == 0) {
      s_wi[warp] = hw ? warp * 32 + __ffs(hw) - 1 : INT32_MAX;
      s_wk[warp] = mw ? (unsigned long long)(warp * 32 + 31 - __clz(mw)) : 0ull;
    }
    __syncthreads();
    if (warp == 0) {
      int32_t first = lane < kCatWarps ? s_wi[lane] : INT32_MAX;
      unsigned long long lastm = lane < kCatWarps ? s_wk[lane] : 0ull;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        first = min(first, __shfl_xor_sync(0xFFFFFFFFu, first, o));
        lastm = max(lastm, __shfl_xor_sync(0xFFFFFFFFu, lastm, o));
      }
      if (lane == 0) s_pick[0] = first != INT32_MAX ? first : (int32_t)lastm;
    }
    __syncthreads();
    if (tid == s_pick[0]) {
      // Walk the chunk; the running sum restarts from 0 to match thread_sum.
      const float r = tl - excl;
      float cum = 0.0f;
      int32_t pick = -1, last = -1;
      for (int32_t u = c0; u < c1 && pick < 0; ++u) {
        const uint4 q = unit_at(u);
#pragma unroll
        for (int e = 0; e < C::kEPU; ++e) {
          const float w = cat_weight(elt<DT, VEC>(q, e), M, k);
          if (w > 0.0f) {
            cum += w;
            last = u * C::kEPU + e;
            if (pick < 0 && r < cum) pick = last;
          }
        }
      }
      p.out_idx[b] = pick >= 0 ? pick : last;
    }
  }
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int DT, bool VEC, bool RES>
void* ck() {
  return reinterpret_cast<void*>(&categorical_kernel<DT, VEC, RES>);
}

void* select_cat(int dtype, bool vec, bool resident) {
  switch (dtype * 4 + (vec ? 2 : 0) + (resident ? 1 : 0)) {
    case 0: return ck<0, false, false>();
    case 1: return ck<0, false, true>();
    case 2: return ck<0, true, false>();
    case 3: return ck<0, true, true>();
    case 4: return ck<1, false, false>();
    case 5: return ck<1, false, true>();
    case 6: return ck<1, true, false>();
    case 7: return ck<1, true, true>();
    case 8: return ck<2, false, false>();
    case 9: return ck<2, false, true>();
    case 10: return ck<2, true, false>();
    default: return ck<2, true, true>();
  }
}

constexpr size_t kCatSmemLimit = 200 * 1024;  // leaves room for the static shared variables

}  // namespace

size_t cat_smem_limit() { return kCatSmemLimit; }

void* cat_kernel(int dtype, bool vec, bool resident, int* threads) {
  *threads = kCatThreads;
  return select_cat(dtype, vec, resident);
}

// One-time per-device setup (as for the HLG kernel): allow clusters of up to
// 16 CTAs and the full slice, then report the largest co-schedulable cluster.
int cat_max_cluster(int dtype, bool vec) {
  for (int res = 0; res < 2; ++res) {
    void* fn = select_cat(dtype, vec, res != 0);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             res ? (int)kCatSmemLimit : 0) != cudaSuccess)
      return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(16);
  cfg.blockDim = dim3(kCatThreads);
  cfg.dynamicSmemBytes = kCatSmemLimit;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 16;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int size = 0;
  if (cudaOccupancyMaxPotentialClusterSize(&size, select_cat(dtype, vec, true), &cfg) !=
      cudaSuccess)
    return 0;
  return size;
}

cudaError_t launch_categorical(const RowClusterParams& p, int dtype, bool vec, cudaStream_t stream) {
  const size_t need = (size_t)p.units_per_cta * 16;
  const bool resident = need <= kCatSmemLimit;
  void* fn = select_cat(dtype, vec, resident);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * p.cluster));
  cfg.blockDim = dim3(kCatThreads);
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
  void* args[] = {const_cast<RowClusterParams*>(&p)};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace gsample
