// Row sampler for small batches: one thread-block cluster per row. The
// computation is the one of sample_kernel ("Softmax-free GPU sampling:
// Gumbel-max categorical sampling kernel", lablup/mlxcel issue #900, Task 1:
// score = x/T + g with g from the per-(row, element) Philox stream, one
// index-carrying max per row; greedy when T <= 0), only laid out for latency.
//
// When a batch has too few units to give every warp of a full wave a few tiles,
// the flat split spends most of each warp's time on its fixed costs: the row
// setup, the first exact candidates, and a chain of L2 round trips to merge.
// Here each CTA of the row's cluster requests its whole slice at once with
// cp.async, scores each thread's largest logit exactly to get the bound L,
// and then runs Philox four groups per thread with the same logit threshold
// and word bound as sample_kernel. The rare survivors are scored exactly. The
// CTAs' best keys are merged by rank 0 over distributed shared memory, which
// writes the answer: no global atomics, no workspace traffic. The only waits
// are hardware CTA and cluster barriers.
#include <cooperative_groups.h>

#include <cstdint>

#include "gsample_internal.h"
#include "gsample_slice.cuh"

namespace cg = cooperative_groups;

namespace gsample {
namespace {

using namespace slice;

constexpr int kRcThreads = 512;
#ifndef GSAMPLE_RC_CHUNKS
#define GSAMPLE_RC_CHUNKS 4
#endif
constexpr int kRcWarps = kRcThreads / 32;

// Packed maxima of two pairs of 16-bit logits (bf16 when DT is 1, else f16).
template <int DT>
__device__ __forceinline__ uint32_t rc_hmax2(uint32_t a, uint32_t b) {
  if constexpr (DT == 1) {
    __nv_bfloat162 m = __hmax2(*reinterpret_cast<__nv_bfloat162*>(&a),
                               *reinterpret_cast<__nv_bfloat162*>(&b));
    return *reinterpret_cast<uint32_t*>(&m);
  } else {
    __half2 m = __hmax2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
    return *reinterpret_cast<uint32_t*>(&m);
  }
}

struct RcBest {
  float s;
  int32_t i;
};

// The rare exact scores of one group, out of line so that the sweep's loop
// code stays small.
__device__ __noinline__ RcBest rc_score_cold(uint32_t g, float x0, float x1, float x2, float x3,
                                             uint4 w, Prune pr, ReachTest rt, float T, float bs,
                                             int32_t bi) {
  score_group(g, x0, x1, x2, x3, w, pr, rt, T, &bs, &bi);
  return RcBest{bs, bi};
}

// Block-wide (score, index) argmax as a packed key; every thread gets it.
__device__ __forceinline__ unsigned long long rc_block_best(float s, int32_t i,
                                                            unsigned long long* red) {
  warp_argmax(s, i);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = (i != INT32_MAX && s > -INFINITY) ? pack_key(s, i) : 0ull;
  __syncthreads();
  const unsigned long long k = warp_max_u64(lane < kRcWarps ? red[lane] : 0ull);
  __syncthreads();  // red may be reused
  return k;
}

template <int DT, bool VEC, bool RESIDENT>
__global__ void __launch_bounds__(kRcThreads, 1) sample_cluster_kernel(const RowClusterParams p) {
  using C = HCfg<DT, VEC>;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ unsigned long long s_red[kRcWarps];
  __shared__ unsigned long long s_best;  // this CTA's best key, read by rank 0

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
  const float T = p.temperature ? __ldg(p.temperature + b) : 0.0f;
  const bool sampled = T > 0.0f;  // NaN and T <= 0: greedy
  // The row's seed and offset are requested now, so their latency hides behind
  // the slice load (greedy launches pass no arrays).
  const uint64_t sd = p.seed ? __ldg(p.seed + b) : 0ull;
  const uint64_t of = p.offset ? __ldg(p.offset + b) : 0ull;

  auto unit_at = [&](int32_t u) -> uint4 {
    if constexpr (RESIDENT)
      return lds128(slice + (uint32_t)(u - u_lo) * 16u);
    else
      return load_unit<DT, VEC>(row, u, p.V, pol);
  };

  // The thread's largest logit, lowest index on ties: the greedy answer, and
  // the first exact candidate of a sampled row. Unit maxima first (packed
  // half2 maxima for 16-bit logits; NaN is ignored unless a whole unit is NaN,
  // and a NaN maximum never wins), then the first element of the best unit
  // that equals it. On the resident path the thread's units are requested in
  // GSAMPLE_RC_CHUNKS groups and each is reduced as it lands.
  float cand_x = -INFINITY;
  int32_t cand_u = -1;
  auto unit_max_of = [&](int32_t u, const uint4& r) {
    float m;
    if constexpr (C::kF32Bits) {
      m = fmaxf(fmaxf(__uint_as_float(r.x), __uint_as_float(r.y)),
                fmaxf(__uint_as_float(r.z), __uint_as_float(r.w)));
    } else {
      const uint32_t h = rc_hmax2<DT>(rc_hmax2<DT>(r.x, r.y), rc_hmax2<DT>(r.z, r.w));
      m = fmaxf(half_to_f32<DT>(h & 0xFFFFu), half_to_f32<DT>(h >> 16));
    }
    if (m > cand_x) {
      cand_x = m;
      cand_u = u;
    }
  };
  if constexpr (RESIDENT) {
    load_slice_then<DT, VEC, kRcThreads, GSAMPLE_RC_CHUNKS>(row, u_lo, u_hi, p.V, slice, pol,
                                                           unit_max_of);
  } else {
    for (int32_t u = u_lo + tid; u < u_hi; u += kRcThreads) unit_max_of(u, unit_at(u));
  }
  int32_t cand_i = INT32_MAX;
  if (cand_u >= 0) {
    const uint4 r = unit_at(cand_u);
#pragma unroll
    for (int e = C::kEPU - 1; e >= 0; --e)
      if (elt<DT, VEC>(r, e) == cand_x) cand_i = cand_u * C::kEPU + e;
  }

  float bs = -INFINITY;
  int32_t bi = INT32_MAX;
  if (!sampled) {
    bs = cand_x;
    bi = cand_x > -INFINITY ? cand_i : INT32_MAX;
  } else {
    const PhiloxRow ph = philox_row((uint32_t)b, (uint32_t)of, (uint32_t)(of >> 32), (uint32_t)sd,
                                    (uint32_t)(sd >> 32));
    if (cand_i != INT32_MAX && cand_x > -INFINITY) {
      const uint4 blk = philox_row_1((uint32_t)cand_i >> 2, ph);
      take_better(exact_score(cand_x, word_of(blk, cand_i & 3), T), cand_i, bs, bi);
    }
    const float L = score_of_key(rc_block_best(bs, bi, s_red));
    const Prune pr = make_prune(L, T);
    const ReachTest rt = make_reach(pr, 1.0f / T);

    // Four 4-element groups per thread at a time (four units of binary32, two
    // of 16-bit), one Philox block each, the word bound, then the rare exact
    // scores.
    constexpr int kUPB = 4 / C::kGPU;
    const int32_t n_iter = (u_hi - u_lo + kRcThreads - 1) / kRcThreads;
    for (int32_t it = 0; it < n_iter; it += kUPB) {
      uint4 r[kUPB];
      float xm[4];
      uint32_t g[4], wt[4];
      bool ok[4];
#pragma unroll
      for (int j = 0; j < kUPB; ++j) {
        const int32_t u = u_lo + tid + (it + j) * kRcThreads;
        const bool valid = u < u_hi;
        r[j] = valid ? unit_at(u) : make_uint4(0, 0, 0, 0);
        if constexpr (C::kF32Bits) {
          xm[j] = fmaxf(fmaxf(__uint_as_float(r[j].x), __uint_as_float(r[j].y)),
                        fmaxf(__uint_as_float(r[j].z), __uint_as_float(r[j].w)));
        } else {
          // Packed maxima of each group's two element pairs, then the larger
          // half (NaN is ignored unless all four are NaN, as with fmaxf).
          const uint32_t m0 = rc_hmax2<DT>(r[j].x, r[j].y), m1 = rc_hmax2<DT>(r[j].z, r[j].w);
          xm[2 * j] = fmaxf(half_to_f32<DT>(m0 & 0xFFFFu), half_to_f32<DT>(m0 >> 16));
          xm[2 * j + 1] = fmaxf(half_to_f32<DT>(m1 & 0xFFFFu), half_to_f32<DT>(m1 >> 16));
        }
#pragma unroll
        for (int h = 0; h < C::kGPU; ++h) {
          const int jj = j * C::kGPU + h;
          ok[jj] = valid && xm[jj] >= pr.thr_x;
          g[jj] = (uint32_t)(u * C::kGPU + h);
        }
      }
      if (!__any_sync(0xFFFFFFFFu, ok[0] || ok[1] || ok[2] || ok[3])) continue;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) wt[jj] = word_threshold(xm[jj], pr, rt);
      uint4 w[4];
      philox_row_x4(g, ph, w);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        if (ok[jj] && max_word(w[jj]) >= wt[jj]) {
          const uint4 rj = r[jj / C::kGPU];
          const int h = jj % C::kGPU;
          if constexpr (DT != 0) {
            // 16-bit rows: the exact scores out of line (measured faster at
            // B = 32-64); binary32 rows keep them inline (faster on the
            // small f32 sweeps).
            const RcBest sb = rc_score_cold(g[jj], elt<DT, VEC>(rj, 4 * h),
                                            elt<DT, VEC>(rj, 4 * h + 1),
                                            elt<DT, VEC>(rj, 4 * h + 2),
                                            elt<DT, VEC>(rj, 4 * h + 3), w[jj], pr, rt, T, bs, bi);
            bs = sb.s;
            bi = sb.i;
          } else {
            score_group(g[jj], elt<DT, VEC>(rj, 4 * h), elt<DT, VEC>(rj, 4 * h + 1),
                        elt<DT, VEC>(rj, 4 * h + 2), elt<DT, VEC>(rj, 4 * h + 3), w[jj], pr, rt, T,
                        &bs, &bi);
          }
        }
      }
    }
  }

  // Rank 0 merges the CTAs' best keys over distributed shared memory; the
  // second barrier keeps every CTA's shared memory alive until it has read.
  const unsigned long long best = rc_block_best(bs, bi, s_red);
  if (tid == 0) s_best = best;
  cluster.sync();
  if (rank == 0 && warp == 0) {
    const unsigned long long k =
        warp_max_u64(lane < p.cluster ? *cluster.map_shared_rank(&s_best, lane) : 0ull);
    if (lane == 0) p.out_idx[b] = index_of_key(k);
  }
  cluster.sync();
}

template <int DT, bool VEC, bool RES>
void* sk() {
  return reinterpret_cast<void*>(&sample_cluster_kernel<DT, VEC, RES>);
}

void* select_rc(int dtype, bool vec, bool resident) {
  switch (dtype * 4 + (vec ? 2 : 0) + (resident ? 1 : 0)) {
    case 0: return sk<0, false, false>();
    case 1: return sk<0, false, true>();
    case 2: return sk<0, true, false>();
    case 3: return sk<0, true, true>();
    case 4: return sk<1, false, false>();
    case 5: return sk<1, false, true>();
    case 6: return sk<1, true, false>();
    case 7: return sk<1, true, true>();
    case 8: return sk<2, false, false>();
    case 9: return sk<2, false, true>();
    case 10: return sk<2, true, false>();
    default: return sk<2, true, true>();
  }
}

constexpr size_t kRcSmemLimit = 200 * 1024;

}  // namespace

size_t rc_smem_limit() { return kRcSmemLimit; }

void* rc_kernel(int dtype, bool vec, bool resident, int* threads) {
  *threads = kRcThreads;
  return select_rc(dtype, vec, resident);
}

int rc_max_cluster(int dtype, bool vec) {
  for (int res = 0; res < 2; ++res) {
    void* fn = select_rc(dtype, vec, res != 0);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             res ? (int)kRcSmemLimit : 0) != cudaSuccess)
      return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(16);
  cfg.blockDim = dim3(kRcThreads);
  cfg.dynamicSmemBytes = kRcSmemLimit;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 16;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int size = 0;
  if (cudaOccupancyMaxPotentialClusterSize(&size, select_rc(dtype, vec, true), &cfg) !=
      cudaSuccess)
    return 0;
  return size;
}

cudaError_t launch_sample_cluster(const RowClusterParams& p, int dtype, bool vec,
                                  cudaStream_t stream) {
  const size_t need = (size_t)p.units_per_cta * 16;
  const bool resident = need <= kRcSmemLimit;
  void* fn = select_rc(dtype, vec, resident);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * p.cluster));
  cfg.blockDim = dim3(kRcThreads);
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
