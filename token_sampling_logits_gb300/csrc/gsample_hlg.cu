// HLG tone-curve sampler ("HLG sampling -- a piecewise tone curve on the
// logits", mlx-bun docs/design/hlg-sampling.md): per-row log-probs l, pivot mu,
// z = l - mu, the C1 toe / linear-mid / shoulder curve g(z) ("The transfer
// function"), then Gumbel-max over g(z)/T + gumbel ("Temperature semantics":
// the temperature folds into the gain, which is the same as dividing the curve
// by T).
//
// Both pivots make the log-normaliser cancel out of z:
//   top     mu = l_max - c       =>  z_i = x_i - max_j x_j + c
//   entropy mu = sum_j p_j l_j   =>  z_i = x_i - sum_j p_j x_j
// so sweep 1 only needs the row max (top) or the softmax-weighted mean of the
// logits (entropy, accumulated online as max / sum e^(x-max) / sum e^(x-max) x).
//
// Layout: one thread-block cluster of `cluster` CTAs per row. Each CTA streams
// its slice of the row from HBM once, keeping it in shared memory (RESIDENT),
// reduces its partial statistics, and the cluster exchanges them through
// distributed shared memory after a hardware cluster barrier. Sweep 2 then
// scores the slice from shared memory. If a slice is too large for shared
// memory the same kernel re-reads it from global memory in sweep 2
// (!RESIDENT). Candidates merge through the same packed-key workspace as the
// plain sampler; no CTA ever spins on another.
#include <cooperative_groups.h>

#include <cstdint>

#include "gsample_internal.h"

namespace cg = cooperative_groups;

namespace gsample {
namespace {

template <int DT, bool VEC>
struct HCfg {
  static constexpr int kEPU = VEC ? (DT == 0 ? 4 : 8) : 4;
  static constexpr int kGPU = kEPU / 4;
  static constexpr bool kF32Bits = DT == 0 || !VEC;
};

template <int DT>
__device__ __forceinline__ float half_to_f32(uint32_t h) {
  return DT == 1 ? bf16_bits_to_f32(h) : f16_bits_to_f32(h);
}

template <int DT, bool VEC>
__device__ __forceinline__ float elt(const uint4& r, int e) {
  if constexpr (HCfg<DT, VEC>::kF32Bits) {
    return __uint_as_float(word_of(r, e));
  } else {
    const uint32_t w = word_of(r, e >> 1);
    return half_to_f32<DT>((e & 1) ? (w >> 16) : (w & 0xFFFFu));
  }
}

template <int DT, bool VEC>
__device__ __forceinline__ uint4 load_unit(const char* row, int32_t u, int32_t V, uint64_t pol) {
  constexpr int EPU = HCfg<DT, VEC>::kEPU;
  const int32_t e0 = u * EPU;
  if constexpr (VEC) {
    if (e0 + EPU <= V) return ld_stream_v4(row + (size_t)u * 16, pol);
  }
  uint32_t w[4];
  if constexpr (HCfg<DT, VEC>::kF32Bits) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float x = -INFINITY;
      if (e0 + e < V) {
        if constexpr (DT == 0)
          x = __ldg(reinterpret_cast<const float*>(row) + e0 + e);
        else
          x = half_to_f32<DT>(__ldg(reinterpret_cast<const unsigned short*>(row) + e0 + e));
      }
      w[e] = __float_as_uint(x);
    }
  } else {
    constexpr uint32_t ninf = DT == 1 ? 0xFF80u : 0xFC00u;
    const unsigned short* h = reinterpret_cast<const unsigned short*>(row);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t lo = (e0 + 2 * k < V) ? (uint32_t)__ldg(h + e0 + 2 * k) : ninf;
      const uint32_t hi = (e0 + 2 * k + 1 < V) ? (uint32_t)__ldg(h + e0 + 2 * k + 1) : ninf;
      w[k] = lo | (hi << 16);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Online softmax moments of finite logits: M = max x, S = sum e^(x-M),
// W = sum e^(x-M) x. Empty: M = -inf, S = W = 0.
struct Moments {
  float M, S, W;
};

__device__ __forceinline__ Moments merge(Moments a, Moments b) {
  if (b.M == -INFINITY) return a;
  if (a.M == -INFINITY) return b;
  const float M = fmaxf(a.M, b.M);
  const float fa = __expf(a.M - M), fb = __expf(b.M - M);
  return Moments{M, a.S * fa + b.S * fb, a.W * fa + b.W * fb};
}

__device__ __forceinline__ void push(Moments& mo, float x) {
  if (x > mo.M) {
    const float f = mo.M == -INFINITY ? 0.0f : __expf(mo.M - x);
    mo.S = mo.S * f + 1.0f;
    mo.W = mo.W * f + x;
    mo.M = x;
  } else {
    const float e = __expf(x - mo.M);
    mo.S += e;
    mo.W += e * x;
  }
}

// The tone curve in binary32 ("The transfer function"). rbt, rbh are 1/beta.
struct Curve {
  float m, w, bt, bh, rbt, rbh;
};

__device__ __forceinline__ float tone(const Curve& c, float z) {
  if (z < -c.w) return -c.m * c.w - c.m * c.bt * log1pf((-z - c.w) * c.rbt);
  if (z > c.w) return c.m * c.w + c.m * c.bh * log1pf((z - c.w) * c.rbh);
  return c.m * z;
}

// z below which the curve stays under Y (the inverse curve), or -inf.
__device__ __forceinline__ float tone_inverse(const Curve& c, float Y) {
  const float mw = c.m * c.w;
  if (Y < -mw) return -c.w - c.bt * expm1f((-Y - mw) / (c.m * c.bt));
  if (Y > mw) return c.w + c.bh * expm1f((Y - mw) / (c.m * c.bh));
  return Y / c.m;
}

struct RowState {
  float shift;   // z = x + shift
  bool pinf;     // the row holds a +inf logit: only +inf entries can win
};

__device__ __forceinline__ float hlg_score(const Curve& c, const RowState& rs, float x,
                                           uint32_t word, float rT) {
  if (x == INFINITY) return INFINITY;
  const float y = tone(c, x + rs.shift);
  return y * rT + gumbel_of_word(word);
}

template <int DT, bool VEC, bool RESIDENT>
__global__ void __launch_bounds__(kThreads) hlg_kernel(const HlgParams p) {
  using C = HCfg<DT, VEC>;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ Moments s_warp[kWarps];
  __shared__ Moments s_part;  // this CTA's partial, read by the whole cluster
  __shared__ int s_pinf;
  __shared__ RowState s_row;

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t b = blockIdx.x / p.cluster;
  const int32_t NU = p.units_per_row;
  const int32_t u_lo = rank * p.units_per_cta;
  const int32_t u_hi = min(NU, u_lo + p.units_per_cta);
  const char* row = p.logits + b * p.ld_bytes;
  uint4* slice = reinterpret_cast<uint4*>(smem);
  const uint64_t pol = evict_first_policy();
  WsRow* ws = p.ws + b;

  const float T = __ldg(p.temperature + b);
  const bool sampled = T > 0.0f;
  const bool entropy = p.pivot_mode == 1;
  if (threadIdx.x == 0) s_pinf = 0;
  __syncthreads();

  // Sweep 1: stream the slice once; statistics (sampled) or argmax (greedy).
  Moments mo{-INFINITY, 0.0f, 0.0f};
  float bs = -INFINITY;
  int32_t bi = INT32_MAX;
  bool pinf = false;
  float cand_x = -INFINITY;
  int32_t cand_i = INT32_MAX;
  for (int32_t u = u_lo + threadIdx.x; u < u_hi; u += kThreads) {
    const uint4 r = load_unit<DT, VEC>(row, u, p.V, pol);
    if constexpr (RESIDENT) slice[u - u_lo] = r;
#pragma unroll
    for (int e = 0; e < C::kEPU; ++e) {
      const float x = elt<DT, VEC>(r, e);
      const int32_t i = u * C::kEPU + e;
      if (x > cand_x) {  // greedy answer, and the first candidate of a sampled row
        cand_x = x;
        cand_i = i;
      }
      if (sampled) {
        if (x == INFINITY) pinf = true;
        if (entropy) {
          if (x > -INFINITY && x < INFINITY) push(mo, x);
        } else if (x < INFINITY) {
          mo.M = fmaxf(mo.M, x);
        }
      }
    }
  }

  if (!sampled) {
    bs = cand_x;
    bi = cand_x > -INFINITY ? cand_i : INT32_MAX;
  } else {
    // Cluster-wide pivot statistics.
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      Moments other;
      other.M = __shfl_xor_sync(0xFFFFFFFFu, mo.M, o);
      other.S = __shfl_xor_sync(0xFFFFFFFFu, mo.S, o);
      other.W = __shfl_xor_sync(0xFFFFFFFFu, mo.W, o);
      mo = entropy ? merge(mo, other) : Moments{fmaxf(mo.M, other.M), 0.0f, 0.0f};
    }
    if (__any_sync(0xFFFFFFFFu, pinf) && lane == 0) atomicOr(&s_pinf, 1);
    if (lane == 0) s_warp[warp] = mo;
    __syncthreads();
    if (threadIdx.x == 0) {
      Moments acc = s_warp[0];
      for (int k = 1; k < kWarps; ++k)
        acc = entropy ? merge(acc, s_warp[k]) : Moments{fmaxf(acc.M, s_warp[k].M), 0.0f, 0.0f};
      if (s_pinf) acc.M = INFINITY;  // flag travels with the partial
      s_part = acc;
    }
    cluster.sync();
    if (warp == 0) {
      Moments acc{-INFINITY, 0.0f, 0.0f};
      bool any_pinf = false;
      // Every CTA merges the same partials in the same (rank) order, so all
      // CTAs of the row get bit-identical pivot statistics.
      for (int k = 0; k < p.cluster; ++k) {
        const Moments* rp = cluster.map_shared_rank(&s_part, k);
        Moments o = *rp;
        if (o.M == INFINITY) {
          any_pinf = true;
          continue;
        }
        acc = entropy ? merge(acc, o) : Moments{fmaxf(acc.M, o.M), 0.0f, 0.0f};
      }
      if (lane == 0) {
        RowState rs;
        rs.pinf = any_pinf;
        rs.shift = entropy ? -(acc.W / acc.S) : (p.pivot_offset - acc.M);
        s_row = rs;
      }
    }
    // Done reading other CTAs' shared memory; the matching wait is at the end.
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    __syncthreads();
    const RowState rs = s_row;

    const Curve cv{p.m, p.w, p.beta_t, p.beta_h, 1.0f / p.beta_t, 1.0f / p.beta_h};
    const float rT = 1.0f / T;
    const uint64_t sd = __ldg(p.seed + b), of = __ldg(p.offset + b);
    const uint32_t k0 = (uint32_t)sd, k1 = (uint32_t)(sd >> 32);
    const uint32_t o0 = (uint32_t)of, o1 = (uint32_t)(of >> 32);
    const uint32_t row_id = (uint32_t)b;

    // First candidate: this thread's largest logit, scored exactly.
    if (cand_i != INT32_MAX && cand_x > -INFINITY && (!rs.pinf || cand_x == INFINITY)) {
      const uint4 blk = philox4x32_10(make_uint4((uint32_t)cand_i >> 2, row_id, o0, o1), k0, k1);
      take_better(hlg_score(cv, rs, cand_x, word_of(blk, cand_i & 3), rT), cand_i, bs, bi);
    }
    float L;
    {
      float s = bs;
      int32_t i = bi;
      warp_argmax(s, i);
      unsigned long long old = 0ull;
      if (lane == 0) {
        if (i != INT32_MAX && s > -INFINITY)
          old = atomicMax(&ws->key, pack_key(s, i));
        else
          old = __ldcg(&ws->key);
      }
      old = __shfl_sync(0xFFFFFFFFu, old, 0);
      L = fmaxf(s, score_of_key(old));
    }
    // Exact pruning in logit space: x < x_thr implies tone(x + shift)/T + max g < L.
    float x_thr = -INFINITY;
    if (rs.pinf || L == INFINITY) {
      x_thr = INFINITY;
    } else if (L > -INFINITY && T >= 1e-20f && T <= 1e20f) {
      const float margin = 1e-3f * (1.0f + fabsf(L));
      const float z_thr = tone_inverse(cv, (L - kGumbelMax - margin) * T);
      x_thr = z_thr - rs.shift - 1e-3f * (1.0f + fabsf(z_thr)) - 1e-3f * (1.0f + fabsf(rs.shift));
      if (!(x_thr == x_thr)) x_thr = -INFINITY;  // NaN guard: no pruning
    }

    // Sweep 2 over the slice, four-element Philox groups.
    for (int32_t u = u_lo + threadIdx.x; u < u_hi; u += kThreads) {
      uint4 r;
      if constexpr (RESIDENT)
        r = slice[u - u_lo];
      else
        r = load_unit<DT, VEC>(row, u, p.V, pol);
#pragma unroll
      for (int h = 0; h < C::kGPU; ++h) {
        float gm = elt<DT, VEC>(r, 4 * h);
#pragma unroll
        for (int e = 1; e < 4; ++e) gm = fmaxf(gm, elt<DT, VEC>(r, 4 * h + e));
        if (!(gm >= x_thr)) continue;
        const uint32_t gid = (uint32_t)(u * C::kGPU + h);
        const uint4 blk = philox4x32_10(make_uint4(gid, row_id, o0, o1), k0, k1);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float x = elt<DT, VEC>(r, 4 * h + t);
          if (!(x >= x_thr) || x == -INFINITY) continue;
          take_better(hlg_score(cv, rs, x, word_of(blk, t), rT), (int32_t)(4 * gid + t), bs, bi);
        }
      }
    }
  }

  // Merge into the row's key; the last CTA of the row writes the answer.
  warp_argmax(bs, bi);
  if (lane == 0 && bi != INT32_MAX && bs > -INFINITY) atomicMax(&ws->key, pack_key(bs, bi));
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned t = atomicAdd(&ws->ticket, 1u);
    if ((int)t == p.cluster - 1) {
      __threadfence();
      const unsigned long long key = atomicExch(&ws->key, 0ull);
      atomicExch(&ws->ticket, 0u);
      p.out_idx[b] = index_of_key(key);
    }
  }
  // Shared memory must outlive the cluster's remote reads of s_part.
  if (sampled) asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int DT, bool VEC, bool RES>
void* hk() {
  return reinterpret_cast<void*>(&hlg_kernel<DT, VEC, RES>);
}

void* select_hlg(int dtype, bool vec, bool resident) {
  switch (dtype * 4 + (vec ? 2 : 0) + (resident ? 1 : 0)) {
    case 0: return hk<0, false, false>();
    case 1: return hk<0, false, true>();
    case 2: return hk<0, true, false>();
    case 3: return hk<0, true, true>();
    case 4: return hk<1, false, false>();
    case 5: return hk<1, false, true>();
    case 6: return hk<1, true, false>();
    case 7: return hk<1, true, true>();
    case 8: return hk<2, false, false>();
    case 9: return hk<2, false, true>();
    case 10: return hk<2, true, false>();
    default: return hk<2, true, true>();
  }
}

constexpr size_t kSmemLimit = 224 * 1024;  // leaves room for the static shared variables

}  // namespace

size_t hlg_smem_limit() { return kSmemLimit; }

size_t hlg_smem_bytes(int, bool, int32_t units_per_cta) { return (size_t)units_per_cta * 16; }

// One-time per-device setup of both variants of (dtype, vec): allow clusters
// of up to 16 CTAs and the full shared-memory slice, then report the largest
// cluster the device can co-schedule when every CTA holds `smem_bytes`.
int hlg_max_cluster(int dtype, bool vec, size_t smem_bytes) {
  for (int res = 0; res < 2; ++res) {
    void* fn = select_hlg(dtype, vec, res != 0);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             res ? (int)kSmemLimit : 0) != cudaSuccess)
      return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(16);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 16;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int size = 0;
  if (cudaOccupancyMaxPotentialClusterSize(&size, select_hlg(dtype, vec, true), &cfg) !=
      cudaSuccess)
    return 0;
  return size;
}

cudaError_t launch_hlg(const HlgParams& p, int dtype, bool vec, cudaStream_t stream) {
  const size_t need = hlg_smem_bytes(dtype, vec, p.units_per_cta);
  const bool resident = need <= kSmemLimit;
  void* fn = select_hlg(dtype, vec, resident);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * p.cluster));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = resident ? need : 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {const_cast<HlgParams*>(&p)};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace gsample
