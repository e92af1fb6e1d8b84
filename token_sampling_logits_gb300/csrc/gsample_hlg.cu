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
// Layout: one thread-block cluster of `cluster` CTAs (512 threads each) per
// row. Each CTA requests its whole slice of the row at once with cp.async into
// shared memory (RESIDENT), reduces its partial statistics, and the cluster
// exchanges them through distributed shared memory after a hardware cluster
// barrier. Sweep 2 scores the slice from shared memory: the logit threshold
// from the inverse curve, then Philox four groups per thread at a time, then a
// word bound (g <= -log(1 - u)) on a fast upper bound of the curve, and the
// exact score only for the rare groups that pass. Each CTA's best (score,
// index) key goes to rank 0 over distributed shared memory, which writes the
// row's answer: the row needs no global atomics and leaves the workspace
// untouched. If a slice is too large for shared memory the same kernel
// re-reads it from global memory in sweep 2 (!RESIDENT). The only waits are
// hardware cluster and CTA barriers.
#include <cooperative_groups.h>

#include <cstdint>

#include "gsample_internal.h"
#include "gsample_slice.cuh"

namespace cg = cooperative_groups;

namespace gsample {
namespace {

using namespace slice;

constexpr int kHlgThreads = 512;
#ifndef GSAMPLE_HLG_CHUNKS
#define GSAMPLE_HLG_CHUNKS 4
#endif
constexpr int kHlgWarps = kHlgThreads / 32;

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

// The tone curve in binary32 ("The transfer function"). rbt, rbh are 1/beta.
struct Curve {
  float m, w, bt, bh, rbt, rbh;
};

__device__ __forceinline__ float tone(const Curve& c, float z) {
  if (z < -c.w) return -c.m * c.w - c.m * c.bt * log1pf((-z - c.w) * c.rbt);
  if (z > c.w) return c.m * c.w + c.m * c.bh * log1pf((z - c.w) * c.rbh);
  return c.m * z;
}

// An upper bound of tone(z) for pruning only: the fast logarithm of 1 + t
// errs by a few 1e-7 relative, far inside the 1e-4 relative slack added.
__device__ __forceinline__ float tone_upper(const Curve& c, float z) {
  float y;
  if (z < -c.w) {
    y = -c.m * c.w - c.m * c.bt * __logf(1.0f + (-z - c.w) * c.rbt);
  } else if (z > c.w) {
    y = c.m * c.w + c.m * c.bh * __logf(1.0f + (z - c.w) * c.rbh);
  } else {
    y = c.m * z;
  }
  return y + 1e-4f * (1.0f + fabsf(y));
}

// The checks the host applies to a launch-wide curve, for per-row curves that
// only the device sees: finite m > 0, w >= 0 (+inf allowed), finite
// beta_t, beta_h > 0, finite pivot offset, pivot mode 0 (top) or 1 (entropy).
__device__ __forceinline__ bool curve_ok(const HlgRowParams& h) {
  return isfinite(h.m) && h.m > 0.0f && h.w >= 0.0f && isfinite(h.beta_t) && h.beta_t > 0.0f &&
         isfinite(h.beta_h) && h.beta_h > 0.0f && isfinite(h.pivot_offset) &&
         (h.pivot_mode == 0 || h.pivot_mode == 1);
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

// The exact score tone(z)/T + g, with an IEEE division as the oracle reads
// "tone(z) / T" (only scored candidates pay for it; pruning multiplies by 1/T
// inside its slack).
__device__ __forceinline__ float hlg_score(const Curve& c, const RowState& rs, float x,
                                           uint32_t word, float T) {
  if (x == INFINITY) return INFINITY;
  const float y = tone(c, x + rs.shift);
  return __fdiv_rn(y, T) + gumbel_of_word(word);
}

// The same score with the Gumbel value g already computed from the word.
__device__ __forceinline__ float hlg_score_g(const Curve& c, const RowState& rs, float x, float g,
                                             float T) {
  if (x == INFINITY) return INFINITY;
  const float y = tone(c, x + rs.shift);
  return __fdiv_rn(y, T) + g;
}

struct HlgBest {
  float s;
  int32_t i;
};

// The exact pass over a warp's listed groups, one group per lane: each
// element's own word bound, then tone(z)/T + g. Out of line: it runs once per
// 32 listed groups, and keeping its logarithms out of sweep 2 keeps that
// loop's code small.
__device__ __noinline__ HlgBest hlg_flush_cold(const uint32_t* rg, const float4* rx, const uint4* rw,
                                               int rcnt, float x_thr, bool word_test, float wa,
                                               float wc, Curve cv, RowState rs, float T, float bs,
                                               int32_t bi) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  if (lane < rcnt) {
    const uint32_t gg = rg[lane];
    const float4 xx = rx[lane];
    const uint4 ww = rw[lane];
    const float xs[4] = {xx.x, xx.y, xx.z, xx.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float x = xs[t];
      if (!(x >= x_thr) || x == -INFINITY) continue;
      if (word_test &&
          !may_reach(tone_upper(cv, x + rs.shift), word_of(ww, t), ReachTest{wa, wc}))
        continue;
      take_better(hlg_score(cv, rs, x, word_of(ww, t), T), (int32_t)(4 * gg + t), bs, bi);
    }
  }
  __syncwarp();
  return HlgBest{bs, bi};
}

// Block-wide (score, index) argmax; every thread gets the result. `red` holds
// kHlgWarps packed keys.
__device__ __forceinline__ unsigned long long block_best(float s, int32_t i,
                                                         unsigned long long* red) {
  warp_argmax(s, i);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = (i != INT32_MAX && s > -INFINITY) ? pack_key(s, i) : 0ull;
  __syncthreads();
  unsigned long long k = lane < kHlgWarps ? red[lane] : 0ull;
  k = warp_max_u64(k);
  __syncthreads();  // red may be reused
  return k;
}

// Packed maxima of two pairs of 16-bit logits (bf16 when DT is 1, else f16).
template <int DT>
__device__ __forceinline__ uint32_t hlg_hmax2(uint32_t a, uint32_t b) {
  if constexpr (DT == 1) {
    __nv_bfloat162 m = __hmax2(*reinterpret_cast<__nv_bfloat162*>(&a),
                               *reinterpret_cast<__nv_bfloat162*>(&b));
    return *reinterpret_cast<uint32_t*>(&m);
  } else {
    __half2 m = __hmax2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
    return *reinterpret_cast<uint32_t*>(&m);
  }
}

template <int DT, bool VEC, bool RESIDENT>
__global__ void __launch_bounds__(kHlgThreads) hlg_kernel(const HlgParams p) {
  using C = HCfg<DT, VEC>;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ Moments s_warp[kHlgWarps];
  __shared__ Moments s_part;            // this CTA's partial, read by the whole cluster
  __shared__ unsigned long long s_red[kHlgWarps];
  __shared__ unsigned long long s_best;  // this CTA's best key, read by rank 0
  __shared__ unsigned long long s_lbest;  // this CTA's best first candidate, read by the cluster
  __shared__ unsigned long long s_lrow;   // the row's best first candidate
  __shared__ int s_pinf;
  __shared__ RowState s_row;
  // Per warp: groups that passed the word test, waiting for an exact pass with
  // one group per lane (row-local group index, its four logits, its words).
  __shared__ uint32_t s_rg[kHlgWarps][32];
  __shared__ float4 s_rx[kHlgWarps][32];
  __shared__ uint4 s_rw[kHlgWarps][32];

  pdl_wait_then_release();
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t b = blockIdx.x / p.cluster;
  const int32_t NU = p.units_per_row;
  const int32_t u_lo = rank * p.units_per_cta;
  const int32_t u_hi = min(NU, u_lo + p.units_per_cta);
  const char* row = p.logits + b * p.ld_bytes;
  const uint32_t slice = (uint32_t)__cvta_generic_to_shared(smem);
  const uint64_t pol = evict_first_policy();

  const float T = __ldg(p.temperature + b);
  // The row's seed and offset are requested now, so their latency hides behind
  // the slice load.
  const uint64_t sd = __ldg(p.seed + b), of = __ldg(p.offset + b);
  // The row's curve: the launch's, or its own from the per-row array.
  HlgRowParams hp{p.m, p.w, p.beta_t, p.beta_h, p.pivot_offset, p.pivot_mode};
  if (p.rows) {
    const HlgRowParams* r = p.rows + b;
    hp = HlgRowParams{__ldg(&r->m), __ldg(&r->w), __ldg(&r->beta_t), __ldg(&r->beta_h),
                      __ldg(&r->pivot_offset), __ldg(&r->pivot_mode)};
  }
  const bool sampled = T > 0.0f;
  if (sampled && !curve_ok(hp)) {  // a per-row curve that fails the checks: no answer
    if (rank == 0 && threadIdx.x == 0) p.out_idx[b] = -1;
    return;  // every CTA of the cluster reads the same row, so all leave here
  }
  const bool entropy = hp.pivot_mode == 1;
  if (threadIdx.x == 0) s_pinf = 0;

  // Sweep 1: stream the slice once. On the resident path the thread's whole
  // share is requested with cp.async into the slice, so the whole slice is in
  // flight together; the thread reads back its own units as they land.
  auto unit_at = [&](int32_t u) -> uint4 {
    if constexpr (RESIDENT)
      return lds128(slice + (uint32_t)(u - u_lo) * 16u);
    else
      return load_unit<DT, VEC>(row, u, p.V, pol);
  };
  // The thread's largest logit (lowest index on ties): the greedy answer, and
  // the first exact candidate of a sampled row. For the pivot, the largest
  // finite logit; +inf is flagged.
  // Unit maxima first (NaN is ignored unless a whole unit is NaN, and a NaN
  // maximum never wins); a unit holding +inf takes its finite maximum element
  // by element; then the first element of the best unit that equals its max.
  float cand_x = -INFINITY;
  int32_t cand_u = -1;
  float fmax_x = -INFINITY;
  bool pinf = false;
  auto sweep1_unit = [&](int32_t u, const uint4& r) {
    float m;
    if constexpr (C::kF32Bits) {
      m = fmaxf(fmaxf(__uint_as_float(r.x), __uint_as_float(r.y)),
                fmaxf(__uint_as_float(r.z), __uint_as_float(r.w)));
    } else {
      const uint32_t h = hlg_hmax2<DT>(hlg_hmax2<DT>(r.x, r.y), hlg_hmax2<DT>(r.z, r.w));
      m = fmaxf(half_to_f32<DT>(h & 0xFFFFu), half_to_f32<DT>(h >> 16));
    }
    if (m > cand_x) {
      cand_x = m;
      cand_u = u;
    }
    if (m == INFINITY) {
      pinf = true;
#pragma unroll
      for (int e = 0; e < C::kEPU; ++e) {
        const float x = elt<DT, VEC>(r, e);
        if (x != INFINITY) fmax_x = fmaxf(fmax_x, x);
      }
    } else {
      fmax_x = fmaxf(fmax_x, m);
    }
  };
  // On the resident path the thread's units are requested in GSAMPLE_HLG_CHUNKS
  // groups (the whole slice is in flight together) and each group is reduced
  // as it lands.
  if constexpr (RESIDENT) {
    load_slice_then<DT, VEC, kHlgThreads, GSAMPLE_HLG_CHUNKS>(row, u_lo, u_hi, p.V, slice, pol,
                                                             sweep1_unit);
  } else {
    for (int32_t u = u_lo + threadIdx.x; u < u_hi; u += kHlgThreads) sweep1_unit(u, unit_at(u));
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
    const uint32_t k0 = (uint32_t)sd, k1 = (uint32_t)(sd >> 32);
    const uint32_t o0 = (uint32_t)of, o1 = (uint32_t)(of >> 32);
    const PhiloxRow ph = philox_row((uint32_t)b, o0, o1, k0, k1);
    // The first candidate's Gumbel value does not depend on the pivot, so its
    // Philox block and logarithms run before the pivot exchange and overlap it.
    float cand_g = 0.0f;
    if (cand_i != INT32_MAX && cand_x > -INFINITY) {
      const uint4 blk = philox_row_1((uint32_t)cand_i >> 2, ph);
      cand_g = gumbel_of_word(word_of(blk, cand_i & 3));
    }
    // Pivot statistics of the slice. Entropy: a second pass over the slice
    // (shared memory) sums e^(x - M) and e^(x - M) x against the thread's max.
    Moments mo{fmax_x, 0.0f, 0.0f};
    if (entropy && fmax_x > -INFINITY) {
      for (int32_t u = u_lo + threadIdx.x; u < u_hi; u += kHlgThreads) {
        const uint4 r = unit_at(u);
#pragma unroll
        for (int e = 0; e < C::kEPU; ++e) {
          const float x = elt<DT, VEC>(r, e);
          if (x > -INFINITY && x < INFINITY) {
            const float ex = __expf(x - fmax_x);
            mo.S += ex;
            mo.W = fmaf(ex, x, mo.W);
          }
        }
      }
    }
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
    if (warp == 0) {
      Moments acc = lane < kHlgWarps ? s_warp[lane] : Moments{-INFINITY, 0.0f, 0.0f};
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        Moments other;
        other.M = __shfl_xor_sync(0xFFFFFFFFu, acc.M, o);
        other.S = __shfl_xor_sync(0xFFFFFFFFu, acc.S, o);
        other.W = __shfl_xor_sync(0xFFFFFFFFu, acc.W, o);
        acc = entropy ? merge(acc, other) : Moments{fmaxf(acc.M, other.M), 0.0f, 0.0f};
      }
      if (lane == 0) {
        if (s_pinf) acc.M = INFINITY;  // the flag travels with the partial
        s_part = acc;
      }
    }
    cluster.sync();
    if (warp == 0) {
      // Lane k reads CTA k's partial; the same butterfly on every CTA gives
      // all CTAs of the row bit-identical pivot statistics.
      Moments o{-INFINITY, 0.0f, 0.0f};
      if (lane < p.cluster) o = *cluster.map_shared_rank(&s_part, lane);
      const bool any_pinf = __any_sync(0xFFFFFFFFu, o.M == INFINITY);
      if (o.M == INFINITY) o = Moments{-INFINITY, 0.0f, 0.0f};
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        Moments other;
        other.M = __shfl_xor_sync(0xFFFFFFFFu, o.M, off);
        other.S = __shfl_xor_sync(0xFFFFFFFFu, o.S, off);
        other.W = __shfl_xor_sync(0xFFFFFFFFu, o.W, off);
        o = entropy ? merge(o, other) : Moments{fmaxf(o.M, other.M), 0.0f, 0.0f};
      }
      if (lane == 0) {
        RowState rs;
        rs.pinf = any_pinf;
        rs.shift = entropy ? -(o.W / o.S) : (hp.pivot_offset - o.M);
        s_row = rs;
      }
    }
    __syncthreads();
    const RowState rs = s_row;

    const Curve cv{hp.m, hp.w, hp.beta_t, hp.beta_h, 1.0f / hp.beta_t, 1.0f / hp.beta_h};
    const float rT = 1.0f / T;

    // First candidate: this thread's largest logit, scored exactly; the CTA's
    // best of them is the bound L that sweep 2 prunes against.
    if (cand_i != INT32_MAX && cand_x > -INFINITY && (!rs.pinf || cand_x == INFINITY))
      take_better(hlg_score_g(cv, rs, cand_x, cand_g, T), cand_i, bs, bi);
    // The bound: the best first candidate of the whole row, over the cluster.
    {
      const unsigned long long kc = block_best(bs, bi, s_red);
      if (threadIdx.x == 0) s_lbest = kc;
    }
    cluster.sync();
    if (warp == 0) {
      unsigned long long k = lane < p.cluster ? *cluster.map_shared_rank(&s_lbest, lane) : 0ull;
      k = warp_max_u64(k);
      if (lane == 0) s_lrow = k;
    }
    __syncthreads();
    const float L = score_of_key(s_lrow);

    // Exact pruning in logit space: x < x_thr implies tone(x + shift)/T + max g < L.
    float x_thr = -INFINITY;
    bool word_test = false;
    float wa = 0.0f, wc = 0.0f;
    if (rs.pinf || L == INFINITY) {
      x_thr = INFINITY;
    } else if (L > -INFINITY && T >= 1e-20f && T <= 1e20f) {
      const float margin = 1e-3f * (1.0f + fabsf(L));
      const float z_thr = tone_inverse(cv, (L - kGumbelMax - margin) * T);
      x_thr = z_thr - rs.shift - 1e-3f * (1.0f + fabsf(z_thr)) - 1e-3f * (1.0f + fabsf(rs.shift));
      if (!(x_thr == x_thr)) x_thr = -INFINITY;  // NaN guard: no pruning
      // Word bound: g <= -log(1 - u), so a group whose curve value is at most
      // y can reach L only if 1 - u(max word) <= 2^((y / T - lm) log2 e).
      constexpr float kLog2e = 1.4426950408889634f;
      const float lm = L - margin - 0.01f;
      word_test = true;
      wa = rT * kLog2e;
      wc = -lm * kLog2e;
    }

    // Sweep 2 over the slice: four 4-element Philox groups per thread at a
    // time (four units of binary32, two of 16-bit), one Philox block each.
    constexpr int kUPB = 4 / C::kGPU;  // units per batch
    const int32_t n_iter = (u_hi - u_lo + kHlgThreads - 1) / kHlgThreads;
    // The warp's listed groups, scored exactly one per lane: the element's own
    // word bound, then tone(z)/T + g.
    int rcnt = 0;
    auto flush = [&]() {
      const HlgBest r = hlg_flush_cold(&s_rg[warp][0], &s_rx[warp][0], &s_rw[warp][0], rcnt, x_thr,
                                       word_test, wa, wc, cv, rs, T, bs, bi);
      bs = r.s;
      bi = r.i;
    };
    for (int32_t it = 0; it < n_iter; it += kUPB) {
      uint4 r[kUPB];
      float xm[4];
      uint32_t g[4];
      bool ok[4];
#pragma unroll
      for (int j = 0; j < kUPB; ++j) {
        const int32_t u = u_lo + threadIdx.x + (it + j) * kHlgThreads;
        const bool valid = u < u_hi;
        r[j] = valid ? unit_at(u) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int h = 0; h < C::kGPU; ++h) {
          float gm = elt<DT, VEC>(r[j], 4 * h);
#pragma unroll
          for (int e = 1; e < 4; ++e) gm = fmaxf(gm, elt<DT, VEC>(r[j], 4 * h + e));
          const int jj = j * C::kGPU + h;
          xm[jj] = gm;
          ok[jj] = valid && gm >= x_thr;
          g[jj] = (uint32_t)(u * C::kGPU + h);
        }
      }
      if (!__any_sync(0xFFFFFFFFu, ok[0] || ok[1] || ok[2] || ok[3])) continue;
      uint4 w[4];
      philox_row_x4(g, ph, w);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        bool need = ok[jj];
        if (need && word_test) {
          const uint32_t wm = max(max(w[jj].x, w[jj].y), max(w[jj].z, w[jj].w));
          need = may_reach(tone_upper(cv, xm[jj] + rs.shift), wm, ReachTest{wa, wc});
        }
        const unsigned m = __ballot_sync(0xFFFFFFFFu, need);
        if (m == 0u) continue;
        const int n = __popc(m);
        if (rcnt + n > 32) {
          flush();
          rcnt = 0;
        }
        if (need) {
          const uint4 rj = r[jj / C::kGPU];
          const int h = jj % C::kGPU;
          const int pos = rcnt + __popc(m & ((1u << lane) - 1u));
          s_rg[warp][pos] = g[jj];
          s_rx[warp][pos] = make_float4(elt<DT, VEC>(rj, 4 * h), elt<DT, VEC>(rj, 4 * h + 1),
                                        elt<DT, VEC>(rj, 4 * h + 2), elt<DT, VEC>(rj, 4 * h + 3));
          s_rw[warp][pos] = w[jj];
        }
        rcnt += n;
      }
    }
    if (rcnt > 0) flush();
  }

  // The row's answer: each CTA's best key, merged by rank 0 over distributed
  // shared memory. The second cluster barrier keeps every CTA's shared memory
  // alive until rank 0 has read it.
  const unsigned long long best = block_best(bs, bi, s_red);
  if (threadIdx.x == 0) s_best = best;
  cluster.sync();
  if (rank == 0 && warp == 0) {
    unsigned long long k = lane < p.cluster ? *cluster.map_shared_rank(&s_best, lane) : 0ull;
    k = warp_max_u64(k);
    if (lane == 0) p.out_idx[b] = index_of_key(k);
  }
  cluster.sync();
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

constexpr size_t kSmemLimit = 204 * 1024;  // leaves room for the static shared variables

// Diagnostics: the exact HLG score of given logits and words with a given
// shift (z = x + shift), as the kernel scores its candidates.
__global__ void debug_hlg_score_kernel(const float* x, const uint32_t* words, int64_t n, Curve c,
                                       float T, float shift, float* out) {
  const RowState rs{shift, false};
  for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n;
       j += (int64_t)gridDim.x * blockDim.x)
    out[j] = hlg_score(c, rs, x[j], words[j], T);
}

}  // namespace

cudaError_t launch_debug_hlg_score(const float* x, const uint32_t* words, int64_t n, float m,
                                   float w, float beta_t, float beta_h, float T, float shift,
                                   float* out, cudaStream_t stream) {
  const Curve c{m, w, beta_t, beta_h, 1.0f / beta_t, 1.0f / beta_h};
  const int64_t blocks = (n + 255) / 256;
  debug_hlg_score_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(
      x, words, n, c, T, shift, out);
  return cudaGetLastError();
}

size_t hlg_smem_limit() { return kSmemLimit; }

void* hlg_kernel_fn(int dtype, bool vec, bool resident, int* threads) {
  *threads = kHlgThreads;
  return select_hlg(dtype, vec, resident);
}

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
  cfg.blockDim = dim3(kHlgThreads);
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
  cfg.blockDim = dim3(kHlgThreads);
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
  void* args[] = {const_cast<HlgParams*>(&p)};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace gsample
