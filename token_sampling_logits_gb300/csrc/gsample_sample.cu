// Row sampler kernel: greedy argmax and Gumbel-max over a [B, V] logits matrix
// in one launch ("Softmax-free GPU sampling: Gumbel-max categorical sampling
// kernel", lablup/mlxcel issue #900, Background and Task 1: score =
// logits/T + g, g = -log(-log u) from a per-(row, element) counter stream,
// one index-carrying max per row, all rows in one grid).
//
// Work split. The B rows are cut into 16-byte units and the B * units_per_row
// units are dealt to exactly one wave of CTAs in near-equal contiguous ranges,
// so the work per CTA is balanced whatever B and V are. A CTA walks the rows its
// range touches; each of its warps takes an equal contiguous piece of the
// row segment and streams it in tiles of 32 lanes x kVPT units (each load
// instruction of a warp covers 512 contiguous bytes).
//
// Merge. A row's candidates meet in its workspace slot: an atomicMax on a packed
// (ordered score, ~index) 64-bit key, then a ticket; the last CTA of the row
// writes out_idx and clears the slot. No CTA ever waits for another.
//
// Exact pruning (sampled rows). Each warp keeps L, the best exact score known
// for the row (its own candidates and whatever other CTAs have published into
// the row's key). An element with x/T + max(g) < L cannot win, so Philox and
// the logarithms are skipped for it. Surviving 4-element groups are compacted
// across the warp through shared memory so that all 32 lanes run Philox on
// useful work.
#include <cstdint>

#include "gsample_internal.h"

namespace gsample {
namespace {

constexpr int kVPT = 8;  // units per lane per tile

template <int DT, bool VEC>
struct Cfg {
  static constexpr int kElt = DT == 0 ? 4 : 2;
  static constexpr int kEPU = VEC ? 16 / kElt : 4;  // elements per unit
  static constexpr int kGPU = kEPU / 4;             // Philox groups per unit
  static constexpr int kTile = 32 * kVPT;           // units per warp tile
  static constexpr int kCap = 32 * kVPT * kGPU;     // compaction entries per warp
  // Unit registers hold binary32 bits (f32 rows, or any dtype on the 4-element
  // scalar path) or raw 16-bit values (bf16/f16 on the 128-bit path).
  static constexpr bool kF32Bits = DT == 0 || !VEC;
  static constexpr int kGroupBytes = kF32Bits ? 16 : 8;
  static constexpr size_t kSmem = (size_t)kWarps * kCap * (4 + kGroupBytes);
};

template <int DT>
__device__ __forceinline__ float half_to_f32(uint32_t h) {
  return DT == 1 ? bf16_bits_to_f32(h) : f16_bits_to_f32(h);
}

// Element e (0 <= e < kEPU) of a unit held in registers.
template <int DT, bool VEC>
__device__ __forceinline__ float unit_elt(const uint4& r, int e) {
  if constexpr (Cfg<DT, VEC>::kF32Bits) {
    return __uint_as_float(word_of(r, e));
  } else {
    const uint32_t w = word_of(r, e >> 1);
    return half_to_f32<DT>((e & 1) ? (w >> 16) : (w & 0xFFFFu));
  }
}

template <int DT>
__device__ __forceinline__ float load_elt(const char* row, int32_t i) {
  if constexpr (DT == 0) {
    return __ldg(reinterpret_cast<const float*>(row) + i);
  } else {
    return half_to_f32<DT>(__ldg(reinterpret_cast<const unsigned short*>(row) + i));
  }
}

template <int DT>
__device__ __forceinline__ uint32_t load_half_bits(const char* row, int32_t i) {
  return __ldg(reinterpret_cast<const unsigned short*>(row) + i);
}

constexpr uint32_t kNegInfF32 = 0xFF800000u;
template <int DT>
__host__ __device__ constexpr uint32_t neg_inf_half() { return DT == 1 ? 0xFF80u : 0xFC00u; }

template <int DT, bool VEC>
__device__ __forceinline__ uint4 empty_unit() {
  if constexpr (Cfg<DT, VEC>::kF32Bits) {
    return make_uint4(kNegInfF32, kNegInfF32, kNegInfF32, kNegInfF32);
  } else {
    const uint32_t w = neg_inf_half<DT>() * 0x10001u;
    return make_uint4(w, w, w, w);
  }
}

// Unit u of a row; elements at or past V read as -inf.
template <int DT, bool VEC>
__device__ __forceinline__ uint4 load_unit(const char* row, int32_t u, int32_t V, uint64_t pol) {
  using C = Cfg<DT, VEC>;
  const int32_t e0 = u * C::kEPU;
  if constexpr (VEC) {
    if (e0 + C::kEPU <= V) return ld_stream_v4(row + (size_t)u * 16, pol);
  }
  uint32_t w[4];
  if constexpr (C::kF32Bits) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w[e] = (e0 + e < V) ? __float_as_uint(load_elt<DT>(row, e0 + e)) : kNegInfF32;
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t lo = (e0 + 2 * k < V) ? load_half_bits<DT>(row, e0 + 2 * k) : neg_inf_half<DT>();
      const uint32_t hi = (e0 + 2 * k + 1 < V) ? load_half_bits<DT>(row, e0 + 2 * k + 1) : neg_inf_half<DT>();
      w[k] = lo | (hi << 16);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int DT, bool VEC>
__device__ __forceinline__ float unit_max(const uint4& r) {
  float m = unit_elt<DT, VEC>(r, 0);
#pragma unroll
  for (int e = 1; e < Cfg<DT, VEC>::kEPU; ++e) m = fmaxf(m, unit_elt<DT, VEC>(r, e));
  return m;  // fmaxf ignores NaN unless every element is NaN
}

// Greedy: running (max, lowest index) over this lane's units, in index order.
template <int DT, bool VEC>
__device__ __forceinline__ void greedy_unit(const uint4& r, int32_t u, float& bs, int32_t& bi) {
  using C = Cfg<DT, VEC>;
  const float m = unit_max<DT, VEC>(r);
  if (m > bs) {
    int32_t e_first = C::kEPU - 1;
#pragma unroll
    for (int e = C::kEPU - 1; e >= 0; --e)
      if (unit_elt<DT, VEC>(r, e) == m) e_first = e;
    bs = m;
    bi = u * C::kEPU + e_first;
  }
}

struct RowCtx {
  const char* row;
  int32_t V;
  uint32_t row_id;
  float T;
  float rT;
  uint32_t k0, k1;      // Philox key
  uint32_t off0, off1;  // Philox counter words 2, 3
  WsRow* ws;
};

__device__ __forceinline__ float exact_score(float x, uint32_t word, float T) {
  return x == INFINITY ? INFINITY : __fdiv_rn(x, T) + gumbel_of_word(word);
}

// Publish the warp's best into the row key and return the row's best known
// score (warp-uniform).
__device__ __forceinline__ float publish_and_bound(WsRow* ws, float bs, int32_t bi, int lane) {
  warp_argmax(bs, bi);
  unsigned long long old = 0ull;
  if (lane == 0) {
    if (bi != INT32_MAX && bs > -INFINITY)
      old = atomicMax(&ws->key, pack_key(bs, bi));
    else
      old = __ldcg(&ws->key);
  }
  old = __shfl_sync(0xFFFFFFFFu, old, 0);
  return fmaxf(bs, score_of_key(old));
}

template <int DT, bool VEC>
__device__ void sample_segment(const RowCtx& rc, int32_t w_lo, int32_t w_hi, uint64_t pol,
                               uint32_t* buf_gid, unsigned char* buf_data, float& bs,
                               int32_t& bi) {
  using C = Cfg<DT, VEC>;
  const int lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1u;
  uint4 r[kVPT];

  auto load_tile = [&](int32_t t0) {
#pragma unroll
    for (int k = 0; k < kVPT; ++k) {
      const int32_t u = t0 + k * 32 + lane;
      r[k] = (u < w_hi) ? load_unit<DT, VEC>(rc.row, u, rc.V, pol) : empty_unit<DT, VEC>();
    }
  };

  if (w_lo >= w_hi) return;
  load_tile(w_lo);
  bool first = true;
  for (int32_t t0 = w_lo; t0 < w_hi; t0 += C::kTile) {
    if (first) {
      // Phase A: each lane scores its largest logit exactly -> a first L.
      float cm = -INFINITY;
      int ck = -1;
#pragma unroll
      for (int k = 0; k < kVPT; ++k) {
        const float m = unit_max<DT, VEC>(r[k]);
        if (m > cm) {
          cm = m;
          ck = k;
        }
      }
      if (ck >= 0) {
        uint4 ru = r[0];
#pragma unroll
        for (int k = 1; k < kVPT; ++k)
          if (k == ck) ru = r[k];
        int ce = C::kEPU - 1;
#pragma unroll
        for (int e = C::kEPU - 1; e >= 0; --e)
          if (unit_elt<DT, VEC>(ru, e) == cm) ce = e;
        const int32_t i = (t0 + ck * 32 + lane) * C::kEPU + ce;
        const uint4 blk = philox4x32_10(make_uint4((uint32_t)i >> 2, rc.row_id, rc.off0, rc.off1),
                                        rc.k0, rc.k1);
        take_better(exact_score(cm, word_of(blk, i & 3), rc.T), i, bs, bi);
      }
      first = false;
    }
    const float L = publish_and_bound(rc.ws, bs, bi, lane);
    const Prune pr = make_prune(L, rc.T);

    // Phase B: append every group that may still win to the warp's buffer.
    int cnt = 0;
#pragma unroll
    for (int k = 0; k < kVPT; ++k) {
      const int32_t u = t0 + k * 32 + lane;
#pragma unroll
      for (int h = 0; h < C::kGPU; ++h) {
        float gm = unit_elt<DT, VEC>(r[k], 4 * h);
#pragma unroll
        for (int e = 1; e < 4; ++e) gm = fmaxf(gm, unit_elt<DT, VEC>(r[k], 4 * h + e));
        const bool keep = gm >= pr.thr_x;
        const unsigned mask = __ballot_sync(0xFFFFFFFFu, keep);
        if (keep) {
          const int pos = cnt + __popc(mask & lt_mask);
          buf_gid[pos] = (uint32_t)(u * C::kGPU + h);
          if constexpr (C::kF32Bits) {
            reinterpret_cast<uint4*>(buf_data)[pos] = r[k];
          } else {
            reinterpret_cast<uint2*>(buf_data)[pos] =
                h == 0 ? make_uint2(r[k].x, r[k].y) : make_uint2(r[k].z, r[k].w);
          }
        }
        cnt += __popc(mask);
      }
    }
    __syncwarp();

    // Start the next tile's loads before the arithmetic on this one.
    if (t0 + C::kTile < w_hi) load_tile(t0 + C::kTile);

    // Phase C: exact scores of the surviving groups, one group per lane.
    for (int p = lane; p < cnt; p += 32) {
      const uint32_t gid = buf_gid[p];
      float x[4];
      if constexpr (C::kF32Bits) {
        const uint4 d = reinterpret_cast<const uint4*>(buf_data)[p];
        x[0] = __uint_as_float(d.x);
        x[1] = __uint_as_float(d.y);
        x[2] = __uint_as_float(d.z);
        x[3] = __uint_as_float(d.w);
      } else {
        const uint2 d = reinterpret_cast<const uint2*>(buf_data)[p];
        x[0] = half_to_f32<DT>(d.x & 0xFFFFu);
        x[1] = half_to_f32<DT>(d.x >> 16);
        x[2] = half_to_f32<DT>(d.y & 0xFFFFu);
        x[3] = half_to_f32<DT>(d.y >> 16);
      }
      const uint4 blk = philox4x32_10(make_uint4(gid, rc.row_id, rc.off0, rc.off1), rc.k0, rc.k1);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float xv = x[t];
        if (!(xv >= pr.thr_x)) continue;
        const uint32_t wd = word_of(blk, t);
        if (pr.use_bound && xv * rc.rT + gumbel_bound_of_word(wd) < pr.lm) continue;
        take_better(exact_score(xv, wd, rc.T), (int32_t)(4 * gid + t), bs, bi);
      }
    }
    __syncwarp();
  }
}

template <int DT, bool VEC>
__device__ void greedy_segment(const RowCtx& rc, int32_t w_lo, int32_t w_hi, uint64_t pol,
                               float& bs, int32_t& bi) {
  using C = Cfg<DT, VEC>;
  const int lane = threadIdx.x & 31;
  for (int32_t t0 = w_lo; t0 < w_hi; t0 += C::kTile) {
    uint4 r[kVPT];
#pragma unroll
    for (int k = 0; k < kVPT; ++k) {
      const int32_t u = t0 + k * 32 + lane;
      r[k] = (u < w_hi) ? load_unit<DT, VEC>(rc.row, u, rc.V, pol) : empty_unit<DT, VEC>();
    }
#pragma unroll
    for (int k = 0; k < kVPT; ++k) greedy_unit<DT, VEC>(r[k], t0 + k * 32 + lane, bs, bi);
  }
}

// First unit of the CTA range that holds unit u (balanced split of U units
// over G CTAs: the first U % G CTAs take one unit more).
__device__ __forceinline__ int64_t owner_cta(int64_t u, int64_t U, int64_t G) {
  const int64_t base = U / G, rem = U % G;
  const int64_t big = rem * (base + 1);
  return u < big ? u / (base + 1) : rem + (u - big) / base;
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads) sample_kernel(const SampleParams p) {
  using C = Cfg<DT, VEC>;
  extern __shared__ __align__(16) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint32_t* buf_gid = reinterpret_cast<uint32_t*>(smem) + warp * C::kCap;
  unsigned char* buf_data = smem + (size_t)kWarps * C::kCap * 4 + (size_t)warp * C::kCap * C::kGroupBytes;
  const uint64_t pol = evict_first_policy();

  const int64_t U = p.total_units, G = p.ctas, NU = p.units_per_row;
  const int64_t c = blockIdx.x;
  const int64_t base = U / G, rem = U % G;
  const int64_t u_begin = c * base + (c < rem ? c : rem);
  const int64_t u_end = u_begin + base + (c < rem ? 1 : 0);

  for (int64_t b = u_begin / NU; b * NU < u_end; ++b) {
    const int64_t row_u0 = b * NU;
    const int32_t lo = (int32_t)((u_begin > row_u0 ? u_begin : row_u0) - row_u0);
    const int32_t hi = (int32_t)((u_end < row_u0 + NU ? u_end : row_u0 + NU) - row_u0);
    const int32_t n = hi - lo;
    const int32_t w_lo = lo + (int32_t)((int64_t)n * warp / kWarps);
    const int32_t w_hi = lo + (int32_t)((int64_t)n * (warp + 1) / kWarps);

    RowCtx rc;
    rc.row = p.logits + b * p.ld_bytes;
    rc.V = p.V;
    rc.row_id = (uint32_t)b;
    rc.ws = p.ws + b;
    rc.T = p.temperature ? __ldg(p.temperature + b) : 0.0f;
    float bs = -INFINITY;
    int32_t bi = INT32_MAX;
    if (rc.T > 0.0f) {  // NaN and T <= 0: greedy
      const uint64_t sd = __ldg(p.seed + b), of = __ldg(p.offset + b);
      rc.k0 = (uint32_t)sd;
      rc.k1 = (uint32_t)(sd >> 32);
      rc.off0 = (uint32_t)of;
      rc.off1 = (uint32_t)(of >> 32);
      rc.rT = 1.0f / rc.T;
      sample_segment<DT, VEC>(rc, w_lo, w_hi, pol, buf_gid, buf_data, bs, bi);
    } else {
      greedy_segment<DT, VEC>(rc, w_lo, w_hi, pol, bs, bi);
    }
    warp_argmax(bs, bi);
    if (lane == 0 && bi != INT32_MAX && bs > -INFINITY) atomicMax(&rc.ws->key, pack_key(bs, bi));
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const int64_t expected = owner_cta(row_u0 + NU - 1, U, G) - owner_cta(row_u0, U, G) + 1;
      const unsigned t = atomicAdd(&rc.ws->ticket, 1u);
      if ((int64_t)t == expected - 1) {
        __threadfence();
        const unsigned long long key = atomicExch(&rc.ws->key, 0ull);
        atomicExch(&rc.ws->ticket, 0u);
        p.out_idx[b] = index_of_key(key);
      }
    }
  }
}

template <int DT, bool VEC>
void* kernel_ptr() {
  return reinterpret_cast<void*>(&sample_kernel<DT, VEC>);
}

void* select_kernel(int dtype, bool vec) {
  switch (dtype * 2 + (vec ? 1 : 0)) {
    case 0: return kernel_ptr<0, false>();
    case 1: return kernel_ptr<0, true>();
    case 2: return kernel_ptr<1, false>();
    case 3: return kernel_ptr<1, true>();
    case 4: return kernel_ptr<2, false>();
    default: return kernel_ptr<2, true>();
  }
}

}  // namespace

size_t sample_smem_bytes(int dtype, bool vec) {
  switch (dtype * 2 + (vec ? 1 : 0)) {
    case 0: return Cfg<0, false>::kSmem;
    case 1: return Cfg<0, true>::kSmem;
    case 2: return Cfg<1, false>::kSmem;
    case 3: return Cfg<1, true>::kSmem;
    case 4: return Cfg<2, false>::kSmem;
    default: return Cfg<2, true>::kSmem;
  }
}

// One-time per-device setup: raise the dynamic shared-memory limit of every
// variant (a function attribute, so it is kept for the life of the context),
// then report how many CTAs of the variant fit on one SM.
int sample_ctas_per_sm(int dtype, bool vec) {
  void* fn = select_kernel(dtype, vec);
  const size_t smem = sample_smem_bytes(dtype, vec);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, smem) != cudaSuccess) return 0;
  return n;
}

cudaError_t launch_sample(const SampleParams& p, int dtype, bool vec, cudaStream_t stream) {
  void* fn = select_kernel(dtype, vec);
  void* args[] = {const_cast<SampleParams*>(&p)};
  return cudaLaunchKernel(fn, dim3((unsigned)p.ctas), dim3(kThreads), args,
                          sample_smem_bytes(dtype, vec), stream);
}

// ---------------------------------------------------------------------------
// Diagnostics: the same device functions, exposed for one-by-one comparison.
// ---------------------------------------------------------------------------
namespace {

__global__ void debug_philox_kernel(uint64_t seed, uint32_t row, uint64_t offset, int64_t group0,
                                    int64_t n, uint32_t* out) {
  for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n;
       j += (int64_t)gridDim.x * blockDim.x) {
    const uint4 v = philox4x32_10(
        make_uint4((uint32_t)(group0 + j), row, (uint32_t)offset, (uint32_t)(offset >> 32)),
        (uint32_t)seed, (uint32_t)(seed >> 32));
    reinterpret_cast<uint4*>(out)[j] = v;
  }
}

__global__ void debug_gumbel_kernel(const uint32_t* words, int64_t n, float* g, float* bound) {
  for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n;
       j += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t w = words[j];
    g[j] = gumbel_of_word(w);
    if (bound) bound[j] = gumbel_bound_of_word(w);
  }
}

unsigned grid_for(int64_t n) {
  const int64_t blocks = (n + 255) / 256;
  return (unsigned)(blocks < 4096 ? (blocks < 1 ? 1 : blocks) : 4096);
}

}  // namespace

cudaError_t launch_debug_philox(uint64_t seed, uint32_t row, uint64_t offset, int64_t group0,
                                int64_t n, uint32_t* out, cudaStream_t stream) {
  debug_philox_kernel<<<grid_for(n), 256, 0, stream>>>(seed, row, offset, group0, n, out);
  return cudaGetLastError();
}

cudaError_t launch_debug_gumbel(const uint32_t* words, int64_t n, float* g, float* bound,
                                cudaStream_t stream) {
  debug_gumbel_kernel<<<grid_for(n), 256, 0, stream>>>(words, n, g, bound);
  return cudaGetLastError();
}

}  // namespace gsample
