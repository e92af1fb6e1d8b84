// Row sampler kernel: greedy argmax and Gumbel-max over a [B, V] logits matrix
// in one launch ("Softmax-free GPU sampling: Gumbel-max categorical sampling
// kernel", lablup/mlxcel issue #900, Background and Task 1: score =
// logits/T + g, g = -log(-log u) from a per-(row, element) counter stream,
// one index-carrying max per row, all rows in one grid).
//
// Work split. The B rows are cut into 16-byte units. All B * units_per_row
// units are dealt to the warps of one wave of CTAs, in near-equal contiguous
// ranges whose ends sit on 128-byte lines of the row. Each warp walks its range
// in tiles of 32 lanes x kVPT units; a tile never crosses a row. Warps never wait for one another: there is no CTA-wide
// barrier in the kernel.
//
// Memory pipeline. Each warp streams its tiles through a ring of kStages tiles
// in shared memory with cp.async (L2 evict-first hint; each warp instruction
// moves 512 contiguous bytes), so kStages-1 tiles are in flight while the warp
// computes on the current one, across row boundaries, without holding the data
// in registers.
//
// Merge. When a warp finishes its part of a row it folds its best (score,
// index) into the row's workspace slot with atomicMax on a packed 64-bit key,
// then takes a ticket; the warp that completes the row's count writes out_idx
// and clears the slot.
//
// Exact pruning (sampled rows). Each warp keeps L, the best exact score known
// for the row (its own candidates and whatever other warps have published). An
// element with x/T + max(g) < L cannot win, so Philox and the logarithms are
// skipped for it: a tile whose logits all sit below L - max(g) is skipped
// whole. In the other tiles every 4-element group gets its Philox block, four
// independent blocks per lane at a time, and a bound on g from the largest
// word of the block (an integer threshold computed from the group's logits
// before the block) rejects almost every group before the two exact
// logarithms. The few survivors wait in a per-warp list and are scored 32 at a
// time, one per lane, out of line. Where only a small share of a tile's groups reaches the
// logit threshold, those groups are compacted first and only they get Philox.
#include <cstdint>
#include <type_traits>

#include <cuda_bf16.h>

#include "gsample_internal.h"

namespace gsample {

#ifdef GSAMPLE_COUNT_BLOCKS
// Diagnostic builds only: Philox blocks the sampler computed, summed over
// launches (dense tiles, compacted batches, first candidates, exact passes).
__device__ unsigned long long g_blocks_computed;
#define GSAMPLE_COUNT(n)                                                          \
  do {                                                                            \
    const unsigned long long c_ = (unsigned long long)__reduce_add_sync(          \
        0xFFFFFFFFu, (unsigned)(n));                                              \
    if ((threadIdx.x & 31) == 0) atomicAdd(&g_blocks_computed, c_);               \
  } while (0)
#else
#define GSAMPLE_COUNT(n) \
  do {                   \
  } while (0)
#endif

namespace {

#ifndef GSAMPLE_VPT
#define GSAMPLE_VPT 8
#endif
#ifndef GSAMPLE_STAGES
#define GSAMPLE_STAGES 2
#endif
#ifndef GSAMPLE_MIN_CTAS_PER_SM
#define GSAMPLE_MIN_CTAS_PER_SM 2
#endif
constexpr int kVPT = GSAMPLE_VPT;        // units per lane per tile
constexpr int kStages = GSAMPLE_STAGES;  // tiles per warp ring

// The rare list of a warp: 32 entries of a row-local group index (4 bytes)
// and the group's four logits as stored in the tile (at most 16 bytes).
constexpr int kRareCap = 32;
constexpr uint32_t kRareRawOff = kRareCap * 4;  // byte offset of the logits array
constexpr int kRareBytes = (int)kRareRawOff + kRareCap * 16;

template <int DT, bool VEC>
struct Cfg {
  static constexpr int kElt = DT == 0 ? 4 : 2;
  static constexpr int kEPU = VEC ? 16 / kElt : 4;  // elements per unit
  static constexpr int kGPU = kEPU / 4;             // Philox groups per unit
  static constexpr int kTile = 32 * kVPT;           // units per warp tile
  static constexpr int kCap = kTile * kGPU;         // groups per tile
  // Units in shared memory hold binary32 bits (f32 rows, or any dtype on the
  // 4-element scalar path) or raw 16-bit values (bf16/f16 on the 128-bit path).
  static constexpr bool kF32Bits = DT == 0 || !VEC;
  static constexpr int kTileBytes = kTile * 16;
  // A warp's list area: the rare list, then a tile's compacted list (one
  // 16-bit tile-local group index per surviving group).
  static constexpr int kListBytes = ((kRareBytes + kCap * 2 + 15) / 16) * 16;
  static constexpr int kWarpBytes = kStages * kTileBytes + kListBytes;
  static constexpr size_t kSmem = (size_t)kWarps * kWarpBytes;
};

// Element e (0 <= e < kEPU) of a unit.
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

// Unit u of a row read with plain loads; elements at or past V read as -inf.
template <int DT, bool VEC>
__device__ __forceinline__ uint4 load_unit_sync(const char* row, int32_t u, int32_t V) {
  using C = Cfg<DT, VEC>;
  const int32_t e0 = u * C::kEPU;
  uint32_t w[4];
  if constexpr (C::kF32Bits) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w[e] = (e0 + e < V) ? __float_as_uint(load_elt<DT>(row, e0 + e)) : kNegInfF32;
  } else {
    const unsigned short* h = reinterpret_cast<const unsigned short*>(row);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t lo = (e0 + 2 * k < V) ? (uint32_t)__ldg(h + e0 + 2 * k) : neg_inf_half<DT>();
      const uint32_t hi = (e0 + 2 * k + 1 < V) ? (uint32_t)__ldg(h + e0 + 2 * k + 1) : neg_inf_half<DT>();
      w[k] = lo | (hi << 16);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// ---------------------------------------------------------------------------
// Packed 16-bit helpers: max of two bf16x2/f16x2 words and "any half >= thr".
// The max ignores a NaN operand (like fmaxf); the compare is ordered (NaN false).
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ uint32_t hmax2_bits(uint32_t a, uint32_t b) {
  if constexpr (DT == 1) {
    __nv_bfloat162 m = __hmax2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<__nv_bfloat162*>(&b));
    return *reinterpret_cast<uint32_t*>(&m);
  } else {
    __half2 m = __hmax2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
    return *reinterpret_cast<uint32_t*>(&m);
  }
}

template <int DT>
__device__ __forceinline__ bool hge2_any(uint32_t a, uint32_t thr2) {
  if constexpr (DT == 1) {
    return __hge2_mask(*reinterpret_cast<__nv_bfloat162*>(&a),
                       *reinterpret_cast<__nv_bfloat162*>(&thr2)) != 0u;
  } else {
    return __hge2_mask(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&thr2)) != 0u;
  }
}

// thr rounded down to the 16-bit type, in both halves: x >= thr implies
// x16 >= thr16, so the packed test never drops a survivor.
template <int DT>
__device__ __forceinline__ uint32_t packed_threshold(float thr) {
  uint32_t h;
  if constexpr (DT == 1) {
    __nv_bfloat16 b = __float2bfloat16_rd(thr);
    h = *reinterpret_cast<unsigned short*>(&b);
  } else {
    __half b = __float2half_rd(thr);
    h = *reinterpret_cast<unsigned short*>(&b);
  }
  return h * 0x10001u;
}

template <int DT, bool VEC>
__device__ __forceinline__ float unit_max(const uint4& r) {
  if constexpr (Cfg<DT, VEC>::kF32Bits) {
    return fmaxf(fmaxf(__uint_as_float(r.x), __uint_as_float(r.y)),
                 fmaxf(__uint_as_float(r.z), __uint_as_float(r.w)));
  } else {
    const uint32_t m = hmax2_bits<DT>(hmax2_bits<DT>(r.x, r.y), hmax2_bits<DT>(r.z, r.w));
    return fmaxf(half_to_f32<DT>(m & 0xFFFFu), half_to_f32<DT>(m >> 16));
  }  // NaN is ignored unless every element is NaN
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
  float T;
  float rT;
  PhiloxRow ph;  // the row's Philox key and counter words, first rounds folded
  WsRow* ws;
};

__device__ __forceinline__ RowCtx row_context(const SampleParams& p, int64_t b) {
  RowCtx rc;
  rc.ws = p.ws + b;
  rc.T = p.temperature ? __ldg(p.temperature + b) : 0.0f;
  rc.rT = 1.0f;
  rc.ph = PhiloxRow{0u, 0u, 0u, 0u, 0u, 0u};
  if (rc.T > 0.0f) {  // NaN and T <= 0: greedy
    const uint64_t sd = __ldg(p.seed + b), of = __ldg(p.offset + b);
    rc.ph = philox_row((uint32_t)b, (uint32_t)of, (uint32_t)(of >> 32), (uint32_t)sd,
                       (uint32_t)(sd >> 32));
    rc.rT = 1.0f / rc.T;
  }
  return rc;
}

// A row's raw parameters, loaded ahead of use (zeros past the last row).
struct RowParams {
  float T;
  uint64_t seed, offset;
};

__device__ __forceinline__ RowParams load_row_params(const SampleParams& p, int64_t b) {
  RowParams r{0.0f, 0ull, 0ull};
  if (b < p.B && p.temperature) {
    r.T = __ldg(p.temperature + b);
    r.seed = __ldg(p.seed + b);
    r.offset = __ldg(p.offset + b);
  }
  return r;
}

__device__ __forceinline__ RowCtx row_context_from(const SampleParams& p, int64_t b,
                                                   const RowParams& r) {
  RowCtx rc;
  rc.ws = p.ws + b;
  rc.T = r.T;
  rc.rT = 1.0f;
  rc.ph = PhiloxRow{0u, 0u, 0u, 0u, 0u, 0u};
  if (rc.T > 0.0f) {
    rc.ph = philox_row((uint32_t)b, (uint32_t)r.offset, (uint32_t)(r.offset >> 32),
                       (uint32_t)r.seed, (uint32_t)(r.seed >> 32));
    rc.rT = 1.0f / rc.T;
  }
  return rc;
}

// The warp whose ticket brought the row's finished-unit count to NU writes the
// row's answer and clears its workspace slot.
__device__ __noinline__ void finish_row_if_last(const SampleParams& p, int64_t b, uint32_t before,
                                                uint32_t mine, int64_t NU) {
  if ((int64_t)before + mine != NU) return;
  WsRow* ws = p.ws + b;
  __threadfence();
  const unsigned long long key = atomicExch(&ws->key, 0ull);
  atomicExch(&ws->ticket, 0u);
  atomicExch(&ws->hint, 0u);
  p.out_idx[b] = index_of_key(key);
}


// Groups that passed the cheap test wait in a per-warp list, across tiles,
// until 32 of them (or the end of the warp's part of the row) make one exact
// pass with every lane busy. An entry holds the row-local group index and the
// group's four logits as stored in the tile (so the ring stage may be reused).
template <int DT, bool VEC>
using RareRaw = typename std::conditional<Cfg<DT, VEC>::kF32Bits, uint4, uint2>::type;

template <int DT, bool VEC>
__device__ __forceinline__ void raw_values(const RareRaw<DT, VEC>& r, float x[4]) {
  if constexpr (Cfg<DT, VEC>::kF32Bits) {
    x[0] = __uint_as_float(r.x);
    x[1] = __uint_as_float(r.y);
    x[2] = __uint_as_float(r.z);
    x[3] = __uint_as_float(r.w);
  } else {
    x[0] = half_to_f32<DT>(r.x & 0xFFFFu);
    x[1] = half_to_f32<DT>(r.x >> 16);
    x[2] = half_to_f32<DT>(r.y & 0xFFFFu);
    x[3] = half_to_f32<DT>(r.y >> 16);
  }
}

// Score the listed groups exactly (one per lane) against the current bound.
// Out of line: it runs once per 32 listed groups, and keeping its logarithms
// out of the tile loop keeps that loop's code small.
struct Best {
  float s;
  int32_t i;
};

template <int DT, bool VEC>
__device__ __noinline__ Best flush_rare_cold(const unsigned char* rbase, int rcnt, float T, float rT,
                                             PhiloxRow ph, Prune pr, float bs, int32_t bi) {
  const int lane = threadIdx.x & 31;
  __syncwarp();  // the entries of every lane are visible
  GSAMPLE_COUNT(lane < rcnt ? 1 : 0);
  if (lane < rcnt) {
    const uint32_t g = reinterpret_cast<const uint32_t*>(rbase)[lane];
    float x[4];
    raw_values<DT, VEC>(reinterpret_cast<const RareRaw<DT, VEC>*>(rbase + kRareRawOff)[lane], x);
    const uint4 w = philox_row_1(g, ph);
    score_group(g, x[0], x[1], x[2], x[3], w, pr, make_reach(pr, rT), T, &bs, &bi);
  }
  __syncwarp();  // every lane has read its entry before the list is refilled
  return Best{bs, bi};
}

template <int DT, bool VEC>
__device__ __forceinline__ void flush_rare(const unsigned char* rbase, int rcnt, const RowCtx& rc,
                                           const Prune& pr, float& bs, int32_t& bi) {
  const Best r = flush_rare_cold<DT, VEC>(rbase, rcnt, rc.T, rc.rT, rc.ph, pr, bs, bi);
  bs = r.s;
  bi = r.i;
}

// Tile-local group q of this lane's i-th group (unit i / kGPU, half i % kGPU).
template <int DT, bool VEC>
__device__ __forceinline__ uint32_t lane_group(int i, int lane) {
  using C = Cfg<DT, VEC>;
  return (uint32_t)(((i / C::kGPU) * 32 + lane) * C::kGPU + i % C::kGPU);
}

// Groups whose word test passed join the rare list: one round per set bit of
// the lane's `need` mask. Bit j stands for tile-local group q[j], or, with N ==
// 0, for the lane's j-th group of the tile.
template <int DT, bool VEC, int N>
__device__ __forceinline__ void append_rare(uint32_t need, const uint32_t* q, uint32_t stage,
                                            uint32_t g0, const RowCtx& rc, const Prune& pr,
                                            unsigned char* rbase, int& rcnt, float& bs,
                                            int32_t& bi) {
  using C = Cfg<DT, VEC>;
  const int lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1u;
  while (__any_sync(0xFFFFFFFFu, need != 0u)) {
    const bool has = need != 0u;
    const unsigned m = __ballot_sync(0xFFFFFFFFu, has);
    const int n = __popc(m);
    if (rcnt + n > kRareCap) {
      flush_rare<DT, VEC>(rbase, rcnt, rc, pr, bs, bi);
      rcnt = 0;
    }
    if (has) {
      const int jj = __ffs(need) - 1;
      need &= need - 1u;
      uint32_t qq;
      if constexpr (N == 0) {
        qq = lane_group<DT, VEC>(jj, lane);
      } else {
        qq = q[0];
#pragma unroll
        for (int j = 1; j < N; ++j)
          if (jj == j) qq = q[j];
      }
      const int s = rcnt + __popc(m & lt_mask);
      reinterpret_cast<uint32_t*>(rbase)[s] = g0 + qq;
      auto* raw = reinterpret_cast<RareRaw<DT, VEC>*>(rbase + kRareRawOff);
      if constexpr (C::kF32Bits) {
        raw[s] = lds128(stage + qq * 16u);
      } else {
        raw[s] = lds64(stage + qq * 8u);
      }
    }
    rcnt += n;
  }
}

// The largest logit of tile-local group q, read back from the stage.
template <int DT, bool VEC>
__device__ __forceinline__ float group_max_at(uint32_t stage, uint32_t q) {
  if constexpr (Cfg<DT, VEC>::kF32Bits) {
    const uint4 d = lds128(stage + q * 16u);
    return fmaxf(fmaxf(__uint_as_float(d.x), __uint_as_float(d.y)),
                 fmaxf(__uint_as_float(d.z), __uint_as_float(d.w)));
  } else {
    const uint2 d = lds64(stage + q * 8u);
    const uint32_t m = hmax2_bits<DT>(d.x, d.y);
    return fmaxf(half_to_f32<DT>(m & 0xFFFFu), half_to_f32<DT>(m >> 16));
  }
}

// One batch of the compacted list: entries [base, base + 32 * N) below cnt,
// N Philox blocks per lane side by side.
template <int DT, bool VEC, int N>
__device__ __forceinline__ void compact_batch(uint32_t stage, const unsigned short* clist, int base,
                                              int cnt, uint32_t g0, const RowCtx& rc,
                                              const Prune& pr, const ReachTest& rt,
                                              unsigned char* rbase, int& rcnt, float& bs,
                                              int32_t& bi) {
  const int lane = threadIdx.x & 31;
  uint32_t q[N], g[N], wt[N];
  bool valid[N];
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const int idx = base + lane + 32 * j;
    valid[j] = idx < cnt;
    q[j] = valid[j] ? (uint32_t)clist[idx] : 0u;
    wt[j] = word_threshold(group_max_at<DT, VEC>(stage, q[j]), pr, rt);
    g[j] = g0 + q[j];
  }
  uint4 w[N];
  philox_row_xn<N>(g, rc.ph, w);
#ifdef GSAMPLE_COUNT_BLOCKS
  {
    int nv = 0;
#pragma unroll
    for (int j = 0; j < N; ++j) nv += valid[j] ? 1 : 0;
    GSAMPLE_COUNT(nv);
  }
#endif
  uint32_t need = 0;
#pragma unroll
  for (int j = 0; j < N; ++j) need |= (valid[j] && max_word(w[j]) >= wt[j]) ? (1u << j) : 0u;
  append_rare<DT, VEC, N>(need, q, stage, g0, rc, pr, rbase, rcnt, bs, bi);
}

#ifndef GSAMPLE_DENSE_NUM
#define GSAMPLE_DENSE_NUM 1  // dense when more than NUM/DEN of the tile's groups survive
#endif
#ifndef GSAMPLE_DENSE_DEN
#define GSAMPLE_DENSE_DEN 8
#endif

// A sampled tile. Each lane first takes the largest logit of each of its
// groups. The share of groups that reach the logit threshold is estimated from
// 128 of them (each lane's first four); when none of those does, the whole
// tile is tested and skipped if no group in the warp reaches it. A large
// share (above GSAMPLE_DENSE_NUM/DEN): every group
// gets its Philox block, four per lane side by side, as straight-line code.
// Otherwise the survivors' tile-local indices are compacted into a list and
// only they get Philox, 128 per warp batch (a short last batch runs one or two
// blocks per lane). Either way the word test follows, and the rare groups that
// pass it join the rare list.
template <int DT, bool VEC>
__device__ __forceinline__ void sampled_tile(uint32_t stage, uint32_t g0, const RowCtx& rc,
                                             const Prune& pr, unsigned char* rbase,
                                             unsigned short* clist, int& rcnt, float& bs,
                                             int32_t& bi) {
  using C = Cfg<DT, VEC>;
  constexpr int NG = kVPT * C::kGPU;  // groups per lane in a tile
  static_assert(NG % 4 == 0 && NG <= 32, "groups per lane must fill four-way Philox batches");
  const int lane = threadIdx.x & 31;
  float xm[NG];
#pragma unroll
  for (int k = 0; k < kVPT; ++k) {
    const uint4 r = lds128(stage + (uint32_t)(k * 32 + lane) * 16u);
    if constexpr (C::kF32Bits) {
      xm[k] = fmaxf(fmaxf(__uint_as_float(r.x), __uint_as_float(r.y)),
                    fmaxf(__uint_as_float(r.z), __uint_as_float(r.w)));
    } else {
      const uint32_t m0 = hmax2_bits<DT>(r.x, r.y), m1 = hmax2_bits<DT>(r.z, r.w);
      xm[2 * k] = fmaxf(half_to_f32<DT>(m0 & 0xFFFFu), half_to_f32<DT>(m0 >> 16));
      xm[2 * k + 1] = fmaxf(half_to_f32<DT>(m1 & 0xFFFFu), half_to_f32<DT>(m1 >> 16));
    }
  }
  // The share of surviving groups, estimated from each lane's first four. Only
  // when none of those survives is the whole tile tested for a skip (at
  // moderate and high temperatures the sample almost always holds survivors,
  // and the tile's maximum is not needed).
  int c4 = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) c4 += xm[i] >= pr.thr_x ? 1 : 0;
  const int sample = (int)__reduce_add_sync(0xFFFFFFFFu, (unsigned)c4);
  if (sample == 0) {
    float tm = xm[0];
#pragma unroll
    for (int i = 1; i < NG; ++i) tm = fmaxf(tm, xm[i]);
    if (!__any_sync(0xFFFFFFFFu, tm >= pr.thr_x)) return;  // nothing here can win
  }
  const ReachTest rt = make_reach(pr, rc.rT);
  if (sample * GSAMPLE_DENSE_DEN > 128 * GSAMPLE_DENSE_NUM) {
    // Every group's word threshold first: it needs only the logits, so its
    // exponential runs ahead of, not after, the Philox chains.
    uint32_t wt[NG];
#pragma unroll
    for (int i = 0; i < NG; ++i) wt[i] = word_threshold(xm[i], pr, rt);
    uint32_t need = 0;
    GSAMPLE_COUNT(NG);
    const uint32_t gl = g0 + lane_group<DT, VEC>(0, lane);
#pragma unroll
    for (int b = 0; b < NG; b += 4) {
      uint32_t g[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        g[j] = gl + (uint32_t)(((b + j) / C::kGPU) * 32 * C::kGPU + (b + j) % C::kGPU);
      uint4 w[4];
      philox_row_x4(g, rc.ph, w);
#pragma unroll
      for (int j = 0; j < 4; ++j) need |= max_word(w[j]) >= wt[b + j] ? (1u << (b + j)) : 0u;
    }
    append_rare<DT, VEC, 0>(need, nullptr, stage, g0, rc, pr, rbase, rcnt, bs, bi);
    return;
  }

  // The survivors' tile-local indices, lane by lane: each lane's mask, an
  // exclusive scan of the lanes' counts, then each lane writes its own.
  uint32_t keep = 0;
#pragma unroll
  for (int i = 0; i < NG; ++i) keep |= xm[i] >= pr.thr_x ? (1u << i) : 0u;
  const int mine = __popc(keep);
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  const int cnt = __shfl_sync(0xFFFFFFFFu, incl, 31);
  int pos = incl - mine;
  while (keep != 0u) {
    const int i = __ffs(keep) - 1;
    keep &= keep - 1u;
    clist[pos++] = (unsigned short)lane_group<DT, VEC>(i, lane);
  }
  __syncwarp();
  for (int base = 0; base < cnt; base += 128) {
    const int r = cnt - base;
    if (r > 64) {
      compact_batch<DT, VEC, 4>(stage, clist, base, cnt, g0, rc, pr, rt, rbase, rcnt, bs, bi);
    } else if (r > 32) {
      compact_batch<DT, VEC, 2>(stage, clist, base, cnt, g0, rc, pr, rt, rbase, rcnt, bs, bi);
    } else {
      compact_batch<DT, VEC, 1>(stage, clist, base, cnt, g0, rc, pr, rt, rbase, rcnt, bs, bi);
    }
  }
  __syncwarp();  // the list is read before the next tile rewrites it
}

// Phase A: this lane's largest logit of the tile, scored exactly.
template <int DT, bool VEC>
__device__ __forceinline__ void lane_candidate(uint32_t stage, int32_t t0, int32_t t_hi,
                                               const RowCtx& rc, float& bs, int32_t& bi) {
  using C = Cfg<DT, VEC>;
  const int lane = threadIdx.x & 31;
  float cm = -INFINITY;
  int ck = -1;
#pragma unroll
  for (int k = 0; k < kVPT; ++k) {
    if (t0 + k * 32 + lane >= t_hi) break;
    const float m = unit_max<DT, VEC>(lds128(stage + (uint32_t)(k * 32 + lane) * 16u));
    if (m > cm) {
      cm = m;
      ck = k;
    }
  }
  GSAMPLE_COUNT(ck < 0 ? 0 : 1);
  if (ck < 0) return;
  const uint4 ru = lds128(stage + (uint32_t)(ck * 32 + lane) * 16u);
  int ce = C::kEPU - 1;
#pragma unroll
  for (int e = C::kEPU - 1; e >= 0; --e)
    if (unit_elt<DT, VEC>(ru, e) == cm) ce = e;
  const int32_t i = (t0 + ck * 32 + lane) * C::kEPU + ce;
  const uint4 blk = philox_row_1((uint32_t)i >> 2, rc.ph);
  take_better(exact_score(cm, word_of(blk, i & 3), rc.T), i, bs, bi);
}

// Warp-uniform cursor over this warp's tiles: row b, row-local units
// [t0, t_hi), and the warp's part of row b, [seg_lo, seg_hi).
struct TileCursor {
  int64_t b;
  int32_t t0, t_hi, seg_lo, seg_hi;
  bool valid;
};

__device__ __forceinline__ TileCursor segment_at(int64_t b, int64_t u_lo, int64_t u_end,
                                                 int64_t NU, int tile) {
  TileCursor c;
  c.b = b;
  c.valid = u_lo < u_end;
  const int64_t row0 = b * NU;
  c.seg_lo = (int32_t)(u_lo - row0);
  c.seg_hi = c.valid ? (int32_t)((u_end < row0 + NU ? u_end : row0 + NU) - row0) : 0;
  c.t0 = c.seg_lo;
  c.t_hi = min(c.t0 + tile, c.seg_hi);
  return c;
}

// The first tile of the next row of this warp's range (rare: once per row).
__device__ __noinline__ TileCursor next_row(int64_t b, int64_t u_end, int64_t NU, int tile) {
  return segment_at(b + 1, (b + 1) * NU, u_end, NU, tile);
}

template <int TILE>
__device__ __forceinline__ TileCursor next_tile(const TileCursor& c, int64_t u_end, int64_t NU) {
  if (!c.valid) return c;
  if (c.t_hi < c.seg_hi) {
    TileCursor n = c;
    n.t0 = c.t_hi;
    n.t_hi = min(n.t0 + TILE, c.seg_hi);
    return n;
  }
  return next_row(c.b, u_end, NU, TILE);
}

// Start copying a tile into a ring stage and close its cp.async group (an empty
// group when there is no tile, so that group counting stays uniform). Units
// past the tile, and elements past V in a row's last unit, read as -inf.
template <int DT, bool VEC>
__device__ __forceinline__ void issue_tile(const SampleParams& p, const TileCursor& c,
                                           uint32_t stage, uint64_t pol) {
  using C = Cfg<DT, VEC>;
  if (c.valid) {
    const int lane = threadIdx.x & 31;
    const char* row = p.logits + c.b * p.ld_bytes;
    if (VEC && c.t_hi - c.t0 == C::kTile && c.t_hi * C::kEPU <= p.V) {
      // A full tile inside the row: kVPT coalesced 512-byte copies, no checks.
      const char* src = row + (size_t)(c.t0 + lane) * 16;
      const uint32_t dst = stage + (uint32_t)lane * 16u;
#pragma unroll
      for (int k = 0; k < kVPT; ++k) cp_async16(dst + k * 512u, src + k * 512, pol);
      cp_async_commit();
      return;
    }
#pragma unroll
    for (int k = 0; k < kVPT; ++k) {
      const int32_t u = c.t0 + k * 32 + lane;
      const uint32_t dst = stage + (uint32_t)(k * 32 + lane) * 16u;
      if (VEC && u < c.t_hi && (u + 1) * C::kEPU <= p.V) {
        cp_async16(dst, row + (size_t)u * 16, pol);
      } else if (u < c.t_hi) {
        sts128(dst, load_unit_sync<DT, VEC>(row, u, p.V));
      } else {
        sts128(dst, empty_unit<DT, VEC>());
      }
    }
  }
  cp_async_commit();
}

__device__ __forceinline__ float warp_max_f32(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// The hint word holds the ordered bits of the best score any warp has seen in
// the row so far (0: none yet).
__device__ __forceinline__ float score_of_hint(uint32_t h) {
  return h == 0u ? -INFINITY : score_of_key((unsigned long long)h << 32 | 1ull);
}

// Start of warp w's range of units (w = NW gives the end of the last). The
// units are dealt in near-equal shares; on the 128-bit path each split point
// then moves down, within its row, to a unit that starts a 128-byte line.
// Host-resident logits (read over the CPU-GPU link) arrive in whole 128-byte
// lines: with ranges that split lines, both neighbours fetch the shared line,
// and host reads measured a third slower. Device reads are unaffected.
template <bool VEC>
__device__ __forceinline__ int64_t split_point(const SampleParams& p, int64_t w) {
  const int64_t U = p.total_units, NW = p.warps;
  const int64_t base = U / NW, rem = U % NW;
  const int64_t u = w * base + (w < rem ? w : rem);
  if (!VEC || u >= U) return u;
  const int64_t NU = p.units_per_row, b = u / NU, l = u - b * NU;
  const uint64_t row_unit = (uint64_t)(uintptr_t)(p.logits + b * p.ld_bytes) / 16u;
  const int64_t la = l - (int64_t)((row_unit + (uint64_t)l) & 7u);
  return b * NU + (la > 0 ? la : 0);
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads, GSAMPLE_MIN_CTAS_PER_SM) sample_kernel(const SampleParams p) {
  using C = Cfg<DT, VEC>;
  extern __shared__ __align__(16) unsigned char smem[];
  pdl_wait_then_release();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  unsigned char* wbase = smem + (size_t)warp * C::kWarpBytes;
  const uint32_t ring = smem_addr(wbase);
  const uint64_t pol = evict_first_policy();

  const int64_t NU = p.units_per_row, NW = p.warps;
  const int64_t gw = (int64_t)blockIdx.x * kWarps + warp;
  if (gw >= NW) return;
  const int64_t u_begin = split_point<VEC>(p, gw), u_end = split_point<VEC>(p, gw + 1);
  if (u_begin >= u_end) return;  // no units (only with fewer than 8 units per warp)

  // Prologue: the first kStages - 1 tiles go in flight.
  TileCursor cur = segment_at(u_begin / NU, u_begin, u_end, NU, C::kTile);
  TileCursor ahead = cur;
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    issue_tile<DT, VEC>(p, ahead, ring + s * C::kTileBytes, pol);
    ahead = next_tile<C::kTile>(ahead, u_end, NU);
  }

  RowCtx rc = row_context(p, cur.b);
  // The next row's parameters, loaded a whole segment before they are needed.
  RowParams next_params = load_row_params(p, cur.b + 1);
  bool seg_first = true;
  float bs = -INFINITY;
  int32_t bi = INT32_MAX;
  // The row's hint word, read one tile ahead of its use so that the load's
  // latency hides behind a tile of work; `seen` is the value in use now.
  uint32_t seen = 0u, pending = 0u;
  // The ticket of the last finished segment is checked a tile later, so that
  // the warp never waits for the atomic's return (lane 0 only).
  bool tk_pending = false;
  uint32_t tk_before = 0u, tk_mine = 0u;
  int64_t tk_row = 0;
  int slot = 0;
  // Rare list (dense path): entries pending an exact pass, and the bound of the
  // tile that listed the last of them.
  unsigned char* rbase = wbase + kStages * C::kTileBytes;
  int rcnt = 0;
  Prune pr_last{INFINITY, -INFINITY, false};

  while (true) {
    // The current tile has landed (this lane's copies, then everyone's).
    cp_async_wait<kStages - 2>();
    __syncwarp();
    const uint32_t stage = ring + slot * C::kTileBytes;
    // Refill the ring slot that the previous tile freed.
    int fill = slot + kStages - 1;
    if (fill >= kStages) fill -= kStages;
    issue_tile<DT, VEC>(p, ahead, ring + fill * C::kTileBytes, pol);
    ahead = next_tile<C::kTile>(ahead, u_end, NU);

    const int32_t t0 = cur.t0, t_hi = cur.t_hi;
    if (rc.T > 0.0f) {
      if (seg_first) {
        lane_candidate<DT, VEC>(stage, t0, t_hi, rc, bs, bi);
        seen = 0u;
      } else {
        seen = pending;
      }
      pending = __ldcg(&rc.ws->hint);
      // The best exact score this warp knows; publish it (fire-and-forget) if
      // it beats what the row had, and prune against the larger of the two.
      const float wbest = warp_max_f32(bs);
      const uint32_t wb = wbest > -INFINITY ? ordered_bits(wbest) : 0u;
      if (lane == 0 && wb > seen) atomicMax(&rc.ws->hint, wb);
      const float L = fmaxf(wbest, score_of_hint(seen));
      const Prune pr = make_prune(L, rc.T);
      pr_last = pr;
      sampled_tile<DT, VEC>(stage, (uint32_t)t0 * C::kGPU, rc, pr, rbase,
                            reinterpret_cast<unsigned short*>(rbase + kRareBytes), rcnt, bs, bi);
    } else {
#pragma unroll
      for (int k = 0; k < kVPT; ++k) {
        const int32_t u = t0 + k * 32 + lane;
        greedy_unit<DT, VEC>(lds128(stage + (uint32_t)(k * 32 + lane) * 16u), u, bs, bi);
      }
    }
    __syncwarp();  // every lane is done with this stage before it is refilled

    if (lane == 0 && tk_pending) {
      finish_row_if_last(p, tk_row, tk_before, tk_mine, NU);
      tk_pending = false;
    }
    if (cur.t_hi == cur.seg_hi) {
      // This warp's part of row b is done: merge its best, then add its units
      // to the row's ticket; the warp that brings the count to NU writes the
      // answer and clears the row's slot (checked one tile later).
      if (rcnt > 0) {
        flush_rare<DT, VEC>(rbase, rcnt, rc, pr_last, bs, bi);
        rcnt = 0;
      }
      warp_argmax(bs, bi);
      if (lane == 0) {
        if (bi != INT32_MAX && bs > -INFINITY) atomicMax(&rc.ws->key, pack_key(bs, bi));
        __threadfence();
        tk_mine = (uint32_t)(cur.seg_hi - cur.seg_lo);
        tk_before = atomicAdd(&rc.ws->ticket, tk_mine);
        tk_row = cur.b;
        tk_pending = true;
      }
      cur = next_tile<C::kTile>(cur, u_end, NU);
      if (!cur.valid) break;
      rc = row_context_from(p, cur.b, next_params);
      next_params = load_row_params(p, cur.b + 1);
      bs = -INFINITY;
      bi = INT32_MAX;
      seg_first = true;
    } else {
      cur = next_tile<C::kTile>(cur, u_end, NU);
      seg_first = false;
    }
    slot = slot + 1 == kStages ? 0 : slot + 1;
  }
  if (lane == 0 && tk_pending) finish_row_if_last(p, tk_row, tk_before, tk_mine, NU);
  cp_async_wait<0>();  // no copy may outlive the warp
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sample_smem_bytes(dtype, vec);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
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

// flags[j]: bit 0 = the element test may_reach(x[j], w[j]), bit 1 = the
// group test w[j] >= word_threshold(x[j]); threshold[j] = that threshold.
__global__ void debug_word_test_kernel(const float* x, const uint32_t* w, int64_t n, float L,
                                       float T, uint32_t* threshold, uint8_t* flags) {
  const Prune pr = make_prune(L, T);
  const ReachTest rt = make_reach(pr, 1.0f / T);
  for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n;
       j += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t t = word_threshold(x[j], pr, rt);
    const bool elem = pr.use_bound ? may_reach(x[j], w[j], rt) : (x[j] >= pr.thr_x);
    threshold[j] = t;
    flags[j] = (uint8_t)((elem ? 1 : 0) | (w[j] >= t ? 2 : 0));
  }
}

// Philox throughput alone: each thread runs `iters` batches of four blocks of
// the kernels' row-folded block code (philox_row_x4) and folds the words into
// sink[thread], so nothing but the blocks is measured.
__global__ void __launch_bounds__(1024, 1) debug_philox_rate_kernel(uint32_t iters, uint32_t* sink) {
  const uint32_t t = blockIdx.x * blockDim.x + threadIdx.x;
  const PhiloxRow pr = philox_row(blockIdx.x, 7u, 0u, 0x12345u + t / 1024u, 0x6789Au);
  uint32_t acc = 0;
  for (uint32_t it = 0; it < iters; ++it) {
    uint32_t g[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) g[j] = t * 4096u + it * 4u + (uint32_t)j;
    uint4 w[4];
    philox_row_x4(g, pr, w);
#pragma unroll
    for (int j = 0; j < 4; ++j) acc ^= w[j].x ^ w[j].y ^ w[j].z ^ w[j].w;
  }
  sink[t] = acc;
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

cudaError_t launch_debug_philox_rate(int ctas, int threads, uint32_t iters, uint32_t* sink,
                                     cudaStream_t stream) {
  debug_philox_rate_kernel<<<ctas, threads, 0, stream>>>(iters, sink);
  return cudaGetLastError();
}

cudaError_t read_blocks_computed(unsigned long long* out, bool reset) {
#ifdef GSAMPLE_COUNT_BLOCKS
  cudaError_t e = cudaMemcpyFromSymbol(out, g_blocks_computed, sizeof *out);
  if (e == cudaSuccess && reset) {
    const unsigned long long z = 0;
    e = cudaMemcpyToSymbol(g_blocks_computed, &z, sizeof z);
  }
  return e;
#else
  (void)out;
  (void)reset;
  return cudaErrorNotSupported;
#endif
}

cudaError_t launch_debug_word_test(const float* x, const uint32_t* w, int64_t n, float L, float T,
                                   uint32_t* threshold, uint8_t* flags, cudaStream_t stream) {
  debug_word_test_kernel<<<grid_for(n), 256, 0, stream>>>(x, w, n, L, T, threshold, flags);
  return cudaGetLastError();
}

}  // namespace gsample
