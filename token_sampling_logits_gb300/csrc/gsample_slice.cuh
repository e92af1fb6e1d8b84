// Helpers shared by the kernels that hold a row slice in shared memory (the
// HLG sampler, the categorical baseline, the small-batch sampler and the
// filtered path): unit shapes, element decoding and unit loads with -inf
// padding. The cp.async / shared-memory primitives live in gsample_device.cuh.
#pragma once

#include <cstdint>

#include "gsample_device.cuh"

namespace gsample {
namespace slice {

template <int DT, bool VEC>
struct HCfg {
  static constexpr int kEPU = VEC ? (DT == 0 ? 4 : 8) : 4;
  static constexpr int kGPU = kEPU / 4;
  static constexpr bool kF32Bits = DT == 0 || !VEC;
};

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

// cp.async.wait_group with a count known only after unrolling.
__device__ __forceinline__ void cp_async_wait_upto(int n) {
  switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    case 4: cp_async_wait<4>(); break;
    case 5: cp_async_wait<5>(); break;
    case 6: cp_async_wait<6>(); break;
    default: cp_async_wait<7>(); break;
  }
}

// The thread's units of the slice [u_lo, u_hi) (u_lo + tid, then every
// THREADS-th unit) are requested into shared memory in CHUNKS commit groups,
// in unit order; then f(u, unit) runs on each unit, in the same order, as soon
// as its chunk has landed, so the work on the first chunks overlaps the
// arrival of the later ones. Units past V read as -inf. Each thread reads back
// only its own units, so its own wait suffices.
template <int DT, bool VEC, int THREADS, int CHUNKS, typename F>
__device__ __forceinline__ void load_slice_then(const char* row, int32_t u_lo, int32_t u_hi,
                                                int32_t V, uint32_t slice, uint64_t pol, F&& f) {
  static_assert(CHUNKS >= 1 && CHUNKS <= 8, "one to eight commit groups");
  constexpr int EPU = HCfg<DT, VEC>::kEPU;
  const int tid = threadIdx.x;
  const int32_t n = u_hi - u_lo > tid ? (u_hi - u_lo - tid + THREADS - 1) / THREADS : 0;
  const int32_t per = (n + CHUNKS - 1) / CHUNKS;
#pragma unroll
  for (int c = 0; c < CHUNKS; ++c) {
    const int32_t i1 = min(n, (c + 1) * per);
    for (int32_t i = c * per; i < i1; ++i) {
      const int32_t u = u_lo + tid + i * THREADS;
      const uint32_t dst = slice + (uint32_t)(u - u_lo) * 16u;
      if (VEC && (u + 1) * EPU <= V)
        cp_async16(dst, row + (size_t)u * 16, pol);
      else
        sts128(dst, load_unit<DT, VEC>(row, u, V, pol));
    }
    cp_async_commit();
  }
#pragma unroll
  for (int c = 0; c < CHUNKS; ++c) {
    cp_async_wait_upto(CHUNKS - 1 - c);
    const int32_t i1 = min(n, (c + 1) * per);
    for (int32_t i = c * per; i < i1; ++i) {
      const int32_t u = u_lo + tid + i * THREADS;
      f(u, lds128(slice + (uint32_t)(u - u_lo) * 16u));
    }
  }
}

}  // namespace slice
}  // namespace gsample
