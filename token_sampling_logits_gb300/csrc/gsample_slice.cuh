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

}  // namespace slice
}  // namespace gsample
