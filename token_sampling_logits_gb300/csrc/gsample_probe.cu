// Diagnostic probe: how ALU work issued beside the Philox multiplies adds to
// their time. Each thread runs `iters` iterations of four Philox4x32-10 blocks
// of the kernels' row-folded block code (philox_row_x4) and/or 4 * STEPS
// independent ALU updates per block (shifts and bitwise operations in four
// chains that do not depend on the Philox words), then folds everything into
// sink[thread] so that nothing is optimised away. Timing the three shapes
// (Philox alone, ALU alone, both) shows how much of the ALU work hides behind
// the multiplies: the sampler's filter (group maxima, the word test) is ALU
// work of this kind.
#include <cstdint>

#include <cuda_runtime.h>

#include "gsample_debug.h"
#include "gsample_device.cuh"

namespace gsample {
namespace {

template <bool PHILOX, int STEPS>
__global__ void __launch_bounds__(1024, 1) probe_mix_kernel(uint32_t iters, uint32_t* sink) {
  const uint32_t t = blockIdx.x * blockDim.x + threadIdx.x;
  const PhiloxRow pr = philox_row(blockIdx.x, 7u, 0u, 0x12345u + t / 1024u, 0x6789Au);
  uint32_t acc = 0;
  uint32_t a0 = t, a1 = t * 3u, a2 = t * 5u, a3 = t * 7u;
  for (uint32_t it = 0; it < iters; ++it) {
    if constexpr (PHILOX) {
      uint32_t g[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) g[j] = t * 4096u + it * 4u + (uint32_t)j;
      uint4 w[4];
      philox_row_x4(g, pr, w);
#pragma unroll
      for (int j = 0; j < 4; ++j) acc ^= w[j].x ^ w[j].y ^ w[j].z ^ w[j].w;
    }
    // STEPS updates of four chains per block, four blocks per iteration.
#pragma unroll
    for (int e = 0; e < 4 * STEPS; ++e) {
      a0 = (a0 ^ (a1 >> 3)) & 0x7FFFFFFFu;
      a1 = (a1 ^ (a2 << 1)) | 1u;
      a2 = a2 ^ a3 ^ it;
      a3 = (a3 >> 1) ^ a0;
    }
  }
  sink[t] = acc ^ a0 ^ a1 ^ a2 ^ a3;
}

cudaError_t launch_probe(bool philox, int steps, int ctas, int threads, uint32_t iters,
                         uint32_t* sink, cudaStream_t stream) {
  if (philox && steps == 0) {
    probe_mix_kernel<true, 0><<<ctas, threads, 0, stream>>>(iters, sink);
  } else if (philox && steps == 2) {
    probe_mix_kernel<true, 2><<<ctas, threads, 0, stream>>>(iters, sink);
  } else if (philox && steps == 4) {
    probe_mix_kernel<true, 4><<<ctas, threads, 0, stream>>>(iters, sink);
  } else if (!philox && steps == 2) {
    probe_mix_kernel<false, 2><<<ctas, threads, 0, stream>>>(iters, sink);
  } else {
    probe_mix_kernel<false, 4><<<ctas, threads, 0, stream>>>(iters, sink);
  }
  return cudaGetLastError();
}

}  // namespace
}  // namespace gsample

extern "C" gsample_status gsample_debug_philox_alu_mix(int32_t warps_per_sm, uint32_t iters,
                                                       int32_t alu_steps, int32_t with_philox,
                                                       uint32_t* sink, gsample_stream_t stream) {
  if (warps_per_sm < 1 || warps_per_sm > 32 || iters < 1 || !sink || (uintptr_t)sink % 4 ||
      !(alu_steps == 0 || alu_steps == 2 || alu_steps == 4) ||
      !(with_philox == 0 || with_philox == 1) || (alu_steps == 0 && with_philox == 0))
    return GSAMPLE_ERR_INVALID_ARG;
  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return GSAMPLE_ERR_CUDA;
  }
  if (!(major == 10 && minor == 3)) return GSAMPLE_ERR_UNSUPPORTED;
  if (gsample::launch_probe(with_philox != 0, alu_steps, sms, warps_per_sm * 32, iters, sink,
                            (cudaStream_t)stream) != cudaSuccess) {
    cudaGetLastError();
    return GSAMPLE_ERR_CUDA;
  }
  return GSAMPLE_OK;
}
