// Internal interface between the host API (gsample_api.cu) and the kernel
// translation units. Not part of the public ABI.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "gsample.h"
#include "gsample_device.cuh"

namespace gsample {

// The launch attribute that pairs with pdl_wait_then_release() in every kernel.
inline cudaLaunchAttribute pdl_attribute() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}


// One launch of the row sampler. Rows are cut into 16-byte units (or 4-element
// units when a row does not start on a 16-byte boundary); the B * units_per_row
// units are split into `ctas` near-equal contiguous ranges, one per CTA.
struct SampleParams {
  const char* logits;
  int64_t ld_bytes;
  int64_t B;
  int32_t V;
  int32_t units_per_row;
  int64_t total_units;
  int32_t ctas;
  int64_t warps;  // warps that get a non-empty range: min(ctas * kWarps, total_units)
  const float* temperature;  // nullptr: every row greedy
  const uint64_t* seed;
  const uint64_t* offset;
  int64_t* out_idx;
  WsRow* ws;
};

// One row's curve; the same layout as the public gsample_hlg_params.
struct HlgRowParams {
  float m, w, beta_t, beta_h, pivot_offset;
  int32_t pivot_mode;
};
static_assert(sizeof(HlgRowParams) == 24, "per-row HLG parameters are six 4-byte fields");

// HLG launch: one thread-block cluster of `cluster` CTAs per row.
struct HlgParams {
  const char* logits;
  int64_t ld_bytes;
  int64_t B;
  int32_t V;
  int32_t units_per_row;
  int32_t cluster;
  int32_t units_per_cta;  // slice of the row held by each CTA of the cluster
  const float* temperature;
  const uint64_t* seed;
  const uint64_t* offset;
  int64_t* out_idx;
  WsRow* ws;
  float m, w, beta_t, beta_h, pivot_offset;
  int32_t pivot_mode;
  const HlgRowParams* rows;  // per-row curves (device), or nullptr: the fields above
};

// Launches with one thread-block cluster of `cluster` CTAs per row (the
// categorical baseline and the small-batch sampler).
struct RowClusterParams {
  const char* logits;
  int64_t ld_bytes;
  int64_t B;
  int32_t V;
  int32_t units_per_row;
  int32_t cluster;
  int32_t units_per_cta;
  const float* temperature;
  const uint64_t* seed;
  const uint64_t* offset;
  int64_t* out_idx;
};

// Top-k / top-p on the Gumbel path, after the plain sampler has written its
// proposals into out_idx: one thread-block cluster of `cluster` CTAs per row
// tests the proposal and, when it is rejected, replaces it by the Gumbel-max
// over the filter set.
struct FilterParams {
  const char* logits;
  int64_t ld_bytes;
  int64_t B;
  int32_t V;
  int32_t units_per_row;
  int32_t cluster;
  int32_t units_per_cta;
  float mass_scale;      // 2^E: fixed-point unit of the top_p masses (a row's sum fits in 63 bits)
  const float* temperature;
  const uint64_t* seed;
  const uint64_t* offset;
  const int32_t* top_k;  // nullptr: no top-k
  const float* top_p;    // nullptr: no top-p
  int64_t* out_idx;
};
// The filter kernel of (dtype, vec, resident) and its block size (occupancy
// queries), the largest cluster the device co-schedules for it, and the
// largest slice it holds in shared memory.
void* filter_kernel_fn(int dtype, bool vec, bool resident, int* threads);
int filter_max_cluster(int dtype, bool vec);
size_t filter_smem_limit();
cudaError_t launch_filter(const FilterParams& p, int dtype, bool vec, cudaStream_t stream);

// Elements per unit for a dtype code (0 f32, 1 bf16, 2 f16) and load path.
inline int units_elems(int dtype, bool vec) { return vec ? (dtype == 0 ? 4 : 8) : 4; }

// Occupancy-derived CTA slots per SM for the sampler kernel of (dtype, vec).
int sample_ctas_per_sm(int dtype, bool vec);
size_t sample_smem_bytes(int dtype, bool vec);
cudaError_t launch_sample(const SampleParams& p, int dtype, bool vec, cudaStream_t stream);

// HLG: the largest cluster size the device can co-schedule for this kernel and
// the shared memory a CTA needs to hold `units_per_cta` units.
int hlg_max_cluster(int dtype, bool vec, size_t smem_bytes);
size_t hlg_smem_bytes(int dtype, bool vec, int32_t units_per_cta);
size_t hlg_smem_limit();
cudaError_t launch_hlg(const HlgParams& p, int dtype, bool vec, cudaStream_t stream);

// The cluster-per-row kernels of (dtype, vec, resident) and their block size,
// for occupancy queries.
void* rc_kernel(int dtype, bool vec, bool resident, int* threads);
void* cat_kernel(int dtype, bool vec, bool resident, int* threads);
void* hlg_kernel_fn(int dtype, bool vec, bool resident, int* threads);

// Small-batch sampler (one cluster per row): largest co-schedulable cluster,
// per-CTA slice limit, launch.
int rc_max_cluster(int dtype, bool vec);
size_t rc_smem_limit();
cudaError_t launch_sample_cluster(const RowClusterParams& p, int dtype, bool vec,
                                  cudaStream_t stream);

// Categorical baseline: largest co-schedulable cluster, per-CTA slice limit.
int cat_max_cluster(int dtype, bool vec);
size_t cat_smem_limit();
cudaError_t launch_categorical(const RowClusterParams& p, int dtype, bool vec, cudaStream_t stream);

// The host-side checks of gsample_gumbel_argmax other than the workspace's
// (arguments, then the device), with nothing enqueued.
gsample_status validate_gumbel_args(const void* logits, gsample_dtype dtype, int64_t B,
                                    int64_t V, int64_t ld, const float* temperature,
                                    const uint64_t* seed, const uint64_t* offset,
                                    const int64_t* out_idx);

cudaError_t launch_debug_philox(uint64_t seed, uint32_t row, uint64_t offset, int64_t group0,
                                int64_t n, uint32_t* out, cudaStream_t stream);
cudaError_t launch_debug_word_test(const float* x, const uint32_t* w, int64_t n, float L, float T,
                                   uint32_t* threshold, uint8_t* flags, cudaStream_t stream);
cudaError_t launch_debug_philox_rate(int ctas, int threads, uint32_t iters, uint32_t* sink,
                                     cudaStream_t stream);
// Blocks counted by a GSAMPLE_COUNT_BLOCKS build; cudaErrorNotSupported otherwise.
cudaError_t read_blocks_computed(unsigned long long* out, bool reset);
cudaError_t launch_debug_hlg_score(const float* x, const uint32_t* words, int64_t n, float m,
                                   float w, float beta_t, float beta_h, float T, float shift,
                                   float* out, cudaStream_t stream);
cudaError_t launch_debug_gumbel(const uint32_t* words, int64_t n, float* g, float* bound,
                                cudaStream_t stream);

}  // namespace gsample
