// Host side of the C ABI declared in include/gsample.h and include/gsample_debug.h:
// argument checks, launch planning and status mapping. Nothing here touches
// device data or synchronises; every entry point only enqueues on the caller's
// stream.
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "gsample.h"
#include "gsample_debug.h"
#include "gsample_internal.h"

namespace {

using gsample::SampleParams;
using gsample::HlgParams;
using gsample::RowClusterParams;
using gsample::WsRow;

// Largest V: element indices, Philox group indices and the packed key's low
// word all stay in 32 bits with room for a 16-byte unit past the end.
constexpr int64_t kMaxV = (int64_t(1) << 31) - 128;
constexpr int64_t kMaxB = INT32_MAX;
constexpr int kMaxDevices = 64;
constexpr int64_t kMinUnitsPerCta = gsample::kThreads;  // at least one unit per thread

struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int sms = 0;
  int sample_slots[6] = {0, 0, 0, 0, 0, 0};  // CTAs per SM, per (dtype, vec)
  int hlg_cluster[6] = {0, 0, 0, 0, 0, 0};   // largest co-schedulable cluster, per (dtype, vec)
  int cat_cluster[6] = {0, 0, 0, 0, 0, 0};   // the same for the categorical baseline
  int rc_cluster[6] = {0, 0, 0, 0, 0, 0};    // the same for the small-batch sampler
  int filt_cluster[6] = {0, 0, 0, 0, 0, 0};  // the same for the top-k / top-p filter
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

gsample_status device_info(const DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return GSAMPLE_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return GSAMPLE_ERR_CUDA;
    }
    d.supported = (major == 10 && minor == 3);
    d.sms = sms;
    if (d.supported) {
      for (int dt = 0; dt < 3; ++dt)
        for (int v = 0; v < 2; ++v) {
          const int n = gsample::sample_ctas_per_sm(dt, v != 0);
          if (n <= 0) {
            cudaGetLastError();
            return GSAMPLE_ERR_CUDA;
          }
          d.sample_slots[dt * 2 + v] = n;
          const int c = gsample::hlg_max_cluster(dt, v != 0, gsample::hlg_smem_limit());
          if (c <= 0) {
            cudaGetLastError();
            return GSAMPLE_ERR_CUDA;
          }
          d.hlg_cluster[dt * 2 + v] = c;
          const int cc = gsample::cat_max_cluster(dt, v != 0);
          if (cc <= 0) {
            cudaGetLastError();
            return GSAMPLE_ERR_CUDA;
          }
          d.cat_cluster[dt * 2 + v] = cc;
          const int rc = gsample::rc_max_cluster(dt, v != 0);
          if (rc <= 0) {
            cudaGetLastError();
            return GSAMPLE_ERR_CUDA;
          }
          d.rc_cluster[dt * 2 + v] = rc;
          const int fc = gsample::filter_max_cluster(dt, v != 0);
          if (fc <= 0) {
            cudaGetLastError();
            return GSAMPLE_ERR_CUDA;
          }
          d.filt_cluster[dt * 2 + v] = fc;
        }
    }
    d.ready = true;
  }
  *out = &d;
  return d.supported ? GSAMPLE_OK : GSAMPLE_ERR_UNSUPPORTED;
}

int64_t elt_bytes(gsample_dtype dt) { return dt == GSAMPLE_F32 ? 4 : 2; }

// How many clusters of `cluster` CTAs of `fn` (with `smem` bytes of dynamic
// shared memory each) the device runs at once; cached per device, kernel,
// cluster size and 16 KB step of shared memory.
int active_clusters(void* fn, int threads, int cluster, size_t smem) {
  static std::map<std::tuple<int, void*, int, size_t>, int> cache;
  const size_t bucket = (smem + 16383) / 16384;
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_tuple(dev, fn, cluster, bucket);
  {
    std::lock_guard<std::mutex> lock(g_mu);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cluster);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = bucket * 16384;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  cache[key] = n;
  return n;
}

// The cluster size for B rows of `nu` units: the largest size (at most
// max_cluster, and no more CTAs than nu / min_units) whose clusters all run in
// one wave; if none does, the one that runs the most rows at a time per CTA.
int pick_cluster(void* (*kernel)(int, bool, bool, int*), int dtype, bool vec, int64_t B,
                 int64_t nu, int max_cluster, int64_t min_units, size_t smem_limit) {
  int64_t cap = (nu + min_units - 1) / min_units;
  if (cap < 1) cap = 1;
  int top = max_cluster < 1 ? 1 : max_cluster;
  if (top > cap) top = (int)cap;
  int best = top;
  double best_rate = -1.0;
  for (int c = top; c >= 1; --c) {
    const size_t smem = (size_t)((nu + c - 1) / c) * 16;
    const bool resident = smem <= smem_limit;
    int threads = 0;
    void* fn = kernel(dtype, vec, resident, &threads);
    const int n = active_clusters(fn, threads, c, resident ? smem : 0);
    if (n <= 0) continue;
    if (B <= n) return c;  // one wave
    // rows finished per unit of time, if time per row scales with units per CTA
    const double rate = (double)n * c;
    if (rate > best_rate) {
      best_rate = rate;
      best = c;
    }
  }
  return best;
}

#ifndef GSAMPLE_FILT_SLICE_BYTES
#define GSAMPLE_FILT_SLICE_BYTES 40960
#endif

// The filter's cluster size for B rows of nu units: the smallest power of two
// (at most max_cluster) whose slices fit in GSAMPLE_FILT_SLICE_BYTES of shared
// memory, so that several CTAs share an SM; then doubled while the whole batch
// still runs in two waves of clusters and every CTA keeps a unit per thread
// (measured at V = 152K bf16: 16 CTAs per row at B = 64, 8 from B = 128).
int pick_filter_cluster(int dtype, bool vec, int64_t B, int64_t nu, int max_cluster) {
  const size_t limit = gsample::filter_smem_limit();
  int c = 1;
  while (c < max_cluster && (nu + c - 1) / c * 16 > GSAMPLE_FILT_SLICE_BYTES)
    c = 2 * c < max_cluster ? 2 * c : max_cluster;
  for (;;) {
    const int c2 = 2 * c < max_cluster ? 2 * c : max_cluster;
    if (c2 == c) break;
    const int64_t upc = (nu + c2 - 1) / c2;
    int threads = 0;
    const size_t smem = (size_t)upc * 16;
    const bool resident = smem <= limit;
    void* fn = gsample::filter_kernel_fn(dtype, vec, resident, &threads);
    if (upc < threads || B > 2 * (int64_t)active_clusters(fn, threads, c2, resident ? smem : 0))
      break;
    c = c2;
  }
  return c;
}

gsample_status check_common(const void* logits, gsample_dtype dtype, int64_t B, int64_t V,
                            int64_t ld, const int64_t* out_idx, const void* ws,
                            bool needs_ws = true) {
  if (dtype != GSAMPLE_F32 && dtype != GSAMPLE_BF16 && dtype != GSAMPLE_F16)
    return GSAMPLE_ERR_INVALID_ARG;
  if (B < 0 || B > kMaxB || V < 1 || V > kMaxV || ld < V) return GSAMPLE_ERR_INVALID_ARG;
  if (B == 0) return GSAMPLE_OK;
  if (!logits || !out_idx || (needs_ws && !ws)) return GSAMPLE_ERR_INVALID_ARG;
  const int64_t e = elt_bytes(dtype);
  if (ld > INT64_MAX / e / B) return GSAMPLE_ERR_INVALID_ARG;
  if ((uintptr_t)logits % (uintptr_t)e) return GSAMPLE_ERR_INVALID_ARG;
  if ((uintptr_t)out_idx % 8) return GSAMPLE_ERR_INVALID_ARG;
  if (needs_ws && (uintptr_t)ws % 16) return GSAMPLE_ERR_WORKSPACE;
  return GSAMPLE_OK;
}

bool vec_path(const void* logits, gsample_dtype dtype, int64_t ld) {
  return ((uintptr_t)logits % 16 == 0) && ((ld * elt_bytes(dtype)) % 16 == 0);
}

// Fill SampleParams and choose the CTA count: one wave of CTAs (SMs x resident
// CTAs per SM), fewer when the batch has too few units to give every thread one.
void plan_sample(const DeviceInfo& d, const void* logits, gsample_dtype dtype, int64_t B,
                 int64_t V, int64_t ld, int32_t ctas_override, SampleParams* p, bool* vec_out) {
  const bool vec = vec_path(logits, dtype, ld);
  const int epu = gsample::units_elems((int)dtype, vec);
  const int64_t nu = (V + epu - 1) / epu;
  const int64_t total = B * nu;
  int64_t g;
  if (ctas_override > 0) {
    g = ctas_override;
  } else {
    const int64_t slots = (int64_t)d.sms * d.sample_slots[(int)dtype * 2 + (vec ? 1 : 0)];
    g = (total + kMinUnitsPerCta - 1) / kMinUnitsPerCta;
    if (g > slots) g = slots;
  }
  if (g > total) g = total;
  if (g < 1) g = 1;
  std::memset(p, 0, sizeof *p);
  p->logits = static_cast<const char*>(logits);
  p->ld_bytes = ld * elt_bytes(dtype);
  p->B = B;
  p->V = (int32_t)V;
  p->units_per_row = (int32_t)nu;
  p->total_units = total;
  p->ctas = (int32_t)g;
  // A warp gets at least 8 units on the 128-bit path, so that its range still
  // holds units after the split points move to 128-byte lines.
  const int64_t max_warps = vec ? (total / 8 > 0 ? total / 8 : 1) : total;
  p->warps = g * gsample::kWarps < max_warps ? g * gsample::kWarps : max_warps;
  *vec_out = vec;
}

// Batches of at most this many rows take the cluster-per-row kernel; a CTA of
// it gets at least this many units.
constexpr int64_t kClusterMaxRows = 64;
constexpr int64_t kClusterUnitsPerCta = 512;

gsample_status run_sample(const void* logits, gsample_dtype dtype, int64_t B, int64_t V,
                          int64_t ld, const float* temperature, const uint64_t* seed,
                          const uint64_t* offset, int64_t* out_idx, void* workspace,
                          int32_t ctas_override, cudaStream_t stream,
                          int32_t cluster_override = 0) {
  gsample_status st = check_common(logits, dtype, B, V, ld, out_idx, workspace);
  if (st != GSAMPLE_OK || B == 0) return st;
  const DeviceInfo* d = nullptr;
  st = device_info(&d);
  if (st != GSAMPLE_OK) return st;
  if (ctas_override == 0 || cluster_override > 0) {
    // Small batches: one cluster per row (latency-bound sizes), unless a CTA
    // count for the flat split was asked for.
    const bool vec = vec_path(logits, dtype, ld);
    const int epu = gsample::units_elems((int)dtype, vec);
    const int64_t nu = (V + epu - 1) / epu;
    const int max_cluster = d->rc_cluster[(int)dtype * 2 + (vec ? 1 : 0)];
    int cluster = cluster_override;
    if (cluster == 0 && B <= kClusterMaxRows) {
      cluster = pick_cluster(gsample::rc_kernel, (int)dtype, vec, B, nu, max_cluster,
                             kClusterUnitsPerCta, gsample::rc_smem_limit());
      if ((nu + cluster - 1) / cluster * 16 > (int64_t)gsample::rc_smem_limit()) cluster = 0;
    }
    if (cluster > 0) {
      if (cluster > 16 || cluster > max_cluster) return GSAMPLE_ERR_INVALID_ARG;
      RowClusterParams q;
      std::memset(&q, 0, sizeof q);
      q.logits = static_cast<const char*>(logits);
      q.ld_bytes = ld * elt_bytes(dtype);
      q.B = B;
      q.V = (int32_t)V;
      q.units_per_row = (int32_t)nu;
      q.cluster = cluster;
      q.units_per_cta = (int32_t)((nu + cluster - 1) / cluster);
      q.temperature = temperature;
      q.seed = seed;
      q.offset = offset;
      q.out_idx = out_idx;
      if (gsample::launch_sample_cluster(q, (int)dtype, vec, stream) != cudaSuccess) {
        cudaGetLastError();
        return GSAMPLE_ERR_CUDA;
      }
      return GSAMPLE_OK;
    }
  }
  SampleParams p;
  bool vec = false;
  plan_sample(*d, logits, dtype, B, V, ld, ctas_override, &p, &vec);
  p.temperature = temperature;
  p.seed = seed;
  p.offset = offset;
  p.out_idx = out_idx;
  p.ws = static_cast<WsRow*>(workspace);
  const cudaError_t err = gsample::launch_sample(p, (int)dtype, vec, stream);
  if (err != cudaSuccess) {
    cudaGetLastError();
    return GSAMPLE_ERR_CUDA;
  }
  return GSAMPLE_OK;
}

// The device address of a page-locked host buffer (cudaHostAlloc,
// cudaMallocHost or cudaHostRegister) on the current device, or null when `p`
// is not one.
const void* mapped_view(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

bool is_device_memory(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice;
}

gsample_status run_categorical(const void* logits, gsample_dtype dtype, int64_t B, int64_t V,
                               int64_t ld, const float* temperature, const uint64_t* seed,
                               const uint64_t* offset, int64_t* out_idx, int32_t cluster_override,
                               cudaStream_t stream) {
  gsample_status st = check_common(logits, dtype, B, V, ld, out_idx, nullptr, false);
  if (st != GSAMPLE_OK) return st;
  if (!temperature || !seed || !offset) return GSAMPLE_ERR_INVALID_ARG;
  if (B == 0) return GSAMPLE_OK;
  const DeviceInfo* d = nullptr;
  st = device_info(&d);
  if (st != GSAMPLE_OK) return st;
  const bool vec = vec_path(logits, dtype, ld);
  const int epu = gsample::units_elems((int)dtype, vec);
  const int64_t nu = (V + epu - 1) / epu;
  const int max_cluster = d->cat_cluster[(int)dtype * 2 + (vec ? 1 : 0)];
  int cluster = cluster_override;
  if (cluster == 0)
    cluster = pick_cluster(gsample::cat_kernel, (int)dtype, vec, B, nu, max_cluster,
                           gsample::kThreads, gsample::cat_smem_limit());
  if (cluster < 1 || cluster > 16 || cluster > max_cluster) return GSAMPLE_ERR_INVALID_ARG;
  RowClusterParams p;
  std::memset(&p, 0, sizeof p);
  p.logits = static_cast<const char*>(logits);
  p.ld_bytes = ld * elt_bytes(dtype);
  p.B = B;
  p.V = (int32_t)V;
  p.units_per_row = (int32_t)nu;
  p.cluster = cluster;
  p.units_per_cta = (int32_t)((nu + cluster - 1) / cluster);
  p.temperature = temperature;
  p.seed = seed;
  p.offset = offset;
  p.out_idx = out_idx;
  if (gsample::launch_categorical(p, (int)dtype, vec, stream) != cudaSuccess) {
    cudaGetLastError();
    return GSAMPLE_ERR_CUDA;
  }
  return GSAMPLE_OK;
}

gsample_status check_hlg(const gsample_hlg_params* h) {
  if (!h) return GSAMPLE_ERR_INVALID_ARG;
  const bool ok = std::isfinite(h->m) && h->m > 0.0f && h->w >= 0.0f && !std::isnan(h->w) &&
                  std::isfinite(h->beta_t) && h->beta_t > 0.0f && std::isfinite(h->beta_h) &&
                  h->beta_h > 0.0f && std::isfinite(h->pivot_offset) &&
                  (h->pivot_mode == GSAMPLE_PIVOT_TOP || h->pivot_mode == GSAMPLE_PIVOT_ENTROPY);
  return ok ? GSAMPLE_OK : GSAMPLE_ERR_INVALID_ARG;
}

gsample_status run_hlg(const void* logits, gsample_dtype dtype, int64_t B, int64_t V, int64_t ld,
                       const float* temperature, const uint64_t* seed, const uint64_t* offset,
                       const gsample_hlg_params* hlg, const gsample_hlg_params* hlg_rows,
                       int64_t* out_idx, void* workspace, int32_t ctas_override,
                       cudaStream_t stream) {
  gsample_status st = check_common(logits, dtype, B, V, ld, out_idx, workspace);
  if (st != GSAMPLE_OK) return st;
  if (hlg_rows) {
    if ((uintptr_t)hlg_rows % 4) return GSAMPLE_ERR_INVALID_ARG;
  } else if (check_hlg(hlg) != GSAMPLE_OK) {
    return GSAMPLE_ERR_INVALID_ARG;
  }
  if (!temperature || !seed || !offset) return GSAMPLE_ERR_INVALID_ARG;
  if (B == 0) return GSAMPLE_OK;
  const DeviceInfo* d = nullptr;
  st = device_info(&d);
  if (st != GSAMPLE_OK) return st;

  const bool vec = vec_path(logits, dtype, ld);
  const int epu = gsample::units_elems((int)dtype, vec);
  const int64_t nu = (V + epu - 1) / epu;
  // Smallest cluster whose CTAs can each hold their slice of the row on chip;
  // if even the largest cluster cannot, the slices stream from memory twice.
  int cluster = ctas_override > 0 ? ctas_override : 0;
  if (cluster == 0)
    cluster = pick_cluster(gsample::hlg_kernel_fn, (int)dtype, vec, B, nu,
                           d->hlg_cluster[(int)dtype * 2 + (vec ? 1 : 0)], gsample::kThreads,
                           gsample::hlg_smem_limit());
  if (cluster > 16 || cluster > d->hlg_cluster[(int)dtype * 2 + (vec ? 1 : 0)])
    return GSAMPLE_ERR_INVALID_ARG;
  HlgParams p;
  std::memset(&p, 0, sizeof p);
  p.logits = static_cast<const char*>(logits);
  p.ld_bytes = ld * elt_bytes(dtype);
  p.B = B;
  p.V = (int32_t)V;
  p.units_per_row = (int32_t)nu;
  p.cluster = cluster;
  p.units_per_cta = (int32_t)((nu + cluster - 1) / cluster);
  p.temperature = temperature;
  p.seed = seed;
  p.offset = offset;
  p.out_idx = out_idx;
  p.ws = static_cast<WsRow*>(workspace);
  if (hlg_rows) {
    static_assert(sizeof(gsample_hlg_params) == sizeof(gsample::HlgRowParams),
                  "the public and internal per-row layouts must agree");
    p.rows = reinterpret_cast<const gsample::HlgRowParams*>(hlg_rows);
  } else {
    p.m = hlg->m;
    p.w = hlg->w;
    p.beta_t = hlg->beta_t;
    p.beta_h = hlg->beta_h;
    p.pivot_offset = hlg->pivot_offset;
    p.pivot_mode = hlg->pivot_mode;
  }
  const cudaError_t err = gsample::launch_hlg(p, (int)dtype, vec, stream);
  if (err != cudaSuccess) {
    cudaGetLastError();
    return GSAMPLE_ERR_CUDA;
  }
  return GSAMPLE_OK;
}

// The proposals (the plain sampler over every row), then the filter: one
// cluster per row tests each proposal and resolves the rejected ones.
gsample_status run_filtered(const void* logits, gsample_dtype dtype, int64_t B, int64_t V,
                            int64_t ld, const float* temperature, const uint64_t* seed,
                            const uint64_t* offset, const int32_t* top_k, const float* top_p,
                            int64_t* out_idx, void* workspace, int32_t cluster_override,
                            cudaStream_t stream) {
  if (B > 0 && (!temperature || !seed || !offset)) return GSAMPLE_ERR_INVALID_ARG;
  if ((uintptr_t)top_k % 4 || (uintptr_t)top_p % 4) return GSAMPLE_ERR_INVALID_ARG;
  if (cluster_override < 0 || cluster_override > 16) return GSAMPLE_ERR_INVALID_ARG;
  gsample_status st = check_common(logits, dtype, B, V, ld, out_idx, workspace);
  if (st != GSAMPLE_OK || B == 0) return st;
  const DeviceInfo* d = nullptr;
  st = device_info(&d);
  if (st != GSAMPLE_OK) return st;
  const bool vec = vec_path(logits, dtype, ld);
  const int epu = gsample::units_elems((int)dtype, vec);
  const int64_t nu = (V + epu - 1) / epu;
  const int max_cluster = d->filt_cluster[(int)dtype * 2 + (vec ? 1 : 0)];
  if (cluster_override > max_cluster) return GSAMPLE_ERR_INVALID_ARG;
  if (B * (cluster_override > 0 ? cluster_override : max_cluster) > (int64_t)INT32_MAX)
    return GSAMPLE_ERR_INVALID_ARG;  // grid size
  st = run_sample(logits, dtype, B, V, ld, temperature, seed, offset, out_idx, workspace, 0,
                  stream);
  if (st != GSAMPLE_OK || (!top_k && !top_p)) return st;
  gsample::FilterParams fp;
  fp.logits = static_cast<const char*>(logits);
  fp.ld_bytes = ld * elt_bytes(dtype);
  fp.B = B;
  fp.V = (int32_t)V;
  fp.units_per_row = (int32_t)nu;
  fp.cluster = cluster_override > 0 ? cluster_override
                                    : pick_filter_cluster((int)dtype, vec, B, nu, max_cluster);
  fp.units_per_cta = (int32_t)((nu + fp.cluster - 1) / fp.cluster);
  // 2^E with a row's V masses of at most 2^E each below 2^63: E = 40 up to
  // V = 2^22, one less per doubling above.
  int lg = 0;
  while ((int64_t(1) << lg) < V) ++lg;
  fp.mass_scale = std::ldexp(1.0f, lg <= 22 ? 40 : 62 - lg);
  fp.temperature = temperature;
  fp.seed = seed;
  fp.offset = offset;
  fp.top_k = top_k;
  fp.top_p = top_p;
  fp.out_idx = out_idx;
  if (gsample::launch_filter(fp, (int)dtype, vec, stream) != cudaSuccess) {
    cudaGetLastError();
    return GSAMPLE_ERR_CUDA;
  }
  return GSAMPLE_OK;
}

}  // namespace

namespace gsample {

// Every host-side check gsample_gumbel_argmax makes before it enqueues
// anything, except the workspace's (the static-workspace entry point owns
// its own): arguments, then the device.
gsample_status validate_gumbel_args(const void* logits, gsample_dtype dtype, int64_t B,
                                    int64_t V, int64_t ld, const float* temperature,
                                    const uint64_t* seed, const uint64_t* offset,
                                    const int64_t* out_idx) {
  gsample_status st = check_common(logits, dtype, B, V, ld, out_idx, nullptr, false);
  if (st != GSAMPLE_OK || B == 0) return st;
  if (!temperature || !seed || !offset) return GSAMPLE_ERR_INVALID_ARG;
  const DeviceInfo* d = nullptr;
  return device_info(&d);
}

}  // namespace gsample

extern "C" {

size_t gsample_workspace_bytes(int64_t B) {
  return B > 0 ? (size_t)B * sizeof(WsRow) : 0;
}

gsample_status gsample_workspace_init(void* workspace, int64_t B, gsample_stream_t stream) {
  if (B < 0 || B > kMaxB) return GSAMPLE_ERR_INVALID_ARG;
  if (B == 0) return GSAMPLE_OK;
  if (!workspace) return GSAMPLE_ERR_INVALID_ARG;
  if ((uintptr_t)workspace % 16) return GSAMPLE_ERR_WORKSPACE;
  if (cudaMemsetAsync(workspace, 0, gsample_workspace_bytes(B), (cudaStream_t)stream) !=
      cudaSuccess) {
    cudaGetLastError();
    return GSAMPLE_ERR_CUDA;
  }
  return GSAMPLE_OK;
}

gsample_status gsample_argmax(const void* logits, gsample_dtype dtype, int64_t B, int64_t V,
                              int64_t ld, int64_t* out_idx, void* workspace,
                              gsample_stream_t stream) {
  return run_sample(logits, dtype, B, V, ld, nullptr, nullptr, nullptr, out_idx, workspace, 0,
                    (cudaStream_t)stream);
}

gsample_status gsample_gumbel_argmax(const void* logits, gsample_dtype dtype, int64_t B,
                                     int64_t V, int64_t ld, const float* temperature,
                                     const uint64_t* seed, const uint64_t* offset,
                                     int64_t* out_idx, void* workspace,
                                     gsample_stream_t stream) {
  if (B > 0 && (!temperature || !seed || !offset)) return GSAMPLE_ERR_INVALID_ARG;
  return run_sample(logits, dtype, B, V, ld, temperature, seed, offset, out_idx, workspace, 0,
                    (cudaStream_t)stream);
}

gsample_status gsample_filtered_gumbel_argmax(const void* logits, gsample_dtype dtype, int64_t B,
                                              int64_t V, int64_t ld, const float* temperature,
                                              const uint64_t* seed, const uint64_t* offset,
                                              const int32_t* top_k, const float* top_p,
                                              int64_t* out_idx, void* workspace,
                                              gsample_stream_t stream) {
  return run_filtered(logits, dtype, B, V, ld, temperature, seed, offset, top_k, top_p, out_idx,
                      workspace, 0, (cudaStream_t)stream);
}

gsample_status gsample_gumbel_argmax_host(const void* logits, gsample_dtype dtype, int64_t B,
                                          int64_t V, int64_t ld, const float* temperature,
                                          const uint64_t* seed, const uint64_t* offset,
                                          int64_t* out_idx, void* workspace,
                                          gsample_stream_t stream) {
  gsample_status st = check_common(logits, dtype, B, V, ld, out_idx, workspace);
  if (st != GSAMPLE_OK || B == 0) return st;
  if (!temperature || !seed || !offset) return GSAMPLE_ERR_INVALID_ARG;
  const DeviceInfo* d = nullptr;
  st = device_info(&d);
  if (st != GSAMPLE_OK) return st;
  const void* x = mapped_view(logits);
  const void* t = mapped_view(temperature);
  const void* s = mapped_view(seed);
  const void* o = mapped_view(offset);
  const void* out = mapped_view(out_idx);
  if (!x || !t || !s || !o || !out) return GSAMPLE_ERR_INVALID_ARG;
  if (!is_device_memory(workspace)) return GSAMPLE_ERR_WORKSPACE;
  return run_sample(x, dtype, B, V, ld, static_cast<const float*>(t),
                    static_cast<const uint64_t*>(s), static_cast<const uint64_t*>(o),
                    static_cast<int64_t*>(const_cast<void*>(out)), workspace, 0,
                    (cudaStream_t)stream);
}

gsample_status gsample_hlg_gumbel_argmax(const void* logits, gsample_dtype dtype, int64_t B,
                                         int64_t V, int64_t ld, const float* temperature,
                                         const uint64_t* seed, const uint64_t* offset,
                                         const gsample_hlg_params* hlg, int64_t* out_idx,
                                         void* workspace, gsample_stream_t stream) {
  return run_hlg(logits, dtype, B, V, ld, temperature, seed, offset, hlg, nullptr, out_idx,
                 workspace, 0, (cudaStream_t)stream);
}

gsample_status gsample_categorical(const void* logits, gsample_dtype dtype, int64_t B, int64_t V,
                                   int64_t ld, const float* temperature, const uint64_t* seed,
                                   const uint64_t* offset, int64_t* out_idx,
                                   gsample_stream_t stream) {
  return run_categorical(logits, dtype, B, V, ld, temperature, seed, offset, out_idx, 0,
                         (cudaStream_t)stream);
}

gsample_status gsample_hlg_gumbel_argmax_rows(const void* logits, gsample_dtype dtype, int64_t B,
                                              int64_t V, int64_t ld, const float* temperature,
                                              const uint64_t* seed, const uint64_t* offset,
                                              const gsample_hlg_params* hlg_rows,
                                              int64_t* out_idx, void* workspace,
                                              gsample_stream_t stream) {
  if (B == 0) return check_common(logits, dtype, B, V, ld, out_idx, workspace);
  if (!hlg_rows) return GSAMPLE_ERR_INVALID_ARG;
  return run_hlg(logits, dtype, B, V, ld, temperature, seed, offset, nullptr, hlg_rows, out_idx,
                 workspace, 0, (cudaStream_t)stream);
}

const char* gsample_status_string(gsample_status status) {
  switch (status) {
    case GSAMPLE_OK: return "GSAMPLE_OK";
    case GSAMPLE_ERR_INVALID_ARG: return "GSAMPLE_ERR_INVALID_ARG: invalid argument";
    case GSAMPLE_ERR_UNSUPPORTED: return "GSAMPLE_ERR_UNSUPPORTED: device is not compute capability 10.3";
    case GSAMPLE_ERR_WORKSPACE: return "GSAMPLE_ERR_WORKSPACE: workspace missing or misaligned";
    case GSAMPLE_ERR_CUDA: return "GSAMPLE_ERR_CUDA: CUDA runtime error";
  }
  return "GSAMPLE_ERR_UNKNOWN";
}

gsample_status gsample_debug_philox(uint64_t seed, uint32_t row, uint64_t offset, int64_t group0,
                                    int64_t n_groups, uint32_t* out, gsample_stream_t stream) {
  if (n_groups < 0 || group0 < 0 || !out || (uintptr_t)out % 16) return GSAMPLE_ERR_INVALID_ARG;
  if (n_groups == 0) return GSAMPLE_OK;
  const DeviceInfo* d = nullptr;
  const gsample_status st = device_info(&d);
  if (st != GSAMPLE_OK) return st;
  if (gsample::launch_debug_philox(seed, row, offset, group0, n_groups, out,
                                   (cudaStream_t)stream) != cudaSuccess) {
    cudaGetLastError();
    return GSAMPLE_ERR_CUDA;
  }
  return GSAMPLE_OK;
}

gsample_status gsample_debug_philox_rate(int32_t warps_per_sm, uint32_t iters, uint32_t* sink,
                                         gsample_stream_t stream) {
  if (warps_per_sm < 1 || warps_per_sm > 32 || iters < 1 || !sink || (uintptr_t)sink % 4)
    return GSAMPLE_ERR_INVALID_ARG;
  const DeviceInfo* d = nullptr;
  const gsample_status st = device_info(&d);
  if (st != GSAMPLE_OK) return st;
  if (gsample::launch_debug_philox_rate(d->sms, warps_per_sm * 32, iters, sink,
                                        (cudaStream_t)stream) != cudaSuccess) {
    cudaGetLastError();
    return GSAMPLE_ERR_CUDA;
  }
  return GSAMPLE_OK;
}

gsample_status gsample_debug_hlg_score(const float* x, const uint32_t* words, int64_t n,
                                       const gsample_hlg_params* hlg, float T, float shift,
                                       float* out, gsample_stream_t stream) {
  if (n < 0 || !(T > 0.0f) || !isfinite(shift)) return GSAMPLE_ERR_INVALID_ARG;
  if (check_hlg(hlg) != GSAMPLE_OK) return GSAMPLE_ERR_INVALID_ARG;
  if (n == 0) return GSAMPLE_OK;
  if (!x || !words || !out) return GSAMPLE_ERR_INVALID_ARG;
  const DeviceInfo* d = nullptr;
  const gsample_status st = device_info(&d);
  if (st != GSAMPLE_OK) return st;
  if (gsample::launch_debug_hlg_score(x, words, n, hlg->m, hlg->w, hlg->beta_t, hlg->beta_h, T,
                                      shift, out, (cudaStream_t)stream) != cudaSuccess) {
    cudaGetLastError();
    return GSAMPLE_ERR_CUDA;
  }
  return GSAMPLE_OK;
}

gsample_status gsample_debug_blocks_computed(uint64_t* count, int32_t reset) {
  if (!count) return GSAMPLE_ERR_INVALID_ARG;
  unsigned long long v = 0;
  const cudaError_t e = gsample::read_blocks_computed(&v, reset != 0);
  if (e == cudaErrorNotSupported) return GSAMPLE_ERR_UNSUPPORTED;
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GSAMPLE_ERR_CUDA;
  }
  *count = v;
  return GSAMPLE_OK;
}

gsample_status gsample_debug_gumbel(const uint32_t* words, int64_t n, float* gumbel, float* bound,
                                    gsample_stream_t stream) {
  if (n < 0 || !words || !gumbel) return GSAMPLE_ERR_INVALID_ARG;
  if (n == 0) return GSAMPLE_OK;
  const DeviceInfo* d = nullptr;
  const gsample_status st = device_info(&d);
  if (st != GSAMPLE_OK) return st;
  if (gsample::launch_debug_gumbel(words, n, gumbel, bound, (cudaStream_t)stream) != cudaSuccess) {
    cudaGetLastError();
    return GSAMPLE_ERR_CUDA;
  }
  return GSAMPLE_OK;
}

gsample_status gsample_debug_word_test(const float* x, const uint32_t* words, int64_t n, float L,
                                       float T, uint32_t* threshold, uint8_t* flags,
                                       gsample_stream_t stream) {
  if (n < 0 || !(T > 0.0f)) return GSAMPLE_ERR_INVALID_ARG;
  if (n == 0) return GSAMPLE_OK;
  if (!x || !words || !threshold || !flags) return GSAMPLE_ERR_INVALID_ARG;
  const DeviceInfo* d = nullptr;
  const gsample_status st = device_info(&d);
  if (st != GSAMPLE_OK) return st;
  if (gsample::launch_debug_word_test(x, words, n, L, T, threshold, flags, (cudaStream_t)stream) !=
      cudaSuccess) {
    cudaGetLastError();
    return GSAMPLE_ERR_CUDA;
  }
  return GSAMPLE_OK;
}

gsample_status gsample_debug_sample_ex(const void* logits, gsample_dtype dtype, int64_t B,
                                       int64_t V, int64_t ld, const float* temperature,
                                       const uint64_t* seed, const uint64_t* offset,
                                       const gsample_hlg_params* hlg, int64_t* out_idx,
                                       void* workspace, int32_t ctas, gsample_stream_t stream) {
  if (ctas < 0) return GSAMPLE_ERR_INVALID_ARG;
  if (hlg)
    return run_hlg(logits, dtype, B, V, ld, temperature, seed, offset, hlg, nullptr, out_idx,
                   workspace, ctas, (cudaStream_t)stream);
  if (B > 0 && (!temperature || !seed || !offset)) return GSAMPLE_ERR_INVALID_ARG;
  return run_sample(logits, dtype, B, V, ld, temperature, seed, offset, out_idx, workspace, ctas,
                    (cudaStream_t)stream);
}

gsample_status gsample_debug_sample_cluster(const void* logits, gsample_dtype dtype, int64_t B,
                                            int64_t V, int64_t ld, const float* temperature,
                                            const uint64_t* seed, const uint64_t* offset,
                                            int64_t* out_idx, void* workspace, int32_t cluster,
                                            gsample_stream_t stream) {
  if (cluster < 1) return GSAMPLE_ERR_INVALID_ARG;
  if (B > 0 && (!temperature || !seed || !offset)) return GSAMPLE_ERR_INVALID_ARG;
  return run_sample(logits, dtype, B, V, ld, temperature, seed, offset, out_idx, workspace, 0,
                    (cudaStream_t)stream, cluster);
}

gsample_status gsample_debug_categorical_ex(const void* logits, gsample_dtype dtype, int64_t B,
                                            int64_t V, int64_t ld, const float* temperature,
                                            const uint64_t* seed, const uint64_t* offset,
                                            int64_t* out_idx, int32_t cluster,
                                            gsample_stream_t stream) {
  if (cluster < 0) return GSAMPLE_ERR_INVALID_ARG;
  return run_categorical(logits, dtype, B, V, ld, temperature, seed, offset, out_idx, cluster,
                         (cudaStream_t)stream);
}

gsample_status gsample_debug_filtered_ex(const void* logits, gsample_dtype dtype, int64_t B,
                                         int64_t V, int64_t ld, const float* temperature,
                                         const uint64_t* seed, const uint64_t* offset,
                                         const int32_t* top_k, const float* top_p,
                                         int64_t* out_idx, void* workspace, int32_t cluster,
                                         gsample_stream_t stream) {
  return run_filtered(logits, dtype, B, V, ld, temperature, seed, offset, top_k, top_p, out_idx,
                      workspace, cluster, (cudaStream_t)stream);
}

int32_t gsample_debug_planned_ctas(gsample_dtype dtype, int64_t B, int64_t V, int64_t ld,
                                   const void* logits, int32_t hlg) {
  if (check_common(logits ? logits : (const void*)16, dtype, B, V, ld, (const int64_t*)16,
                   (const void*)16) != GSAMPLE_OK || B == 0 || hlg)
    return 0;
  const DeviceInfo* d = nullptr;
  if (device_info(&d) != GSAMPLE_OK) return 0;
  SampleParams p;
  bool vec = false;
  plan_sample(*d, logits ? logits : (const void*)16, dtype, B, V, ld, 0, &p, &vec);
  return p.ctas;
}

}  // extern "C"
