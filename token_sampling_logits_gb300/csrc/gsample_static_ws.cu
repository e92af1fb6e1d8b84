// gsample_gumbel_argmax_static: Gumbel-max sampling with a library-owned,
// statically allocated workspace, for callers that cannot allocate device
// memory themselves (see include/gsample.h for who they are).
//
// The workspace is a file-scope __device__ array, so every GPU that loads this
// library holds it (GSAMPLE_STATIC_WS_MAX_ROWS * 16 bytes) until the process
// exits. In host code the array's name is only a host-side stand-in; its device
// address is fetched once per device with cudaGetSymbolAddress while that
// device is current, then passed to the regular entry point.
#include <cstdint>
#include <mutex>

#include "gsample.h"
#include "gsample_internal.h"

namespace {

static __device__ __align__(256) gsample::WsRow g_static_ws[GSAMPLE_STATIC_WS_MAX_ROWS];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ws_addr[kMaxDevices] = {};

// One-time per-device set-up (first call on each device): look up the
// array's device address and zero it. Returns nullptr on failure.
void* static_workspace_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_ws_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_ws) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return nullptr;
    }
    if (cudaMemset(ptr, 0, sizeof(g_static_ws)) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_ws_addr[dev] = ptr;
  }
  return g_ws_addr[dev];
}

}  // namespace

extern "C" gsample_status gsample_gumbel_argmax_static(
    const void* logits, gsample_dtype dtype, int64_t B, int64_t V, int64_t ld,
    const float* temperature, const uint64_t* seed, const uint64_t* offset, int64_t* out_idx,
    gsample_stream_t stream) {
  if (B < 0 || B > GSAMPLE_STATIC_WS_MAX_ROWS) return GSAMPLE_ERR_INVALID_ARG;
  if (B == 0) return GSAMPLE_OK;
  void* ws = static_workspace_for_current_device();
  if (ws == nullptr) return GSAMPLE_ERR_CUDA;
  // The rows this call uses start from zero even if an earlier launch on the
  // array never completed; a completed launch leaves them zero anyway.
  if (cudaMemsetAsync(ws, 0, (size_t)B * sizeof(gsample::WsRow), (cudaStream_t)stream) !=
      cudaSuccess) {
    cudaGetLastError();
    return GSAMPLE_ERR_CUDA;
  }
  return gsample_gumbel_argmax(logits, dtype, B, V, ld, temperature, seed, offset, out_idx, ws,
                               stream);
}
