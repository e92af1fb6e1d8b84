// gsample_gumbel_argmax_static: Gumbel-max sampling with a library-owned,
// statically allocated workspace, for callers that cannot allocate device
// memory themselves (see include/gsample.h for who they are).
//
// The workspace is a file-scope __device__ array, so every GPU that loads this
// library holds it (GSAMPLE_STATIC_WS_MAX_ROWS * 16 bytes) until the process
// exits. In host code the array's name is only a host-side stand-in; its device
// address is fetched once per device with cudaGetSymbolAddress while that
// device is current, then passed to the regular entry point. Like every
// static __device__ variable it is zero when the module loads.
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
// array's device address. It is only a lookup: nothing is enqueued or
// synchronised, and the array needs no clearing, since it starts at zero and
// every call clears the rows it uses. A first call on a device while `stream`
// is being captured is refused (GSAMPLE_ERR_UNSUPPORTED), so that the lookup,
// which may load the library's device code, never runs inside a capture.
gsample_status static_workspace_for_current_device(cudaStream_t stream, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return GSAMPLE_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_ws_addr[dev] == nullptr) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
      cudaGetLastError();
      return GSAMPLE_ERR_CUDA;
    }
    if (cap != cudaStreamCaptureStatusNone) return GSAMPLE_ERR_UNSUPPORTED;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_ws) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return GSAMPLE_ERR_CUDA;
    }
    g_ws_addr[dev] = ptr;
  }
  *out = g_ws_addr[dev];
  return GSAMPLE_OK;
}

}  // namespace

extern "C" gsample_status gsample_gumbel_argmax_static(
    const void* logits, gsample_dtype dtype, int64_t B, int64_t V, int64_t ld,
    const float* temperature, const uint64_t* seed, const uint64_t* offset, int64_t* out_idx,
    gsample_stream_t stream) {
  if (B < 0 || B > GSAMPLE_STATIC_WS_MAX_ROWS) return GSAMPLE_ERR_INVALID_ARG;
  // Every argument check of the regular entry point runs before anything is
  // set up or enqueued.
  gsample_status st = gsample::validate_gumbel_args(logits, dtype, B, V, ld, temperature, seed,
                                                    offset, out_idx);
  if (st != GSAMPLE_OK || B == 0) return st;
  void* ws = nullptr;
  st = static_workspace_for_current_device((cudaStream_t)stream, &ws);
  if (st != GSAMPLE_OK) return st;
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
