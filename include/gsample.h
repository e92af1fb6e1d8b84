/*
 * gsample -- batch Gumbel-max token sampling on GB300 (sm_103a).
 *
 * One launch samples one token per row of a [B, V] logits matrix. For every
 * element it forms
 *
 *     score_i = logits[i] / T + g_i,     g_i = -log(-log u_i),
 *
 * and returns the index of the largest score of each row. That index is an
 * exact sample of softmax(logits / T), with no softmax and no sort
 * ("Softmax-free GPU sampling: Gumbel-max categorical sampling kernel",
 * lablup/mlxcel issue #900, sections Background and Task 1). The uniform u_i
 * comes from a stateless Philox4x32-10 stream (Salmon et al., "Parallel Random
 * Numbers: As Easy as 1, 2, 3", SC'11) keyed by the row's 64-bit seed, with
 * counter (i >> 2, row, offset_lo32, offset_hi32); element i takes output word
 * i & 3; u_i = ((word >> 9) + 0.5) * 2^-23. Equal scores go to the lowest index.
 *
 * Conventions shared by every entry point:
 *   - logits: device pointer to B rows of V elements (dtype below); row b starts
 *     at element b * ld (ld >= V). Any element alignment is accepted; rows that
 *     start on a 16-byte boundary use 128-bit loads.
 *   - out_idx: device int64[B], written with the sampled index of each row, or
 *     -1 for a row with no candidate (every logit -inf or NaN).
 *   - NaN logits are never drawn; a +inf logit scores +inf (so the lowest +inf
 *     index of a row wins); scores are formed in binary32.
 *   - temperature / seed / offset: device arrays of B entries. A row whose
 *     temperature is <= 0 or NaN is sampled greedily (plain argmax of the raw
 *     logits, lowest index on ties), as the issue's Task 3 keeps greedy on argmax.
 *   - workspace: device buffer of gsample_workspace_bytes(B) bytes, zeroed once
 *     (gsample_workspace_init or a memset) before first use. Every launch that
 *     completes leaves it zeroed again, so it needs no clearing between calls.
 *     Two launches that are in flight at the same time (different streams) must
 *     not share a workspace.
 *   - stream: a cudaStream_t (NULL = legacy default stream). Calls only enqueue
 *     work on it and never synchronise; GSAMPLE_OK means "launched". Kernels are
 *     launched with programmatic stream serialization: each may be scheduled
 *     while the previous kernel of the stream drains, waits for it to complete
 *     before touching memory, and lets the next kernel be scheduled early. A
 *     kernel that follows on the stream with that launch attribute must wait
 *     (griddepcontrol.wait / cudaGridDependencySynchronize) before reading the
 *     indices; one launched without it sees the usual stream order.
 *   - The caller owns every buffer; the library allocates nothing and keeps no
 *     global state apart from cached device attributes.
 *   - Errors: arguments are checked on the host before anything is launched and
 *     a bad argument returns GSAMPLE_ERR_INVALID_ARG with nothing enqueued.
 *     Device data (temperatures, logits) is never validated. A launch failure
 *     returns GSAMPLE_ERR_CUDA. GSAMPLE_ERR_UNSUPPORTED means the current device
 *     is not a compute-capability 10.3 GPU.
 */
#ifndef GSAMPLE_H_
#define GSAMPLE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* gsample_stream_t;

typedef enum {
  GSAMPLE_F32 = 0,  /* IEEE binary32 */
  GSAMPLE_BF16 = 1, /* bfloat16, widened to binary32 exactly */
  GSAMPLE_F16 = 2   /* IEEE binary16, widened to binary32 exactly */
} gsample_dtype;

typedef enum {
  GSAMPLE_OK = 0,
  GSAMPLE_ERR_INVALID_ARG = 1,
  GSAMPLE_ERR_UNSUPPORTED = 2,
  GSAMPLE_ERR_WORKSPACE = 3,
  GSAMPLE_ERR_CUDA = 4
} gsample_status;

/* HLG pivot modes ("HLG sampling -- a piecewise tone curve on the logits",
 * section "The pivot"). */
typedef enum {
  GSAMPLE_PIVOT_TOP = 0,    /* mu = l_max - pivot_offset */
  GSAMPLE_PIVOT_ENTROPY = 1 /* mu = sum_i p_i l_i (minus the entropy) */
} gsample_pivot_mode;

/* HLG tone-curve parameters, in nats ("HLG sampling", sections "The transfer
 * function" and "Knobs"). With z = l - mu (l = log-softmax of the row):
 *   z < -w  : -m*w - m*beta_t*ln(1 + (-z - w)/beta_t)   (toe)
 *   |z| <= w:  m*z                                      (linear mid)
 *   z > w   :  m*w + m*beta_h*ln(1 + (z - w)/beta_h)    (shoulder)
 * Requirements: m > 0 finite; w >= 0 (w = +inf turns the rolloff off);
 * beta_t, beta_h > 0 finite; pivot_offset finite (used by the top mode). */
typedef struct {
  float m;
  float w;
  float beta_t;
  float beta_h;
  float pivot_offset;
  int32_t pivot_mode; /* gsample_pivot_mode */
} gsample_hlg_params;

/* Bytes of workspace needed for B rows (16 bytes per row). */
size_t gsample_workspace_bytes(int64_t B);

/* Zero the first gsample_workspace_bytes(B) bytes of `workspace` on `stream`. */
gsample_status gsample_workspace_init(void* workspace, int64_t B, gsample_stream_t stream);

/* Greedy decoding: out_idx[b] = lowest index of the largest logit of row b
 * (NaN and -inf never chosen; -1 if none). The issue keeps temperature 0 on a
 * plain argmax ("Softmax-free GPU sampling", Background and Task 3); the HLG
 * page's section "Greedy is untouched" says the same of the tone curve. */
gsample_status gsample_argmax(const void* logits, gsample_dtype dtype, int64_t B, int64_t V,
                              int64_t ld, int64_t* out_idx, void* workspace,
                              gsample_stream_t stream);

/* Gumbel-max sampling of every row in one launch ("Softmax-free GPU sampling",
 * Task 1: per-row RNG (seed, offset), temperature, batch-wide grid).
 * temperature[b] <= 0 or NaN selects greedy argmax for row b. */
gsample_status gsample_gumbel_argmax(const void* logits, gsample_dtype dtype, int64_t B,
                                     int64_t V, int64_t ld, const float* temperature,
                                     const uint64_t* seed, const uint64_t* offset,
                                     int64_t* out_idx, void* workspace,
                                     gsample_stream_t stream);

/* Top-k / top-p sampling on the Gumbel path, the follow-up "Softmax-free GPU
 * sampling" (Background) names as rejection-based top-k/top-p. Per row b the
 * filter set K is the first r candidates (logits that are neither NaN nor
 * -inf) in the order (logit descending, index ascending), where r is the
 * smaller of
 *   - top_k[b], when top_k[b] >= 1 (else no limit), and
 *   - the smallest prefix whose softmax(x / T) mass reaches top_p[b] * (row
 *     mass), when top_p[b] < 1 (top_p[b] <= 0 keeps the first candidate only;
 *     top_p[b] >= 1 or NaN: no limit);
 * and out_idx[b] is the Gumbel-max over K with the same noise as
 * gsample_gumbel_argmax: argmax over i in K of x_i / T + g_i, lowest index on
 * ties. It is an exact draw of softmax(x / T) restricted to K.
 *   - Rejection: the unfiltered draw (gsample_gumbel_argmax) is a proposal; a
 *     second pass over each filtered row keeps it when it lies in K (it is
 *     then the argmax over K); rejected rows are resolved exactly by a radix
 *     select of K's last element and the Gumbel-max over K. Three launches on
 *     `stream`, no host synchronisation.
 *   - top_k and top_p are device arrays of B entries (int32, float); either
 *     may be NULL (that filter off for every row). Both NULL: the same as
 *     gsample_gumbel_argmax.
 *   - Rows with temperature <= 0 or NaN are greedy (K always holds the top
 *     element). A row with a +inf logit returns its lowest +inf index.
 *   - The nucleus masses are binary32 sums on the GPU: a row whose top_p lands
 *     within ~1e-5 of the row mass from a prefix boundary may take one element
 *     more or less than an exact computation would.
 *   - Workspace, layout, validation and asynchrony as gsample_gumbel_argmax; a
 *     misaligned top_k/top_p (4 bytes) returns GSAMPLE_ERR_INVALID_ARG. */
gsample_status gsample_filtered_gumbel_argmax(const void* logits, gsample_dtype dtype, int64_t B,
                                              int64_t V, int64_t ld, const float* temperature,
                                              const uint64_t* seed, const uint64_t* offset,
                                              const int32_t* top_k, const float* top_p,
                                              int64_t* out_idx, void* workspace,
                                              gsample_stream_t stream);

/* HLG tone curve on the row's log-probs, then Gumbel-max ("HLG sampling",
 * sections "The transfer function", "The pivot", "Temperature semantics"):
 *     score_i = g(l_i - mu) / T + g_i,
 * where l = log_softmax(logits) and mu is the pivot of `hlg->pivot_mode`.
 * Dividing the curve by T is the pages' folding of temperature into the gain.
 * Rows with temperature <= 0 or NaN are greedy on the raw logits (the curve is
 * monotone, so it cannot move the argmax). `hlg` is a host pointer read during
 * the call. */
gsample_status gsample_hlg_gumbel_argmax(const void* logits, gsample_dtype dtype, int64_t B,
                                         int64_t V, int64_t ld, const float* temperature,
                                         const uint64_t* seed, const uint64_t* offset,
                                         const gsample_hlg_params* hlg, int64_t* out_idx,
                                         void* workspace, gsample_stream_t stream);

/* gsample_hlg_gumbel_argmax with one curve per row ("HLG sampling", section
 * "Where it lands in the code": each batched row owns its sampler, so the
 * curve parameters batch per request). hlg_rows: DEVICE array of B
 * gsample_hlg_params (24 bytes each, 4-byte aligned), read by the kernel.
 * Device data cannot be checked at the call, so a row whose parameters fail
 * the checks of gsample_hlg_gumbel_argmax (finite m > 0, w >= 0 (may be
 * +inf), finite beta_t > 0 and beta_h > 0, finite pivot_offset, a known
 * pivot_mode) gets out_idx[b] = -1; rows with temperature <= 0 or NaN are
 * greedy whatever their curve. Everything else as gsample_hlg_gumbel_argmax. */
gsample_status gsample_hlg_gumbel_argmax_rows(const void* logits, gsample_dtype dtype, int64_t B,
                                              int64_t V, int64_t ld, const float* temperature,
                                              const uint64_t* seed, const uint64_t* offset,
                                              const gsample_hlg_params* hlg_rows,
                                              int64_t* out_idx, void* workspace,
                                              gsample_stream_t stream);

/* The categorical baseline the issue measures Gumbel-max against ("Softmax-free
 * GPU sampling", Background and Performance validation): a normalisation of
 * softmax(logits / T) and one inverse-CDF draw per row,
 *     out_idx[b] = smallest i with e_0 + ... + e_i > u * S,
 * e_i = exp((x_i - M) / T) (0 for -inf and NaN), M the largest finite logit,
 * S = sum e_i, u the uniform of element 0's Philox word of the row's
 * (seed, offset) stream (the same word gsample_gumbel_argmax gives element 0).
 * temperature <= 0 or NaN is greedy; a +inf logit takes all the mass (lowest
 * +inf index); -1 if the row has no candidate. The sums are binary32: the
 * index is the inverse CDF of a target within about 1e-6 of S of u * S (not
 * bit-exact against a double-precision CDF). Needs no workspace. Device
 * pointers, caller stream, asynchronous, host-side validation as above. */
gsample_status gsample_categorical(const void* logits, gsample_dtype dtype, int64_t B, int64_t V,
                                   int64_t ld, const float* temperature, const uint64_t* seed,
                                   const uint64_t* offset, int64_t* out_idx,
                                   gsample_stream_t stream);

/* Static, human-readable name of a status code. */
const char* gsample_status_string(gsample_status status);

/* Largest batch gsample_gumbel_argmax_static accepts. */
#define GSAMPLE_STATIC_WS_MAX_ROWS 4096

/* gsample_gumbel_argmax without a workspace argument: the merge state lives in
 * a fixed array inside the library (GSAMPLE_STATIC_WS_MAX_ROWS rows, 64 KiB),
 * so the call allocates no device memory. The source pages have no counterpart
 * to this entry point; it exists for callers that cannot allocate: code that
 * runs inside a host framework or engine plugin which owns all device memory
 * and forbids allocations while it executes, code with a device-memory budget
 * fixed at start-up, and decode loops where cudaMalloc/cudaFree would stall the
 * GPU with their implicit synchronisation.
 *   - The caller still passes the inputs and out_idx (same meaning as in
 *     gsample_gumbel_argmax); B > GSAMPLE_STATIC_WS_MAX_ROWS returns
 *     GSAMPLE_ERR_INVALID_ARG with nothing enqueued; B == 0 is a no-op.
 *   - Every other argument is checked as gsample_gumbel_argmax checks it, and
 *     a bad one returns that entry point's status with nothing enqueued.
 *   - The array is held by every GPU that loads the library until the process
 *     exits, and is zero when the library's device code loads. The first call
 *     on each device looks up its device address (cudaGetSymbolAddress) and
 *     keeps it for the life of the process: do not call this entry point again
 *     on a device after cudaDeviceReset. That first call must not be made while
 *     `stream` is being captured: it returns GSAMPLE_ERR_UNSUPPORTED, with
 *     nothing enqueued. A failed look-up returns GSAMPLE_ERR_CUDA.
 *   - Every call clears the rows it uses (an asynchronous memset on `stream`)
 *     before sampling, and calls no cudaMalloc, cudaFree or other allocating
 *     routine.
 *   - All calls on a device share the one array: calls whose work overlaps on
 *     the GPU (different streams, or host threads racing) race on it and may
 *     return wrong indices. Serialise them, for example on one stream. */
gsample_status gsample_gumbel_argmax_static(const void* logits, gsample_dtype dtype, int64_t B,
                                            int64_t V, int64_t ld, const float* temperature,
                                            const uint64_t* seed, const uint64_t* offset,
                                            int64_t* out_idx, gsample_stream_t stream);

/* gsample_gumbel_argmax on host-resident data, with no staging copy: logits,
 * temperature, seed, offset and out_idx are page-locked HOST buffers
 * (cudaHostAlloc / cudaMallocHost, or cudaHostRegister), which the kernel
 * reads and writes through their mapping into the current device. On a GB300
 * the loads cross the CPU-GPU link once per logit; no device copy of the
 * logits is made. workspace stays a DEVICE buffer.
 *   - Each of the five host pointers is looked up with cudaPointerGetAttributes.
 *     One that is not page-locked host memory mapped into the current device
 *     returns GSAMPLE_ERR_INVALID_ARG, a workspace that is not device memory
 *     GSAMPLE_ERR_WORKSPACE; nothing is enqueued in either case. Buffer sizes
 *     cannot be checked: the caller guarantees B rows of ld elements, and B
 *     entries of the per-row arrays.
 *   - Asynchronous on `stream`: out_idx holds the indices once `stream` has been
 *     synchronised, and the host must not write the inputs before then.
 *   - Shapes, ld, alignment, NaN/inf handling, greedy rows and the workspace
 *     contract are those of gsample_gumbel_argmax, and so are the indices.
 *   - Its rate is the link's (host-to-device reads measured about 0.21 TB/s on
 *     GB300, the same as cudaMemcpyAsync), not the kernel's. */
gsample_status gsample_gumbel_argmax_host(const void* logits, gsample_dtype dtype, int64_t B,
                                          int64_t V, int64_t ld, const float* temperature,
                                          const uint64_t* seed, const uint64_t* offset,
                                          int64_t* out_idx, void* workspace,
                                          gsample_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GSAMPLE_H_ */
