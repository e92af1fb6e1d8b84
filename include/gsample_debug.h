/*
 * gsample diagnostic entry points. They expose the building blocks the
 * sampling kernels use, so that tests can compare them one by one with an
 * independent implementation, and let a caller fix the launch shape.
 * Same conventions as gsample.h (device pointers, caller stream, no sync).
 */
#ifndef GSAMPLE_DEBUG_H_
#define GSAMPLE_DEBUG_H_

#include "gsample.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Raw Philox4x32-10 blocks of one row's stream (Salmon et al., SC'11):
 * out[4*j + w] = word w of the block with counter
 * (group0 + j, row, lo32(offset), hi32(offset)) under key (lo32(seed), hi32(seed)),
 * for j in [0, n_groups). out: device uint32[4 * n_groups]. */
gsample_status gsample_debug_philox(uint64_t seed, uint32_t row, uint64_t offset,
                                    int64_t group0, int64_t n_groups, uint32_t* out,
                                    gsample_stream_t stream);

/* The kernels' binary32 Gumbel transform of raw words, and the upper bound on it
 * that the exact pruning relies on: gumbel[j] = g(words[j]) and
 * bound[j] = -log(1 - u(words[j])), which is >= g(words[j]) in exact arithmetic.
 * words, gumbel, bound: device arrays of n entries; bound may be NULL. */
gsample_status gsample_debug_gumbel(const uint32_t* words, int64_t n, float* gumbel,
                                    float* bound, gsample_stream_t stream);

/* The two word tests of the sampled path's exact pruning, for a row whose best
 * known score is L at temperature T > 0 ("Softmax-free GPU sampling",
 * Background: an element can win only if x/T + g reaches L, and g is at most
 * -log(1 - u)). For each j:
 *   flags[j] bit 0: the element test, 1 - u(words[j]) <= 2^((x[j]/T - lm)*log2 e)
 *                   (x[j] >= the logit threshold when L is not finite);
 *   flags[j] bit 1: the group test the kernels run first, words[j] >= threshold[j];
 *   threshold[j]:   the integer word threshold computed from x[j] alone.
 * The group test must pass wherever the element test does. x, words: device
 * arrays of n entries; threshold (uint32) and flags (uint8): device outputs. */
gsample_status gsample_debug_word_test(const float* x, const uint32_t* words, int64_t n, float L,
                                       float T, uint32_t* threshold, uint8_t* flags,
                                       gsample_stream_t stream);

/* gsample_gumbel_argmax / gsample_hlg_gumbel_argmax with an explicit number
 * of CTAs (0 = the library's choice). ctas is clamped to [1, number of 16-byte
 * units in the batch]. hlg == NULL selects the plain sampler; a positive ctas
 * then always takes the flat split (sample_kernel), whatever the batch size. */
gsample_status gsample_debug_sample_ex(const void* logits, gsample_dtype dtype, int64_t B,
                                       int64_t V, int64_t ld, const float* temperature,
                                       const uint64_t* seed, const uint64_t* offset,
                                       const gsample_hlg_params* hlg, int64_t* out_idx,
                                       void* workspace, int32_t ctas,
                                       gsample_stream_t stream);

/* gsample_gumbel_argmax on the cluster-per-row kernel with `cluster` CTAs per
 * row (1..16), whatever the batch size (the library picks it for small
 * batches only). */
gsample_status gsample_debug_sample_cluster(const void* logits, gsample_dtype dtype, int64_t B,
                                            int64_t V, int64_t ld, const float* temperature,
                                            const uint64_t* seed, const uint64_t* offset,
                                            int64_t* out_idx, void* workspace, int32_t cluster,
                                            gsample_stream_t stream);

/* gsample_categorical with an explicit cluster size (CTAs per row, 1..16;
 * 0 = the library's choice). */
gsample_status gsample_debug_categorical_ex(const void* logits, gsample_dtype dtype, int64_t B,
                                            int64_t V, int64_t ld, const float* temperature,
                                            const uint64_t* seed, const uint64_t* offset,
                                            int64_t* out_idx, int32_t cluster,
                                            gsample_stream_t stream);

/* gsample_filtered_gumbel_argmax with an explicit cluster size for the
 * filter (CTAs per row, 1..16, at most what the device co-schedules;
 * 0 = the library's choice). A CTA whose slice exceeds the filter's shared
 * memory re-reads it from global memory in every phase. */
gsample_status gsample_debug_filtered_ex(const void* logits, gsample_dtype dtype, int64_t B,
                                         int64_t V, int64_t ld, const float* temperature,
                                         const uint64_t* seed, const uint64_t* offset,
                                         const int32_t* top_k, const float* top_p,
                                         int64_t* out_idx, void* workspace, int32_t cluster,
                                         gsample_stream_t stream);

/* Philox4x32-10 throughput of the kernels' block code alone (Salmon et al.,
 * SC'11; the row-folded first two rounds and four blocks per thread side by
 * side, as in the sampler). One CTA per SM of warps_per_sm warps (1..32); each
 * thread computes 4 * iters blocks and folds their words into sink[thread].
 * sink: device uint32[SMs * warps_per_sm * 32]. Time it on `stream` to get the
 * measured Philox rate the sampler's second roofline is reported against. */
gsample_status gsample_debug_philox_rate(int32_t warps_per_sm, uint32_t iters, uint32_t* sink,
                                         gsample_stream_t stream);

/* How ALU work adds to the Philox multiplies (a measurement probe, no page
 * counterpart): one CTA per SM of warps_per_sm warps (1..32); each thread runs
 * `iters` iterations of four blocks of the kernels' Philox block code (when
 * with_philox is 1) and/or 4 * alu_steps independent ALU updates per block
 * (alu_steps 0, 2 or 4; shifts and bitwise operations in four chains that do
 * not depend on the Philox words), folding everything into sink[thread].
 * sink: device uint32[SMs * warps_per_sm * 32]. Time the Philox-only,
 * ALU-only and mixed shapes on `stream`: the mixed time minus the Philox-only
 * time, over the ALU-only time, is the share of the ALU work that does not
 * hide behind the multiplies. GSAMPLE_ERR_INVALID_ARG for other values or
 * for alu_steps 0 without Philox. */
gsample_status gsample_debug_philox_alu_mix(int32_t warps_per_sm, uint32_t iters,
                                            int32_t alu_steps, int32_t with_philox,
                                            uint32_t* sink, gsample_stream_t stream);

/* Philox blocks the row sampler computed since the last reset (dense tiles,
 * compacted batches, first candidates and exact passes, summed over
 * launches), in a library built with -DGSAMPLE_COUNT_BLOCKS; reset != 0 sets
 * the count back to zero after reading it. The regular build returns
 * GSAMPLE_ERR_UNSUPPORTED. Synchronous (reads a device counter). */
gsample_status gsample_debug_blocks_computed(uint64_t* count, int32_t reset);

/* The HLG kernel's exact candidate score ("HLG sampling", "The transfer
 * function"): out[j] = tone(x[j] + shift) / T + g(words[j]) in binary32, the
 * tone curve of `hlg` (pivot fields unused), the shift standing for the row's
 * pivot (z = x + shift). x, words, out: device arrays of n entries; T > 0 and
 * shift finite, else GSAMPLE_ERR_INVALID_ARG. */
gsample_status gsample_debug_hlg_score(const float* x, const uint32_t* words, int64_t n,
                                       const gsample_hlg_params* hlg, float T, float shift,
                                       float* out, gsample_stream_t stream);

/* Number of CTAs the library would launch for this problem (0 on bad args). */
int32_t gsample_debug_planned_ctas(gsample_dtype dtype, int64_t B, int64_t V, int64_t ld,
                                   const void* logits, int32_t hlg);

#ifdef __cplusplus
}
#endif

#endif /* GSAMPLE_DEBUG_H_ */
