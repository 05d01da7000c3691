/*
 * kd_topk_kl_testing.h — test hooks of libkdtopk. Not part of the loss API.
 *
 * They expose the pieces the loss is built from so that tests can check each
 * one on its own: the tcgen05 GEMM mainloop as a plain GEMM, the work
 * schedule as host arithmetic, and the bounded-wait error path.
 * Ownership, stream and error rules are those of kd_topk_kl.h.
 */
#ifndef KD_TOPK_KL_TESTING_H
#define KD_TOPK_KL_TESTING_H

#include "kd_topk_kl.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * C[m][n] = sum_k A(m,k) * B(n,k) in fp32 through the same persistent
 * tcgen05/TMA mainloop the loss kernels use (bf16 operands, fp32 accumulate).
 * a_mn = 0: A is [M x K] row-major (K contiguous); a_mn = 1: A is [K x M]
 * row-major (M contiguous). b_mn likewise for B ([N x K] or [K x N]).
 * C is [M x N] fp32 row-major. Device pointers, 16-byte aligned; M, N and K
 * must be multiples of 8.
 * cta_pair != 0 runs the CTA-pair form the loss uses (cta_group::2, 256-row
 * tiles); 0 runs the single-CTA form (128-row tiles).
 */
kd_status kd_debug_gemm_bf16(const uint16_t* A, const uint16_t* B, float* C, int M, int N, int K,
                             int a_mn, int b_mn, int cta_pair, kd_stream_t stream);

/*
 * Launches one block whose pipeline wait can never be satisfied (nothing
 * arrives on its barrier). The wait gives up after timeout_ns nanoseconds
 * (capped at 2 s), records KD_ERR_TIMEOUT in the status word and the kernel
 * returns normally. Read the result with kd_get_status.
 */
kd_status kd_debug_wait_timeout(uint64_t timeout_ns, kd_stream_t stream);

/*
 * Host-side description of the work schedule the library would use.
 * kind: 0 = forward / dZ recompute (rows x vocabulary tiles),
 *       1 = dH (tokens x hidden tiles, split over the vocabulary),
 *       2 = dW (vocabulary x hidden tiles).
 * rows, cols, depth: the GEMM's M, N (columns) and K extents; grid_units:
 * the number of persistent workers to plan for (SMs, or CTA pairs);
 * tile_rows: 128 (single CTA) or 256 (CTA pair). counts (optional, length
 * MB*NB*KBLOCKS, where MB = ceil(rows/tile_rows), NB = number of column
 * tiles, KBLOCKS = ceil(depth/64)) is incremented once per (m-tile, n-tile,
 * k-block) the schedule visits. info (length 8) receives {units, grid, MB,
 * NB, KBLOCKS, BN, max_slots, k_splits}. Returns KD_ERR_ARG for bad sizes.
 */
kd_status kd_debug_schedule(int kind, int64_t rows, int64_t cols, int64_t depth, int grid_units,
                            int tile_rows, int32_t* counts, int64_t* info);

/*
 * Per-kernel timing. enable != 0 starts recording a CUDA event pair on the
 * launching stream around every kernel the library launches (clearing earlier
 * records); enable = 0 stops. kd_debug_profile_read waits for the recorded
 * events and returns, per category, the summed milliseconds and the launch
 * count (arrays of length n; categories: 0 prep, 1 forward GEMM, 2 combine,
 * 3 dZ GEMM, 4 dH GEMM, 5 dH split sum, 6 dW GEMM, 7 loss from logits,
 * 8 teacher-logit GEMMs, 9 top-K selection and thresholds, 10 the backward's
 * transposes of H and the teacher cache's gather of W rows), then clears the
 * records.
 * Event objects are created on first use and kept for the process lifetime.
 */
kd_status kd_debug_profile(int enable);
kd_status kd_debug_profile_read(double* total_ms, int64_t* launches, int n);

#ifdef __cplusplus
}
#endif

#endif /* KD_TOPK_KL_TESTING_H */
