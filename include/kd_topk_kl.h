/*
 * kd_topk_kl.h — C ABI of the fused top-K KL distillation head (B300, sm_103a).
 *
 * What it computes (Efficient Knowledge Distillation for LLMs: Offline Top-K
 * Logits and a Fused Chunked KL Loss — abstract, and the blog post "Making
 * Knowledge Distillation Cheap Enough to Run at Scale", section "Two systems
 * changes"): the student's output projection Z = H W^T is fused into the
 * KL-divergence loss against a cached teacher top-K, so that no tokens x
 * vocabulary tensor is ever written to memory. The forward projects the
 * hidden states tile by tile and folds each tile into a running logsumexp and
 * a gather of the logits at the teacher's cached ids; the backward recomputes
 * each chunk of logits instead of storing them.
 *
 * Per counted row n (mask[n] = 1), with temperature T > 0:
 *   q    = softmax(Z[n] / T) over all V tokens            (student)
 *   P    = softmax(t[n] / T) placed at idx[n], 0 elsewhere (teacher grid;
 *          a repeated id gets the sum of its entries)
 *   loss = sum_j P_j (log P_j - log q_j)
 *   lse  = logsumexp(Z[n] / T)                             (natural log)
 * A masked row gets loss 0 and zero gradient, and its idx/t are never read.
 * The mean loss is sum(loss) / n_valid, formed by the caller.
 *
 * Conventions shared by every call:
 *   - All pointers are DEVICE pointers owned by the caller, into memory of the
 *     CURRENT device (cudaSetDevice) or managed memory; anything else (host
 *     memory, another device's memory) is refused with KD_ERR_ARG before any
 *     launch. The library never allocates, frees or synchronises
 *     (kd_get_status is the one exception: it synchronises the given stream).
 *   - Every compute call is asynchronous on `stream` (a cudaStream_t; 0 is the
 *     legacy default stream).
 *   - Layouts are row-major and contiguous. bf16 tensors are passed as
 *     uint16_t bit patterns.
 *   - H, W, dH and the workspace must be 16-byte aligned; the other arrays
 *     4-byte aligned (mask 1-byte). D must be a multiple of 8, 1 <= K <= 256,
 *     V >= 1, T finite and > 0.
 *   - Argument errors are returned synchronously and nothing is launched.
 *     Errors found on the device (an id outside [0, V) at a counted row, a
 *     bounded wait that ran out) are recorded in a per-device status word and
 *     returned by kd_get_status.
 *   - No C++ exception crosses this interface.
 */
#ifndef KD_TOPK_KL_H
#define KD_TOPK_KL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KD_OK = 0,
  KD_ERR_ARG = 1,          /* bad size, NULL pointer, bad T, or memory not on the current device */
  KD_ERR_ALIGN = 2,        /* a pointer breaks the alignment rules above */
  KD_ERR_UNSUPPORTED = 3,  /* shape outside what the kernels handle, or no sm_103 device */
  KD_ERR_WORKSPACE = 4,    /* ws_bytes smaller than kd_topk_kl_workspace_size() */
  KD_ERR_INDEX = 5,        /* device: a teacher id outside [0, V) at a counted row */
  KD_ERR_TIMEOUT = 6,      /* device: a bounded pipeline wait ran out; results invalid */
  KD_ERR_CUDA = 7,         /* a CUDA runtime/driver call failed */
  KD_ERR_BOUNDS = 8        /* device, checked build only: a bounds check failed and the access
                              was skipped (libkdtopk_checked.so; see the build's -DKD_CHECKED) */
} kd_status;

/* Opaque stream handle; pass a cudaStream_t. */
typedef struct CUstream_st* kd_stream_t;

/*
 * Bytes of device workspace that kd_topk_kl_fwd and kd_topk_kl_bwd need for
 * these sizes (one buffer serves both calls). The only vocabulary-sized parts
 * are two chunks of dZ (chunk_tokens x V bf16 each; one when N fits in one
 * chunk); beside them the backward keeps the transposed hidden states of two
 * chunks (D x 2 chunk_tokens bf16) and the k-split partials of dH (at most
 * 8 x chunk_tokens x D fp32), all fixed in N, so the size grows linearly in N
 * and never as N x V. chunk_tokens is the backward's row-chunk C (rounded up
 * to a multiple of 256 internally; <= 0 selects 4096). Returns 0 for invalid
 * sizes. Host arithmetic (it reads the current device's SM count when there
 * is one); safe without a GPU.
 */
size_t kd_topk_kl_workspace_size(int64_t N, int D, int V, int K, int64_t chunk_tokens);

/*
 * Forward. Inputs: H [N x D] bf16 (final hidden states), W [V x D] bf16
 * (lm-head weight), topk_idx [N x K] int32 teacher ids, topk_logit [N x K]
 * fp32 teacher logits, mask [N] uint8 (NULL = every row counted).
 * Outputs: loss [N] fp32 per-row KL (0 at masked rows), lse [N] fp32
 * logsumexp of Z/T for every row, n_valid [1] int64 count of counted rows.
 * ws: workspace of at least kd_topk_kl_workspace_size(N, D, V, K, 0) bytes;
 * its contents on entry do not matter and are clobbered.
 */
kd_status kd_topk_kl_fwd(const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                         const float* topk_logit, const uint8_t* mask, int64_t N, int D, int V,
                         int K, float T, float* loss, float* lse, int64_t* n_valid, void* ws,
                         size_t ws_bytes, kd_stream_t stream);

/*
 * Backward of L = sum_n dloss[n] * loss[n]. Takes the forward's inputs plus
 * lse [N] from kd_topk_kl_fwd and dloss [N] fp32 (for the mean loss:
 * 1/n_valid at counted rows). Recomputes the logits chunk by chunk
 * (chunk_tokens rows at a time; the result does not depend on it) and writes
 *   dH [N x D] bf16  = dZ W
 *   dW [V x D] fp32  = dZ^T H   (added to the existing dW if accumulate_dW != 0,
 *                                 overwritten otherwise)
 * with dZ = (dloss/T) (q - P) at counted rows and 0 elsewhere.
 * ws: at least kd_topk_kl_workspace_size(N, D, V, K, chunk_tokens) bytes.
 */
kd_status kd_topk_kl_bwd(const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                         const float* topk_logit, const uint8_t* mask, const float* lse,
                         const float* dloss, int64_t N, int D, int V, int K, float T,
                         int64_t chunk_tokens, int accumulate_dW, uint16_t* dH, float* dW,
                         void* ws, size_t ws_bytes, kd_stream_t stream);

/*
 * Upstream gradient of the mean loss, computed on the device from the count
 * the forward wrote (no host round trip): dloss[n] = 1 / n_valid at counted
 * rows (mask[n] != 0, or every row when mask is NULL) and 0 elsewhere, all 0
 * when n_valid is 0 (reading: the mean over no rows is 0). loss_sum[0] (fp64,
 * device) receives sum_n loss[n], summed in a fixed order. Either output may
 * be NULL (loss may be NULL when loss_sum is). n_valid is a device int64; in
 * token-sharded data parallelism it is the count summed over all ranks, so
 * each rank's rows get the gradient of the global mean.
 */
kd_status kd_topk_kl_mean_grad(const float* loss, const uint8_t* mask, int64_t N,
                               const int64_t* n_valid, float* dloss, double* loss_sum,
                               kd_stream_t stream);

/*
 * Vocabulary shards: the head split over the vocabulary (W's rows), each shard
 * held by one rank, as tensor-parallel heads are. The pages name multi-GPU
 * communication as the method's open question (news article "Offline Top-K
 * Distillation Removes the Need for a Resident Teacher Model...", closing
 * caveats); this is the plainest split of the same computation: every
 * per-row quantity is a sum or a logsumexp over vocabulary columns, so a shard
 * computes its part and the parts are combined exactly.
 *
 * A shard covers ids [v0, v0 + V_shard) of a vocabulary of V; W_shard is
 * those rows of W ([V_shard x D] bf16). topk_idx holds GLOBAL ids in [0, V)
 * (checked as in kd_topk_kl_fwd); each shard uses the teacher entries that
 * fall in its range, and the teacher softmax always runs over all K.
 *
 *   kd_topk_kl_fwd_shard: parts [N x 2] fp32 = per row (logsumexp over the
 *     shard's columns of Z/T, sum_k P_k z_k over the teacher entries in the
 *     shard, z unscaled), ent [N] fp32 = sum_j P_j log P_j of the row's
 *     teacher grid (the same on every shard; 0 at masked rows), n_valid as in
 *     kd_topk_kl_fwd.
 *   kd_topk_kl_shard_merge: parts [R x N x 2] = the R shards' parts stacked in
 *     shard order (e.g. an all-gather), ent from any shard -> loss [N] and
 *     lse [N] exactly as kd_topk_kl_fwd defines them. Shards are combined in
 *     index order, so every rank merging the same parts gets the same bits.
 *   kd_topk_kl_bwd_shard: with the MERGED lse and dloss, the shard's part of
 *     the gradients: dH [N x D] fp32 = dZ_shard W_shard (added to dH's
 *     contents if accumulate_dH != 0; the full dH is the sum over shards) and
 *     dW_shard [V_shard x D] fp32 = dZ_shard^T H (added if accumulate_dW).
 *   ws: kd_topk_kl_shard_workspace_size(N, D, V_shard, K, chunk_tokens) bytes
 *     (fwd and bwd of a shard).
 * Layout, alignment and error rules are those of kd_topk_kl_fwd / _bwd;
 * parts must be 8-byte aligned. A range outside [0, V) is KD_ERR_ARG.
 */
size_t kd_topk_kl_shard_workspace_size(int64_t N, int D, int V_shard, int K, int64_t chunk_tokens);

kd_status kd_topk_kl_fwd_shard(const uint16_t* H, const uint16_t* W_shard, int v0, int V_shard,
                               int V, const int32_t* topk_idx, const float* topk_logit,
                               const uint8_t* mask, int64_t N, int D, int K, float T, float* parts,
                               float* ent, int64_t* n_valid, void* ws, size_t ws_bytes,
                               kd_stream_t stream);

kd_status kd_topk_kl_shard_merge(const float* parts, int R, const float* ent, const uint8_t* mask,
                                 int64_t N, float T, float* loss, float* lse, kd_stream_t stream);

kd_status kd_topk_kl_bwd_shard(const uint16_t* H, const uint16_t* W_shard, int v0, int V_shard,
                               int V, const int32_t* topk_idx, const float* topk_logit,
                               const uint8_t* mask, const float* lse, const float* dloss,
                               int64_t N, int D, int K, float T, int64_t chunk_tokens,
                               int accumulate_dW, int accumulate_dH, float* dH, float* dW_shard,
                               void* ws, size_t ws_bytes, kd_stream_t stream);

/*
 * The loss from logits the caller has already computed, and optionally its
 * gradient with respect to those logits: the forward-chunked form (blog "Making
 * Knowledge Distillation Cheap Enough to Run at Scale", section "Two systems
 * changes", forward-chunked KL bullet: the teacher stays sparse and the loss is
 * computed one slice of sequence positions at a time, from student logits the
 * output layer produced beforehand). Call it once per slice of rows to bound
 * memory; rows are independent.
 *   Z      [N x V] bf16 logits, row stride ldz elements (ldz >= V).
 *   dloss  [N] fp32 upstream gradient (1/n_valid at counted rows for the mean
 *          loss), or NULL to compute the loss only.
 *   dZ     [N x V] bf16 output dZ = (dloss/T)(softmax(Z/T) - P), 0 at masked
 *          rows; row stride lddz; or NULL. It may be Z itself: the gradient
 *          then overwrites the logits (each row is read completely before its
 *          gradient is written).
 *   loss, lse, n_valid, topk_idx, topk_logit, mask, T: as in kd_topk_kl_fwd
 *          (lse = logsumexp(Z/T) for every row).
 *   ws     at least kd_topk_kl_logits_workspace_size(N, K) bytes.
 * V, ldz and lddz must be multiples of 8 (16-byte row starts; KD_ERR_ALIGN
 * otherwise); V up to about 460,000 (KD_ERR_UNSUPPORTED beyond). Z, dZ 16-byte
 * aligned, ws 256-byte aligned. dZ given without dloss is KD_ERR_ARG.
 */
size_t kd_topk_kl_logits_workspace_size(int64_t N, int K);

kd_status kd_topk_kl_logits(const uint16_t* Z, int64_t ldz, const int32_t* topk_idx,
                            const float* topk_logit, const uint8_t* mask, const float* dloss,
                            int64_t N, int V, int K, float T, float* loss, float* lse,
                            int64_t* n_valid, uint16_t* dZ, int64_t lddz, void* ws,
                            size_t ws_bytes, kd_stream_t stream);

/*
 * The teacher's top-K cache: per row, the K largest logits of Z = H W^T and
 * their token ids, in descending order of logit (ties: lower id first). This
 * is the offline step of the method (blog "Making Knowledge Distillation Cheap
 * Enough to Run at Scale", section "Two systems changes", offline-distillation
 * paragraph: the teacher's top-K logits are cached once so the teacher never
 * has to be resident while the student trains; the pages cache the top 100).
 * Its output is the topk_idx / topk_logit input of the loss calls above.
 *   H [N x D] bf16 teacher hidden states, W [V x D] bf16 teacher lm-head weight.
 *   topk_idx [N x K] int32, topk_logit [N x K] fp32 outputs (raw logits; the
 *   loss applies the temperature).
 *   ws: kd_teacher_topk_workspace_size(N, D, V, K) bytes (one chunk of at most
 *   4,096 rows of fp32 logits, plus for V >= 16,384 a sample of W's rows and
 *   per-row candidate lists; fixed in N beyond 4,096 rows).
 * D a multiple of 8, 1 <= K <= min(V, 256). The logits are accumulated in fp32
 * on the tensor cores and the selection is exact on those fp32 values. For
 * V >= 16,384 the chunk's logits are not written out: a strided sample of W's
 * rows sets a threshold per row, the GEMM keeps the logits that reach it, and
 * the K largest are picked from those; a row where the threshold keeps fewer
 * than K or too many logits sends its chunk through the materialising path,
 * so the result is the same either way.
 */
size_t kd_teacher_topk_workspace_size(int64_t N, int D, int V, int K);

kd_status kd_teacher_topk(const uint16_t* H, const uint16_t* W, int64_t N, int D, int V, int K,
                          int32_t* topk_idx, float* topk_logit, void* ws, size_t ws_bytes,
                          kd_stream_t stream);

/*
 * Forward with no workspace argument and no allocation, for callers that
 * cannot obtain device memory themselves (a plugin inside a process whose own
 * allocator already holds the GPU's memory, or a hot path where cudaMalloc,
 * which can synchronise the device, is not allowed). The paper has no
 * counterpart; this is a convenience of this library.
 *   - Same arguments and results as kd_topk_kl_fwd, minus ws / ws_bytes. The
 *     caller still owns and passes every input and output.
 *   - Scratch comes from a fixed 64 MiB array inside the library's device
 *     image, held by every GPU that loads the library until the process exits.
 *     The forward needs N * (12 K + 4 + 8 min(ceil(V / 256), 64)) bytes of it
 *     (plus 256-byte alignment per region), i.e. at most about 52K tokens at
 *     K = 64, V = 201,088. Larger sizes are rejected with KD_ERR_WORKSPACE
 *     before anything is launched.
 *   - The first call on each device looks up the array's device address (with
 *     that device current), and so does the first call after the device's
 *     context has been replaced (cudaDeviceReset); make that first call before
 *     any stream capture.
 *   - All calls on a device share the one array and it keeps the last call's
 *     contents (nothing in it has to start at zero: every cell a call reads is
 *     written earlier in that call). Calls that can overlap on the GPU, e.g. on
 *     two streams without ordering between them, race on it.
 *   - Calls no cudaMalloc, cudaFree or allocating library routine.
 */
kd_status kd_topk_kl_fwd_noalloc(const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                                 const float* topk_logit, const uint8_t* mask, int64_t N, int D,
                                 int V, int K, float T, float* loss, float* lse, int64_t* n_valid,
                                 kd_stream_t stream);

/*
 * Synchronises `stream`, then returns and clears the current device's status
 * word (KD_OK, KD_ERR_INDEX or KD_ERR_TIMEOUT), or KD_ERR_CUDA if the
 * synchronisation itself failed.
 */
kd_status kd_get_status(kd_stream_t stream);

/* Static, NUL-terminated description of a status code. */
const char* kd_status_string(kd_status status);

#ifdef __cplusplus
}
#endif

#endif /* KD_TOPK_KL_H */
