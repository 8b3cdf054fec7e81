/*
 * foak_ce.h -- C ABI of the GB300 (sm_103a) fused cross-entropy library.
 *
 * The operation is the loss the fms-acceleration FOAK plugin swaps into a causal
 * LM head: "Fast Cross Entropy Triton Kernels" on the fms-acceleration-foak 0.7.4
 * page (list of fused operations and kernels), called FastCrossEntropyLoss in
 * fms-acceleration PR #79 "Allow Kernels for Full FT and Non-Quantized PEFT"
 * (Description, items 4 and 5).  The pages name the kernel but print no formula;
 * this library computes the textbook softmax cross-entropy over the rows of an
 * N x V logits matrix with mean reduction over rows whose label is not
 * ignore_index:
 *
 *     lse_i = log sum_j exp(x_ij)          l_i = lse_i - x_{i, y_i}
 *     loss  = sum_{valid i} l_i / D        D = denom > 0 ? denom : n_valid
 *     dx_ij = (g / D) * (exp(x_ij - lse_i) - [j == y_i])   (0 on ignored rows)
 *
 * The chunked linear + CE call is the fused-linear form the pages name as
 * LigerFusedLinearCrossEntropy ("Running Liger Kernel Benchmarks", foak page),
 * "chunked loss" (PR #79, TODO) and FusedCrossEntropyLoss (fms-hf-tuning PR #280,
 * "Notes on FastKernels").  A caller-supplied denom is the per-token mean across
 * data-parallel ranks that PR #280 lists under LossAccelerationPlugin
 * ("--loss_across_gpus mean token"): the caller all-reduces n_valid and passes it.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Pointers marked (device) are device memory owned by the caller; the library
 *   never allocates or frees.  Host pointers are marked (host).
 * - Logits are row-major: element (i, j) is at logits[i * ld + j], ld >= V, in
 *   FOAK_BF16 (bfloat16) or FOAK_F32.  fp16 is not accepted.
 * - labels (device) are int64[N]; a label equal to ignore_index marks an ignored
 *   row.  A label outside [0, V) that is not ignore_index is an error found on the
 *   device: the row is treated as ignored and the error word gets
 *   FOAK_ERRBIT_LABEL_RANGE.  Nothing traps.
 * - stream is a cudaStream_t passed as void* (NULL = legacy default stream).  All
 *   work is enqueued asynchronously on it; nothing synchronises unless the
 *   environment variable FOAK_SYNC_CHECK=1 is set, in which case the call waits
 *   for its own work and turns a non-zero error word into FOAK_ERR_LABEL_RANGE or
 *   FOAK_ERR_TIMEOUT.
 * - Problems checkable on the host return a status before anything is enqueued.
 *   A failed launch returns FOAK_ERR_CUDA.  No C++ exception crosses the ABI.
 * - Scalar outputs (loss, n_valid, err) are single device elements written by the
 *   last kernel of the call.  With n_valid == 0 and denom <= 0 the loss is 0/0 =
 *   NaN (as torch's mean reduction gives) and every gradient row is +0.0.
 * - The result is deterministic for a given input and device: the loss is the
 *   sum of the per-row float32 terms in a fixed order (each of 512 threads adds
 *   rows t, t + 512, ...; then a fixed tree) carried as a double-float (hi + lo,
 *   about 48 significant bits, Knuth's TwoSum), divided by D and rounded to float.
 */
#ifndef FOAK_CE_H
#define FOAK_CE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FOAK_CE_ABI_VERSION 1

typedef enum foak_status {
    FOAK_OK = 0,
    FOAK_ERR_INVALID_ARG = 1,   /* null/negative/misaligned argument, ld < V, ... */
    FOAK_ERR_UNSUPPORTED = 2,   /* dtype or size outside what the kernels handle */
    FOAK_ERR_LABEL_RANGE = 3,   /* (FOAK_SYNC_CHECK only) a label was out of range */
    FOAK_ERR_WORKSPACE = 4,     /* workspace missing, misaligned or too small */
    FOAK_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed */
    FOAK_ERR_TIMEOUT = 6        /* (FOAK_SYNC_CHECK only) a device wait gave up */
} foak_status;

typedef enum foak_dtype { FOAK_F32 = 0, FOAK_BF16 = 1 } foak_dtype;

/* Bits of the device error word (int32) that calls write when err != NULL. */
#define FOAK_ERRBIT_LABEL_RANGE 1
#define FOAK_ERRBIT_TIMEOUT 2

/* Human-readable name of a status code (static string, never NULL). */
const char* foak_status_string(int32_t status);

/* ABI version of the loaded library (FOAK_CE_ABI_VERSION at build time). */
int32_t foak_abi_version(void);

/* Largest V the row calls accept for a dtype: 2^31 - 1 (rows past 8 CTAs x 64 KB,
 * the one-pass plans' reach, are streamed twice by one CTA).  The chunked linear +
 * CE calls take V <= 262144. */
int64_t foak_ce_max_vocab(int32_t dtype);

/*
 * Bytes of device workspace that foak_ce_forward / foak_ce_fwd_bwd need for N rows
 * (a 256-byte header plus N float32 per-row loss terms).  The workspace must be
 * 256-byte aligned and zero-filled before its first use; every call leaves the
 * header zeroed again when its work completes, so one buffer can serve any number
 * of stream-ordered calls.  Calls that share a workspace must not overlap on the
 * GPU (same stream, or ordered by events).
 */
size_t foak_ce_workspace_size(int64_t N);

/*
 * Forward: one read of each non-ignored row (an ignored row is never read).
 *   logits (device)   N x V, row stride ld (elements)
 *   dtype             FOAK_BF16 or FOAK_F32
 *   labels (device)   int64[N]
 *   ignore_index      label value of ignored rows (usually -100)
 *   denom             > 0: divide by denom (global valid-token count under data
 *                     parallelism); <= 0: divide by this call's n_valid
 *   loss (device)     float[1]: the mean loss
 *   lse (device)      float[N] or NULL: log-sum-exp per row (0 for ignored rows);
 *                     foak_ce_backward needs it
 *   row_loss (device) float[N] or NULL: per-row terms lse_i - x_{i,y_i} (0 for
 *                     ignored rows), i.e. reduction 'none'
 *   n_valid (device)  int32[1] or NULL: rows with a label in [0, V)
 *   err (device)      int32[1] or NULL: FOAK_ERRBIT_* of this call (0 = clean)
 *   workspace (device) foak_ce_workspace_size(N) bytes, see above
 */
foak_status foak_ce_forward(const void* logits, int32_t dtype, int64_t ld, const int64_t* labels,
                            int64_t N, int64_t V, int64_t ignore_index, float denom, float* loss,
                            float* lse, float* row_loss, int32_t* n_valid, int32_t* err,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward: dlogits = (exp(logits - lse) - onehot) * g / D, ignored rows +0.0.
 *   dlogits (device)  N x V with the same ld and dtype; may equal logits (in place)
 *   logits (device)   as in forward (not read on ignored rows)
 *   lse (device)      float[N] from foak_ce_forward
 *   grad_out (device) float[1]: g, the upstream gradient of the loss; NULL = 1.0
 *   denom             as in forward (<= 0: count n_valid again from labels)
 *   err (device)      int32[1] or NULL: FOAK_ERRBIT_LABEL_RANGE if a label is bad
 * Needs no workspace.
 */
foak_status foak_ce_backward(void* dlogits, const void* logits, int32_t dtype, int64_t ld,
                             const int64_t* labels, int64_t N, int64_t V, int64_t ignore_index,
                             const float* lse, const float* grad_out, float denom, int32_t* err,
                             void* stream);

/*
 * Fused forward + backward, in place: each non-ignored row is read once and its
 * gradient written over it; ignored rows are only written (+0.0).  The logits are
 * destroyed; a caller that still needs them calls forward + backward instead.
 *   g (host)          upstream gradient of the loss (1.0 for a plain mean loss,
 *                     or a loss-scale / accumulation factor)
 *   lse (device)      float[N] or NULL, as in forward
 *   other arguments   as in forward
 */
foak_status foak_ce_fwd_bwd(void* logits, int32_t dtype, int64_t ld, const int64_t* labels,
                            int64_t N, int64_t V, int64_t ignore_index, float g, float denom,
                            float* loss, float* lse, int32_t* n_valid, int32_t* err,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * The data-parallel per-token mean (fms-hf-tuning PR #280, "Early Version Of This
 * Plugin": LossAccelerationPlugin, --loss_across_gpus mean token) divides every
 * rank's share by the number of valid tokens of ALL ranks, which each rank knows
 * only after an all-reduce.  These two calls keep that exchange on the device:
 * a rank counts its valid labels into device memory, the caller sums the counts
 * across ranks in place (e.g. an NCCL all-reduce of one int64), and the fused
 * call reads the total from device memory, with no host synchronisation between.
 *
 * foak_ce_count_valid: number of rows whose label is not ignore_index and lies in
 * [0, V).
 *   labels (device)   int64[N] (may be NULL when N == 0)
 *   n_valid (device)  int64[1], 8-byte aligned: the count
 *   err (device)      int32[1] or NULL: FOAK_ERRBIT_LABEL_RANGE if a label is
 *                     neither ignore_index nor in [0, V), else 0
 * Errors: FOAK_ERR_INVALID_ARG for N < 0, V < 1, a null or misaligned pointer.
 */
foak_status foak_ce_count_valid(const int64_t* labels, int64_t N, int64_t V, int64_t ignore_index,
                                int64_t* n_valid, int32_t* err, void* stream);

/*
 * foak_ce_fwd_bwd with the denominator read from device memory: D = *denom_count
 * (int64, e.g. the all-reduced sum of every rank's foak_ce_count_valid), read by
 * the kernel when it runs, so the count may still be in flight on `stream` when
 * the call is made.  loss is then this rank's share sum_{valid i} l_i / D (the
 * ranks' losses add up to the global mean); n_valid is this call's own count.
 * With D == 0 the loss is NaN and every gradient row +0.0, as in foak_ce_fwd_bwd.
 *   denom_count (device)  int64[1], 8-byte aligned
 *   other arguments       as for foak_ce_fwd_bwd (there is no host denom)
 */
foak_status foak_ce_fwd_bwd_devdenom(void* logits, int32_t dtype, int64_t ld, const int64_t* labels,
                                     int64_t N, int64_t V, int64_t ignore_index, float g,
                                     const int64_t* denom_count, float* loss, float* lse, int32_t* n_valid,
                                     int32_t* err, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Bytes of device workspace foak_ce_fwd_bwd_host needs for N rows: a 256-byte
 * header, N float32 per-row loss terms and 256 bytes of per-chunk error words and
 * results.  256-byte aligned, zero-filled before first use, left reusable by every
 * call (the same rules as foak_ce_workspace_size).
 */
size_t foak_ce_host_workspace_size(int64_t N);

/*
 * Fused forward + backward on logits that live in HOST memory: the call copies
 * the labels and then the logits to the device in row chunks on a copy stream of
 * its own and runs the fused kernel of foak_ce_fwd_bwd on each chunk as soon as it
 * has landed (on `stream`), so the arithmetic hides under the host-to-device copy;
 * every chunk divides by the n_valid of all N rows (or denom), and one reduction
 * over all N rows in the same order as foak_ce_fwd_bwd's gives the loss.
 * This is the same mean-reduced cross-entropy and in-place gradient as the
 * FastCrossEntropyLoss kernel of the FOAK pages (fms-acceleration PR #79,
 * Description item 4); the pages fix no host interface, so this one is ours.
 *   host_logits (host)   N x V in dtype, row stride ld elements; pinned memory
 *                        (cudaHostAlloc / torch pin_memory) for a full-speed copy.
 *                        Only the first V elements of each row are copied.
 *   host_labels (host)   int64[N]
 *   dev_logits (device)  N x ld in dtype, 16-byte aligned: receives the logits and
 *                        ends holding dlogits (ignored rows +0.0)
 *   dev_labels (device)  int64[N], receives the labels
 *   host_loss (host)     float[1]; host_n_valid, host_err (host) int32[1] or NULL:
 *                        written by device-to-host copies at the end of the work on
 *                        `stream` (pinned memory keeps the call asynchronous;
 *                        read them after synchronising the stream)
 *   workspace (device)   foak_ce_host_workspace_size(N) bytes
 *   other arguments      as for foak_ce_fwd_bwd
 * Errors: as foak_ce_fwd_bwd for the arguments; FOAK_ERR_INVALID_ARG for a null
 * host or device buffer when N > 0.  Calls for the same device from several host
 * threads are serialised internally (they share the copy stream).
 */
foak_status foak_ce_fwd_bwd_host(const void* host_logits, int32_t dtype, int64_t ld, const int64_t* host_labels,
                                 int64_t N, int64_t V, int64_t ignore_index, float g, float denom,
                                 void* dev_logits, int64_t* dev_labels, float* host_loss, int32_t* host_n_valid,
                                 int32_t* host_err, void* workspace, size_t workspace_bytes, void* stream);

/*
 * RMSNorm, the "Fast RMS LayerNorm" kernel the FOAK pages list among their fused
 * operations (fms-acceleration-foak 0.7.4 page; its patch rule swaps a decoder's
 * RMSNorm module for fast_rms_layernorm).  The pages print no formula; the
 * operation is the Llama / Mistral / Granite RMSNorm, in fp32, rounded once:
 *     r_i = 1 / sqrt(mean_j X_ij^2 + eps),   Y_ij = X_ij * r_i * gamma_j
 *   X (device)      N x D in dtype (bf16 or fp32), row stride ldx elements
 *   gamma (device)  D in dtype
 *   Y (device)      N x D in dtype, row stride ldy (may equal X)
 *   rstd (device)   float[N] or NULL: r_i, needed by the backward
 * D % 8 == 0; X, Y, gamma 16-byte aligned with 16-byte row strides; eps >= 0.
 */
foak_status foak_rmsnorm_forward(const void* X, int32_t dtype, int64_t ldx, const void* gamma, int64_t N, int64_t D,
                                 float eps, void* Y, int64_t ldy, float* rstd, void* stream);

/* Bytes of device workspace foak_rmsnorm_backward needs for dgamma (512 x D floats of partial sums). */
size_t foak_rmsnorm_workspace_size(int64_t D);

/*
 * RMSNorm backward: with xh = X * r and u = gamma * dY (per row),
 *     dX = r * (u - xh * mean(xh * u)),    dgamma_j = sum_i dY_ij * xh_ij
 *   dY, X (device)  N x D in dtype (row strides lddy, ldx); rstd from the forward
 *   dX (device)     N x D in dtype, row stride lddx (may equal dY)
 *   dgamma (device) float32[D], overwritten, or NULL to skip it; it is summed in a
 *                   fixed order (deterministic) through `workspace`
 *                   (foak_rmsnorm_workspace_size(D) bytes, 256-byte aligned)
 * Alignment as for the forward.
 */
foak_status foak_rmsnorm_backward(const void* dY, int64_t lddy, const void* X, int64_t ldx, const void* gamma,
                                  const float* rstd, int32_t dtype, int64_t N, int64_t D, void* dX, int64_t lddx,
                                  float* dgamma, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Bytes of device workspace foak_rmsnorm_linear_ce_chunked needs: the chunked
 * linear + CE workspace, the normalised hidden states H and their gradient dH
 * (bf16 N x D each), r (float[N]) and the dgamma partials.
 */
size_t foak_rmsnorm_linear_ce_workspace_size(int64_t N, int64_t V, int64_t D, int64_t chunk);

/*
 * The decoder's tail: final RMSNorm -> LM head -> cross-entropy, the norm and the
 * chunked linear + CE of the FOAK pages composed on the device (the norm as the
 * chunked path's prologue and its backward as the epilogue; H and dH never leave
 * the device, the logits are never materialised):
 *     H = rmsnorm(X, gamma, eps) (bf16), loss / dH / dW as foak_linear_ce_chunked on
 *     H, then dX, dgamma through the norm (the rounding of H to bf16 is passed
 *     through as the identity).
 *   X (device)       bf16 [N][D] dense (row stride D), D % 8 == 0
 *   gamma (device)   bf16 [D]
 *   W, labels, chunk, g, denom, loss, dW, n_valid, err: as foak_linear_ce_chunked
 *   eps              >= 0 (1e-5 for Mistral and Llama-3)
 *   dX (device)      bf16 [N][D], overwritten
 *   dgamma (device)  float32 [D], overwritten
 * All pointers 16-byte aligned (loss, dgamma, n_valid, err: 4-byte).
 */
foak_status foak_rmsnorm_linear_ce_chunked(const void* X, const void* gamma, const void* W, const int64_t* labels,
                                           int64_t N, int64_t V, int64_t D, int64_t ignore_index, int64_t chunk,
                                           float eps, float g, float denom, float* loss, void* dX, float* dgamma,
                                           float* dW, int32_t* n_valid, int32_t* err, void* workspace,
                                           size_t workspace_bytes, void* stream);

/*
 * Rotary position embedding, the "Fast RoPE" kernel the FOAK pages list among
 * their fused operations (fms-acceleration-foak 0.7.4 page), with the explicit
 * position ids the pages note the FOAK version lacks (foak page, Known Issues;
 * fms-hf-tuning PR #280, Notes on FastKernels).  The pages print no formula; the
 * operation is the Llama / Mistral rotary embedding, "rotate half" pairing: for
 * head dimension d and i < d/2, elements i and i + d/2 of every head vector of
 * token t turn by theta = positions[t] * base^(-2i/d).
 *
 * Bytes of the cos/sin table for positions [0, max_pos) and head dimension d
 * (two fp32 planes of max_pos x d/2); 0 for an unsupported d (d % 16 != 0).
 */
size_t foak_rope_cache_size(int64_t max_pos, int64_t d);

/*
 * Build the table on the device: cos and sin of every (position, frequency),
 * the angle and its reduction in float64, stored as fp32.  base > 1 (10000 for
 * Llama-2 / Mistral, 500000 for Llama-3).  cache (device): 256-byte aligned,
 * foak_rope_cache_size(max_pos, d) bytes, owned by the caller; build it once per
 * (base, d, max_pos) and reuse it.
 */
foak_status foak_rope_build_cache(double base, int64_t d, int64_t max_pos, void* cache, size_t cache_bytes,
                                  void* stream);

/*
 * Apply the rotation in place (inverse != 0: turn by -theta, the backward: the
 * gradient of sum(G * rope(X)) is rope(G, inverse)).
 *   X (device)          T tokens x H heads x d in dtype (bf16 or fp32); heads of a
 *                       token contiguous, token stride ldt >= H*d elements (so Q
 *                       and K may be views into a fused QKV buffer); 16-byte
 *                       aligned, ldt * sizeof(dtype) % 16 == 0
 *   positions (device)  int64[T]: the token's position id (restarting at 0 per
 *                       sequence in a packed batch)
 *   cache (device)      the table of foak_rope_build_cache for max_pos, d
 *   err (device)        int32[1] or NULL: FOAK_ERRBIT_LABEL_RANGE when a position
 *                       is outside [0, max_pos); that token is left unchanged
 * d % 16 == 0 (FOAK_ERR_UNSUPPORTED otherwise).
 */
foak_status foak_rope_apply(void* X, int32_t dtype, int64_t T, int64_t H, int64_t ldt, int64_t d,
                            const int64_t* positions, const void* cache, int64_t max_pos, int32_t inverse,
                            int32_t* err, void* stream);

/*
 * foak_rope_apply on the Q and K of one layer in a single launch: Q is T x Hq x d
 * (token stride ldq), K is T x Hk x d (token stride ldk), both in dtype, same
 * positions and table; either may be empty (H = 0, pointer may be NULL).  Rules
 * and errors as foak_rope_apply.
 */
foak_status foak_rope_apply_qk(void* Q, int64_t Hq, int64_t ldq, void* K, int64_t Hk, int64_t ldk, int32_t dtype,
                               int64_t T, int64_t d, const int64_t* positions, const void* cache, int64_t max_pos,
                               int32_t inverse, int32_t* err, void* stream);

/*
 * Bytes of device workspace foak_linear_ce_chunked needs: the batch's label
 * count, N float32 per-row loss terms, a few error words, one chunk's per-tile
 * softmax statistics (chunk x ceil(V / 256) float pairs), its label logits and
 * log-sum-exps, and eight chunks of bf16 logits (min(8 chunk, N) x V, rows padded
 * to 64 elements: dW is updated once per group of four chunks, and one group is
 * computed while the last one is used).  256-byte aligned; its
 * contents need no initialisation and every call may reuse it.
 */
size_t foak_linear_ce_workspace_size(int64_t N, int64_t V, int64_t D, int64_t chunk);

/*
 * Chunked linear + cross-entropy: loss, dH and dW of CE(H W^T) computed chunk by
 * chunk (Z = H_c W^T, dZ = (softmax(Z) - onehot) g / D, dH_c = dZ W,
 * dW += dZ^T H_c) without materialising the N x V logits; the products run on the
 * tcgen05 tensor cores with fp32 accumulation, Z/dZ are kept in bf16.  The Z
 * product's epilogue reduces its fp32 accumulator to per-row, per-tile softmax
 * statistics and the label's logit, so the loss and log-sum-exp come from the
 * unrounded logits and dZ is one streaming pass over Z.
 *   H (device)        bf16 [N][D] row-major (hidden states), D % 8 == 0
 *   W (device)        bf16 [V][D] row-major (LM-head weight, no bias)
 *   labels (device)   int64[N]; ignore_index as for the CE calls
 *   chunk             rows per chunk (e.g. 1024), >= 1
 *   g (host), denom   as for foak_ce_fwd_bwd; D = denom > 0 ? denom : n_valid of
 *                     all N rows, the same for every chunk
 *   loss (device)     float[1]
 *   dH (device)       bf16 [N][D], overwritten
 *   dW (device)       float32 [V][D], overwritten (not accumulated into)
 *   n_valid, err      as for foak_ce_forward (err also reports GEMM wait timeouts)
 * All pointers 16-byte aligned.
 */
foak_status foak_linear_ce_chunked(const void* H, const void* W, const int64_t* labels, int64_t N, int64_t V,
                                   int64_t D, int64_t ignore_index, int64_t chunk, float g, float denom,
                                   float* loss, void* dH, float* dW, int32_t* n_valid, int32_t* err,
                                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * Building block of the chunked linear + CE: C[M x N] (+)= A[M x K] * B[N x K]^T on
 * the tcgen05 tensor cores, bf16 operands, fp32 accumulation (exposed so the
 * three products of the chunked call can be tested and timed alone).
 *   a, b (device)     bf16.  With *_mn_major = 0 the operand is stored row-major
 *                     as [rows][K] (K contiguous, row stride lda/ldb elements);
 *                     with 1 as [K][rows] (rows contiguous).  16-byte aligned
 *                     pointers and row strides; row strides >= the contiguous extent.
 *   out (device)      row-major [M][ldo]: bf16 for out_mode FOAK_GEMM_BF16, fp32 for
 *                     FOAK_GEMM_F32 (overwrite) and FOAK_GEMM_F32_ACC (add into it);
 *                     16-byte aligned pointer and row stride.
 *   err (device)      int32[1] or NULL: FOAK_ERRBIT_TIMEOUT is OR-ed in if a
 *                     device wait gave up (never set on a healthy GPU).
 */
#define FOAK_GEMM_BF16 0
#define FOAK_GEMM_F32 1
#define FOAK_GEMM_F32_ACC 2
foak_status foak_gemm_bf16(const void* a, int64_t lda, int32_t a_mn_major, const void* b, int64_t ldb,
                           int32_t b_mn_major, int64_t M, int64_t N, int64_t K, void* out, int64_t ldo,
                           int32_t out_mode, int32_t* err, void* stream);

/*
 * Up to FOAK_GEMM_GROUP_MAX independent products of foak_gemm_bf16's form in one
 * persistent launch: the SM pairs take a list of (product, 256 x 256 output unit)
 * entries balanced by estimated cost, longest units first, so a product with fewer
 * units than the GPU has SM pairs (dH of the chunked call: 4 x 16 units on 76 pairs)
 * shares the machine with another instead of leaving pairs idle.  This is how the
 * chunked call issues its dH products (with the next chunk's logits product).
 *   problems (host)   n descriptors, fields and rules as for foak_gemm_bf16; read
 *                     before the call returns.  No product may write memory that
 *                     another one reads or writes.
 *   n                 0 .. FOAK_GEMM_GROUP_MAX
 *   err (device)      as for foak_gemm_bf16, shared by the products
 * Products with M <= 128 (single-CTA tiles), or more than 8192 output units in all,
 * are launched one after another in the order given, with the same results.
 */
#define FOAK_GEMM_GROUP_MAX 3
typedef struct foak_gemm_problem {
    const void* a;
    int64_t lda;
    int32_t a_mn_major;
    const void* b;
    int64_t ldb;
    int32_t b_mn_major;
    int64_t M, N, K;
    void* out;
    int64_t ldo;
    int32_t out_mode;
} foak_gemm_problem;
foak_status foak_gemm_bf16_group(const foak_gemm_problem* problems, int32_t n, int32_t* err, void* stream);

/*
 * Largest N that foak_ce_fwd_bwd_noalloc accepts (its fixed scratch holds one
 * float per row: 1 MiB plus a 256-byte header on every device that loads the
 * library, kept until the process exits).
 */
#define FOAK_CE_NOALLOC_MAX_ROWS 262144

/*
 * Fused forward + backward without any workspace from the caller.  The pages
 * have no counterpart to this call; it exists for callers that must not allocate
 * device memory while they run -- e.g. code on a latency-critical path, where
 * cudaMalloc/cudaFree can synchronise the whole device, or a plugin inside a
 * runtime that owns all device memory and forbids allocations during execution.
 * It computes exactly what foak_ce_fwd_bwd computes, with the same arguments
 * minus the workspace, and allocates nothing: its scratch is a fixed array in the
 * library's device image.
 *   N                 at most FOAK_CE_NOALLOC_MAX_ROWS; larger N returns
 *                     FOAK_ERR_WORKSPACE before anything is enqueued
 *   stream            besides the kernel, the call enqueues a 256-byte
 *                     cudaMemsetAsync that clears the scratch header
 * The scratch used is the CURRENT device's: make the device that holds the
 * buffers and owns `stream` current before the call.  The first call on a device
 * looks up the scratch array's device address (once per device, with that device
 * current); make that first call before any stream capture begins.  Every call on a device shares the one scratch array, so calls
 * that overlap on the GPU (different streams without ordering) race and give
 * wrong results: serialise them.
 */
foak_status foak_ce_fwd_bwd_noalloc(void* logits, int32_t dtype, int64_t ld, const int64_t* labels,
                                    int64_t N, int64_t V, int64_t ignore_index, float g, float denom,
                                    float* loss, float* lse, int32_t* n_valid, int32_t* err,
                                    void* stream);

/*
 * Test hook: the next `count` launches made by this library fail with
 * FOAK_ERR_CUDA before anything is enqueued (host-side fault injection).
 */
void foak_test_fail_next_launches(int32_t count);

/*
 * Test hooks for the device-side failure path (no fault is involved): the row
 * kernels' shared-memory barrier waits give up after `ns` nanoseconds (0 restores
 * the default of 4 s), and the row kernels' producers never load row `row`'s data
 * (-1 disables), so the wait for that row is sure to run out.  A call that hits a
 * run-out wait stops loading, finishes its barriers, leaves the workspace reusable
 * and reports FOAK_ERRBIT_TIMEOUT in its error word (FOAK_ERR_TIMEOUT under
 * FOAK_SYNC_CHECK=1); its loss and gradient are then undefined.
 */
void foak_test_set_wait_limit_ns(uint64_t ns);
void foak_test_skip_row_load(int64_t row);

/*
 * Test hook: which row kernel the forward and fused calls use.  0 (default):
 * automatic -- aligned rows that fit one CTA's 64 KB slice go to the kernel whose
 * 16 warps each stream a 4 KB region of every row on their own, other rows of one
 * slice are swept once by one CTA in step, longer rows are streamed twice by one
 * CTA (log-sum-exp, then gradient); 1: one pass with the CTA in step, longer rows
 * split over a cluster of 2, 4 or 8 CTAs; 2: the two-pass streaming kernel for
 * every row length; 3: as 0 (the independent-warp kernel wherever it applies).
 * Results agree up to fp32 summation order.  Other values are treated as 0.
 */
void foak_test_set_row_path(int32_t path);

/*
 * Test hook (host only, no device work): the unit list foak_gemm_bf16_group would
 * give products of these shapes on `pairs` SM pairs.
 *   mnk      host int64[3 n]: M, N, K of each product (every M > 128), n in 1 .. 3
 *   start    host int32[pairs + 1]: cluster c takes entries start[c] .. start[c+1] - 1
 *   ent      host int32[ent_cap]: entries, product << 14 | output unit
 * Returns the number of clusters used (<= pairs), or -1 for bad arguments or when
 * ent_cap is too small.
 */
int32_t foak_test_gemm_group_schedule(const int64_t* mnk, int32_t n, int32_t pairs, int32_t* start, int32_t* ent,
                                      int32_t ent_cap);

#ifdef __cplusplus
}
#endif

#endif /* FOAK_CE_H */
