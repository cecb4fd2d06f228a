/*
 * lce.h -- C ABI of liblce.so: fused, chunked LM-head linear + cross-entropy
 * (forward and backward) on one GB300 (sm_103a).
 *
 * The operation ("XTuner on Ascend 910C: Qwen3.5-2B training optimisation",
 * section 3.1.4, Liger chunked cross-entropy, Fig. 12 and Fig. 13): the LM-head
 * logits z = H W^T of an N-token batch over a V-word vocabulary feed a
 * token-level cross-entropy, and the backward produces d_input (dH) and
 * d_weight (dW) without ever writing the full [N, V] logits or d_logits to
 * memory. With valid_i = [y_i != ignore_index], n = sum_i valid_i:
 *
 *   lse_i  = log sum_v exp(z_iv)
 *   loss   = sum_i valid_i (lse_i - z_{i,y_i}) / n        (LCE_MEAN; no /n for LCE_SUM)
 *   G_iv   = valid_i g (exp(z_iv - lse_i) - [v = y_i]) / n (g = upstream gradient)
 *   dH     = G W,   dW = G^T H
 *
 * Tokens are processed in chunks ("XTuner V1 introduction", memory
 * optimisation section: the loss graph is computed chunk by chunk), so the
 * extra device memory is O(chunk * V), never O(N * V).
 *
 * Conventions for every entry point
 *   - Pointers named "device" are CUDA device pointers owned by the caller;
 *     the library never allocates, frees or keeps them.
 *   - H [N, d] and W [V, d] are bf16, row-major and contiguous; dH [N, d] is
 *     bf16; dW [V, d], loss [1], lse [N] are fp32; y [N] is int64. d is a
 *     multiple of 8. Alignment: H, W, dH, dW (and x, dx of the norm calls,
 *     the shard statistics) 16 bytes, because the kernels move them with TMA
 *     or 16-byte vector accesses; y 8 bytes; lse, loss, grad_loss 4 bytes. A
 *     slice of rows [a, b) of contiguous H and y therefore always qualifies,
 *     since a row of H is d * 2 bytes.
 *   - ws / ws_bytes: caller-allocated device workspace of at least
 *     lce_workspace_size(op, ...) bytes, 256-byte aligned. Its contents on
 *     entry do not matter; two calls running at the same time need two
 *     workspaces.
 *   - stream: a cudaStream_t (passed as void*); NULL is the legacy default
 *     stream. All device work is ordered on it. No call synchronises the host
 *     unless opts->sync_check is set.
 *   - Return value: LCE_OK or an LCE_ERR_* code. Argument errors are detected
 *     on the host before any launch. Device-detected problems (a label outside
 *     {ignore_index} U [0, V), a wait that timed out) set bits in the
 *     workspace's status word; the affected row is then treated as ignored
 *     (never an out-of-bounds read). They become return codes when
 *     opts->sync_check is set, or through lce_read_device_status().
 *   - Thread safety: calls with distinct workspaces may run concurrently.
 */
#ifndef LCE_H_
#define LCE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LCE_VERSION 1

/* status codes */
#define LCE_OK 0
#define LCE_ERR_INVALID_ARG 1        /* null pointer, N < 0, d/V <= 0, d % 8 != 0, bad option */
#define LCE_ERR_ALIGNMENT 2          /* a pointer below the alignment stated below (workspace: 256 bytes) */
#define LCE_ERR_WORKSPACE 3          /* ws_bytes smaller than lce_workspace_size() */
#define LCE_ERR_UNSUPPORTED_DEVICE 4 /* the current device is not an sm_103 GPU */
#define LCE_ERR_CUDA 5               /* a CUDA runtime / driver call failed */
#define LCE_ERR_LABEL_RANGE 6        /* a label is neither ignore_index nor in [0, V) */
#define LCE_ERR_TIMEOUT 7            /* a device-side wait exceeded its limit */
#define LCE_ERR_BOUNDS 8             /* (a library built with LCE_CHECKS only) a kernel computed an
                                        index or tile coordinate outside its buffer; the access
                                        was skipped, so the outputs are not valid */

/* reductions */
#define LCE_MEAN 0
#define LCE_SUM 1

/* ops for lce_workspace_size */
#define LCE_OP_FORWARD 0
#define LCE_OP_BACKWARD 1
#define LCE_OP_FWD_BWD 2
#define LCE_OP_VSHARD_COMBINE 3
#define LCE_OP_NORM_FWD_BWD 4
#define LCE_OP_VSHARD_CHUNK 5

/* device status bits returned by lce_read_device_status */
#define LCE_DEVICE_LABEL_RANGE 1
#define LCE_DEVICE_TIMEOUT 2
#define LCE_DEVICE_BOUNDS 4   /* set only by a library built with LCE_CHECKS (see LCE_ERR_BOUNDS) */

typedef struct lce_opts {
  int64_t chunk_tokens;     /* tokens per chunk; 0 = automatic (4096, capped at N) */
  int64_t ignore_index;     /* label value that is ignored; default -100 */
  int64_t n_valid_override; /* < 0: count valid labels of this call; >= 0: use as the
                               denominator n (data-parallel shards pass the global count) */
  int32_t reduction;        /* LCE_MEAN (default) or LCE_SUM */
  int32_t accumulate_dW;    /* 0: dW = G^T H; 1: dW += G^T H (gradient accumulation) */
  int32_t sync_check;       /* 1: synchronise the stream at the end and turn device
                               status bits into the return code */
  int32_t reserved;         /* 0, or LCE_TEST_FORCE_TIMEOUT (tests only, see below) */
} lce_opts;

/* Test value for lce_opts.reserved: lce_forward's logits kernel then loads
 * no operands, so its bounded device waits run out (about 2 s); the kernel
 * records LCE_DEVICE_TIMEOUT, releases its resources and returns, and the
 * call reports LCE_ERR_TIMEOUT (with sync_check, or via
 * lce_read_device_status). Outputs are meaningless. It exists to test the
 * timeout path without faulting or hanging the GPU; other calls reject it. */
#define LCE_TEST_FORCE_TIMEOUT 0x7E57

/* Fill *opts with the defaults above. */
void lce_opts_init(lce_opts* opts);

/* Bytes of device workspace one call of the given op needs (LCE_OP_*). opts
 * may be NULL (defaults). Returns 0 for invalid sizes. */
size_t lce_workspace_size(int op, int64_t N, int64_t d, int64_t V, const lce_opts* opts);

/* Automatic chunk size ("XTuner V1 introduction", memory optimisation
 * section: the loss graph is chunked automatically to bound its memory): the
 * largest multiple of 256 tokens, at most 4096 and at most N rounded up to
 * 256, whose LCE_OP_FWD_BWD workspace fits in budget_bytes (with opts'
 * other fields). Larger chunks do not run faster on this GPU (W is read once
 * per chunk either way), so 4096 is the cap. Returns 0 if not even 256
 * tokens fit or the sizes are invalid. Host-only; touches no device. */
int64_t lce_auto_chunk(int64_t N, int64_t d, int64_t V, size_t budget_bytes, const lce_opts* opts);

/* Forward: loss [1] and lse [N] (fp32, device). lse of ignored rows is
 * computed too (the backward needs it for nothing, callers may use it).
 * N = 0 gives loss = 0. */
int lce_forward(const void* H, const void* W, const int64_t* y, int64_t N, int64_t d, int64_t V,
                float* loss, float* lse, const lce_opts* opts, void* ws, size_t ws_bytes, void* stream);

/* Backward from a saved lse [N] (device, from lce_forward of the same inputs)
 * and the upstream gradient grad_loss [1] (device fp32; NULL means 1.0).
 * Recomputes the logits chunk by chunk. Writes dH [N, d] (bf16) and dW [V, d]
 * (fp32; overwritten, or accumulated into when opts->accumulate_dW). */
int lce_backward(const void* H, const void* W, const int64_t* y, int64_t N, int64_t d, int64_t V,
                 const float* lse, const float* grad_loss, void* dH, float* dW, const lce_opts* opts,
                 void* ws, size_t ws_bytes, void* stream);

/* Forward and backward in one call (the training step's loss head).
 * grad_loss: device fp32 [1] or NULL for 1.0. lse may be NULL (kept in the
 * workspace). Outputs as in lce_forward and lce_backward. */
int lce_fwd_bwd(const void* H, const void* W, const int64_t* y, int64_t N, int64_t d, int64_t V,
                const float* grad_loss, float* loss, float* lse, void* dH, float* dW, const lce_opts* opts,
                void* ws, size_t ws_bytes, void* stream);

/* lce_fwd_bwd with dW finished in vocabulary slices, so that its reduction
 * over data-parallel ranks (FSDP's reduce-scatter of the weight gradient)
 * can run on another stream while the backward is still computing. FSDP
 * shards every parameter evenly over the ranks and hides its communication
 * behind computation ("XTuner V1 introduction", communication masking
 * section; "XTuner on Ascend 910C: Qwen3.5-2B training optimisation",
 * section 3.2.1, for the gather of the parameters); the gradient reduction
 * is the mirror step of the backward.
 *
 * Same arguments and workspace as lce_fwd_bwd (LCE_OP_FWD_BWD) plus:
 *   n_slices      1 .. LCE_MAX_SLICES
 *   slice_bounds  host int64 [n_slices + 1]: 0 = b_0 <= b_1 <= ... <= b_n = V;
 *                 every interior bound a multiple of LCE_SLICE_ALIGN (the dW
 *                 tile height). Slice s is dW rows [b_s, b_{s+1}).
 *   slice_events  host array of n_slices cudaEvent_t (as void*), created by
 *                 the caller, or NULL. events[s] is recorded on the stream
 *                 right after the last launch that writes slice s; a
 *                 cudaStreamWaitEvent on it orders later work (a collective
 *                 on another stream) after the final values of that slice.
 *                 All events are recorded before this call returns.
 *   sm_limit      0 = all SMs; else the CTA-pair GEMM launches of this call
 *                 use at most sm_limit SMs (rounded down to even, >= 2), so
 *                 that kernels on other streams (collectives) find free SMs.
 * The last chunk's backward runs as n_slices launches in slice order: dW
 * rows of slices 0 .. n-2 alone, then slice n-1 together with the chunk's
 * dH. Earlier chunks are unchanged. Every output (loss, lse, dH, dW) is
 * bitwise identical to lce_fwd_bwd's: each output tile is computed by the
 * same arithmetic, whichever launch it falls in. */
#define LCE_MAX_SLICES 4096
#define LCE_SLICE_ALIGN 256
int lce_fwd_bwd_sliced(const void* H, const void* W, const int64_t* y, int64_t N, int64_t d, int64_t V,
                       const float* grad_loss, float* loss, float* lse, void* dH, float* dW, int32_t n_slices,
                       const int64_t* slice_bounds, void* const* slice_events, int32_t sm_limit,
                       const lce_opts* opts, void* ws, size_t ws_bytes, void* stream);

/* Forward that allocates nothing and takes no workspace, for callers that
 * cannot allocate device memory: their memory is wholly owned by another
 * allocator (a framework's caching pool or a runtime's arena), or they must
 * not call cudaMalloc / cudaFree, which can block or synchronise the device.
 * The pages have no counterpart to this entry point; it is a deployment aid.
 * Same arguments and results as lce_forward, minus ws / ws_bytes. Its scratch
 * is a fixed 32 MiB array inside the library's device image, held on every
 * GPU that loads the library until the process exits; a call whose forward
 * workspace (lce_workspace_size(LCE_OP_FORWARD, ...)) exceeds 32 MiB returns
 * LCE_ERR_WORKSPACE (pass a smaller opts->chunk_tokens). The array's device
 * address belongs to one CUDA context (the device's primary context, a
 * context the caller created with the driver API, or the new primary context
 * after cudaDeviceReset each hold their own copy of the library's device
 * image): the first call in each context looks it up, with that context
 * current, and caches it under the context's id, so make the first call in a
 * context before any stream capture in it. All calls share the one array: calls whose work overlaps on the
 * GPU (other streams, other host threads) race and must be serialised by the
 * caller. Nothing in the array needs to be zero on entry; each call
 * overwrites what it reads, and lce_read_device_status() does not apply. */
int lce_forward_noalloc(const void* H, const void* W, const int64_t* y, int64_t N, int64_t d, int64_t V,
                        float* loss, float* lse, const lce_opts* opts, void* stream);

/*
 * Vocabulary-parallel use (W split by rows over R ranks; each rank holds
 * W_shard = W[vocab_offset : vocab_offset + V_shard], all of H and the global
 * labels). The token-level cross-entropy needs, per token, the log-sum-exp
 * over the whole vocabulary; it is assembled from per-shard statistics with
 * the streaming max / sum-exp rule ("MindSpeed fusion optimisation: principles
 * and practice", section 3.2, applied across vocabulary shards):
 *   1. lce_vshard_forward_stats on each rank -> stats [N, 4] fp32 (device):
 *      (max over the shard, sum of exp(z - max) over the shard, the label's
 *      logit if the label lies in the shard else 0, 1 if it does else 0);
 *   2. the caller gathers the R stats arrays into one [R, N, 4] array in rank
 *      order (an all-gather), and every rank calls lce_vshard_combine ->
 *      lse [N] and loss [1] (merged in rank order: identical on all ranks);
 *   3. lce_vshard_backward on each rank with that lse -> dW_shard
 *      [V_shard, d] (complete for the shard) and dH_partial [N, d] fp32, whose
 *      sum over ranks (an all-reduce) is dH.
 * Labels are global ids in [0, V_total) or ignore_index; the denominator n is
 * the count of valid labels (all ranks see all labels) unless overridden.
 * Workspaces: lce_workspace_size(LCE_OP_FORWARD / LCE_OP_BACKWARD, N, d,
 * V_shard, opts) and (LCE_OP_VSHARD_COMBINE, N, d, V_total, opts).
 * Requirements: 0 <= vocab_offset, vocab_offset + V_shard <= V_total.
 */
int lce_vshard_forward_stats(const void* H, const void* W_shard, const int64_t* y, int64_t N, int64_t d,
                             int64_t V_shard, int64_t vocab_offset, int64_t V_total, float* stats,
                             const lce_opts* opts, void* ws, size_t ws_bytes, void* stream);
int lce_vshard_combine(const float* stats, int64_t R, const int64_t* y, int64_t N, int64_t V_total, float* lse,
                       float* loss, const lce_opts* opts, void* ws, size_t ws_bytes, void* stream);
int lce_vshard_backward(const void* H, const void* W_shard, const int64_t* y, int64_t N, int64_t d, int64_t V_shard,
                        int64_t vocab_offset, int64_t V_total, const float* lse, const float* grad_loss,
                        float* dH_partial, float* dW_shard, const lce_opts* opts, void* ws, size_t ws_bytes,
                        void* stream);

/*
 * Vocabulary-parallel use without recomputing the logits: 6 N V_shard d flops
 * per rank instead of the 8 N V_shard d of the three calls above. Per chunk of
 * rows [c0, c0 + rows) (rows <= the chunk size of opts; c0 = 0 first, chunks
 * in order):
 *   1. lce_vshard_chunk_stats -> stats [rows, 4] fp32, the same statistics as
 *      lce_vshard_forward_stats for those rows; the shard's exp tile
 *      exp(z - m~) (m~: the row's maximum over the shard's first 128 columns)
 *      stays in ws for step 3;
 *   2. the caller all-gathers the R ranks' stats into [R, rows, 4] (rank order);
 *   3. lce_vshard_chunk_backward with that array and the SAME ws (untouched in
 *      between) -> lse rows [c0, c0 + rows) of lse [N], dH_partial rows of
 *      [N, d] fp32 (summed over ranks by the caller: an all-reduce), and
 *      dW_shard [V_shard, d] fp32, written for c0 == 0 (unless
 *      opts->accumulate_dW) and added to for later chunks.
 * The merge in step 3 is lce_vshard_combine's, so the loss of the whole batch
 * is lce_vshard_combine on the gathered statistics of all chunks [R, N, 4].
 * The exp tile is exact only within a range: a chunk where it would exceed its
 * row reference by more than ~e^60 (found in step 1), or where the merged lse
 * of a row whose label lies in this shard exceeds that row's reference by more
 * than 60 nats (found in step 3), gets the exact gradient tile recomputed.
 * Workspace: lce_workspace_size(LCE_OP_VSHARD_CHUNK, N, d, V_shard, opts)
 * (the chunk's exp tile, its statistics and alpha-scaled rows of H).
 * Requirements as for the calls above, and 0 <= c0, 0 <= rows, c0 + rows <= N,
 * 1 <= R <= 4096; stats arrays 16-byte aligned. rows == 0 does nothing.
 */
int lce_vshard_chunk_stats(const void* H, const void* W_shard, const int64_t* y, int64_t N, int64_t d,
                           int64_t V_shard, int64_t vocab_offset, int64_t V_total, int64_t c0, int64_t rows,
                           float* stats, const lce_opts* opts, void* ws, size_t ws_bytes, void* stream);
int lce_vshard_chunk_backward(const void* H, const void* W_shard, const int64_t* y, int64_t N, int64_t d,
                              int64_t V_shard, int64_t vocab_offset, int64_t V_total, int64_t c0, int64_t rows,
                              const float* stats_all, int64_t R, const float* grad_loss, float* lse,
                              float* dH_partial, float* dW_shard, const lce_opts* opts, void* ws, size_t ws_bytes,
                              void* stream);

/*
 * The final zero-centred RMSNorm that produces H ("XTuner on Ascend 910C:
 * Qwen3.5-2B training optimisation", section 3.1.1: one pass over the bf16
 * input with the (1 + w) scale folded into an fp32 gamma and one bf16
 * rounding of the output):
 *   r_i = 1 / sqrt(mean_k x_ik^2 + eps),  H_ik = bf16(x_ik r_i (1 + w_k)).
 * x, H, dH, dx: [N, d] bf16 row-major; w (the zero-centred weight), dw: [d]
 * fp32; rstd: [N] fp32 (r_i, saved by the forward for the backward).
 * d % 8 == 0 and d <= 32768; x, H, dH, dx, w 16-byte aligned.
 * lce_rmsnorm_backward: dx = d(loss)/dx and dw = d(loss)/dw (overwritten) from
 * dH; dw is summed in a fixed order. Its scratch: lce_rmsnorm_workspace_size.
 * lce_norm_fwd_bwd: norm forward -> lce_fwd_bwd on H -> norm backward in one
 * call (H, rstd and dH stay in the workspace, lce_workspace_size with
 * LCE_OP_NORM_FWD_BWD); outputs loss, lse (may be NULL), dx, dw_norm, dW.
 */
size_t lce_rmsnorm_workspace_size(int64_t N, int64_t d);
int lce_rmsnorm_forward(const void* x, const float* w, int64_t N, int64_t d, float eps, void* H, float* rstd,
                        void* stream);
int lce_rmsnorm_backward(const void* x, const float* w, const float* rstd, const void* dH, int64_t N, int64_t d,
                         void* dx, float* dw, void* ws, size_t ws_bytes, void* stream);
int lce_norm_fwd_bwd(const void* x, const float* w_norm, float eps, const void* W, const int64_t* y, int64_t N,
                     int64_t d, int64_t V, const float* grad_loss, float* loss, float* lse, void* dx, float* dw_norm,
                     float* dW, const lce_opts* opts, void* ws, size_t ws_bytes, void* stream);

/* Scale gradients computed for an upstream gradient of 1 by the actual one,
 * in place: dH [N, d] bf16 and dW [V, d] fp32 (either may be NULL) times
 * *grad_loss (device fp32). When *grad_loss == 1 the kernel returns without
 * touching memory. For frameworks whose loss node computes the gradients in
 * its forward pass (as the fused Liger loss does) and receives the upstream
 * gradient only in its backward. No host synchronisation. */
int lce_scale_grads(void* dH, float* dW, int64_t N, int64_t d, int64_t V, const float* grad_loss, void* stream);

/* Synchronise the stream and copy the workspace's device status bits
 * (LCE_DEVICE_*) of the last call that used ws into *flags. */
int lce_read_device_status(const void* ws, void* stream, int* flags);

/* Static, human-readable text for a status code. */
const char* lce_status_string(int status);

/* LCE_VERSION of the built library. */
int lce_version(void);

/*
 * Measurement hook (for benchmarks; off by default). Between
 * lce_profile_begin() and lce_profile_end(), every kernel the library
 * launches is bracketed by two CUDA events recorded on the launch stream, so
 * each kernel's device time is measured where it runs, inside the caller's
 * step. lce_profile_end() synchronises those events and returns, per kernel
 * kind, the number of launches, their summed device time and their summed
 * algorithmic work (bytes for memory-bound kinds, flops for the GEMMs).
 * Every kind is a library kernel except "memset" (dW zeroed by a
 * cudaMemsetAsync when a call has no tokens). Events come from a pool the library owns (created on first use, no device
 * memory is allocated). Not thread-safe: one profiling thread at a time.
 */
#define LCE_KERNEL_KINDS 11
typedef struct lce_profile {
  int32_t launches[LCE_KERNEL_KINDS];
  double ms[LCE_KERNEL_KINDS];      /* summed device time per kind */
  double work[LCE_KERNEL_KINDS];    /* summed algorithmic flops (GEMMs) or bytes (others) */
} lce_profile;

int lce_profile_begin(void);
int lce_profile_end(lce_profile* out);
/* Name of a kernel kind (0 .. LCE_KERNEL_KINDS-1), or NULL. */
const char* lce_kernel_name(int kind);

#ifdef __cplusplus
}
#endif

#endif /* LCE_H_ */
