/*
 * flce.h - C ABI of the fused linear cross-entropy library for GB300 (sm_103a).
 *
 * The operation (source: "Long-Sequence MoE RL Training: From First Principles
 * to MI300X", section 3 "Linear cross-entropy: don't build a 32 GB tensor to
 * get a scalar"): the language-model head forms logits Z = H W^T over
 * [tokens x vocab] and reduces every row through the softmax to a per-token
 * cross-entropy.  The fused method never stores Z: tokens are processed in
 * blocks, each block's logits are formed tile by tile and merged straight
 * into a per-row maximum and sum of exponentials, so a row keeps a handful of
 * scalars.  The backward forms the same logit tiles again, turns them into
 * dZ = softmax(Z) - onehot(target) (scaled by the upstream per-token gradient)
 * and contracts dZ into dH = dZ W and dW = dZ^T H, so no more than a
 * [block x vocab] slice of dZ exists at a time.
 * Section 2.3, Step 1 of "让长序列 MoE RL 训练更好调：Megatron-Lite / bumblebee
 * 的优化实践" describes the same loss as streaming along the vocab dimension.
 *
 * Notation: T tokens, Hd hidden size, V vocabulary size.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers of the current CUDA device and
 *     stay owned by the caller.  The library never allocates device memory:
 *     the caller passes a workspace of at least the size the matching
 *     *_workspace_size() function returns.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL means the legacy default stream).  Outputs are overwritten, never
 *     accumulated into.  Outputs must not overlap one another, the inputs or
 *     the workspace (not checked; overlapping buffers give undefined values).
 *     One workspace serves one call at a time: calls that share a workspace
 *     must be ordered on one stream.
 *   - Argument errors are detected on the host and returned before anything
 *     is launched.  Errors that depend on device data (a target outside
 *     [0, V) that is not ignore_index; a bounded wait inside a kernel that
 *     ran out) are written to a status word at the start of the workspace;
 *     read it with flce_read_device_status().  Each call clears that word
 *     first, so it reports the latest call made with this workspace.  Rows
 *     whose target is out of range are treated as ignored.
 *   - H and W are bf16, row-major: H [T, Hd], W [V, Hd], each row contiguous.
 *     Hd must be a positive multiple of 64; H, W, dH and dW must be 16-byte
 *     aligned; the workspace 256-byte aligned; every other array aligned to
 *     its element type (4 bytes for float, 8 for int64_t).  T may be 0.  V >= 1.
 *     T, V < 2^30.
 *   - Rows whose target equals ignore_index contribute zero loss and zero
 *     gradient and are not counted in n_valid.  ignore_index must lie outside
 *     [0, V).
 *   - Reductions: MEAN = sum over valid rows / n_valid (0 when n_valid == 0),
 *     SUM = sum over valid rows, NONE = one loss per token.
 *   - Results are deterministic: the same inputs and workspace size give
 *     bit-identical outputs on the same device.
 */
#ifndef FLCE_H_
#define FLCE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 1: the first interface.  2: the backward skips rows with a zero upstream
 * weight (its workspace holds the row list and the chunk's H rows),
 * flce_forward_valid, flce_score_valid and flce_backward_workspace_size_for_chunk
 * added, kernel kinds 6-8 added to the timing aid. */
#define FLCE_ABI_VERSION 2

#if defined(__GNUC__)
#define FLCE_API __attribute__((visibility("default")))
#else
#define FLCE_API
#endif

typedef enum flce_status {
  FLCE_OK = 0,
  FLCE_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad reduction, ignore_index in [0, V) */
  FLCE_ERR_UNSUPPORTED = 2,  /* Hd not a multiple of 64, or the device is not sm_103 */
  FLCE_ERR_ALIGNMENT = 3,    /* H, W, dH, dW not 16-byte aligned, the workspace not 256-byte, or a
                                per-token array not aligned to its element type */
  FLCE_ERR_WORKSPACE = 4,    /* workspace missing or smaller than required */
  FLCE_ERR_CUDA = 5,         /* a CUDA runtime / driver call failed; see flce_last_error() */
  FLCE_ERR_TARGET_RANGE = 6, /* device status: a target outside [0, V) and != ignore_index */
  FLCE_ERR_TIMEOUT = 7       /* device status: a bounded wait inside a kernel ran out */
} flce_status;

typedef enum flce_reduction {
  FLCE_REDUCTION_NONE = 0,
  FLCE_REDUCTION_MEAN = 1,
  FLCE_REDUCTION_SUM = 2
} flce_reduction;

/* Bytes of workspace flce_forward() needs for these sizes (>= 256). */
FLCE_API size_t flce_forward_workspace_size(int64_t T, int64_t Hd, int64_t V);

/* Bytes of workspace flce_backward() needs to run with its default token
 * chunk.  The backward skips the rows whose upstream gradient g_t is zero
 * (ignored targets; their dZ rows vanish) and works on chunks of `chunk` of
 * the remaining rows, in token order; the workspace holds one [chunk x V] bf16
 * slice of dZ (the page's [block x vocab] residency), the chunk's rows of H
 * ([chunk x Hd] bf16) and O(T) scalars.  The default chunk is T rounded up to
 * 128 for T <= 256, else min(8192, T/2 rounded down to 128), so for T > 256 and
 * Hd < V/2 the workspace stays below the T*V*2 bytes of one dense bf16 logits
 * tensor.  A larger or smaller workspace is accepted:
 * the backward then uses the largest chunk (a multiple of 128 rows, at least
 * 128) that fits. */
FLCE_API size_t flce_backward_workspace_size(int64_t T, int64_t Hd, int64_t V);

/* Bytes of backward workspace for chunks of `chunk` rows (a positive multiple
 * of 128; chunks above T rounded up to 128 are capped there); 0 for an invalid
 * chunk or size. */
FLCE_API size_t flce_backward_workspace_size_for_chunk(int64_t T, int64_t Hd, int64_t V, int64_t chunk);

/* The token chunk flce_backward() uses with a workspace of `workspace_bytes`;
 * 0 if the workspace is too small. */
FLCE_API int64_t flce_backward_chunk_tokens(int64_t T, int64_t Hd, int64_t V, size_t workspace_bytes);

/* Forward.  Source: "Long-Sequence MoE RL Training: From First Principles to
 * MI300X", section 3 (logits H W^T reduced row-wise through the running-max /
 * log-sum-exp recurrence; loss per token).
 *   H        [T, Hd] bf16              hidden states
 *   W        [V, Hd] bf16              LM-head weight
 *   targets  [T] int64                 class per token, or ignore_index
 *   loss     [1] fp32 (MEAN, SUM) or [T] fp32 (NONE)
 *   lse      [T] fp32                  log sum_v exp(z_{t,v}) on every row
 *   logp     [T] fp32                  z_{t,y_t} - lse_t; 0 on ignored rows
 *   n_valid  [1] int64 or NULL         number of rows with a valid target
 *   workspace, workspace_bytes         >= flce_forward_workspace_size(T, Hd, V)
 * No [T x V] buffer exists at any time. */
FLCE_API flce_status flce_forward(const void* H, const void* W, const int64_t* targets, int64_t T, int64_t Hd,
                                  int64_t V, int64_t ignore_index, int32_t reduction, float* loss, float* lse,
                                  float* logp, int64_t* n_valid, void* workspace, size_t workspace_bytes,
                                  void* stream);

/* Forward for training: the same arguments and results as flce_forward(),
 * except that rows with an ignored target are left out of the contraction
 * altogether (their lse is written as 0; their loss and logp are 0 as always).
 * The rows with a valid target are listed in token order, their rows of H
 * gathered into the workspace, and the logit tiles run over that list only,
 * so masked tokens (padding, prompt prefixes) cost nothing but the copy; loss,
 * logp and the lse of listed rows are bit-identical to flce_forward()'s.  The
 * lse it returns is what flce_backward() needs (the backward reads it only on
 * rows with a non-zero upstream weight, which are valid rows).
 *   workspace, workspace_bytes  >= flce_forward_valid_workspace_size(T, Hd, V)
 *                               (the forward's, plus 8 bytes per token and the
 *                               [T x Hd] bf16 rows of H) */
FLCE_API size_t flce_forward_valid_workspace_size(int64_t T, int64_t Hd, int64_t V);
FLCE_API flce_status flce_forward_valid(const void* H, const void* W, const int64_t* targets, int64_t T, int64_t Hd,
                                        int64_t V, int64_t ignore_index, int32_t reduction, float* loss, float* lse,
                                        float* logp, int64_t* n_valid, void* workspace, size_t workspace_bytes,
                                        void* stream);

/* Backward.  Source: the same page and section (each logit tile is formed
 * again, turned into dZ = softmax - onehot and contracted into dH and dW
 * straight away).
 *   dloss    [1] fp32 (MEAN, SUM) or [T] fp32 (NONE): gradient of the loss output
 *   H, W, targets, T, Hd, V, ignore_index, reduction: as passed to flce_forward
 *   lse      [T] fp32                  the lse output of flce_forward (or flce_forward_valid)
 *                                      for these inputs
 *   dH       [T, Hd] bf16              overwritten with dL/dH (fp32 accumulation, rounded)
 *   dW       [V, Hd] fp32              overwritten with dL/dW, accumulated in fp32 over
 *                                      token chunks in a fixed order
 *   workspace, workspace_bytes         see flce_backward_workspace_size()
 * Per token, the upstream weight is g_t = dloss/n_valid (MEAN), dloss (SUM) or
 * dloss[t] (NONE), and 0 on ignored rows; dZ_{t,v} = g_t (exp(z_{t,v} - lse_t) - [v = y_t]). */
FLCE_API flce_status flce_backward(const float* dloss, const void* H, const void* W, const int64_t* targets,
                                   const float* lse, int64_t T, int64_t Hd, int64_t V, int64_t ignore_index,
                                   int32_t reduction, void* dH, float* dW, void* workspace, size_t workspace_bytes,
                                   void* stream);

/* Backward with a gradient on the logp output as well.  RL trainers build
 * their objective from the per-token log-probabilities (policy-gradient and
 * ratio terms), so the upstream gradient can arrive on logp instead of, or as
 * well as, on the loss.  On valid rows logp_t = -loss_t, so dlogp_t enters the
 * per-token weight as g_t = (gradient of the loss output at t) - dlogp_t.
 *   dloss   as flce_backward, or NULL (no gradient on the loss output)
 *   dlogp   [T] fp32, or NULL (no gradient on logp); ignored rows get g_t = 0
 * Everything else as flce_backward. */
FLCE_API flce_status flce_backward_logp(const float* dloss, const float* dlogp, const void* H, const void* W,
                                        const int64_t* targets, const float* lse, int64_t T, int64_t Hd, int64_t V,
                                        int64_t ignore_index, int32_t reduction, void* dH, float* dW,
                                        void* workspace, size_t workspace_bytes, void* stream);

/* Forward without any allocation by the caller or the library.  The pages
 * have no counterpart to this entry point; it exists for callers that cannot
 * allocate device memory at the point where they need the loss: code whose
 * framework allocator owns all of device memory, plugin hooks of inference or
 * training engines that are not allowed to allocate, and latency-critical
 * paths that forbid allocation.  Such callers pass only inputs and outputs.
 *
 * Arguments and results are those of flce_forward(); instead of a workspace,
 * the call uses a scratch array built into the library: a 32 MiB device array
 * that every GPU which loads the library holds until the process exits.  That
 * limits T to at most 253,952 tokens (any Hd and V); larger T is rejected with
 * FLCE_ERR_WORKSPACE before anything is launched.  The device status word of
 * the call (0, FLCE_ERR_TARGET_RANGE or FLCE_ERR_TIMEOUT) is copied into
 * *device_status (a device int32) unless it is NULL.
 *
 * The first call on a device looks up that device's address of the scratch
 * array (cudaGetSymbolAddress) with the device current; make that first call
 * before any stream capture.  All calls share the one array, and each call
 * overwrites what it needs from it, so calls whose kernels overlap on the GPU
 * (different streams, or different host threads on the same device) race and
 * give wrong results: order them on one stream. */
FLCE_API flce_status flce_forward_noalloc(const void* H, const void* W, const int64_t* targets, int64_t T,
                                          int64_t Hd, int64_t V, int64_t ignore_index, int32_t reduction,
                                          float* loss, float* lse, float* logp, int64_t* n_valid,
                                          int32_t* device_status, void* stream);

/* Scoring: per-token log p(target) and the greedy token, without a loss.
 * Serves comparing a trainer's token log-probabilities with a rollout
 * engine's (the token-level agreement checks of the pages' RL write-ups,
 * e.g. "Long-Sequence MoE RL Training: From First Principles to MI300X"
 * section 1: rollout then train).  Same logit tiles and log-sum-exp
 * recurrence as flce_forward; no reduction.
 *   logp    [T] fp32         z_{t,y_t} - lse_t; 0 on ignored rows
 *   lse     [T] fp32 or NULL
 *   argmax  [T] int64 or NULL  argmax_v z_{t,v} over the fp32-accumulated
 *                              logits, lowest id on ties
 *   workspace >= flce_score_workspace_size(T, Hd, V) */
FLCE_API size_t flce_score_workspace_size(int64_t T, int64_t Hd, int64_t V);
FLCE_API flce_status flce_score(const void* H, const void* W, const int64_t* targets, int64_t T, int64_t Hd, int64_t V,
                                int64_t ignore_index, float* logp, float* lse, int64_t* argmax, void* workspace,
                                size_t workspace_bytes, void* stream);

/* Scoring over the rows with a valid target only: the same arguments and results
 * as flce_score(), except that rows with an ignored target are left out of the
 * contraction (lse 0, logp 0 and argmax -1 there); on every other row lse, logp
 * and argmax are bit-identical to flce_score()'s.  For scoring a rollout's
 * response tokens with the prompt masked.
 *   workspace, workspace_bytes  >= flce_score_valid_workspace_size(T, Hd, V) */
FLCE_API size_t flce_score_valid_workspace_size(int64_t T, int64_t Hd, int64_t V);
FLCE_API flce_status flce_score_valid(const void* H, const void* W, const int64_t* targets, int64_t T, int64_t Hd,
                                      int64_t V, int64_t ignore_index, float* logp, float* lse, int64_t* argmax,
                                      void* workspace, size_t workspace_bytes, void* stream);

/* ---- vocab-parallel split ---------------------------------------------------
 * The vocabulary split into shards of consecutive rows, as when the LM head is
 * tensor-parallel over the vocab ("让长序列 MoE RL 训练更好调：Megatron-Lite /
 * bumblebee 的优化实践", section 2.3 Step 1: a 248,320-row vocab over two ranks
 * gives 124,160 columns per rank).  Each shard reduces its own logit columns to
 * a per-row log-sum-exp; the shards' partials combine exactly as the vocab
 * ranges inside one flce_forward call do (running max / log-sum-exp merge), so
 * the combined results equal flce_forward on the whole vocabulary.  Moving the
 * partials between ranks (an all-gather of 2 floats per token) and summing the
 * dH partials (an all-reduce) are the caller's collectives.
 *
 * Forward of one shard: W_shard [V_shard, Hd] holds global vocab rows
 * [vocab_offset, vocab_offset + V_shard) of a V_total vocabulary.
 *   shard_lse [T] fp32   log sum_{v in shard} exp(z_{t,v})
 *   shard_zy  [T] fp32   z_{t,y_t} when y_t lies in the shard, else 0
 *   workspace            >= flce_forward_workspace_size(T, Hd, V_shard)
 * ignore_index must lie outside [0, V_total). */
FLCE_API flce_status flce_forward_shard(const void* H, const void* W_shard, const int64_t* targets, int64_t T,
                                        int64_t Hd, int64_t V_shard, int64_t vocab_offset, int64_t V_total,
                                        int64_t ignore_index, float* shard_lse, float* shard_zy, void* workspace,
                                        size_t workspace_bytes, void* stream);

/* Bytes of workspace flce_combine_shards() needs (0 if n_shards is outside [1, 64]). */
FLCE_API size_t flce_combine_workspace_size(int64_t T, int32_t n_shards);

/* Combine the partials of n_shards shards (1..64), merged in shard order:
 *   shard_lse, shard_zy  [n_shards, T] fp32 (shard r's rows at offset r*T)
 * Outputs and reductions as flce_forward over the V_total vocabulary; targets
 * outside [0, V_total) that are not ignore_index set FLCE_ERR_TARGET_RANGE in
 * the workspace status word. */
FLCE_API flce_status flce_combine_shards(const float* shard_lse, const float* shard_zy, int32_t n_shards,
                                         const int64_t* targets, int64_t T, int64_t V_total, int64_t ignore_index,
                                         int32_t reduction, float* loss, float* lse, float* logp, int64_t* n_valid,
                                         void* workspace, size_t workspace_bytes, void* stream);

/* Backward of one shard, given the combined lse [T]: dW_shard [V_shard, Hd]
 * fp32 is this shard's rows of dW; dH_partial [T, Hd] bf16 is this shard's
 * term sum_{v in shard} dZ_{t,v} w_v of dH (the shards' partials sum to dH).
 * g_t counts valid rows against the whole vocabulary.  Workspace as
 * flce_backward_workspace_size(T, Hd, V_shard). */
FLCE_API flce_status flce_backward_shard(const float* dloss, const void* H, const void* W_shard,
                                         const int64_t* targets, const float* lse, int64_t T, int64_t Hd,
                                         int64_t V_shard, int64_t vocab_offset, int64_t V_total, int64_t ignore_index,
                                         int32_t reduction, void* dH_partial, float* dW_shard, void* workspace,
                                         size_t workspace_bytes, void* stream);

/* Synchronizes `stream`, then reads the device status word of the latest call
 * made with `workspace` into *out (an flce_status value). */
FLCE_API flce_status flce_read_device_status(const void* workspace, void* stream, int32_t* out);

/* Self-test of the kernels' bounded waits (no counterpart on the pages): one
 * thread waits on an mbarrier that nothing ever completes, with the same
 * bounded wait every GEMM role uses, and writes FLCE_ERR_TIMEOUT to the status
 * word of `workspace` (>= 256 bytes) once `timeout_ns` (1e6 .. 1e10) has
 * passed.  Read it with flce_read_device_status(); the context stays usable. */
FLCE_API flce_status flce_selftest_wait_timeout(void* workspace, uint64_t timeout_ns, void* stream);

/* Human-readable name of a status code (static storage). */
FLCE_API const char* flce_status_string(int32_t status);

/* Text of the last FLCE_ERR_CUDA / argument error raised on this host thread. */
FLCE_API const char* flce_last_error(void);

/* FLCE_ABI_VERSION of the loaded library. */
FLCE_API int32_t flce_abi_version(void);

/* Limit, in nanoseconds, of every bounded wait inside the kernels.  Values
 * below 1e6 are raised to 1e6.  Affects later launches only.  Until this is
 * called the limit of each launch is max(4e9, 16 x K) ns, K being the longest
 * contraction of one output tile in that launch (Hd in the forward and dZ
 * kernels; V for dH tiles and the token chunk for dW tiles), since the longest
 * wait spans one tile's K loop (about 8 SM-pair clocks per unit of K); once it
 * is called, the given value is used for every launch. */
FLCE_API void flce_set_wait_timeout_ns(uint64_t ns);

/* ---- per-kernel timing, a profiling aid ------------------------------------
 * While enabled, every kernel launch of the library is bracketed by CUDA
 * events recorded on its launch stream.  flce_profile_collect() synchronizes
 * on those events and returns, per kernel kind, the launches, the summed
 * device time and the summed algorithmic work (FLOPs and bytes the kernel's
 * mathematics requires, independent of how it is executed).  The backward's
 * work is counted over the rows it does not skip; that count is read from the
 * backward workspace at collection time, so collect while the workspaces of
 * the profiled calls still exist (each reports its latest call). */
typedef struct flce_kernel_stats {
  int32_t kind;     /* flce_kernel_kind value */
  int32_t launches;
  double total_ms;
  double flops;     /* algorithmic FLOPs summed over the launches */
  double bytes;     /* algorithmic DRAM bytes summed over the launches */
} flce_kernel_stats;

typedef enum flce_kernel_kind {
  FLCE_KERNEL_FWD_LOGITS_LSE = 0, /* logit tiles H W^T + running max / sum-exp epilogue */
  FLCE_KERNEL_FWD_FINALIZE = 1,   /* per-row lse / loss / logp and block partial sums */
  FLCE_KERNEL_FWD_REDUCE = 2,     /* fixed-order scalar loss and n_valid */
  FLCE_KERNEL_BWD_PREP = 3,       /* n_valid and the per-token upstream weights g */
  FLCE_KERNEL_BWD_DZ = 4,         /* recomputed logit tiles + dZ epilogue, bf16 dZ chunk */
  FLCE_KERNEL_BWD_DH_DW = 5,      /* dH chunk = dZ W and dW (+)= dZ^T H, one launch per chunk */
  FLCE_KERNEL_BWD_GATHER = 6,     /* the chunk's rows of H gathered through the row list */
  FLCE_KERNEL_BWD_SCATTER = 7,    /* not launched: the dH tiles write their rows straight to their tokens */
  FLCE_KERNEL_FWD_LIST = 8,       /* flce_forward_valid: the list of rows with a valid target */
  FLCE_KERNEL_KINDS = 9
} flce_kernel_kind;

FLCE_API void flce_profile_enable(int32_t on);
/* Fills up to `max_entries` records (one per kind that launched), sets *n_out,
 * and clears the records.  Returns FLCE_ERR_CUDA if an event query fails. */
FLCE_API flce_status flce_profile_collect(flce_kernel_stats* out, int32_t max_entries, int32_t* n_out);
FLCE_API const char* flce_kernel_name(int32_t kind);

#ifdef __cplusplus
}
#endif

#endif /* FLCE_H_ */
