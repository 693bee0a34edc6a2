/*
 * ce.h -- C ABI of libgbce, the fused vocabulary cross-entropy pass for
 * NVIDIA GB300 (sm_103a).
 *
 * One call runs, on one GPU and on the caller's stream, the whole pass the
 * TENPU "Parallel Cross Entropy (Triton)" issue (Ascend/TransformerEngineNPU
 * #29) describes in its section 1 "Interface":
 *
 *     loss = parallel_cross_entropy(inp, target, label_smoothing, reduce_loss,
 *                                   dist_process_group, ignore_idx)
 *
 *   - inp: logits (B,SQ,V) or (SQ,B,V), FP32 / BF16 (FP16 also accepted);
 *   - target: (B,SQ) or (SQ,B), global vocabulary indices (int64 here);
 *   - softmax and loss accumulate in FP32, the loss is FP32, the gradient is
 *     written back in the input dtype (same section), in place over the
 *     logits (section 6 "Memory": in-place gradient staging);
 *   - loss of a row = logsumexp(x) - x[target] (CSDN "Ascend CANN ops-nn
 *     cross-entropy fusion: from three kernel launches to one", section
 *     "Fusion scheme: log_softmax + NLL"), with PyTorch-style label smoothing
 *     (1-a)*nll + a*mean_j(-log_softmax_j);
 *   - gradient of a row = (softmax - (1-a)*onehot(target) - a/V) * dloss
 *     (same article, section "Backward" and pitfall 3, with the smoothing mass
 *     spread over all V classes as torch F.cross_entropy does);
 *   - rows whose target equals ignore_idx (default -100) get loss 0 and a
 *     zero gradient and are left out of the mean (TENPU #29 section 1;
 *     mindspore/hyper-parallel #269 section 3.1);
 *   - reduce_loss: the mean over kept rows, produced on the device by a
 *     fixed-order reduction (TENPU #29 counts n_non_ignore on the host,
 *     section 7 "Known limitations"; here the count runs on the device).
 *
 * dist_process_group has no counterpart: the vocabulary-parallel combine of
 * (max, sum-exp, target logit) that hyper-parallel #269 section 3.1 runs as
 * MAX/SUM all-reduces plus a gather runs here between vocabulary chunks of
 * one GPU (thread-block clusters over distributed shared memory, or a second
 * kernel).
 *
 * Conventions for every entry point:
 *   - every pointer argument is a DEVICE pointer unless it says "host";
 *   - the caller owns all memory; the library allocates nothing, keeps no
 *     pointer after the call returns and never synchronises the stream
 *     (ce_get_error excepted);
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream); all work is enqueued on it in order;
 *   - dims: the logits have shape (dim0, dim1, V); (B,SQ,V) and (SQ,B,V)
 *     differ only in which of dim0/dim1 is the batch; row (i, j) is the
 *     flattened row r = i*dim1 + j; element (i, j, v) sits at
 *     logits + (i*strides[0] + j*strides[1] + v*strides[2]) elements;
 *     strides[2] must be 1 (non-unit vocabulary stride: make the tensor
 *     contiguous first, as TENPU #29 "Problems and solutions" does);
 *   - targets: int64, target of row (i, j) at targets[i*target_strides[0] +
 *     j*target_strides[1]];
 *   - logits (and a separate gradient) must sit on a multiple of their element
 *     size (CE_ERR_INVALID_ARG otherwise); rows need no further alignment:
 *     rows on the 16-byte grid take the TMA kernels, others 16-byte loads
 *     between a scalar head and tail (CE_PATH_VECROW, the two-stage kernels,
 *     ce_bwd, ce_vp_partials);
 *   - errors found on the host are returned before anything is launched;
 *     a target outside [0, V) that is not ignore_idx is found on the device:
 *     that row gets loss NaN and a zero gradient, and the device error word
 *     in the workspace gets CE_DEVERR_TARGET_RANGE (read it with
 *     ce_get_error).  Kernels never trap.
 */
#ifndef GBCE_CE_H
#define GBCE_CE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { CE_F32 = 0, CE_BF16 = 1, CE_F16 = 2 } ce_dtype;

/* (B,SQ,V): dim0 = B, dim1 = SQ.  (SQ,B,V): dim0 = SQ, dim1 = B. */
typedef enum { CE_LAYOUT_BSV = 0, CE_LAYOUT_SBV = 1 } ce_layout;

typedef enum {
    CE_OK = 0,
    CE_ERR_INVALID_ARG = 1,        /* null pointer, bad size, smoothing outside [0,1],
                                      logits off their element size, ... */
    CE_ERR_UNSUPPORTED_DTYPE = 2,
    CE_ERR_BAD_STRIDE = 3,         /* strides[2] != 1, a negative stride, or (ce_fwd_bwd)
                                      rows that share memory */
    CE_ERR_WORKSPACE_TOO_SMALL = 4,
    CE_ERR_LAUNCH = 5,             /* a CUDA launch or attribute call failed */
    CE_ERR_TARGET_RANGE = 6,       /* reported by ce_get_error only */
    CE_ERR_DEVICE_TIMEOUT = 7,     /* reported by ce_get_error only */
    CE_ERR_UNSUPPORTED_PATH = 8    /* a forced path cannot run this shape */
} ce_status;

/* Bits of the device error word (ce_get_error). */
#define CE_DEVERR_TARGET_RANGE 0x1u
#define CE_DEVERR_TIMEOUT 0x2u     /* a bounded wait inside a kernel gave up */

typedef enum {
    CE_PATH_AUTO = 0,
    CE_PATH_ROW = 1,       /* one CTA holds a whole row in shared memory and registers */
    CE_PATH_CLUSTER = 2,   /* a thread-block cluster splits each row; combine over DSMEM */
    CE_PATH_TWO_STAGE = 3, /* per-chunk statistics kernel, then combine + gradient kernel */
    CE_PATH_STREAM = 4,    /* one CTA streams whole rows twice through a TMA ring (rows
                              claimed from a counter in the workspace); the second read
                              of a row is served by L2, or for rows of at least twice
                              the ring by the ring's last tiles still in shared memory.
                              Default shape: rows up to 128 KB 16 KB tiles, 6 deep, two
                              CTAs per SM; wider rows 32 KB tiles, 6 deep, one CTA.
                              Rows off the 16-byte grid (the default for such rows over
                              32 KB): the ring takes each row's aligned body, and the at
                              most 2 (16/sizeof(T) - 1) elements before and after it are
                              read and written one per thread (256 consuming threads).
                              A vocabulary split (num_vocab_chunks = K, the default path
                              for a split of aligned rows into at most 32 non-empty
                              chunks; 16 KB tiles, two CTAs per SM): each chunk streams
                              as its own run of tiles with the warps' running max shared,
                              the
                              chunks' (max, sum-exp, sum, target logit) partials are
                              combined in chunk order (256 consuming threads) */
    CE_PATH_WARP = 5,      /* one warp per row, the row held in one shared-memory tile
                              (rows up to 32 KB) */
    CE_PATH_VECROW = 6     /* rows off the 16-byte grid (any alignment): a persistent
                              grid, two passes of plain 16-byte loads per row between a
                              scalar head and tail, the second served by L2; a warp per
                              row up to 32 KB, else a CTA per row (512 threads two per
                              SM, rows over 320 KB 1024 threads one per SM); no
                              vocabulary split, no class weights */
} ce_path;

typedef struct {
    int force_path;         /* ce_path; CE_PATH_AUTO lets the planner choose */
    int num_vocab_chunks;   /* 0: planner chooses; K > 0: cut V into K contiguous
                               chunks of ceil(V/K) (rounded up to 16 bytes on the
                               row, cluster and stream paths, so fewer chunks may be
                               non-empty) whose partials are combined on the device:
                               the stream path for aligned rows cut into up to 32
                               non-empty chunks, else the two-stage path (the
                               cluster path when forced, up to 16 chunks) */
    void* event_begin;      /* cudaEvent_t or NULL: recorded on `stream` right
                               before the main kernel of the pass */
    void* event_end;        /* cudaEvent_t or NULL: recorded right after it */
    int tune_threads;       /* 0 = default; otherwise CTA size (256 or 512; on the stream
                               path the number of consuming threads); CE_PATH_VECROW
                               also takes 1024 (one CTA per SM) and 32 (a row per warp),
                               which the stream, row and cluster paths refuse */
    int tune_stages;        /* 0 = default; otherwise TMA pipeline depth (2..4 rows on the
                               row/cluster paths, 2..12 tiles on the stream path, 6 or 12
                               tiles on the warp path: 12 = two tiles per consumer warp,
                               the default for 16 KB tiles from 8192 rows on) */
    int tune_ctas_per_sm;   /* 0 = as many as fit; otherwise a cap */
    int tune_l2_keep;       /* stream path: 0 = default (1), 1 = the first read asks L2 to
                               keep the row for the second (evict-last), 2 = evict-first */
    int tune_tile_kb;       /* stream and warp paths: 0 = default, else the ring tile size
                               (16 or 32 KB) */
    const float* class_weights; /* NULL, or device float32[V]: per-class weights as in
                               torch F.cross_entropy(weight=...): the smoothed target's
                               class j term is weighted by w_j and the mean divides by
                               the summed weight of the kept rows' targets.  Runs on the
                               stream path when the rows and this vector are 16-byte
                               aligned and no vocabulary split is asked for (256
                               consuming threads), else on the two-stage path;
                               CE_PATH_ROW, CE_PATH_CLUSTER and CE_PATH_WARP are refused
                               with CE_ERR_UNSUPPORTED_PATH (ce_fwd_bwd, ce_fwd_only;
                               not ce_bwd) */
    int reserved[2];        /* must be zero */
} ce_options;

/* Bytes of device workspace a call with these sizes needs (either entry
 * point, any path, reduce_loss or not).  Host only; returns 0 for invalid
 * sizes.  opts may be NULL. */
size_t ce_workspace_bytes(int64_t dim0, int64_t dim1, int64_t V, ce_dtype dtype,
                          const ce_options* opts);

/* Forward and backward in one pass.
 *   logits          (dim0, dim1, V) in `dtype`; read, then overwritten with the
 *                   gradient (grad_inplace must equal logits).
 *   label_smoothing a in [0, 1].
 *   ignore_idx      target value that marks a row as ignored (usually -100).
 *   reduce_loss     0: per-row losses; 1: mean over rows whose target is not
 *                   ignore_idx.
 *   dloss           float32 upstream gradient: one value (reduce_loss = 1; the
 *                   gradient of the mean, each kept row is scaled by dloss/n)
 *                   or one value per flattened row (reduce_loss = 0); NULL
 *                   means 1.
 *   loss_out        float32: one value (reduce_loss = 1; NaN when every row is
 *                   ignored) or dim0*dim1 values in flattened row order.
 *   n_non_ignore_out  int64 count of rows whose target != ignore_idx, or NULL.
 *   workspace       at least ce_workspace_bytes(...) bytes, 256-byte aligned;
 *                   its contents need no initialisation and must not be
 *                   shared by calls that may run concurrently.
 *   opts            NULL for defaults.
 * Returns CE_OK once every kernel is enqueued. */
ce_status ce_fwd_bwd(void* logits, ce_dtype dtype, ce_layout layout, int64_t dim0, int64_t dim1,
                     int64_t V, const int64_t strides[3], const int64_t* targets,
                     const int64_t target_strides[2], float label_smoothing, int64_t ignore_idx,
                     int reduce_loss, const float* dloss, float* loss_out, void* grad_inplace,
                     int64_t* n_non_ignore_out, void* workspace, size_t workspace_bytes,
                     const ce_options* opts, void* stream);

/* Forward only: the logits are read, never written.  Same arguments as
 * ce_fwd_bwd minus dloss and the gradient, plus
 *   lse_out   float32 logsumexp of every row (NaN for ignored or out-of-range
 *             rows), or NULL. */
ce_status ce_fwd_only(const void* logits, ce_dtype dtype, ce_layout layout, int64_t dim0,
                      int64_t dim1, int64_t V, const int64_t strides[3], const int64_t* targets,
                      const int64_t target_strides[2], float label_smoothing, int64_t ignore_idx,
                      int reduce_loss, float* loss_out, float* lse_out, int64_t* n_non_ignore_out,
                      void* workspace, size_t workspace_bytes, const ce_options* opts,
                      void* stream);

/* Backward only, from the logsumexp a forward-only pass saved: for callers
 * that learn the upstream gradient after the forward (autograd).  Writes
 *   grad_j = g * (exp(x_j - lse) - a/V) - g * (1-a) * [j == target]
 * for every kept row (CSDN "Ascend CANN ops-nn cross-entropy fusion",
 * section "Backward", pitfall 3; smoothing over all V classes) and zeros for
 * ignored or out-of-range rows; g = dloss[0] / n_non_ignore (reduce_loss) or
 * dloss[row] (otherwise; NULL means 1).
 *   logits, targets, sizes, strides, label_smoothing, ignore_idx: as given to
 *                  ce_fwd_only; the logits must be unchanged since then.
 *   lse            float32 per flattened row, from ce_fwd_only's lse_out.
 *   n_non_ignore   int64 count from ce_fwd_only's n_non_ignore_out; required
 *                  when reduce_loss.
 *   grad           gradient in the logits dtype with its own strides
 *                  (grad_strides[2] == 1): either the logits themselves (same
 *                  strides; the TENPU in-place staging) or memory that does
 *                  not overlap them.
 * One read of the logits and one write of the gradient per element; no
 * workspace.  Returns CE_OK once the kernel is enqueued on `stream`. */
ce_status ce_bwd(const void* logits, ce_dtype dtype, ce_layout layout, int64_t dim0, int64_t dim1,
                 int64_t V, const int64_t strides[3], const int64_t* targets,
                 const int64_t target_strides[2], const float* lse, float label_smoothing,
                 int64_t ignore_idx, int reduce_loss, const float* dloss,
                 const int64_t* n_non_ignore, void* grad, const int64_t grad_strides[3],
                 void* stream);

/* Vocabulary-parallel cross-entropy (mindspore/hyper-parallel #269, section
 * 3.1: each tensor-parallel rank holds a ceil(V/tp) slice of the vocabulary;
 * per-row (max, sum-exp) statistics of the slice, a MAX all-reduce and a SUM
 * all-reduce of the rescaled sums and a gather of the target logit -- TENPU
 * #29 section 6's m_d_Xy gather -- then a backward without collectives).  The
 * three calls below are the three steps; a caller with one GPU runs them over
 * vocabulary shards held as separate tensors, a caller with several ranks
 * would all-gather the partials between steps 1 and 2.
 *
 * Step 1: statistics of one shard.
 *   shard_logits   (dim0, dim1, V_shard) columns [vocab_offset, vocab_offset +
 *                  V_shard) of the vocabulary; strides as for ce_fwd_bwd.
 *   targets        global vocabulary indices, as for ce_fwd_bwd.
 *   partials       float32 [dim0*dim1][4], 16-byte aligned: per flattened row
 *                  {max, sum of exp(x - max), sum of x, target logit if the
 *                  target lies in this shard else 0}; ignored rows get
 *                  {-inf, 0, 0, 0}. */
ce_status ce_vp_partials(const void* shard_logits, ce_dtype dtype, int64_t dim0, int64_t dim1,
                         int64_t V_shard, const int64_t strides[3], const int64_t* targets,
                         const int64_t target_strides[2], int64_t vocab_offset, int64_t ignore_idx,
                         float* partials, void* stream);

/* Step 2: combine the partials of all shards, in shard order.
 *   partials       num_shards consecutive blocks of [dim0*dim1][4] (shard k's
 *                  block k), 1 <= num_shards <= 64.
 *   shard_offsets  HOST array of num_shards + 1 increasing column offsets:
 *                  shard k covers [shard_offsets[k], shard_offsets[k+1]);
 *                  shard_offsets[0] = 0, shard_offsets[num_shards] = V.
 *   loss_out, reduce_loss, n_non_ignore_out, workspace: as for ce_fwd_bwd
 *                  (workspace of ce_workspace_bytes(dim0, dim1, V, dtype, NULL)).
 *   lse_out        float32 logsumexp per flattened row (required: step 3 needs
 *                  it); NaN for ignored or out-of-range rows.
 * Out-of-range targets set CE_DEVERR_TARGET_RANGE in the workspace. */
ce_status ce_vp_combine(const float* partials, int num_shards, const int64_t* shard_offsets,
                        int64_t dim0, int64_t dim1, const int64_t* targets,
                        const int64_t target_strides[2], float label_smoothing, int64_t ignore_idx,
                        int reduce_loss, float* loss_out, float* lse_out,
                        int64_t* n_non_ignore_out, void* workspace, size_t workspace_bytes,
                        void* stream);

/* Step 3: the gradient of one shard from the combined lse -- ce_bwd for the
 * columns [vocab_offset, vocab_offset + V_shard) of a V_total vocabulary (the
 * smoothing share is a / V_total; the one-hot term lands in the shard that
 * holds the target).  Other arguments as for ce_bwd. */
ce_status ce_vp_bwd(const void* shard_logits, ce_dtype dtype, int64_t dim0, int64_t dim1,
                    int64_t V_shard, const int64_t strides[3], const int64_t* targets,
                    const int64_t target_strides[2], int64_t vocab_offset, int64_t V_total,
                    const float* lse, float label_smoothing, int64_t ignore_idx, int reduce_loss,
                    const float* dloss, const int64_t* n_non_ignore, void* grad,
                    const int64_t grad_strides[3], void* stream);

/* lm_head + cross-entropy, chunked over token rows (the sequence-chunked
 * lm_head + loss of the TorchTitan ChunkedLossWrapper that hyper-parallel
 * #269 describes: the full (N, V) logits never exist).  For each chunk of
 * chunk_rows rows: logits = hidden . weight^T into the workspace -- for
 * bf16 / fp16 with H a multiple of 8 and 16-byte aligned hidden and weight,
 * this library's tcgen05 GEMM, whose epilogue also folds every (row,
 * 256-column tile) into softmax statistics that a per-row combine turns into
 * lse and the loss, then the backward from lse writes the gradient in place;
 * otherwise a cuBLAS GEMM and this library's fused pass -- scaled with the
 * kept-row count of the whole batch; then grad_hidden = dlogits . weight and
 * grad_weight += dlogits^T . hidden (cuBLAS GEMMs, fp32 accumulation).
 * GBCE_LINEAR_GEMM=library in the environment (read once, at the first
 * call) takes the cuBLAS branch for every dtype and shape, for comparison.
 *   hidden       (N, H) row-major, dtype; weight (V, H) row-major, dtype.
 *   targets      int64 [N], contiguous.
 *   loss_out     one value (reduce_loss) or N values.
 *   grad_hidden  (N, H) row-major, dtype, written; or NULL.
 *   grad_weight  (V, H) row-major float32, ACCUMULATED into (zero it first for
 *                a fresh gradient); or NULL.
 *   workspace    ce_linear_workspace_bytes(N, H, V, dtype, chunk_rows) bytes,
 *                256-byte aligned; it holds one chunk of logits (rows padded
 *                to a multiple of 8 elements), their statistics and cuBLAS's
 *                workspace.  cuBLAS creates one handle per host thread and
 *                device on first use (its own small allocation).
 * Returns CE_OK once every kernel and GEMM is enqueued on `stream`. */
size_t ce_linear_workspace_bytes(int64_t N, int64_t H, int64_t V, ce_dtype dtype,
                                 int64_t chunk_rows);
ce_status ce_linear_fwd_bwd(const void* hidden, const void* weight, ce_dtype dtype, int64_t N,
                            int64_t H, int64_t V, const int64_t* targets, float label_smoothing,
                            int64_t ignore_idx, int reduce_loss, const float* dloss,
                            float* loss_out, void* grad_hidden, float* grad_weight,
                            int64_t* n_non_ignore_out, int64_t chunk_rows, void* workspace,
                            size_t workspace_bytes, void* stream);

/* ce_fwd_bwd without a workspace argument: the pass keeps its scratch in a
 * fixed 2 MiB array of device memory that the library itself reserves on
 * every GPU where it is loaded (held until the process exits).  The pages have
 * no counterpart of this entry point; it exists for callers that must not
 * allocate device memory for a call: runtimes that plan every byte of device
 * memory before they start and give custom operators no workspace, and
 * latency-critical loops where cudaMalloc (which may synchronise the device or
 * fail on a fragmented heap) is not acceptable.  The caller still passes the
 * logits, targets and outputs, as for ce_fwd_bwd; this call allocates nothing.
 *
 * Limit: the scratch must hold 256 bytes + 4*dim0*dim1 bytes rounded up to
 * 256 (per-row losses), plus 16*dim0*dim1*K bytes rounded up to 256 when the
 * planner takes the two-stage path with K chunks.  Larger problems are
 * rejected with CE_ERR_WORKSPACE_TOO_SMALL before anything is launched
 * (about 520,000 rows on the row, cluster, stream, warp and plain-load
 * paths).
 *
 * Set-up: the first call on a device looks up the scratch's device address
 * with that device current (the caller's current device); make that first
 * call before any stream capture.  No part of the scratch needs clearing:
 * every pass writes what it later reads.  All calls on a device share the one
 * array and it keeps the last call's contents, so calls that may overlap on
 * the GPU (different streams, or threads enqueuing at once) race on it:
 * serialise them.  The error word lives in that internal scratch, so
 * ce_get_error cannot read it; ce_noalloc_get_error (below) reads it
 * instead.  Out-of-range targets also show as NaN row losses; a bounded wait
 * inside a kernel that gave up (CE_DEVERR_TIMEOUT, see ce_wait_timeout_probe)
 * shows only there: the call has already returned CE_OK, and some loss and
 * gradient rows may be left unwritten. */
ce_status ce_fwd_bwd_noalloc(void* logits, ce_dtype dtype, ce_layout layout, int64_t dim0,
                             int64_t dim1, int64_t V, const int64_t strides[3],
                             const int64_t* targets, const int64_t target_strides[2],
                             float label_smoothing, int64_t ignore_idx, int reduce_loss,
                             const float* dloss, float* loss_out, void* grad_inplace,
                             int64_t* n_non_ignore_out, const ce_options* opts, void* stream);

/* ce_get_error for ce_fwd_bwd_noalloc: waits for `stream`, then copies the
 * error word of the last no-alloc pass on the current device (the one its
 * fixed scratch array holds) into *host_err (host pointer) and decodes it as
 * ce_get_error does.  Serialise it with the no-alloc passes like they are
 * serialised with each other: a pass enqueued on another stream meanwhile
 * rewrites the word.  Returns CE_ERR_INVALID_ARG if host_err is NULL,
 * CE_ERR_LAUNCH if the scratch's address cannot be looked up or the copy
 * fails. */
ce_status ce_noalloc_get_error(void* stream, uint32_t* host_err);

/* Waits for `stream`, then copies the device error word of the last pass that
 * used `workspace` into *host_err (host pointer).  Returns CE_OK,
 * CE_ERR_TARGET_RANGE or CE_ERR_DEVICE_TIMEOUT from its bits, CE_ERR_LAUNCH if
 * the copy fails.  Diagnostic use: this is the only call that synchronises. */
ce_status ce_get_error(const void* workspace, void* stream, uint32_t* host_err);

/* Failure detection check (no counterpart on the pages).  Every wait inside
 * this library's kernels -- on a TMA copy landing, on a ring slot, on a row
 * handed between warps -- is bounded: after ~1.5 s it gives up, sets
 * CE_DEVERR_TIMEOUT in the workspace error word and lets the kernel return,
 * so a lost copy is reported instead of hanging the GPU.  This call runs that
 * same bounded wait once, in a one-thread kernel, on an mbarrier that nothing
 * arrives on, and writes the result as the error word of `workspace`
 * (>= 256 bytes, 16-byte aligned): ce_get_error then returns
 * CE_ERR_DEVICE_TIMEOUT after ~1.5 s, and the stream stays usable.  Returns
 * CE_OK once the kernel is enqueued, CE_ERR_INVALID_ARG for a bad workspace. */
ce_status ce_wait_timeout_probe(void* workspace, size_t workspace_bytes, void* stream);

/* Static English description of a status code. */
const char* ce_status_string(ce_status status);

/* Path the planner would take for these arguments (host only): CE_PATH_ROW,
 * CE_PATH_CLUSTER, CE_PATH_TWO_STAGE, CE_PATH_STREAM, CE_PATH_WARP or
 * CE_PATH_VECROW, with the vocabulary chunk count in *chunks_out (host
 * pointer, may be NULL).  Returns -1 for arguments
 * ce_fwd_bwd would reject, -2 for a forced path that cannot run them. */
int ce_plan_path(const void* logits, ce_dtype dtype, int64_t dim0, int64_t dim1, int64_t V,
                 const int64_t strides[3], const ce_options* opts, int* chunks_out);

#ifdef __cplusplus
}
#endif

#endif /* GBCE_CE_H */
