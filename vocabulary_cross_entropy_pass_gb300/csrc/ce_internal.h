// ce_internal.h -- host-side structures shared by the C-ABI layer and the
// kernel launchers of libgbce.  Not part of the public interface.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/ce.h"

namespace gbce {

// Workspace layout (byte offsets from the caller's workspace pointer):
//   [0, 4)      uint32 device error word
//   [8, 16)     int64 n_non_ignore of the last pass
//   [16, 20)    uint32 count of CTAs done (the stream kernel's in-kernel mean)
//   [24, 32)    double summed class weight of the kept rows' targets (weighted pass)
//   [32, 40)    double summed class weight over the vocabulary (weighted pass)
//   [40, 44)    uint32 rows claimed beyond each CTA's first two (stream kernel)
//   [44, 48)    uint32 CTAs done claiming (the last one zeroes both words)
//   [256, ...)  float per-row losses (N) -- used when reduce_loss
//   [...]       float4 per-(row, chunk) partials of the two-stage path
constexpr size_t kWsErrOffset = 0;
constexpr size_t kWsCountOffset = 8;
constexpr size_t kWsTicketOffset = 16;
constexpr size_t kWsWeightDenomOffset = 24;
constexpr size_t kWsWeightSumOffset = 32;
constexpr size_t kWsRowClaimOffset = 40;
constexpr size_t kWsRowDoneOffset = 44;
constexpr size_t kWsHeaderBytes = 256;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Problem {
    char* logits;              // byte address of element (0,0,0)
    int dtype;                 // ce_dtype
    int es;                    // element size in bytes
    int64_t dim0, dim1, N, V;
    int64_t s0, s1;            // element strides of dims 0 and 1
    const int64_t* targets;
    int64_t ts0, ts1;
    float a;                   // label smoothing
    int64_t ignore_idx;
    int reduce;
    const float* dloss;
    float* loss_rows;          // per-row loss destination (loss_out or workspace)
    float* lse_out;            // optional
    bool grad;                 // write the gradient in place
    uint32_t* err;             // device error word
    int64_t* n_dev;            // device count
    uint32_t* ticket;          // CTAs-done counter, zeroed by the count kernel
    float* mean_out;           // stream path with reduce_loss: the mean, written in-kernel
    const float* cw;           // class weights [V] or NULL
    double* wdenom;            // summed weight of kept targets (weighted pass)
    double* wsum;              // summed weight over the vocabulary (weighted pass)
    uint32_t* row_claim;       // stream kernel: shared row counter (NULL: static rows)
    uint32_t* row_done;        // stream kernel: CTAs done claiming
};

// Rows and targets laid out so that flattened row r sits at r * s1 and its
// target at r * ts1 (s0 = dim1 * s1, ts0 = dim1 * ts1: every contiguous
// (B,SQ,V) or (SQ,B,V) tensor; or dim0 = 1, where r = j): the kernels then
// skip the 64-bit division r / dim1 per row.
inline bool rows_flat(const Problem& p) {
    const int64_t lim = (int64_t)1 << 31;
    if (p.dim1 < 1 || p.dim1 >= lim || p.s1 < 0 || p.s1 >= lim || p.ts1 < 0 || p.ts1 >= lim) return false;
    return p.dim0 == 1 || (p.s0 == p.dim1 * p.s1 && p.ts0 == p.dim1 * p.ts1);
}

// Plan of the fused (row / cluster) kernel.
struct FusedPlan {
    int threads;               // 256 or 512
    int cluster;               // CTAs per row (1 = row path)
    int chunk;                 // elements per CTA slice, multiple of the 16-byte vector
    int stages;                // TMA pipeline depth
    int ctas_per_sm_cap;       // 0 = no cap
};

// Row geometries of the row-streaming kernel: rows on the 16-byte grid;
// rows anywhere (an aligned body through the ring, a scalar head and tail);
// rows cut into vocabulary chunks whose partials are combined in order.
constexpr int kStreamAligned = 0;
constexpr int kStreamEdges = 1;
constexpr int kStreamChunks = 2;
constexpr int kMaxStreamChunks = 32;  // chunks per row the stream kernel combines

// Plan of the row-streaming kernel.
struct StreamPlan {
    int threads;               // consumer threads: 256 or 512
    int tile_kb;               // ring tile size: 16 or 32 KB
    int stages;                // ring depth in tiles
    int ctas_per_sm_cap;       // 0 = no cap
    int l2_keep;               // 1: first-pass copies use an L2 evict-last policy
    int geo;                   // kStreamAligned / kStreamEdges / kStreamChunks
    int64_t chunk_elems;       // kStreamChunks: elements per chunk (16-byte multiple)
    int nchunks;               // kStreamChunks: non-empty chunks, <= kMaxStreamChunks
};

// Plan of the warp-per-row kernel (rows that fit one shared-memory tile).
struct RowsPlan {
    int tile_kb;               // 16 or 32
    int stages;                // ring depth in tiles
    int ctas_per_sm_cap;       // 0 = no cap
};

// Plan of the kernel for rows off the 16-byte grid.
struct VecRowPlan {
    int threads;               // a row per CTA: 512 (two CTAs per SM), 256 (three), 1024 (one)
    bool warp_rows;            // a row per warp instead (512-thread CTAs, two per SM)
    int ctas_per_sm_cap;       // 0 = no cap
};

// Plan of the two-stage kernels.
struct SplitPlan {
    int chunks;                // K
    int64_t chunk;             // elements per chunk (ceil(V/K))
};

// The backward from a saved logsumexp.
struct BwdProblem {
    const char* logits;
    char* grad;
    int dtype;
    int64_t dim1, N, V;
    int64_t s0, s1, gs0, gs1;  // element strides of logits and gradient rows
    const int64_t* targets;
    int64_t ts0, ts1, ignore_idx;
    const float* lse;
    float a;
    int reduce;
    const float* dloss;
    const int64_t* n_dev;
    bool vec_ok;               // gradient rows at the logits rows' offset from 16 bytes
    int64_t vocab_offset;      // global index of column 0 (a vocabulary shard), else 0
    int64_t V_total;           // vocabulary size the targets index, else V
};

// Vocabulary-parallel partials of one shard.
constexpr int kVpMaxShards = 64;
struct VpPartProblem {
    const char* logits;
    int dtype;
    int64_t s0, s1, dim1, N, V, vocab_offset;
    const int64_t* targets;
    int64_t ts0, ts1, ignore_idx;
    float4* part;
};
struct VpCombineProblem {
    const float4* part;
    int R;
    const int64_t* off;        // host, R + 1 entries
    int64_t dim1, N;
    const int64_t* targets;
    int64_t ts0, ts1, ignore_idx;
    float a;
    float* loss;
    float* lse;
};

int elem_size(int dtype);
bool fused_aligned(const Problem& p);
int fused_capacity(int dtype, int threads);  // elements one CTA can hold
int split_auto_chunks(int64_t V);

cudaError_t launch_count(const Problem& p, int64_t* n_out, cudaStream_t s);
// one bounded mbarrier wait that runs out; writes the error word
cudaError_t launch_wait_probe(uint32_t* err, cudaStream_t s);
// the count kernel and the pass after it overlap (programmatic dependent launch)
void set_pdl_attr(cudaLaunchAttribute* attr);
cudaError_t launch_reduce_mean(const Problem& p, float* loss_out, cudaStream_t s);
cudaError_t launch_fused(const Problem& p, const FusedPlan& plan, cudaStream_t s);
cudaError_t launch_stream(const Problem& p, const StreamPlan& plan, cudaStream_t s);
// rows with a scalar head and tail, or cut into chunks (partials: per-(row,
// chunk) {m, d, S, x_y}, N * plan.nchunks of them, or NULL)
cudaError_t launch_stream_geo(const Problem& p, const StreamPlan& plan, float4* partials,
                              cudaStream_t s);
cudaError_t launch_rows(const Problem& p, const RowsPlan& plan, cudaStream_t s);
cudaError_t launch_vecrow(const Problem& p, const VecRowPlan& plan, cudaStream_t s);
cudaError_t launch_bwd(const BwdProblem& bp, cudaStream_t s);
cudaError_t launch_vp_partials(const VpPartProblem& vp, cudaStream_t s);
cudaError_t launch_vp_combine(const VpCombineProblem& vc, cudaStream_t s);
cudaError_t launch_split(const Problem& p, const SplitPlan& plan, float4* partials,
                         cudaStream_t s);

// lm_head logits of one chunk of rows on the tensor cores (ce_lmhead.cu), with
// the cross-entropy statistics of every (row, 256-column tile) in the GEMM's
// epilogue, then combined per row into lse and the row's loss.
struct LmHeadProblem {
    const void* hidden;        // (rows, H) row-major, 16-byte aligned
    const void* weight;        // (V, H) row-major, 16-byte aligned
    int dtype;                 // CE_BF16 or CE_F16
    int64_t rows, H, V;
    int64_t ldl;               // elements between rows of the logits output (multiple of 8)
    void* logits;              // out: (rows, ldl), the logits rounded to the dtype
    float4* part;              // scratch: [rows][ceil(V/256)] {m, d, S, x_y}
    const int64_t* targets;    // [rows], contiguous
    int64_t ignore_idx;
    float a;                   // label smoothing
    float* loss_rows;          // out: per-row loss (0 ignored, NaN out of range)
    float* lse;                // out: per-row logsumexp (NaN ignored / out of range)
    uint32_t* err;             // device error word
};
bool lmhead_supported(int dtype, int64_t H, int64_t V, const void* hidden, const void* weight);
size_t lmhead_part_bytes(int64_t rows, int64_t V);
int64_t lmhead_ldl(int64_t V);
cudaError_t launch_lmhead(const LmHeadProblem& lp, cudaStream_t s);

// Used by the lm_head + cross-entropy orchestration (ce_linear.cu).
cudaError_t launch_main_pass(Problem& pb, const ce_options* o, float4* partials, size_t partial_bytes,
                             cudaStream_t s);
size_t partial_bytes_for(int64_t N, int64_t V);
void problem_init(Problem& pb, const void* logits, int dtype, int64_t dim0, int64_t dim1, int64_t V,
                  const int64_t* strides, const int64_t* targets, const int64_t* tstrides, float a,
                  int64_t ignore_idx, int reduce);

}  // namespace gbce
