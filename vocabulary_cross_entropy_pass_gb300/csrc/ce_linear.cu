// ce_linear.cu -- lm_head + cross-entropy, chunked over token rows.
//
// hyper-parallel #269 (background, and its TorchTitan comparison) describes
// the ChunkedLossWrapper: the lm_head projection and the cross-entropy run a
// chunk of the sequence at a time so that the full (B*L, V) logits never
// exist, bounding their O(B*L*V) peak memory.  Here, for each chunk of rows:
//
//   1. bf16 / fp16 (hidden size a multiple of 8, 16-byte aligned operands):
//      this library's tcgen05 GEMM (ce_lmhead.cu) writes logits_c = hidden_c .
//      weight^T into a chunk buffer of the workspace and the cross-entropy
//      statistics of every (row, 256-column tile) from its epilogue; a
//      per-row combine turns them into lse and the row's loss; then the
//      backward from the saved lse (ce_bwd's kernel) writes the gradient in
//      place over the chunk's logits;
//      otherwise: a cuBLAS GEMM into the chunk buffer, then the fused
//      cross-entropy pass of this library on it;
//      either way scaled with the kept-row count of the whole batch (counted
//      once, up front);
//   2. grad_hidden_c = dlogits_c . weight    cuBLAS GEMM;
//      grad_weight  += dlogits_c^T . hidden_c cuBLAS GEMM, float32 accumulation.
//
// At a hidden size in the thousands the GEMMs dominate (about 6*H flops per
// logit against a few bytes of logits traffic), so the chunk buffer's round
// trip through memory costs little.
#include <cublas_v2.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "ce_internal.h"

namespace gbce {
namespace {

constexpr size_t kCublasWorkspaceBytes = (size_t)32 << 20;
constexpr int kLinMaxDevices = 64;

// Launched in plain stream order between the logits GEMM and the pass.  The
// pass kernels go out under programmatic dependent launch and their producers
// issue the first logits copies before they wait on the preceding grid (in
// ce_fwd_bwd that grid is the count kernel, which writes no logits).  A
// library GEMM may signal its dependents before its last stores, so the pass
// follows this empty kernel instead, which starts only once the GEMM has
// completed.
__global__ void ce_order_kernel() {}

// One cuBLAS handle per host thread and device (handles are not shared
// between threads that may run at the same time).
cublasHandle_t thread_handle(int dev) {
    thread_local cublasHandle_t handles[kLinMaxDevices] = {};
    if (dev < 0 || dev >= kLinMaxDevices) return nullptr;
    if (!handles[dev] && cublasCreate(&handles[dev]) != CUBLAS_STATUS_SUCCESS) handles[dev] = nullptr;
    return handles[dev];
}

// GBCE_LINEAR_GEMM=library in the environment (read once, at the first call)
// puts the logits GEMM on cuBLAS even where this library's tcgen05 kernel
// applies: the same step with the library GEMM, for comparison.
bool library_gemm_asked() {
    static const bool asked = [] {
        const char* e = getenv("GBCE_LINEAR_GEMM");
        return e != nullptr && strcmp(e, "library") == 0;
    }();
    return asked;
}

cudaDataType_t cuda_type(int dtype) {
    return dtype == CE_F32 ? CUDA_R_32F : (dtype == CE_BF16 ? CUDA_R_16BF : CUDA_R_16F);
}

struct LinLayout {
    size_t rows_off, chunk_off, lse_off, part_off, cublas_off, total;
};

// Workspace: header, per-row losses (N), one chunk of logits (rows padded to
// a multiple of 8 elements), the chunk's lse, partials (two-stage path, or
// the tensor-core path's per-tile statistics), cuBLAS's workspace.
LinLayout lin_layout(int64_t N, int64_t V, int es, int64_t chunk_rows) {
    LinLayout L;
    L.rows_off = kWsHeaderBytes;
    L.chunk_off = L.rows_off + align_up((size_t)N * sizeof(float), 256);
    L.lse_off = L.chunk_off + align_up((size_t)chunk_rows * (size_t)lmhead_ldl(V) * es, 256);
    L.part_off = L.lse_off + align_up((size_t)chunk_rows * sizeof(float), 256);
    const size_t parts = partial_bytes_for(chunk_rows, V);
    const size_t tiles = lmhead_part_bytes(chunk_rows, V);
    L.cublas_off = L.part_off + (parts > tiles ? parts : tiles);
    L.total = L.cublas_off + kCublasWorkspaceBytes;
    return L;
}

}  // namespace
}  // namespace gbce

using namespace gbce;

extern "C" {

size_t ce_linear_workspace_bytes(int64_t N, int64_t H, int64_t V, ce_dtype dtype,
                                 int64_t chunk_rows) {
    if (N < 0 || H < 1 || V < 1 || chunk_rows < 1 || (int)dtype < CE_F32 || (int)dtype > CE_F16)
        return 0;
    return lin_layout(N, V, elem_size(dtype), chunk_rows).total;
}

ce_status ce_linear_fwd_bwd(const void* hidden, const void* weight, ce_dtype dtype, int64_t N,
                            int64_t H, int64_t V, const int64_t* targets, float label_smoothing,
                            int64_t ignore_idx, int reduce_loss, const float* dloss,
                            float* loss_out, void* grad_hidden, float* grad_weight,
                            int64_t* n_non_ignore_out, int64_t chunk_rows, void* workspace,
                            size_t workspace_bytes, void* stream) {
    if ((int)dtype < CE_F32 || (int)dtype > CE_F16) return CE_ERR_UNSUPPORTED_DTYPE;
    if (N < 0 || H < 1 || V < 1 || V > 0x7fffffffLL || H > 0x7fffffffLL || chunk_rows < 1)
        return CE_ERR_INVALID_ARG;
    if (!(label_smoothing >= 0.f && label_smoothing <= 1.f)) return CE_ERR_INVALID_ARG;
    if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256) return CE_ERR_INVALID_ARG;
    if (N > 0 && (!hidden || !weight || !targets || !loss_out)) return CE_ERR_INVALID_ARG;
    if (N == 0 && reduce_loss && !loss_out) return CE_ERR_INVALID_ARG;
    const int es = elem_size(dtype);
    if (chunk_rows > N && N > 0) chunk_rows = N;
    const LinLayout L = lin_layout(N, V, es, chunk_rows);
    if (workspace_bytes < L.total) return CE_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* w = static_cast<char*>(workspace);

    // kept-row count and range check over the whole batch
    static const int64_t no_strides[3] = {0, 0, 1};
    const int64_t t_strides[2] = {N, 1};
    Problem all;
    problem_init(all, hidden, dtype, 1, N, V, no_strides, targets, t_strides, label_smoothing,
                 ignore_idx, reduce_loss);
    all.err = reinterpret_cast<uint32_t*>(w + kWsErrOffset);
    all.n_dev = reinterpret_cast<int64_t*>(w + kWsCountOffset);
    all.ticket = reinterpret_cast<uint32_t*>(w + kWsTicketOffset);
    all.row_claim = reinterpret_cast<uint32_t*>(w + kWsRowClaimOffset);
    all.row_done = reinterpret_cast<uint32_t*>(w + kWsRowDoneOffset);
    all.loss_rows = reduce_loss ? reinterpret_cast<float*>(w + L.rows_off) : loss_out;
    if (launch_count(all, n_non_ignore_out, s) != cudaSuccess) return CE_ERR_LAUNCH;
    if (N == 0) {
        if (reduce_loss && launch_reduce_mean(all, loss_out, s) != cudaSuccess) return CE_ERR_LAUNCH;
        return CE_OK;
    }

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CE_ERR_LAUNCH;
    cublasHandle_t h = thread_handle(dev);
    if (!h) return CE_ERR_LAUNCH;
    if (cublasSetStream(h, s) != CUBLAS_STATUS_SUCCESS) return CE_ERR_LAUNCH;
    if (cublasSetWorkspace(h, w + L.cublas_off, kCublasWorkspaceBytes) != CUBLAS_STATUS_SUCCESS)
        return CE_ERR_LAUNCH;
    const cudaDataType_t ty = cuda_type(dtype);
    const float one = 1.f, zero = 0.f;
    char* chunk = w + L.chunk_off;
    const char* hid = static_cast<const char*>(hidden);
    const bool grads = grad_hidden != nullptr || grad_weight != nullptr;
    // the tensor-core path: this library's GEMM with the statistics in its
    // epilogue; its chunk rows are padded to a multiple of 8 elements
    const bool tc = !library_gemm_asked() && lmhead_supported(dtype, H, V, hidden, weight);
    const int64_t ld = tc ? lmhead_ldl(V) : V;

    for (int64_t r0 = 0; r0 < N; r0 += chunk_rows) {
        const int64_t rows = (N - r0 < chunk_rows) ? N - r0 : chunk_rows;
        if (tc) {
            // 1. logits of the chunk and their per-tile statistics, then lse
            //    and the row losses
            LmHeadProblem lp;
            memset(&lp, 0, sizeof lp);
            lp.hidden = hid + (size_t)r0 * H * es;
            lp.weight = weight;
            lp.dtype = dtype;
            lp.rows = rows;
            lp.H = H;
            lp.V = V;
            lp.ldl = ld;
            lp.logits = chunk;
            lp.part = reinterpret_cast<float4*>(w + L.part_off);
            lp.targets = targets + r0;
            lp.ignore_idx = ignore_idx;
            lp.a = label_smoothing;
            lp.loss_rows = all.loss_rows + r0;
            lp.lse = reinterpret_cast<float*>(w + L.lse_off);
            lp.err = all.err;
            if (launch_lmhead(lp, s) != cudaSuccess) return CE_ERR_LAUNCH;
            //    the gradient in place over the chunk's logits, from lse
            if (grads) {
                BwdProblem bp;
                memset(&bp, 0, sizeof bp);
                bp.logits = chunk;
                bp.grad = chunk;
                bp.dtype = dtype;
                bp.dim1 = rows;
                bp.N = rows;
                bp.V = V;
                bp.s0 = rows * ld;
                bp.s1 = ld;
                bp.gs0 = rows * ld;
                bp.gs1 = ld;
                bp.targets = targets + r0;
                bp.ts0 = rows;
                bp.ts1 = 1;
                bp.ignore_idx = ignore_idx;
                bp.lse = lp.lse;
                bp.a = label_smoothing;
                bp.reduce = reduce_loss ? 1 : 0;
                bp.dloss = reduce_loss ? dloss : (dloss ? dloss + r0 : nullptr);
                bp.n_dev = all.n_dev;
                bp.vec_ok = true;
                bp.vocab_offset = 0;
                bp.V_total = V;
                if (launch_bwd(bp, s) != cudaSuccess) return CE_ERR_LAUNCH;
            }
        } else {
            // 1. logits of the chunk, row-major (rows, V): column-major C[V, rows] = W^T-op . h
            if (cublasGemmEx(h, CUBLAS_OP_T, CUBLAS_OP_N, (int)V, (int)rows, (int)H, &one, weight, ty,
                             (int)H, hid + (size_t)r0 * H * es, ty, (int)H, &zero, chunk, ty, (int)V,
                             CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
                return CE_ERR_LAUNCH;
            //    the cross-entropy pass over the chunk, gradient in place,
            //    after the GEMM has completed (see ce_order_kernel)
            ce_order_kernel<<<1, 32, 0, s>>>();
            if (cudaGetLastError() != cudaSuccess) return CE_ERR_LAUNCH;
            const int64_t c_strides[3] = {rows * V, V, 1};
            const int64_t ct_strides[2] = {rows, 1};
            Problem pb;
            problem_init(pb, chunk, dtype, 1, rows, V, c_strides, targets + r0, ct_strides,
                         label_smoothing, ignore_idx, reduce_loss);
            pb.err = all.err;
            pb.n_dev = all.n_dev;
            pb.ticket = all.ticket;
            pb.row_claim = all.row_claim;  // zeroed by the count kernel, then by each pass's last CTA
            pb.row_done = all.row_done;
            pb.dloss = reduce_loss ? dloss : (dloss ? dloss + r0 : nullptr);
            pb.loss_rows = all.loss_rows + r0;
            pb.grad = grads;
            if (launch_main_pass(pb, nullptr, reinterpret_cast<float4*>(w + L.part_off),
                                 L.cublas_off - L.part_off, s) != cudaSuccess)
                return CE_ERR_LAUNCH;
        }
        // 2. gradients through the projection
        if (grad_hidden &&
            cublasGemmEx(h, CUBLAS_OP_N, CUBLAS_OP_N, (int)H, (int)rows, (int)V, &one, weight, ty,
                         (int)H, chunk, ty, (int)ld, &zero,
                         static_cast<char*>(grad_hidden) + (size_t)r0 * H * es, ty, (int)H,
                         CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
            return CE_ERR_LAUNCH;
        if (grad_weight &&
            cublasGemmEx(h, CUBLAS_OP_N, CUBLAS_OP_T, (int)H, (int)V, (int)rows, &one,
                         hid + (size_t)r0 * H * es, ty, (int)H, chunk, ty, (int)ld, &one, grad_weight,
                         CUDA_R_32F, (int)H, CUBLAS_COMPUTE_32F,
                         CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
            return CE_ERR_LAUNCH;
    }
    if (reduce_loss && launch_reduce_mean(all, loss_out, s) != cudaSuccess) return CE_ERR_LAUNCH;
    return CE_OK;
}

}  // extern "C"
