// ce_aux.cu -- the small kernels around the main pass.
//
// ce_count_kernel: the ignore mask count n_non_ignore and the target range
//   check.  TENPU "Parallel Cross Entropy (Triton)" issue #29 (section 7,
//   "Known limitations") counts n_non_ignore on the host because atomic adds
//   were unreliable there; here one CTA counts on the device with a
//   fixed-order integer reduction, before the gradient pass needs dloss/n.
// ce_wait_probe_kernel: a bounded wait that is left to run out, so a host
//   can check that a kernel which would otherwise hang reports a timeout.
// ce_mean_kernel: reduce_loss -- the mean of the per-row losses over the kept
//   rows (or over their summed class weight), summed in a fixed order (fixed per-thread strides, then a fixed
//   butterfly and a fixed cross-warp order), so the result is bitwise the same
//   on every run.
#include "ce_device.cuh"
#include "ce_internal.h"

namespace gbce {
namespace {

constexpr int kAuxThreads = 1024;
constexpr int kAuxBatch = 8;  // loads in flight per thread

__global__ void __launch_bounds__(kAuxThreads)
ce_count_kernel(const int64_t* __restrict__ targets, int64_t ts0, int64_t ts1, int64_t dim1,
                int64_t N, int64_t V, int64_t ignore_idx, int64_t* n_ws, int64_t* n_out,
                uint32_t* err, uint32_t* ticket, const float* __restrict__ cw, double* wdenom,
                double* wsum, uint32_t* row_claim, uint32_t* row_done) {
    // the pass launched after this kernel may start now: it waits for this
    // kernel's results itself (griddepcontrol.wait) before it reads them
    griddep_launch_dependents();
    __shared__ long long s_n[kAuxThreads / 32];
    __shared__ unsigned s_e[kAuxThreads / 32];
    __shared__ double s_wd[kAuxThreads / 32], s_ws[kAuxThreads / 32];
    long long n = 0;
    unsigned e = 0;
    double wd = 0.0, ws = 0.0;
    // thread t takes rows t, t + T, t + 2T, ... in that order, kAuxBatch loads
    // in flight at a time
    for (int64_t r0 = threadIdx.x; r0 < N; r0 += (int64_t)kAuxThreads * kAuxBatch) {
        int64_t yb[kAuxBatch];
#pragma unroll
        for (int u = 0; u < kAuxBatch; ++u) {
            const int64_t r = r0 + (int64_t)u * kAuxThreads;
            if (r < N) {
                const int64_t i = r / dim1, j = r - i * dim1;
                yb[u] = targets[i * ts0 + j * ts1];
            }
        }
#pragma unroll
        for (int u = 0; u < kAuxBatch; ++u) {
            if (r0 + (int64_t)u * kAuxThreads >= N) break;
            const int64_t y = yb[u];
            if (y == ignore_idx) continue;
            ++n;
            if (y < 0 || y >= V)
                e |= CE_DEVERR_TARGET_RANGE;
            else if (cw)
                wd += (double)__ldg(cw + y);
        }
    }
    if (cw) {
        for (int64_t v0 = threadIdx.x; v0 < V; v0 += (int64_t)kAuxThreads * kAuxBatch) {
            float wb[kAuxBatch];
#pragma unroll
            for (int u = 0; u < kAuxBatch; ++u) {
                const int64_t v = v0 + (int64_t)u * kAuxThreads;
                wb[u] = v < V ? __ldg(cw + v) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < kAuxBatch; ++u)
                if (v0 + (int64_t)u * kAuxThreads < V) ws += (double)wb[u];
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        n += __shfl_xor_sync(kFull, n, off);
        e |= __shfl_xor_sync(kFull, e, off);
        wd += __shfl_xor_sync(kFull, wd, off);
        ws += __shfl_xor_sync(kFull, ws, off);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        s_n[warp] = n;
        s_e[warp] = e;
        s_wd[warp] = wd;
        s_ws[warp] = ws;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        long long tn = 0;
        unsigned te = 0;
        double twd = 0.0, tws = 0.0;
        for (int w = 0; w < kAuxThreads / 32; ++w) {
            tn += s_n[w];
            te |= s_e[w];
            twd += s_wd[w];
            tws += s_ws[w];
        }
        *n_ws = tn;
        if (n_out) *n_out = tn;
        *err = te;     // starts the error word of this pass
        *ticket = 0u;  // no CTA of the pass has finished yet
        if (row_claim) {  // no row of the pass claimed yet
            *row_claim = 0u;
            *row_done = 0u;
        }
        if (cw) {
            *wdenom = twd;
            *wsum = tws;
        }
    }
}

__global__ void __launch_bounds__(kAuxThreads)
ce_mean_kernel(const float* __restrict__ loss_rows, int64_t N, const int64_t* n_dev,
               const double* wdenom, float* out) {
    __shared__ double s_sum[kAuxThreads / 32];
    double acc = strided_sum_fixed(loss_rows, N, threadIdx.x, kAuxThreads);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) s_sum[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int w = 0; w < kAuxThreads / 32; ++w) t += s_sum[w];
        // the mean over kept rows, or over their summed class weight
        const double den = wdenom ? *wdenom : (double)(*n_dev);
        out[0] = (float)(t / den);  // 0/0 = NaN when every row is ignored
    }
}

// The bounded wait every kernel uses, on an mbarrier no one arrives on: it
// gives up after the wait limit and records CE_DEVERR_TIMEOUT, exactly as a
// kernel whose copy never lands would.  One thread; nothing else runs.
__global__ void ce_wait_probe_kernel(uint32_t* err) {
    __shared__ __align__(8) uint64_t bar;
    mbar_init(&bar, 1);
    fence_barrier_init();
    uint32_t e = 0u;
    if (!mbar_wait_bounded(&bar, 0u)) e |= CE_DEVERR_TIMEOUT;  // phase 0 never completes
    *err = e;
}

}  // namespace

cudaError_t launch_wait_probe(uint32_t* err, cudaStream_t s) {
    ce_wait_probe_kernel<<<1, 1, 0, s>>>(err);
    return cudaGetLastError();
}

cudaError_t launch_count(const Problem& p, int64_t* n_out, cudaStream_t s) {
    ce_count_kernel<<<1, kAuxThreads, 0, s>>>(p.targets, p.ts0, p.ts1, p.dim1, p.N, p.V,
                                              p.ignore_idx, p.n_dev, n_out, p.err, p.ticket, p.cw,
                                              p.wdenom, p.wsum, p.row_claim, p.row_done);
    return cudaGetLastError();
}

void set_pdl_attr(cudaLaunchAttribute* attr) {
    attr->id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr->val.programmaticStreamSerializationAllowed = 1;
}

cudaError_t launch_reduce_mean(const Problem& p, float* loss_out, cudaStream_t s) {
    ce_mean_kernel<<<1, kAuxThreads, 0, s>>>(p.loss_rows, p.N, p.n_dev, p.cw ? p.wdenom : nullptr,
                                             loss_out);
    return cudaGetLastError();
}

}  // namespace gbce
