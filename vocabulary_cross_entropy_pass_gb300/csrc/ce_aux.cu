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
constexpr int kCountMaxCluster = 8;  // CTAs of the count kernel's cluster (portable maximum)

// One CTA's totals, read by rank 0 of the cluster through distributed shared
// memory (two 16-byte words).
struct __align__(16) CountPart {
    long long n;
    double wd, ws;
    unsigned e, pad;
};

__device__ __forceinline__ uint4 ld_dsmem_u4(const void* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    uint4 v;
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(remote)
                 : "memory");
    return v;
}

// A cluster of up to kCountMaxCluster CTAs (one for few rows): every thread
// of the cluster takes rows t, t + T, t + 2T, ... (T threads in the cluster)
// in that order, kAuxBatch loads in flight (contiguous int64 targets two per
// 16-byte load; rows of contiguous tensors addressed without a division);
// each CTA folds its threads in a fixed order, and rank 0 folds the CTAs in
// rank order through distributed shared memory, so every total is the same
// from call to call.
__global__ void __launch_bounds__(kAuxThreads)
ce_count_kernel(const int64_t* __restrict__ targets, int64_t ts0, int64_t ts1, int64_t dim1,
                int64_t N, int64_t V, int64_t ignore_idx, int64_t* n_ws, int64_t* n_out,
                uint32_t* err, uint32_t* ticket, const float* __restrict__ cw, double* wdenom,
                double* wsum, uint32_t* row_claim, uint32_t* row_done, int flat) {
    // the pass launched after this kernel may start now: it waits for this
    // kernel's results itself (griddepcontrol.wait) before it reads them
    griddep_launch_dependents();
    __shared__ long long s_n[kAuxThreads / 32];
    __shared__ unsigned s_e[kAuxThreads / 32];
    __shared__ double s_wd[kAuxThreads / 32], s_ws[kAuxThreads / 32];
    __shared__ CountPart s_part;
    const uint32_t crank = cluster_ctarank(), csize = cluster_nctarank();
    const int64_t T = (int64_t)kAuxThreads * csize;
    const int64_t tg = (int64_t)crank * kAuxThreads + threadIdx.x;
    long long n = 0;
    unsigned e = 0;
    double wd = 0.0, ws = 0.0;
    auto take = [&](int64_t y) {
        if (y == ignore_idx) return;
        ++n;
        if (y < 0 || y >= V)
            e |= CE_DEVERR_TARGET_RANGE;
        else if (cw)
            wd += (double)__ldg(cw + y);
    };
    if (flat && ts1 == 1 && reinterpret_cast<uintptr_t>(targets) % 16 == 0) {
        const longlong2* t2 = reinterpret_cast<const longlong2*>(targets);
        const int64_t np = N / 2;
        for (int64_t q0 = tg; q0 < np; q0 += T * kAuxBatch) {
            longlong2 yb[kAuxBatch];
#pragma unroll
            for (int u = 0; u < kAuxBatch; ++u) {
                const int64_t q = q0 + (int64_t)u * T;
                if (q < np) yb[u] = t2[q];
            }
#pragma unroll
            for (int u = 0; u < kAuxBatch; ++u) {
                if (q0 + (int64_t)u * T < np) {
                    take(yb[u].x);
                    take(yb[u].y);
                }
            }
        }
        if ((N & 1) && tg == 0) take(targets[N - 1]);
    } else {
        for (int64_t r0 = tg; r0 < N; r0 += T * kAuxBatch) {
            int64_t yb[kAuxBatch];
#pragma unroll
            for (int u = 0; u < kAuxBatch; ++u) {
                const int64_t r = r0 + (int64_t)u * T;
                if (r < N) {
                    if (flat) {
                        yb[u] = targets[r * ts1];
                    } else {
                        const int64_t i = r / dim1, j = r - i * dim1;
                        yb[u] = targets[i * ts0 + j * ts1];
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kAuxBatch; ++u)
                if (r0 + (int64_t)u * T < N) take(yb[u]);
        }
    }
    if (cw) {
        for (int64_t v0 = tg; v0 < V; v0 += T * kAuxBatch) {
            float wb[kAuxBatch];
#pragma unroll
            for (int u = 0; u < kAuxBatch; ++u) {
                const int64_t v = v0 + (int64_t)u * T;
                wb[u] = v < V ? __ldg(cw + v) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < kAuxBatch; ++u)
                if (v0 + (int64_t)u * T < V) ws += (double)wb[u];
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
        CountPart c;
        c.n = 0;
        c.e = 0u;
        c.pad = 0u;
        c.wd = 0.0;
        c.ws = 0.0;
        for (int w = 0; w < kAuxThreads / 32; ++w) {
            c.n += s_n[w];
            c.e |= s_e[w];
            c.wd += s_wd[w];
            c.ws += s_ws[w];
        }
        s_part = c;
    }
    cluster_sync();  // every CTA's totals are in its shared memory
    if (crank == 0 && threadIdx.x == 0) {
        long long tn = 0;
        unsigned te = 0;
        double twd = 0.0, tws = 0.0;
        for (uint32_t c = 0; c < csize; ++c) {
            const uint4 a = ld_dsmem_u4(&s_part, c);
            const uint4 b = ld_dsmem_u4(reinterpret_cast<const char*>(&s_part) + 16, c);
            tn += (long long)(((unsigned long long)a.y << 32) | a.x);
            twd += __hiloint2double((int)a.w, (int)a.z);
            tws += __hiloint2double((int)b.y, (int)b.x);
            te |= b.z;
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
    cluster_sync();  // rank 0 has read every CTA's totals
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
    // one CTA per 8192 rows, up to a cluster of kCountMaxCluster
    int64_t cl = (p.N + 8191) / 8192;
    if (cl < 1) cl = 1;
    if (cl > kCountMaxCluster) cl = kCountMaxCluster;
    const int64_t lim = (int64_t)1 << 31;
    const int flat = (p.dim1 >= 1 && p.dim1 < lim && p.ts1 >= 0 && p.ts1 < lim &&
                      (p.N == p.dim1 || p.ts0 == p.dim1 * p.ts1))
                         ? 1
                         : 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)cl, 1, 1);
    cfg.blockDim = dim3(kAuxThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, ce_count_kernel, p.targets, p.ts0, p.ts1, p.dim1, p.N, p.V,
                              p.ignore_idx, p.n_dev, n_out, p.err, p.ticket, p.cw, p.wdenom, p.wsum,
                              p.row_claim, p.row_done, flat);
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
