// ce_fused.cu -- the one-read, one-write fused cross-entropy kernel.
//
// Each token row is read from HBM once and its gradient written once, in
// place (TENPU "Parallel Cross Entropy (Triton)" issue #29, section 6: the
// gradient is staged in the input buffer).  A row is cut into `cluster`
// contiguous vocabulary slices; CTA `rank` of a thread-block cluster owns
// slice `rank` of every row the cluster visits:
//
//   1. a 1-D TMA bulk copy brings the slice into shared memory (a pipeline of
//      `stages` rows is kept in flight per CTA, rows whose target is ignored
//      are never loaded);
//   2. each thread pulls its 16-byte vectors into registers, takes the warp
//      max, and keeps p = exp(x - m_warp) of every element in registers
//      (one exponential per element for the whole pass);
//   3. warps reduce (m, d = sum p, S = sum x) and the CTA writes its partial to
//      shared memory; the cluster barrier makes every CTA's partial visible and
//      each warp combines the `cluster` partials it reads over distributed
//      shared memory in a fixed butterfly order -- the (max, sum-exp, target
//      logit) combine that mindspore/hyper-parallel #269 section 3.1 runs
//      across vocabulary-parallel ranks, run here across the CTAs of a
//      cluster;
//   4. lse = m + log d; loss = lse - (1-a) x_y - (a/V) S (CSDN "Ascend CANN
//      ops-nn cross-entropy fusion", section "Fusion scheme" with PyTorch-style
//      smoothing); the gradient g (p e^(m_warp - lse) - a/V) - g (1-a) [j==y]
//      (same article, "Backward" and pitfall 3) is rounded to the storage
//      dtype and stored straight from registers.
//
// cluster == 1 is the row path (one CTA per row, no cluster barrier).
// Every wait is bounded; a wait that gives up sets CE_DEVERR_TIMEOUT, stops
// issuing copies, keeps taking part in every cluster barrier so that no peer
// is left waiting, and before exit waits (bounded) for its copies in flight.
#include <cuda.h>

#include "ce_device.cuh"
#include "ce_internal.h"

namespace gbce {
namespace {

struct FusedArgs {
    char* logits;
    int64_t s0, s1, dim1, N;
    int32_t V, chunk;
    int32_t stages;
    uint32_t stage_bytes;
    const int64_t* targets;
    int64_t ts0, ts1, ignore_idx;
    float a, a_over_v;
    int reduce;
    const float* dloss;
    float* loss;
    float* lse_out;
    const int64_t* n_dev;
    uint32_t* err;
};

template <typename T, int NT, int NV, bool GRAD>
__global__ void __launch_bounds__(NT, NT == 256 ? (sizeof(T) == 4 ? 2 : 3) : 1) ce_fused_kernel(const __grid_constant__ FusedArgs p) {
    using VT = Vec<T>;
    constexpr int VEC = VT::kElems;
    constexpr int ES = sizeof(T);
    constexpr int NW = NT / 32;

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* stage_buf = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)p.stages * p.stage_bytes);
    float4* red = reinterpret_cast<float4*>(bars + 8);  // [2][NW]
    float4* part = red + 2 * NW;                        // [2]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(part + 2);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t C = cluster_nctarank();
    const uint32_t rank = cluster_ctarank();
    // cluster index and count (a launch without clusters: one CTA per cluster)
    const int64_t cid = (C > 1) ? (int64_t)cluster_id_x() : (int64_t)blockIdx.x;
    const int64_t ncl = (C > 1) ? (int64_t)ncluster_x() : (int64_t)gridDim.x;

    const int32_t c0 = (int32_t)rank * p.chunk;                        // first column of my slice
    const int32_t clen = max(0, min(p.chunk, p.V - c0));                // may be 0
    const int nvec = clen / VEC;
    const uint32_t cbytes = (uint32_t)clen * ES;

    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) mbar_init(&bars[s], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    const uint64_t policy = l2_evict_first_policy();
    auto row_target = [&](int64_t r) -> int64_t {
        const int64_t i = r / p.dim1, j = r - (r / p.dim1) * p.dim1;
        return __ldg(p.targets + i * p.ts0 + j * p.ts1);
    };
    auto row_ptr = [&](int64_t r) -> char* {
        const int64_t i = r / p.dim1, j = r - (r / p.dim1) * p.dim1;
        return p.logits + (i * p.s0 + j * p.s1) * ES;
    };
    auto is_loaded = [&](int64_t y) -> bool {
        return y != p.ignore_idx && y >= 0 && y < (int64_t)p.V;
    };

    // Producer state, used by thread 0 only.
    int64_t prow = cid;     // next row the producer examines
    int issued = 0;         // copies issued so far
    auto issue_next = [&]() {
        while (prow < p.N && !is_loaded(row_target(prow))) prow += ncl;
        if (prow >= p.N) return;
        const int s = issued % p.stages;
        fence_proxy_async_smem();  // earlier generic reads of this stage come first
        mbar_arrive_expect_tx(&bars[s], cbytes);
        tma_load_1d(stage_buf + (size_t)s * p.stage_bytes, row_ptr(prow) + (size_t)c0 * ES, cbytes,
                    &bars[s], policy);
        ++issued;
        prow += ncl;
    };
    if (tid == 0 && cbytes > 0)
        for (int s = 0; s < p.stages; ++s) issue_next();

    float g_reduce = 1.f;
    if (p.reduce) {
        const float dl = p.dloss ? __ldg(p.dloss) : 1.f;
        g_reduce = dl / (float)(*p.n_dev);
    }

    int consumed = 0;
    for (int64_t r = cid; r < p.N; r += ncl) {
        const int64_t y = row_target(r);
        char* rowp = row_ptr(r);
        if (!is_loaded(y)) {
            // ignored (loss 0) or out of range (loss NaN): zero gradient, no read
            if (GRAD) {
                const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    const int v = tid + k * NT;
                    if (v < nvec) stg128_stream(rowp + ((size_t)c0 + (size_t)v * VEC) * ES, z);
                }
            }
            if (rank == 0 && tid == 0) {
                p.loss[r] = (y == p.ignore_idx) ? 0.f : __int_as_float(0x7fc00000);
                if (p.lse_out) p.lse_out[r] = __int_as_float(0x7fc00000);
            }
            continue;
        }

        const int slot = consumed & 1;
        const int stage = consumed % p.stages;
        const uint32_t parity = (uint32_t)(consumed / p.stages) & 1u;
        const float g = p.reduce ? g_reduce : (p.dloss ? __ldg(p.dloss + r) : 1.f);
        const unsigned char* sbuf = stage_buf + (size_t)stage * p.stage_bytes;

        if (cbytes > 0 && !*abort_flag) {
            if (!mbar_wait_bounded(&bars[stage], parity)) {
                atomicOr(p.err, CE_DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
        }

        // 2. registers: warp max, then p = exp(x - m_warp)
        uint4 raw[NV];
        float mt = -INFINITY;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = tid + k * NT;
            if (v < nvec) {
                raw[k] = lds128(sbuf + (size_t)v * 16);
                mt = fmaxf(mt, VT::vmax(raw[k]));
            }
        }
        const float mw = warp_allmax(mt);
        const float mwl = (mw == -INFINITY) ? 0.f : mw * kLog2e;
        float pv[NV][GRAD ? VEC : 1];
        float dt = 0.f, st = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = tid + k * NT;
            if (v < nvec) {
                float x[VEC];
                VT::unpack(raw[k], x);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float q = ex2_approx(fmaf(x[e], kLog2e, -mwl));
                    if (GRAD) pv[k][GRAD ? e : 0] = q;
                    dt += q;
                    st += x[e];
                }
            }
        }
        const float dw = warp_allsum(dt);
        const float sw = (p.a != 0.f) ? warp_allsum(st) : 0.f;
        if (lane == 0) red[slot * NW + warp] = make_float4(mw, dw, sw, 0.f);

        // target logit, read by the CTA that owns it before the stage is refilled
        const int64_t ky = y / p.chunk;
        float xy_own = 0.f;
        if (tid == 0 && ky == (int64_t)rank) xy_own = VT::load1(sbuf + (size_t)(y - c0) * ES);
        __syncthreads();

        // 1'. the stage is free: refill it with the next row this CTA will need
        if (tid == 0 && cbytes > 0 && !*abort_flag) issue_next();

        // 3. CTA partial
        if (warp == 0) {
            Part q = part_identity();
            if (lane < NW) {
                const float4 w = red[slot * NW + lane];
                q = Part{w.x, w.y, w.z};
            }
            q = warp_allreduce_part(q);
            if (lane == 0) part[slot] = make_float4(q.m, q.d, q.S, xy_own);
        }
        if (C > 1)
            cluster_sync();
        else
            __syncthreads();

        // every warp combines the cluster's partials in the same fixed order
        float4 pk = make_float4(-INFINITY, 0.f, 0.f, 0.f);
        if (lane < (int)C) pk = (C > 1) ? ld_dsmem_f4(&part[slot], (uint32_t)lane) : part[slot];
        const Part G = warp_allreduce_part(Part{pk.x, pk.y, pk.z});
        const float xy = __shfl_sync(kFull, pk.w, (int)ky);
        const float lse = G.m + logf(G.d);

        // 4. gradient from the registers, one 16-byte store per vector
        if (GRAD) {
            const float cw = g * ex2_approx((mw - lse) * kLog2e);
            const float bb = g * p.a_over_v;
            const int vy = (ky == (int64_t)rank) ? (int)((y - c0) / VEC) : -1;
            const int ey = (int)((y - c0) % VEC);
            const float hit = g * (1.f - p.a);
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int v = tid + k * NT;
                if (v < nvec) {
                    float o[VEC];
#pragma unroll
                    for (int e = 0; e < VEC; ++e) o[e] = fmaf(pv[k][GRAD ? e : 0], cw, -bb);
                    if (v == vy) {
#pragma unroll
                        for (int e = 0; e < VEC; ++e)
                            if (e == ey) o[e] -= hit;
                    }
                    stg128_stream(rowp + ((size_t)c0 + (size_t)v * VEC) * ES, VT::pack(o));
                }
            }
        }
        if (rank == 0 && tid == 0) {
            p.loss[r] = lse - (1.f - p.a) * xy - p.a_over_v * G.S;
            if (p.lse_out) p.lse_out[r] = lse;
        }
        ++consumed;
    }

    // a CTA's shared memory must outlive every peer read of it
    if (C > 1) cluster_sync();
    // copies that a timed-out wait left behind must land before the CTA exits
    if (tid == 0 && cbytes > 0 && *abort_flag) {
        for (int s = 0; s < p.stages; ++s) {
            // the last phase issued on stage s
            if (issued > s) {
                const int last = (issued - 1 - s) / p.stages;
                const uint32_t par = (uint32_t)last & 1u;
                (void)mbar_wait_bounded(&bars[s], par);
            }
        }
    }
}

template <typename T, int NT, int NV, bool GRAD>
cudaError_t launch_one(const Problem& pb, const FusedPlan& plan, cudaStream_t s) {
    auto kern = ce_fused_kernel<T, NT, NV, GRAD>;
    constexpr int NW = NT / 32;
    FusedArgs a;
    a.logits = pb.logits;
    a.s0 = pb.s0;
    a.s1 = pb.s1;
    a.dim1 = pb.dim1;
    a.N = pb.N;
    a.V = (int32_t)pb.V;
    a.chunk = plan.chunk;
    a.stages = plan.stages;
    a.stage_bytes = (uint32_t)align_up((size_t)plan.chunk * sizeof(T), 128);
    a.targets = pb.targets;
    a.ts0 = pb.ts0;
    a.ts1 = pb.ts1;
    a.ignore_idx = pb.ignore_idx;
    a.a = pb.a;
    a.a_over_v = pb.a / (float)pb.V;
    a.reduce = pb.reduce;
    a.dloss = pb.dloss;
    a.loss = pb.loss_rows;
    a.lse_out = pb.lse_out;
    a.n_dev = pb.n_dev;
    a.err = pb.err;

    const size_t smem = (size_t)plan.stages * a.stage_bytes + 8 * sizeof(uint64_t) +
                        (2 * NW + 2) * sizeof(float4) + 16;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (plan.cluster > 8) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }

    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)plan.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = plan.cluster > 1 ? 1 : 0;

    // persistent grid: as many clusters as can be resident at once, capped by rows
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, smem);
    if (e != cudaSuccess) return e;
    if (plan.ctas_per_sm_cap > 0 && per_sm > plan.ctas_per_sm_cap) per_sm = plan.ctas_per_sm_cap;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    int64_t clusters = 0;
    if (plan.cluster == 1) {
        clusters = (int64_t)per_sm * sms;
    } else {
        cfg.gridDim = dim3((unsigned)(plan.cluster * sms), 1, 1);
        int active = 0;
        e = cudaOccupancyMaxActiveClusters(&active, kern, &cfg);
        if (e != cudaSuccess) return e;
        if (active < 1) return cudaErrorInvalidConfiguration;
        clusters = active;
        if (plan.ctas_per_sm_cap > 0) {
            const int64_t cap = (int64_t)plan.ctas_per_sm_cap * sms / plan.cluster;
            if (cap >= 1 && clusters > cap) clusters = cap;
        }
    }
    if (clusters > pb.N) clusters = pb.N;
    if (clusters < 1) clusters = 1;
    cfg.gridDim = dim3((unsigned)(clusters * plan.cluster), 1, 1);
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename T, bool GRAD>
cudaError_t launch_typed(const Problem& pb, const FusedPlan& plan, cudaStream_t s) {
    // NV vectors of 16 bytes per thread: 32 elements per thread for every dtype
    constexpr int NV = 32 / Vec<T>::kElems;
    if (plan.threads == 256) return launch_one<T, 256, NV, GRAD>(pb, plan, s);
    return launch_one<T, 512, NV, GRAD>(pb, plan, s);
}

}  // namespace

int fused_capacity(int dtype, int threads) {
    (void)dtype;
    return threads * 32;  // 32 elements per thread
}

bool fused_aligned(const Problem& p) {
    const uintptr_t base = reinterpret_cast<uintptr_t>(p.logits);
    if (base % 16) return false;
    if ((p.s0 * p.es) % 16 || (p.s1 * p.es) % 16) return false;
    if ((p.V * p.es) % 16) return false;
    return true;
}

cudaError_t launch_fused(const Problem& p, const FusedPlan& plan, cudaStream_t s) {
    switch (p.dtype) {
        case CE_F32:
            return p.grad ? launch_typed<float, true>(p, plan, s) : launch_typed<float, false>(p, plan, s);
        case CE_BF16:
            return p.grad ? launch_typed<__nv_bfloat16, true>(p, plan, s)
                          : launch_typed<__nv_bfloat16, false>(p, plan, s);
        default:
            return p.grad ? launch_typed<__half, true>(p, plan, s) : launch_typed<__half, false>(p, plan, s);
    }
}

}  // namespace gbce
