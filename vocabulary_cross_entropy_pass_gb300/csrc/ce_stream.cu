// ce_stream.cu -- the row-streaming fused cross-entropy kernel.
//
// One CTA owns whole token rows (a persistent grid walks rows r = cta,
// cta + grid, ...), so no CTA ever waits for another.  Each row goes twice
// through a ring of shared-memory tiles fed by 1-D TMA bulk copies:
//
//   pass 1 (statistics): a running (max m, sum-exp d, sum S) per thread, the
//     online-softmax update of the TENPU "Parallel Cross Entropy (Triton)"
//     issue #29 (experience report: the online-softmax two-stage kernel), taken
//     over tiles: per tile the thread's max is found first, so one rescale per
//     tile suffices; the target logit is picked up on the way;
//   CTA combine: warp butterflies, then every warp combines the per-warp
//     partials in the same fixed order -> lse = m + log d (CSDN "Ascend CANN
//     ops-nn cross-entropy fusion", pitfall 1);
//   pass 2 (gradient): the tiles are loaded again -- the row was read moments
//     before, so these reads are served by L2, not HBM -- and g*(exp(x-lse) -
//     a/V) - g*(1-a)[j==y] (same article, "Backward", pitfall 3, smoothing over
//     V) is rounded to the storage dtype and stored in place with 16-byte
//     streaming stores (TENPU #29 section 6: in-place gradient staging).
//
// Warp specialisation: warps 0..NC/32-1 consume tiles; the last warp only
// issues copies.  `full[s]` completes when tile s has landed (TMA transaction
// count); `empty[s]` completes when every consumer warp is done with it.  Both
// waits are bounded; a wait that gives up sets CE_DEVERR_TIMEOUT and the CTA
// drains without further copies (the producer then waits, bounded, for the
// copies it already issued before the CTA exits).
#include "ce_device.cuh"
#include "ce_internal.h"

namespace gbce {
namespace {

struct StreamArgs {
    char* logits;
    int64_t s0, s1, dim1, N;
    int32_t V;
    int32_t stages;
    uint32_t tile_bytes;   // bytes per ring tile, multiple of 16
    int32_t ntiles;        // tiles per row
    uint32_t last_bytes;   // bytes of the last tile of a row
    const int64_t* targets;
    int64_t ts0, ts1, ignore_idx;
    float a, a_over_v;
    int reduce;
    const float* dloss;
    float* loss;
    float* lse_out;
    const int64_t* n_dev;
    uint32_t* err;
    int l2_keep;           // 1: pass-1 copies ask L2 to keep the row for pass 2
};

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

template <typename T, int NC, int NV, bool GRAD>
__global__ void __launch_bounds__(NC + 32, 1)
ce_stream_kernel(const __grid_constant__ StreamArgs p) {
    using VT = Vec<T>;
    constexpr int VEC = VT::kElems;
    constexpr int ES = sizeof(T);
    constexpr int NW = NC / 32;  // consumer warps

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)p.stages * p.tile_bytes);
    uint64_t* empty = full + 8;
    float4* red = reinterpret_cast<float4*>(empty + 8);   // [2][NW]
    float* xy_s = reinterpret_cast<float*>(red + 2 * NW);  // [2]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(xy_s + 2);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

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
    const int npass = GRAD ? 2 : 1;

    // ------------------------------------------------------------ producer warp
    if (warp == NW) {
        if (lane == 0) {
            const uint64_t pol_keep = p.l2_keep ? l2_evict_last_policy() : l2_evict_first_policy();
            const uint64_t pol_drop = l2_evict_first_policy();
            uint32_t k = 0;
            for (int64_t r = blockIdx.x; r < p.N && !*abort_flag; r += gridDim.x) {
                if (!is_loaded(row_target(r))) continue;
                const char* row = row_ptr(r);
                for (int pass = 0; pass < npass && !*abort_flag; ++pass) {
                    for (int t = 0; t < p.ntiles; ++t, ++k) {
                        const int s = (int)(k % (uint32_t)p.stages);
                        const uint32_t ph = (k / (uint32_t)p.stages) & 1u;
                        if (!mbar_wait_bounded(&empty[s], ph ^ 1u)) {
                            atomicOr(p.err, CE_DEVERR_TIMEOUT);
                            *abort_flag = 1;
                            break;
                        }
                        const uint32_t bytes = (t == p.ntiles - 1) ? p.last_bytes : p.tile_bytes;
                        mbar_arrive_expect_tx(&full[s], bytes);
                        tma_load_1d(ring + (size_t)s * p.tile_bytes, row + (size_t)t * p.tile_bytes,
                                    bytes, &full[s], pass == 0 ? pol_keep : pol_drop);
                    }
                }
            }
            if (*abort_flag) {
                // let every copy already issued land before the CTA goes away
                for (int s = 0; s < p.stages; ++s) {
                    if (k > (uint32_t)s) {
                        const uint32_t last = (k - 1u - (uint32_t)s) / (uint32_t)p.stages;
                        (void)mbar_wait_bounded(&full[s], last & 1u);
                    }
                }
            }
        }
        return;
    }

    // ------------------------------------------------------------ consumer warps
    float g_reduce = 1.f;
    if (p.reduce) g_reduce = (p.dloss ? __ldg(p.dloss) : 1.f) / (float)(*p.n_dev);
    uint32_t k = 0;
    int par = 0;
    for (int64_t r = blockIdx.x; r < p.N; r += gridDim.x) {
        const int64_t y = row_target(r);
        char* rowp = row_ptr(r);
        if (!is_loaded(y)) {
            if (GRAD) {
                const uint4 z = make_uint4(0, 0, 0, 0);
                const int64_t nv = (int64_t)p.V / VEC;
                for (int64_t v = tid; v < nv; v += NC) stg128_stream(rowp + v * 16, z);
            }
            if (tid == 0) {
                p.loss[r] = (y == p.ignore_idx) ? 0.f : __int_as_float(0x7fc00000);
                if (p.lse_out) p.lse_out[r] = __int_as_float(0x7fc00000);
            }
            continue;
        }
        const float g = p.reduce ? g_reduce : (p.dloss ? __ldg(p.dloss + r) : 1.f);
        const int64_t ybyte = y * ES;

        // pass 1: running statistics over the tiles
        float m = -INFINITY, d = 0.f, S = 0.f;
        for (int t = 0; t < p.ntiles; ++t, ++k) {
            const int s = (int)(k % (uint32_t)p.stages);
            const uint32_t ph = (k / (uint32_t)p.stages) & 1u;
            if (!*abort_flag && !mbar_wait_bounded(&full[s], ph)) {
                atomicOr(p.err, CE_DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
            const unsigned char* tile = ring + (size_t)s * p.tile_bytes;
            const int nvec = (int)(((t == p.ntiles - 1) ? p.last_bytes : p.tile_bytes) / 16);
            uint4 raw[NV];
            float tm = -INFINITY;
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int v = tid + i * NC;
                if (v < nvec) {
                    raw[i] = lds128(tile + (size_t)v * 16);
                    tm = fmaxf(tm, VT::vmax(raw[i]));
                }
            }
            // the target logit lives in this tile at byte offset ybyte - t*tile_bytes
            const int64_t yoff = ybyte - (int64_t)t * p.tile_bytes;
            if (tid == 0 && yoff >= 0 && yoff < (int64_t)nvec * 16)
                xy_s[par] = VT::load1(tile + yoff);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            if (tm > m) {
                if (m != -INFINITY) d *= ex2_approx((m - tm) * kLog2e);
                m = tm;
            }
            const float ml = (m == -INFINITY) ? 0.f : m * kLog2e;
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int v = tid + i * NC;
                if (v < nvec) {
                    float x[VEC];
                    VT::unpack(raw[i], x);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        d += ex2_approx(fmaf(x[e], kLog2e, -ml));
                        S += x[e];
                    }
                }
            }
        }

        // CTA combine, fixed order
        Part q = warp_allreduce_part(Part{m, d, S});
        if (lane == 0) red[par * NW + warp] = make_float4(q.m, q.d, q.S, 0.f);
        named_bar_sync(1, NC);
        Part G = part_identity();
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float4 v4 = red[par * NW + w];
            G = part_combine(G, Part{v4.x, v4.y, v4.z});
        }
        const float lse = G.m + logf(G.d);
        if (tid == 0) {
            p.loss[r] = lse - (1.f - p.a) * xy_s[par] - p.a_over_v * G.S;
            if (p.lse_out) p.lse_out[r] = lse;
        }

        // pass 2: gradient
        if (GRAD) {
            const float lsel = lse * kLog2e;
            const float bb = g * p.a_over_v;
            const float hit = g * (1.f - p.a);
            for (int t = 0; t < p.ntiles; ++t, ++k) {
                const int s = (int)(k % (uint32_t)p.stages);
                const uint32_t ph = (k / (uint32_t)p.stages) & 1u;
                if (!*abort_flag && !mbar_wait_bounded(&full[s], ph)) {
                    atomicOr(p.err, CE_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                }
                const unsigned char* tile = ring + (size_t)s * p.tile_bytes;
                const int nvec = (int)(((t == p.ntiles - 1) ? p.last_bytes : p.tile_bytes) / 16);
                char* gdst = rowp + (size_t)t * p.tile_bytes;
                const int64_t yoff = ybyte - (int64_t)t * p.tile_bytes;
                const int64_t yv = (yoff >= 0 && yoff < (int64_t)nvec * 16) ? yoff / 16 : -1;
                const int ye = (int)(y % VEC);
                uint4 raw[NV];
#pragma unroll
                for (int i = 0; i < NV; ++i) {
                    const int v = tid + i * NC;
                    if (v < nvec) raw[i] = lds128(tile + (size_t)v * 16);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
                for (int i = 0; i < NV; ++i) {
                    const int v = tid + i * NC;
                    if (v < nvec) {
                        float x[VEC], o[VEC];
                        VT::unpack(raw[i], x);
#pragma unroll
                        for (int e = 0; e < VEC; ++e)
                            o[e] = fmaf(ex2_approx(fmaf(x[e], kLog2e, -lsel)), g, -bb);
                        if ((int64_t)v == yv) {
#pragma unroll
                            for (int e = 0; e < VEC; ++e)
                                if (e == ye) o[e] -= hit;
                        }
                        stg128_stream(gdst + (size_t)v * 16, VT::pack(o));
                    }
                }
            }
        }
        par ^= 1;
    }
}

template <typename T, int NC, int NV, bool GRAD>
cudaError_t launch_stream_one(const Problem& pb, const StreamPlan& plan, cudaStream_t s) {
    auto kern = ce_stream_kernel<T, NC, NV, GRAD>;
    constexpr int NW = NC / 32;
    StreamArgs a;
    a.logits = pb.logits;
    a.s0 = pb.s0;
    a.s1 = pb.s1;
    a.dim1 = pb.dim1;
    a.N = pb.N;
    a.V = (int32_t)pb.V;
    a.stages = plan.stages;
    a.tile_bytes = (uint32_t)(NC * NV * 16);
    const int64_t row_bytes = pb.V * (int64_t)sizeof(T);
    a.ntiles = (int32_t)((row_bytes + a.tile_bytes - 1) / a.tile_bytes);
    a.last_bytes = (uint32_t)(row_bytes - (int64_t)(a.ntiles - 1) * a.tile_bytes);
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
    a.l2_keep = plan.l2_keep;
    const size_t smem = (size_t)plan.stages * a.tile_bytes + 16 * sizeof(uint64_t) +
                        2 * NW * sizeof(float4) + 2 * sizeof(float) + 16;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NC + 32, smem);
    if (e != cudaSuccess) return e;
    if (plan.ctas_per_sm_cap > 0 && per_sm > plan.ctas_per_sm_cap) per_sm = plan.ctas_per_sm_cap;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    int64_t grid = (int64_t)per_sm * sms;
    if (grid > pb.N) grid = pb.N;
    if (grid < 1) grid = 1;
    kern<<<(unsigned)grid, NC + 32, smem, s>>>(a);
    return cudaGetLastError();
}

template <typename T, bool GRAD>
cudaError_t launch_stream_typed(const Problem& pb, const StreamPlan& plan, cudaStream_t s) {
    if (plan.threads == 512) return launch_stream_one<T, 512, 2, GRAD>(pb, plan, s);
    return launch_stream_one<T, 256, 4, GRAD>(pb, plan, s);
}

}  // namespace

cudaError_t launch_stream(const Problem& p, const StreamPlan& plan, cudaStream_t s) {
    switch (p.dtype) {
        case CE_F32:
            return p.grad ? launch_stream_typed<float, true>(p, plan, s)
                          : launch_stream_typed<float, false>(p, plan, s);
        case CE_BF16:
            return p.grad ? launch_stream_typed<__nv_bfloat16, true>(p, plan, s)
                          : launch_stream_typed<__nv_bfloat16, false>(p, plan, s);
        default:
            return p.grad ? launch_stream_typed<__half, true>(p, plan, s)
                          : launch_stream_typed<__half, false>(p, plan, s);
    }
}

}  // namespace gbce
