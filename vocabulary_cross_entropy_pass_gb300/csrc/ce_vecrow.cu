// ce_vecrow.cu -- the fused pass for rows off the 16-byte grid.
//
// Rows whose first element does not sit on a 16-byte boundary (vocabulary
// widths such as 50257 or 100277 in 16-bit types, padded or shifted views)
// cannot be copied by TMA, which the stream and warp kernels use.  This kernel
// streams such rows with plain 16-byte loads instead: a persistent grid, one
// row per CTA (or per warp, for rows up to 32 KB) at a time, two passes per
// row as in the online-softmax fusion of TENPU "Parallel Cross Entropy
// (Triton)" #29 (section 6):
//   pass 1: the row's (max, sum-exp, sum) -- a scalar head up to the first
//           16-byte boundary, whole 16-byte vectors (kVrBatch loads in flight
//           per thread, one rescale per batch with a new max), a scalar tail
//           (ce_span.cuh) -- then a fixed-order combine of the warps' partials
//           (a warp's butterfly alone when a warp owns the row),
//           lse = m + log d, loss = lse - (1-a) x_y - (a/V) S;
//   pass 2: the gradient g (exp(x - lse) - a/V) - g (1-a) [j == y] written in
//           place, reading the row again.
// Two CTAs per SM (512 threads) keep 2 x 152 rows between their passes, so
// for rows up to ~300 KB the second read comes from L2 and HBM sees one read
// and one write per element (the two-stage kernels read the logits twice
// from HBM).  Every access stays inside its row, and head and tail elements
// are stored one by one, so a row's neighbours are never touched.
#include "ce_device.cuh"
#include "ce_internal.h"
#include "ce_span.cuh"

namespace gbce {
namespace {

constexpr int kVrBatch = 4;  // 16-byte loads in flight per thread

// Shapes.  A row per CTA: 512 threads two CTAs per SM (default), 256
// threads three per SM, or 1024 threads one per SM (rows over 320 KB: half
// the rows wait in L2 between their passes).  A row per warp (rows up to
// 32 KB): 512 threads, two CTAs per SM, 32 rows in flight per SM and no CTA
// barrier.
template <int THREADS>
struct VrShape;
template <>
struct VrShape<1024> {
    static constexpr int kCtasPerSm = 1;
};
template <>
struct VrShape<512> {
    static constexpr int kCtasPerSm = 2;
};
template <>
struct VrShape<256> {
    static constexpr int kCtasPerSm = 3;
};

struct VecRowArgs {
    char* logits;
    int64_t s0, s1, dim1, N, V;
    const int64_t* targets;
    int64_t ts0, ts1, ignore_idx;
    float a, a_over_v;
    int reduce;
    const float* dloss;
    float* loss;       // per-row losses
    float* lse_out;    // optional
    const int64_t* n_dev;
    int flat;          // row r at r * s1, its target at r * ts1
};

// Pass 1's 16-byte load, with an L2 evict-last policy: the row's second pass
// rereads the line (and takes it with __ldcs, the row's last use).
__device__ __forceinline__ uint4 ldg128_keep(const uint4* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// WARPROW: each warp takes its own rows (kVrThreads below is then the 32
// lanes of a row's group, tid the lane); otherwise the whole CTA takes a row.
template <typename T, bool GRAD, int THREADS, bool WARPROW>
__global__ void __launch_bounds__(THREADS, VrShape<THREADS>::kCtasPerSm)
    ce_vecrow_kernel(const __grid_constant__ VecRowArgs p) {
    constexpr int kVrThreads = WARPROW ? 32 : THREADS;  // threads on one row
    constexpr int kVrWarps = THREADS / 32;
    using VT = Vec<T>;
    constexpr int VEC = VT::kElems;
    constexpr int ES = sizeof(T);
    constexpr int PP = VEC / 2;
    // double-buffered so that a warp already in the next row's combine cannot
    // overwrite partials a slower warp is still reading
    __shared__ float4 s_part[WARPROW ? 1 : 2][kVrWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int tid = WARPROW ? lane : (int)threadIdx.x;
    const uint64_t keep = l2_evict_last_policy();
    const float2 L2 = make_float2(kLog2e, kLog2e);
    griddep_wait();  // the count kernel's n_non_ignore
    int buf = 0;
    const int64_t r0 = WARPROW ? (int64_t)blockIdx.x * kVrWarps + warp : (int64_t)blockIdx.x;
    const int64_t rstep = WARPROW ? (int64_t)gridDim.x * kVrWarps : (int64_t)gridDim.x;
    for (int64_t r = r0; r < p.N; r += rstep) {
        int64_t y;
        char* row;
        if (p.flat) {
            y = __ldg(p.targets + r * p.ts1);
            row = p.logits + r * p.s1 * (int64_t)ES;
        } else {
            const int64_t i = r / p.dim1, j = r - i * p.dim1;
            y = __ldg(p.targets + i * p.ts0 + j * p.ts1);
            row = p.logits + (i * p.s0 + j * p.s1) * (int64_t)ES;
        }
        const Span16 sp = span16<ES>(row, 0, p.V);
        const int64_t ee = span16_edge(sp, 0, p.V, tid);
        uint4* rv = reinterpret_cast<uint4*>(row + sp.h1 * ES);
        const int nv = (int)sp.nv;  // V < 2^31 elements

        if (y == p.ignore_idx || y < 0 || y >= p.V) {  // the same branch for the row's threads
            if (GRAD) {
                if (ee >= 0) VT::store1(row + ee * ES, 0.f);
                const uint4 z = make_uint4(0, 0, 0, 0);
                for (int v = tid; v < nv; v += kVrThreads) stg128_stream(rv + v, z);
            }
            if (tid == 0) {
                p.loss[r] = (y == p.ignore_idx) ? 0.f : __int_as_float(0x7fc00000);
                if (p.lse_out) p.lse_out[r] = __int_as_float(0x7fc00000);
            }
            continue;
        }

        // pass 1: statistics; the target logit is read before any thread
        // can overwrite it in pass 2
        const float xy = tid == 0 ? VT::load1(row + y * ES) : 0.f;
        float m = -INFINITY;
        float2 d2 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
        if (ee >= 0) {  // the thread's first element: exp(x - m) = 1 (nothing for -inf)
            const float x = VT::load1(row + ee * ES);
            if (x > m) {
                m = x;
                d2.x = 1.f;
            }
            s2.x = x;
        }
        for (int vb = tid; vb < nv; vb += kVrThreads * kVrBatch) {
            uint4 raw[kVrBatch];
            float vm = -INFINITY;
#pragma unroll
            for (int u = 0; u < kVrBatch; ++u) {
                const int v = vb + u * kVrThreads;
                if (v < nv) {
                    raw[u] = ldg128_keep(rv + v, keep);
                    vm = fmaxf(vm, VT::vmax(raw[u]));
                }
            }
            if (vm > m) {
                if (m != -INFINITY) {
                    const float c = ex2_approx((m - vm) * kLog2e);
                    d2.x *= c;
                    d2.y *= c;
                }
                m = vm;
            }
            const float nml = -m * kLog2e;
            const float2 NM = make_float2(nml, nml);
#pragma unroll
            for (int u = 0; u < kVrBatch; ++u) {
                if (vb + u * kVrThreads < nv) {
                    float2 x[PP];
                    VT::unpack2(raw[u], x);
#pragma unroll
                    for (int q = 0; q < PP; ++q) {
                        const float2 e = __ffma2_rn(x[q], L2, NM);
                        d2 = __fadd2_rn(d2, make_float2(ex2_approx(e.x), ex2_approx(e.y)));
                        s2 = __fadd2_rn(s2, x[q]);
                    }
                }
            }
        }
        const Part q = warp_allreduce_part(Part{m, d2.x + d2.y, s2.x + s2.y});
        Part G = q;
        if constexpr (!WARPROW) {
            if (lane == 0) s_part[buf][warp] = make_float4(q.m, q.d, q.S, 0.f);
            __syncthreads();
            // every thread combines the warps' partials in the same order
            G = part_identity();
#pragma unroll
            for (int w = 0; w < kVrWarps; ++w) {
                const float4 f = s_part[buf][w];
                G = part_combine(G, Part{f.x, f.y, f.z});
            }
            buf ^= 1;
        } else {
            // orders lane 0's read of the target logit before any lane's
            // pass-2 store (every lane of the warp walks the same rows)
            __syncwarp();
        }
        const float lse = G.m + logf(G.d);
        if (tid == 0) {
            p.loss[r] = lse - (1.f - p.a) * xy - p.a_over_v * G.S;
            if (p.lse_out) p.lse_out[r] = lse;
        }
        if (!GRAD) continue;

        // pass 2: the gradient, in place
        float g;
        if (p.reduce)
            g = (p.dloss ? __ldg(p.dloss) : 1.f) / (float)(*p.n_dev);
        else
            g = p.dloss ? __ldg(p.dloss + r) : 1.f;
        const float nll = -lse * kLog2e;
        const float ga = g * p.a_over_v;
        const float hit = g * (1.f - p.a);
        if (ee >= 0) {
            const float x = VT::load1(row + ee * ES);
            float o = fmaf(ex2_approx(fmaf(x, kLog2e, nll)), g, -ga);
            if (ee == y) o -= hit;
            VT::store1(row + ee * ES, o);
        }
        const float2 NL = make_float2(nll, nll), G2 = make_float2(g, g), NB = make_float2(-ga, -ga);
        const int yb = (int)(y - sp.h1);  // the target's place in the body
        for (int vb = tid; vb < nv; vb += kVrThreads * kVrBatch) {
            uint4 raw[kVrBatch];
#pragma unroll
            for (int u = 0; u < kVrBatch; ++u) {
                const int v = vb + u * kVrThreads;
                if (v < nv) raw[u] = __ldcs(rv + v);
            }
#pragma unroll
            for (int u = 0; u < kVrBatch; ++u) {
                const int v = vb + u * kVrThreads;
                if (v >= nv) continue;
                float2 x[PP], o[PP];
                VT::unpack2(raw[u], x);
#pragma unroll
                for (int q2 = 0; q2 < PP; ++q2) {
                    const float2 e = __ffma2_rn(x[q2], L2, NL);
                    o[q2] = __ffma2_rn(make_float2(ex2_approx(e.x), ex2_approx(e.y)), G2, NB);
                }
                const int ey = yb - v * VEC;
                if (ey >= 0 && ey < VEC) {
#pragma unroll
                    for (int q2 = 0; q2 < PP; ++q2) {
                        if (2 * q2 == ey) o[q2].x -= hit;
                        if (2 * q2 + 1 == ey) o[q2].y -= hit;
                    }
                }
                stg128_stream(rv + v, VT::pack2(o));
            }
        }
    }
}

template <typename T, int THREADS, bool WARPROW>
cudaError_t launch_vecrow_shaped(const VecRowArgs& a, const Problem& pb, int ctas_cap, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int per_sm = VrShape<THREADS>::kCtasPerSm;
    if (ctas_cap > 0 && ctas_cap < per_sm) per_sm = ctas_cap;
    int64_t grid = (int64_t)sms * per_sm;
    const int64_t rows_per_cta = WARPROW ? THREADS / 32 : 1;
    const int64_t need = (pb.N + rows_per_cta - 1) / rows_per_cta;
    if (grid > need) grid = need;
    if (grid < 1) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    set_pdl_attr(&attr[0]);
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (pb.grad) return cudaLaunchKernelEx(&cfg, ce_vecrow_kernel<T, true, THREADS, WARPROW>, a);
    return cudaLaunchKernelEx(&cfg, ce_vecrow_kernel<T, false, THREADS, WARPROW>, a);
}

template <typename T>
cudaError_t launch_vecrow_typed(const Problem& pb, const VecRowPlan& plan, cudaStream_t s) {
    VecRowArgs a;
    a.logits = pb.logits;
    a.s0 = pb.s0;
    a.s1 = pb.s1;
    a.dim1 = pb.dim1;
    a.N = pb.N;
    a.V = pb.V;
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
    a.flat = rows_flat(pb) ? 1 : 0;
    if (plan.warp_rows) return launch_vecrow_shaped<T, 512, true>(a, pb, plan.ctas_per_sm_cap, s);
    if (plan.threads == 256) return launch_vecrow_shaped<T, 256, false>(a, pb, plan.ctas_per_sm_cap, s);
    if (plan.threads == 1024) return launch_vecrow_shaped<T, 1024, false>(a, pb, plan.ctas_per_sm_cap, s);
    return launch_vecrow_shaped<T, 512, false>(a, pb, plan.ctas_per_sm_cap, s);
}

}  // namespace

cudaError_t launch_vecrow(const Problem& p, const VecRowPlan& plan, cudaStream_t s) {
    switch (p.dtype) {
        case CE_F32:
            return launch_vecrow_typed<float>(p, plan, s);
        case CE_BF16:
            return launch_vecrow_typed<__nv_bfloat16>(p, plan, s);
        default:
            return launch_vecrow_typed<__half>(p, plan, s);
    }
}

}  // namespace gbce
