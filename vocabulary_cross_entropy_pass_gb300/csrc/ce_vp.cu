// ce_vp.cu -- vocabulary-parallel cross-entropy, one shard at a time.
//
// mindspore/hyper-parallel #269 (section 3.1) describes the vocab-sharded
// cross-entropy that tensor-parallel training runs when each rank holds a
// ceil(V/tp) slice of the logits: per-row (max, sum-exp) statistics of the
// slice, a MAX all-reduce and a SUM all-reduce of the rescaled sums plus a
// gather of the target logit (the m_d_Xy gather of TENPU "Parallel Cross
// Entropy (Triton)" #29, section 6), then a backward that needs no collective.
// On one GPU the ranks become vocabulary shards (separate tensors) and the
// collectives become a fixed-order combine over the gathered partials:
//
//   ce_vp_partials_kernel: per row of one shard, {m, d, S, x_y} (x_y when the
//     global target falls in the shard, else 0); ignored rows get the empty
//     partial {-inf, 0, 0, 0};
//   ce_vp_combine_kernel:  per row, the partials of all shards in shard order
//     -> lse = m + log d, loss = lse - (1-a) x_y - (a/V) S;
//   the gradient of each shard: ce_bwd's kernels with the shard's vocabulary
//     offset (ce_bwd.cu).
#include "ce_device.cuh"
#include "ce_internal.h"
#include "ce_span.cuh"

namespace gbce {
namespace {

constexpr int kVpThreads = 256;
constexpr int kVpWarps = kVpThreads / 32;

struct VpPartArgs {
    const char* logits;
    int64_t s0, s1, dim1, N, V;        // V: columns of this shard
    int64_t vocab_offset;              // global index of the shard's column 0
    const int64_t* targets;
    int64_t ts0, ts1, ignore_idx;
    float4* part;                      // [N]
    int flat;                          // row r at r * s1, its target at r * ts1
};

// One CTA per row: a running (max, sum-exp, sum) per thread over 16-byte
// vectors, kVpBatch loads in flight per thread (one rescale per batch whose
// max is new), then the CTA combine.
constexpr int kVpBatch = 8;

template <typename T>
// Eight loads in flight per thread at four CTAs per SM (64 registers, no
// spills): 128 KB of loads in flight per SM.  Four loads at six CTAs per SM
// (96 KB; 40 registers, small spills) measured 2.010 / 1.876 ms for 8 / 2
// shards of the bench workload against 2.004 / 1.852 ms, six loads at five
// CTAs per SM (spills) 2.089 ms for 8 shards; four loads at the unbounded 54
// registers (four CTAs per SM, 64 KB in flight) had measured 2.134 ms.
__global__ void __launch_bounds__(kVpThreads, 4) ce_vp_partials_kernel(const __grid_constant__ VpPartArgs p) {
    using VT = Vec<T>;
    constexpr int VEC = VT::kElems;
    constexpr int ES = sizeof(T);
    constexpr int PP = VEC / 2;
    __shared__ float4 s_red[kVpWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float2 L2 = make_float2(kLog2e, kLog2e);
    for (int64_t r = blockIdx.x; r < p.N; r += gridDim.x) {
        int64_t y;
        const char* row;
        if (p.flat) {
            y = __ldg(p.targets + r * p.ts1);
            row = p.logits + r * p.s1 * ES;
        } else {
            const int64_t i = r / p.dim1, j = r - i * p.dim1;
            y = __ldg(p.targets + i * p.ts0 + j * p.ts1);
            row = p.logits + (i * p.s0 + j * p.s1) * ES;
        }
        if (y == p.ignore_idx) {
            if (threadIdx.x == 0) p.part[r] = make_float4(-INFINITY, 0.f, 0.f, 0.f);
            continue;
        }
        float m = -INFINITY;
        float2 d2 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
        // head and tail (rows off a 16-byte boundary) one element per thread
        const Span16 sp = span16<ES>(row, 0, p.V);
        const int64_t ee = span16_edge(sp, 0, p.V, threadIdx.x);
        if (ee >= 0) {  // the thread's first element: exp(x - m) = 1 (nothing for -inf)
            const float x = VT::load1(row + ee * ES);
            if (x > m) {
                m = x;
                d2.x = 1.f;
            }
            s2.x = x;
        }
        const uint4* rv = reinterpret_cast<const uint4*>(row + sp.h1 * ES);
        for (int64_t vb = threadIdx.x; vb < sp.nv; vb += kVpThreads * kVpBatch) {
            uint4 raw[kVpBatch];
            float vm = -INFINITY;
#pragma unroll
            for (int u = 0; u < kVpBatch; ++u) {
                const int64_t v = vb + (int64_t)u * kVpThreads;
                if (v < sp.nv) {
                    raw[u] = __ldcs(rv + v);
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
            for (int u = 0; u < kVpBatch; ++u) {
                if (vb + (int64_t)u * kVpThreads < sp.nv) {
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
        Part q = warp_allreduce_part(Part{m, d2.x + d2.y, s2.x + s2.y});
        if (lane == 0) s_red[warp] = make_float4(q.m, q.d, q.S, 0.f);
        __syncthreads();
        if (threadIdx.x == 0) {
            Part G = part_identity();
            for (int w = 0; w < kVpWarps; ++w) G = part_combine(G, Part{s_red[w].x, s_red[w].y, s_red[w].z});
            const int64_t yl = y - p.vocab_offset;
            const float xy = (yl >= 0 && yl < p.V) ? VT::load1(row + yl * ES) : 0.f;
            p.part[r] = make_float4(G.m, G.d, G.S, xy);
        }
        __syncthreads();
    }
}

struct VpCombineArgs {
    const float4* part;                // [R][N]
    int R;
    int64_t off[kVpMaxShards + 1];     // shard column offsets, off[R] = V total
    int64_t dim1, N;
    const int64_t* targets;
    int64_t ts0, ts1, ignore_idx;
    float a, a_over_v;
    float* loss;                       // [N]
    float* lse;                        // [N]
};

// One thread per row: combine the shards' partials in shard order.
__global__ void __launch_bounds__(256) ce_vp_combine_kernel(const __grid_constant__ VpCombineArgs p) {
    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= p.N) return;
    const int64_t i = r / p.dim1, j = r - i * p.dim1;
    const int64_t y = __ldg(p.targets + i * p.ts0 + j * p.ts1);
    const float nan = __int_as_float(0x7fc00000);
    if (y == p.ignore_idx || y < 0 || y >= p.off[p.R]) {
        p.loss[r] = (y == p.ignore_idx) ? 0.f : nan;
        p.lse[r] = nan;
        return;
    }
    Part G = part_identity();
    float xy = 0.f;
    for (int k = 0; k < p.R; ++k) {
        const float4 w = p.part[(int64_t)k * p.N + r];
        G = part_combine(G, Part{w.x, w.y, w.z});
        if (y >= p.off[k] && y < p.off[k + 1]) xy = w.w;  // the target's owner
    }
    const float lse = G.m + logf(G.d);
    p.lse[r] = lse;
    p.loss[r] = lse - (1.f - p.a) * xy - p.a_over_v * G.S;
}

template <typename T>
cudaError_t launch_vp_partials_typed(const VpPartArgs& a, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t grid = a.N;
    if (grid > (int64_t)sms * 16) grid = (int64_t)sms * 16;
    if (grid < 1) return cudaSuccess;
    ce_vp_partials_kernel<T><<<(unsigned)grid, kVpThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_vp_partials(const VpPartProblem& vp, cudaStream_t s) {
    VpPartArgs a;
    a.logits = vp.logits;
    a.s0 = vp.s0;
    a.s1 = vp.s1;
    a.dim1 = vp.dim1;
    a.N = vp.N;
    a.V = vp.V;
    a.vocab_offset = vp.vocab_offset;
    a.targets = vp.targets;
    a.ts0 = vp.ts0;
    a.ts1 = vp.ts1;
    a.ignore_idx = vp.ignore_idx;
    a.part = vp.part;
    {
        const int64_t lim = (int64_t)1 << 31;
        a.flat = (vp.dim1 >= 1 && vp.dim1 < lim && vp.s1 >= 0 && vp.s1 < lim && vp.ts1 >= 0 && vp.ts1 < lim &&
                  vp.s0 == vp.dim1 * vp.s1 && vp.ts0 == vp.dim1 * vp.ts1)
                     ? 1
                     : 0;
    }
    switch (vp.dtype) {
        case CE_F32:
            return launch_vp_partials_typed<float>(a, s);
        case CE_BF16:
            return launch_vp_partials_typed<__nv_bfloat16>(a, s);
        default:
            return launch_vp_partials_typed<__half>(a, s);
    }
}

cudaError_t launch_vp_combine(const VpCombineProblem& vc, cudaStream_t s) {
    VpCombineArgs a;
    a.part = vc.part;
    a.R = vc.R;
    for (int k = 0; k <= vc.R; ++k) a.off[k] = vc.off[k];
    a.dim1 = vc.dim1;
    a.N = vc.N;
    a.targets = vc.targets;
    a.ts0 = vc.ts0;
    a.ts1 = vc.ts1;
    a.ignore_idx = vc.ignore_idx;
    a.a = vc.a;
    a.a_over_v = vc.a / (float)vc.off[vc.R];
    a.loss = vc.loss;
    a.lse = vc.lse;
    if (vc.N < 1) return cudaSuccess;
    const int64_t blocks = (vc.N + 255) / 256;
    ce_vp_combine_kernel<<<(unsigned)blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace gbce
