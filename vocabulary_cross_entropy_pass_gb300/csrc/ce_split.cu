// ce_split.cu -- the two-stage split-vocabulary path.
//
// Stage 1 (ce_split_stats_kernel): one CTA per (row, chunk) computes the
// chunk's (max, sum-exp, sum, target logit) partial and writes it to the
// workspace.  Stage 2 (ce_split_grad_kernel): one CTA per (row, chunk)
// combines the row's K partials in chunk order -- the MAX all-reduce, SUM
// all-reduce and target gather that mindspore/hyper-parallel #269 (section
// 3.1) runs between vocabulary-parallel ranks, with the uneven ceil(V/K)
// split it describes -- then rereads its chunk and writes the gradient in
// place.  The kernel boundary orders every read of a row before any write.
//
// This path takes any row alignment and any row strides: each chunk moves in
// 16-byte vectors between a scalar head and tail (ce_span.cuh), or, when the
// rows and every chunk boundary sit on the 16-byte grid, in vectors indexed
// from the row start (unweighted; 1.86 against 2.09 ms for the two-stage
// pass on the bench workload); the other fused paths need 16-byte aligned
// rows.  It reads the logits
// twice, so it is the fallback, the forced second implementation of the
// vocabulary-split workloads, and the path of the class-weighted pass
// (weights as in torch F.cross_entropy(weight=...)).
#include "ce_device.cuh"
#include "ce_internal.h"
#include "ce_span.cuh"

namespace gbce {
namespace {

constexpr int kSplitThreads = 256;
constexpr int kSplitWarps = kSplitThreads / 32;
constexpr int kSplitBatch = 4;  // 16-byte loads in flight per thread

struct SplitArgs {
    char* logits;
    int64_t s0, s1, dim1, N, V, chunk;
    int K;
    const int64_t* targets;
    int64_t ts0, ts1, ignore_idx;
    float a, a_over_v;
    int reduce;
    const float* dloss;
    float* loss;
    float* lse_out;
    const int64_t* n_dev;
    float4* part;  // [N][K]
    const float* cw;         // class weights [V] (weighted pass) or NULL
    const double* wdenom;    // summed weight of the kept rows' targets
    const double* wsum;      // summed weight over the vocabulary
};

__device__ __forceinline__ void row_of(const SplitArgs& p, int64_t r, int64_t& y, int64_t& off) {
    const int64_t i = r / p.dim1, j = r - i * p.dim1;
    y = p.targets[i * p.ts0 + j * p.ts1];
    off = i * p.s0 + j * p.s1;
}

// The class weights of one 16-byte vector of logits (VEC of them, from
// base): 16-byte loads when base sits on the 16-byte grid (it stays there from
// vector to vector: VEC * 4 bytes apart), one float at a time otherwise.
template <int VEC>
__device__ __forceinline__ void weights_of(const float* base, bool vec16, float (&w)[VEC]) {
    if (vec16) {
#pragma unroll
        for (int k = 0; k < VEC / 4; ++k) {
            const float4 f = __ldg(reinterpret_cast<const float4*>(base) + k);
            w[4 * k] = f.x;
            w[4 * k + 1] = f.y;
            w[4 * k + 2] = f.z;
            w[4 * k + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) w[e] = __ldg(base + e);
    }
}

// Stage 1.  WT: the class-weighted pass, whose third statistic is
// sum_j w_j x_j.  The chunk's elements outside whole 16-byte vectors (a row
// that starts off a 16-byte boundary, a ragged chunk end) go one per thread;
// the rest in 16-byte vectors, kSplitBatch loads in flight per thread and one
// rescale per batch with a new max.  VECOK: the rows and every chunk
// boundary on the 16-byte grid, so the chunk is whole vectors indexed from
// the row start (the head/tail form measured 26 % slower on such rows).
// The weighted pass always takes the head/tail form.
template <typename T, bool WT, bool VECOK>
__global__ void __launch_bounds__(kSplitThreads) ce_split_stats_kernel(const __grid_constant__ SplitArgs p) {
    static_assert(!(WT && VECOK), "the weighted pass takes the head/tail form");
    using VT = Vec<T>;
    constexpr int VEC = VT::kElems;
    constexpr int ES = sizeof(T);
    __shared__ float4 s_part[kSplitWarps];
    const int64_t b = blockIdx.x;
    const int64_t r = b / p.K;
    const int k = (int)(b - r * p.K);
    int64_t y, off;
    row_of(p, r, y, off);
    if (y == p.ignore_idx || y < 0 || y >= p.V) return;
    const int64_t k0 = (int64_t)k * p.chunk;
    const int64_t k1 = min(p.V, k0 + p.chunk);
    const char* row = p.logits + off * (int64_t)ES;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const Span16 sp = span16<ES>(row, k0, k1);

    float m = -INFINITY, d = 0.f, S = 0.f;
    if constexpr (VECOK) {
        const uint4* rv = reinterpret_cast<const uint4*>(row);
        const int64_t vend = k1 / VEC;
        for (int64_t vb = k0 / VEC + threadIdx.x; vb < vend; vb += kSplitThreads * kSplitBatch) {
            uint4 raw[kSplitBatch];
            float vm = -INFINITY;
#pragma unroll
            for (int u = 0; u < kSplitBatch; ++u) {
                const int64_t v = vb + (int64_t)u * kSplitThreads;
                if (v < vend) {
                    raw[u] = __ldcs(rv + v);
                    vm = fmaxf(vm, VT::vmax(raw[u]));
                }
            }
            if (vm > m) {
                if (m != -INFINITY) d *= ex2_approx((m - vm) * kLog2e);
                m = vm;
            }
            const float nml = -m * kLog2e;
#pragma unroll
            for (int u = 0; u < kSplitBatch; ++u) {
                const int64_t v = vb + (int64_t)u * kSplitThreads;
                if (v < vend) {
                    float x[VEC];
                    VT::unpack(raw[u], x);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        d += ex2_approx(fmaf(x[e], kLog2e, nml));
                        S += x[e];
                    }
                }
            }
        }
    } else {
    const int64_t ee = span16_edge(sp, k0, k1, threadIdx.x);
    if (ee >= 0) {
        const float x = VT::load1(row + ee * ES);  // the thread's first element
        if (x > m) {
            m = x;
            d = 1.f;  // exp(x - m); a -inf element adds nothing
        }
        S = WT ? __ldg(p.cw + ee) * x : x;
    }
    const uint4* rv = reinterpret_cast<const uint4*>(row + sp.h1 * ES);
    const float* cwb = WT ? p.cw + sp.h1 : nullptr;
    const bool wvec = WT && reinterpret_cast<uintptr_t>(cwb) % 16 == 0;
    for (int64_t vb = threadIdx.x; vb < sp.nv; vb += kSplitThreads * kSplitBatch) {
        uint4 raw[kSplitBatch];
        float vm = -INFINITY;
#pragma unroll
        for (int u = 0; u < kSplitBatch; ++u) {
            const int64_t v = vb + (int64_t)u * kSplitThreads;
            if (v < sp.nv) {
                raw[u] = __ldcs(rv + v);
                vm = fmaxf(vm, VT::vmax(raw[u]));
            }
        }
        if (vm > m) {
            if (m != -INFINITY) d *= ex2_approx((m - vm) * kLog2e);
            m = vm;
        }
        const float nml = -m * kLog2e;
#pragma unroll
        for (int u = 0; u < kSplitBatch; ++u) {
            const int64_t v = vb + (int64_t)u * kSplitThreads;
            if (v < sp.nv) {
                float x[VEC], w[VEC];
                VT::unpack(raw[u], x);
                if (WT) weights_of<VEC>(cwb + v * VEC, wvec, w);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    d += ex2_approx(fmaf(x[e], kLog2e, nml));
                    S = WT ? fmaf(w[e], x[e], S) : S + x[e];
                }
            }
        }
    }
    }
    Part q = warp_allreduce_part(Part{m, d, S});
    if (lane == 0) s_part[warp] = make_float4(q.m, q.d, q.S, 0.f);
    __syncthreads();
    if (threadIdx.x == 0) {
        Part G = part_identity();
        for (int w = 0; w < kSplitWarps; ++w)
            G = part_combine(G, Part{s_part[w].x, s_part[w].y, s_part[w].z});
        const float xy = (y >= k0 && y < k1) ? VT::load1(row + y * ES) : 0.f;
        p.part[r * p.K + k] = make_float4(G.m, G.d, G.S, xy);
    }
}

// Stage 2: the row's K partials combined by one warp in a fixed order (lane
// l takes partials l, l+32, ... in turn, then a butterfly), then the loss and
// the gradient of this CTA's chunk (head and tail one element per thread, the
// body in 16-byte vectors, as in stage 1).
template <typename T, bool GRAD, bool WT, bool VECOK>
__global__ void __launch_bounds__(kSplitThreads) ce_split_grad_kernel(const __grid_constant__ SplitArgs p) {
    static_assert(!(WT && VECOK), "the weighted pass takes the head/tail form");
    using VT = Vec<T>;
    constexpr int VEC = VT::kElems;
    constexpr int ES = sizeof(T);
    constexpr int PP = VEC / 2;
    __shared__ float s_lse, s_S;
    const int kper = GRAD ? p.K : 1;  // without a gradient one CTA per row
    const int64_t b = blockIdx.x;
    const int64_t r = b / kper;
    const int k = (int)(b - r * kper);
    int64_t y, off;
    row_of(p, r, y, off);
    const int64_t k0 = (int64_t)k * p.chunk;
    const int64_t k1 = min(p.V, k0 + p.chunk);
    char* row = p.logits + off * (int64_t)ES;
    const Span16 sp = span16<ES>(row, k0, k1);
    const int64_t ee = span16_edge(sp, k0, k1, threadIdx.x);
    uint4* rv = reinterpret_cast<uint4*>(row + sp.h1 * ES);

    if (y == p.ignore_idx || y < 0 || y >= p.V) {
        if (GRAD) {
            if (ee >= 0) VT::store1(row + ee * ES, 0.f);
            const uint4 z = make_uint4(0, 0, 0, 0);
            for (int64_t v = threadIdx.x; v < sp.nv; v += kSplitThreads) stg128_stream(rv + v, z);
        }
        if (k == 0 && threadIdx.x == 0) {
            p.loss[r] = (y == p.ignore_idx) ? 0.f : __int_as_float(0x7fc00000);
            if (p.lse_out) p.lse_out[r] = __int_as_float(0x7fc00000);
        }
        return;
    }

    const int lane = threadIdx.x & 31;
    if (threadIdx.x < 32) {
        const float4* pr = p.part + r * p.K;
        Part G = part_identity();
        for (int q = lane; q < p.K; q += 32) {
            const float4 w = pr[q];
            G = part_combine(G, Part{w.x, w.y, w.z});
        }
        G = warp_allreduce_part(G);
        if (lane == 0) {
            const float lse = G.m + logf(G.d);
            const float xy = pr[y / p.chunk].w;
            s_lse = lse;
            s_S = G.S;
            if (k == 0) {
                float loss;
                if (WT)  // (1-a) w_y (lse - x_y) + (a/V) (W lse - sum_j w_j x_j)
                    loss = (1.f - p.a) * __ldg(p.cw + y) * (lse - xy) +
                           p.a_over_v * ((float)(*p.wsum) * lse - G.S);
                else
                    loss = lse - (1.f - p.a) * xy - p.a_over_v * G.S;
                p.loss[r] = loss;
                if (p.lse_out) p.lse_out[r] = lse;
            }
        }
    }
    if (!GRAD) return;
    __syncthreads();
    const float lse = s_lse;
    float g;
    if (p.reduce)
        g = (p.dloss ? p.dloss[0] : 1.f) / (WT ? (float)(*p.wdenom) : (float)(*p.n_dev));
    else
        g = p.dloss ? p.dloss[r] : 1.f;
    const float nll = -lse * kLog2e;
    // gradient = c * softmax - b_j, minus the one-hot term at the target:
    //   unweighted c = g, b_j = g a/V;  weighted c = g ((1-a) w_y + (a/V) W),
    //   b_j = g (a/V) w_j, one-hot term g (1-a) w_y
    const float wy = WT ? __ldg(p.cw + y) : 1.f;
    const float c = WT ? g * ((1.f - p.a) * wy + p.a_over_v * (float)(*p.wsum)) : g;
    const float ga = g * p.a_over_v;
    const float hit = g * (1.f - p.a) * wy;
    if constexpr (VECOK) {
        const float2 L2 = make_float2(kLog2e, kLog2e), NL = make_float2(nll, nll);
        const float2 C2 = make_float2(c, c), NB = make_float2(-ga, -ga);
        uint4* rw = reinterpret_cast<uint4*>(row);
        const int64_t vend = k1 / VEC;
        for (int64_t vb = k0 / VEC + threadIdx.x; vb < vend; vb += kSplitThreads * kSplitBatch) {
            uint4 raw[kSplitBatch];
#pragma unroll
            for (int u = 0; u < kSplitBatch; ++u) {
                const int64_t v = vb + (int64_t)u * kSplitThreads;
                if (v < vend) raw[u] = __ldcs(rw + v);
            }
#pragma unroll
            for (int u = 0; u < kSplitBatch; ++u) {
                const int64_t v = vb + (int64_t)u * kSplitThreads;
                if (v >= vend) continue;
                float2 x[PP], o[PP];
                VT::unpack2(raw[u], x);
#pragma unroll
                for (int q = 0; q < PP; ++q) {
                    const float2 e = __ffma2_rn(x[q], L2, NL);
                    const float2 pe = make_float2(ex2_approx(e.x), ex2_approx(e.y));
                    o[q] = __ffma2_rn(pe, C2, NB);
                }
                if (v == y / VEC) {
                    const int ey = (int)(y % VEC);
#pragma unroll
                    for (int q = 0; q < PP; ++q) {
                        if (2 * q == ey) o[q].x -= hit;
                        if (2 * q + 1 == ey) o[q].y -= hit;
                    }
                }
                stg128_stream(rw + v, VT::pack2(o));
            }
        }
        return;
    }
    if (ee >= 0) {
        const float x = VT::load1(row + ee * ES);
        const float bj = WT ? ga * __ldg(p.cw + ee) : ga;
        float o = fmaf(ex2_approx(fmaf(x, kLog2e, nll)), c, -bj);
        if (ee == y) o -= hit;
        VT::store1(row + ee * ES, o);
    }
    const float2 L2 = make_float2(kLog2e, kLog2e), NL = make_float2(nll, nll);
    const float2 C2 = make_float2(c, c), NB = make_float2(-ga, -ga);
    const float* cwb = WT ? p.cw + sp.h1 : nullptr;
    const bool wvec = WT && reinterpret_cast<uintptr_t>(cwb) % 16 == 0;
    const int64_t yb = y - sp.h1;  // the target's place in the body
    for (int64_t vb = threadIdx.x; vb < sp.nv; vb += kSplitThreads * kSplitBatch) {
        uint4 raw[kSplitBatch];
#pragma unroll
        for (int u = 0; u < kSplitBatch; ++u) {
            const int64_t v = vb + (int64_t)u * kSplitThreads;
            if (v < sp.nv) raw[u] = __ldcs(rv + v);
        }
#pragma unroll
        for (int u = 0; u < kSplitBatch; ++u) {
            const int64_t v = vb + (int64_t)u * kSplitThreads;
            if (v >= sp.nv) continue;
            float2 x[PP], o[PP];
            float w[VEC];
            VT::unpack2(raw[u], x);
            if (WT) weights_of<VEC>(cwb + v * VEC, wvec, w);
#pragma unroll
            for (int q = 0; q < PP; ++q) {
                const float2 e = __ffma2_rn(x[q], L2, NL);
                const float2 pe = make_float2(ex2_approx(e.x), ex2_approx(e.y));
                if (WT) {
                    o[q] = __ffma2_rn(pe, C2, make_float2(-ga * w[2 * q], -ga * w[2 * q + 1]));
                } else {
                    o[q] = __ffma2_rn(pe, C2, NB);
                }
            }
            const int64_t ey = yb - v * VEC;
            if (ey >= 0 && ey < VEC) {
#pragma unroll
                for (int q = 0; q < PP; ++q) {
                    if (2 * q == ey) o[q].x -= hit;
                    if (2 * q + 1 == ey) o[q].y -= hit;
                }
            }
            stg128_stream(rv + v, VT::pack2(o));
        }
    }
}

template <typename T>
cudaError_t launch_split_typed(const Problem& pb, const SplitPlan& plan, float4* partials,
                               cudaStream_t s) {
    SplitArgs a;
    a.logits = pb.logits;
    a.s0 = pb.s0;
    a.s1 = pb.s1;
    a.dim1 = pb.dim1;
    a.N = pb.N;
    a.V = pb.V;
    a.chunk = plan.chunk;
    a.K = plan.chunks;
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
    a.part = partials;
    a.cw = pb.cw;
    a.wdenom = pb.wdenom;
    a.wsum = pb.wsum;
    const int64_t blocks = pb.N * plan.chunks;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const bool wt = pb.cw != nullptr;
    // whole 16-byte vectors when every row and chunk boundary is on the grid
    const bool vec = reinterpret_cast<uintptr_t>(pb.logits) % 16 == 0 &&
                     (pb.s0 * (int64_t)sizeof(T)) % 16 == 0 && (pb.s1 * (int64_t)sizeof(T)) % 16 == 0 &&
                     (pb.V * (int64_t)sizeof(T)) % 16 == 0 && (plan.chunk * (int64_t)sizeof(T)) % 16 == 0;
    const unsigned gs = (unsigned)blocks, gr = (unsigned)(pb.grad ? blocks : pb.N);
#define CE_SPLIT_LAUNCH(W, VK)                                                     \
    do {                                                                           \
        ce_split_stats_kernel<T, W, VK><<<gs, kSplitThreads, 0, s>>>(a);           \
        cudaError_t e_ = cudaGetLastError();                                       \
        if (e_ != cudaSuccess) return e_;                                          \
        if (pb.grad)                                                               \
            ce_split_grad_kernel<T, true, W, VK><<<gr, kSplitThreads, 0, s>>>(a);  \
        else                                                                       \
            ce_split_grad_kernel<T, false, W, VK><<<gr, kSplitThreads, 0, s>>>(a); \
    } while (0)
    // (the weighted pass measured 1.7 % faster in the head/tail form, even on
    // aligned rows: 3.90 against 3.97 ms on the bench workload)
    if (wt)
        CE_SPLIT_LAUNCH(true, false);
    else if (vec)
        CE_SPLIT_LAUNCH(false, true);
    else
        CE_SPLIT_LAUNCH(false, false);
#undef CE_SPLIT_LAUNCH
    return cudaGetLastError();
}

}  // namespace

int split_auto_chunks(int64_t V) {
    int64_t k = (V + 16383) / 16384;  // 64 elements per thread
    if (k < 1) k = 1;
    if (k > 4096) k = 4096;
    return (int)k;
}

cudaError_t launch_split(const Problem& p, const SplitPlan& plan, float4* partials, cudaStream_t s) {
    switch (p.dtype) {
        case CE_F32:
            return launch_split_typed<float>(p, plan, partials, s);
        case CE_BF16:
            return launch_split_typed<__nv_bfloat16>(p, plan, partials, s);
        default:
            return launch_split_typed<__half>(p, plan, partials, s);
    }
}

}  // namespace gbce
