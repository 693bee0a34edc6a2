// ce_bwd.cu -- the backward pass from a saved logsumexp.
//
// When the upstream gradient is known only after the forward (autograd), the
// forward-only pass saves lse = logsumexp(x) per row and this kernel writes
//   grad_j = g * (exp(x_j - lse) - a/V) - g * (1-a) * [j == y]
// (CSDN "Ascend CANN ops-nn cross-entropy fusion", section "Backward" and
// pitfall 3, smoothing spread over all V classes), g the row's upstream
// scale: dloss/n for the mean, dloss[r] per row.  Ignored and out-of-range
// rows get zeros.  One read of the logits and one write of the gradient per
// element, no reduction: a plain streaming kernel, 16-byte vectors between
// a scalar head and tail when the gradient rows sit at the logits rows'
// offset from a 16-byte boundary, element by element otherwise.  The
// gradient may overwrite the logits (TENPU "Parallel Cross Entropy (Triton)"
// #29 section 6, in-place staging) or go to a separate tensor.
#include "ce_device.cuh"
#include "ce_internal.h"
#include "ce_span.cuh"

namespace gbce {
namespace {

constexpr int kBwdThreads = 256;
constexpr int kBwdVecs = 4;  // 16-byte vectors per thread per chunk

struct BwdArgs {
    const char* logits;
    char* grad;
    int64_t s0, s1, gs0, gs1, dim1, N, V;
    int64_t chunk;         // elements per CTA-chunk
    int64_t nchunks;       // chunks per row
    const int64_t* targets;
    int64_t ts0, ts1, ignore_idx;
    const float* lse;
    float a, a_over_v;
    int reduce;
    const float* dloss;
    const int64_t* n_dev;
    int64_t voff, Vtot;    // vocabulary offset of column 0, and the size targets index
    int flat;              // row r at r * s1 (r * gs1), its target at r * ts1
};

// Rows of the logits and the gradient at the same offset from a 16-byte
// boundary (always so in place): each chunk's head and tail one element per
// thread, its body in 16-byte vectors.  ALIGNED: both tensors' rows on the
// 16-byte grid and V a whole number of vectors, so a chunk is whole vectors
// indexed from the row start (the head/tail form measured 4 % slower on the
// backward of the bench workload).
template <typename T, bool ALIGNED>
__global__ void __launch_bounds__(kBwdThreads) ce_bwd_vec_kernel(const __grid_constant__ BwdArgs p) {
    using VT = Vec<T>;
    constexpr int VEC = VT::kElems;
    constexpr int ES = sizeof(T);
    constexpr int PP = VEC / 2;
    const float2 L2 = make_float2(kLog2e, kLog2e);
    const int64_t total = p.N * p.nchunks;
    for (int64_t b = blockIdx.x; b < total; b += gridDim.x) {
        const int64_t r = b / p.nchunks;
        const int64_t c = b - r * p.nchunks;
        int64_t y;
        const char* srow;
        char* drow;
        if (p.flat) {
            y = __ldg(p.targets + r * p.ts1);
            srow = p.logits + r * p.s1 * ES;
            drow = p.grad + r * p.gs1 * ES;
        } else {
            const int64_t i = r / p.dim1, j = r - i * p.dim1;
            y = __ldg(p.targets + i * p.ts0 + j * p.ts1);
            srow = p.logits + (i * p.s0 + j * p.s1) * ES;
            drow = p.grad + (i * p.gs0 + j * p.gs1) * ES;
        }
        const int64_t e0 = c * p.chunk, e1 = min(p.V, (c + 1) * p.chunk);
        if constexpr (ALIGNED) {
            const uint4* src = reinterpret_cast<const uint4*>(srow);
            uint4* dst = reinterpret_cast<uint4*>(drow);
            const int64_t v0 = e0 / VEC, v1 = e1 / VEC;
            if (y == p.ignore_idx || y < 0 || y >= p.Vtot) {
                const uint4 z = make_uint4(0, 0, 0, 0);
                for (int64_t v = v0 + threadIdx.x; v < v1; v += kBwdThreads) stg128_stream(dst + v, z);
                continue;
            }
            float g;
            if (p.reduce)
                g = (p.dloss ? __ldg(p.dloss) : 1.f) / (float)(*p.n_dev);
            else
                g = p.dloss ? __ldg(p.dloss + r) : 1.f;
            const float nll = -__ldg(p.lse + r) * kLog2e;
            const float bb = g * p.a_over_v;
            const float2 NL = make_float2(nll, nll), G2 = make_float2(g, g), NB = make_float2(-bb, -bb);
            const int64_t yl = y - p.voff;  // the target's column in these logits
            const int64_t vy = (yl >= 0 && yl < p.V) ? yl / VEC : -1;
            const int ey = (int)(yl >= 0 ? yl % VEC : 0);
            const float hit = g * (1.f - p.a);
            for (int64_t vb = v0 + threadIdx.x; vb < v1; vb += kBwdThreads * kBwdVecs) {
                uint4 raw[kBwdVecs];
#pragma unroll
                for (int u = 0; u < kBwdVecs; ++u) {
                    const int64_t v = vb + (int64_t)u * kBwdThreads;
                    if (v < v1) raw[u] = __ldcs(src + v);
                }
#pragma unroll
                for (int u = 0; u < kBwdVecs; ++u) {
                    const int64_t v = vb + (int64_t)u * kBwdThreads;
                    if (v < v1) {
                        float2 x[PP], o[PP];
                        VT::unpack2(raw[u], x);
#pragma unroll
                        for (int q = 0; q < PP; ++q) {
                            const float2 e = __ffma2_rn(x[q], L2, NL);
                            o[q] = __ffma2_rn(make_float2(ex2_approx(e.x), ex2_approx(e.y)), G2, NB);
                        }
                        if (v == vy) {
#pragma unroll
                            for (int q = 0; q < PP; ++q) {
                                if (2 * q == ey) o[q].x -= hit;
                                if (2 * q + 1 == ey) o[q].y -= hit;
                            }
                        }
                        stg128_stream(dst + v, VT::pack2(o));
                    }
                }
            }
            continue;
        }
        const Span16 sp = span16<ES>(srow, e0, e1);
        const int64_t ee = span16_edge(sp, e0, e1, threadIdx.x);
        const uint4* src = reinterpret_cast<const uint4*>(srow + sp.h1 * ES);
        uint4* dst = reinterpret_cast<uint4*>(drow + sp.h1 * ES);
        if (y == p.ignore_idx || y < 0 || y >= p.Vtot) {
            if (ee >= 0) VT::store1(drow + ee * ES, 0.f);
            const uint4 z = make_uint4(0, 0, 0, 0);
            for (int64_t v = threadIdx.x; v < sp.nv; v += kBwdThreads) stg128_stream(dst + v, z);
            continue;
        }
        float g;
        if (p.reduce)
            g = (p.dloss ? __ldg(p.dloss) : 1.f) / (float)(*p.n_dev);
        else
            g = p.dloss ? __ldg(p.dloss + r) : 1.f;
        const float nll = -__ldg(p.lse + r) * kLog2e;
        const float bb = g * p.a_over_v;
        const float hit = g * (1.f - p.a);
        const int64_t yl = y - p.voff;  // the target's column in these logits
        if (ee >= 0) {
            const float x = VT::load1(srow + ee * ES);
            float o = fmaf(ex2_approx(fmaf(x, kLog2e, nll)), g, -bb);
            if (ee == yl) o -= hit;
            VT::store1(drow + ee * ES, o);
        }
        const float2 NL = make_float2(nll, nll), G2 = make_float2(g, g), NB = make_float2(-bb, -bb);
        const int64_t yb = yl - sp.h1;  // the target's place in the body
        for (int64_t vb = threadIdx.x; vb < sp.nv; vb += kBwdThreads * kBwdVecs) {
            uint4 raw[kBwdVecs];
#pragma unroll
            for (int u = 0; u < kBwdVecs; ++u) {
                const int64_t v = vb + (int64_t)u * kBwdThreads;
                if (v < sp.nv) raw[u] = __ldcs(src + v);
            }
#pragma unroll
            for (int u = 0; u < kBwdVecs; ++u) {
                const int64_t v = vb + (int64_t)u * kBwdThreads;
                if (v < sp.nv) {
                    float2 x[PP], o[PP];
                    VT::unpack2(raw[u], x);
#pragma unroll
                    for (int q = 0; q < PP; ++q) {
                        const float2 e = __ffma2_rn(x[q], L2, NL);
                        o[q] = __ffma2_rn(make_float2(ex2_approx(e.x), ex2_approx(e.y)), G2, NB);
                    }
                    const int64_t ey = yb - v * VEC;
                    if (ey >= 0 && ey < VEC) {
#pragma unroll
                        for (int q = 0; q < PP; ++q) {
                            if (2 * q == ey) o[q].x -= hit;
                            if (2 * q + 1 == ey) o[q].y -= hit;
                        }
                    }
                    stg128_stream(dst + v, VT::pack2(o));
                }
            }
        }
    }
}

// Rows of the two tensors at different offsets from a 16-byte boundary:
// element by element.
template <typename T>
__global__ void __launch_bounds__(kBwdThreads) ce_bwd_scalar_kernel(const __grid_constant__ BwdArgs p) {
    using VT = Vec<T>;
    constexpr int ES = sizeof(T);
    const int64_t total = p.N * p.nchunks;
    for (int64_t b = blockIdx.x; b < total; b += gridDim.x) {
        const int64_t r = b / p.nchunks;
        const int64_t c = b - r * p.nchunks;
        const int64_t i = r / p.dim1, j = r - i * p.dim1;
        const int64_t y = __ldg(p.targets + i * p.ts0 + j * p.ts1);
        const char* src = p.logits + (i * p.s0 + j * p.s1) * ES;
        char* dst = p.grad + (i * p.gs0 + j * p.gs1) * ES;
        const int64_t e0 = c * p.chunk, e1 = min(p.V, (c + 1) * p.chunk);
        if (y == p.ignore_idx || y < 0 || y >= p.Vtot) {
            for (int64_t e = e0 + threadIdx.x; e < e1; e += kBwdThreads) VT::store1(dst + e * ES, 0.f);
            continue;
        }
        float g;
        if (p.reduce)
            g = (p.dloss ? __ldg(p.dloss) : 1.f) / (float)(*p.n_dev);
        else
            g = p.dloss ? __ldg(p.dloss + r) : 1.f;
        const float nll = -__ldg(p.lse + r) * kLog2e;
        const float bb = g * p.a_over_v;
        for (int64_t e = e0 + threadIdx.x; e < e1; e += kBwdThreads) {
            const float x = VT::load1(src + e * ES);
            float o = fmaf(ex2_approx(fmaf(x, kLog2e, nll)), g, -bb);
            if (e + p.voff == y) o -= g * (1.f - p.a);
            VT::store1(dst + e * ES, o);
        }
    }
}

template <typename T>
cudaError_t launch_bwd_typed(const BwdProblem& bp, cudaStream_t s) {
    BwdArgs a;
    a.logits = bp.logits;
    a.grad = bp.grad;
    a.s0 = bp.s0;
    a.s1 = bp.s1;
    a.gs0 = bp.gs0;
    a.gs1 = bp.gs1;
    a.dim1 = bp.dim1;
    a.N = bp.N;
    a.V = bp.V;
    a.chunk = (int64_t)kBwdThreads * kBwdVecs * Vec<T>::kElems;
    a.nchunks = (bp.V + a.chunk - 1) / a.chunk;
    a.targets = bp.targets;
    a.ts0 = bp.ts0;
    a.ts1 = bp.ts1;
    a.ignore_idx = bp.ignore_idx;
    a.lse = bp.lse;
    a.a = bp.a;
    a.voff = bp.vocab_offset;
    a.Vtot = bp.V_total;
    a.a_over_v = bp.a / (float)bp.V_total;
    a.reduce = bp.reduce;
    a.dloss = bp.dloss;
    a.n_dev = bp.n_dev;
    {
        const int64_t lim = (int64_t)1 << 31;
        a.flat = (bp.dim1 >= 1 && bp.dim1 < lim && bp.s1 >= 0 && bp.s1 < lim && bp.gs1 >= 0 && bp.gs1 < lim &&
                  bp.ts1 >= 0 && bp.ts1 < lim && bp.s0 == bp.dim1 * bp.s1 && bp.gs0 == bp.dim1 * bp.gs1 &&
                  bp.ts0 == bp.dim1 * bp.ts1)
                     ? 1
                     : 0;
    }
    constexpr int64_t ES = sizeof(T);
    const bool aligned = bp.vec_ok && reinterpret_cast<uintptr_t>(bp.logits) % 16 == 0 &&
                         reinterpret_cast<uintptr_t>(bp.grad) % 16 == 0 && (bp.s0 * ES) % 16 == 0 &&
                         (bp.s1 * ES) % 16 == 0 && (bp.gs0 * ES) % 16 == 0 && (bp.gs1 * ES) % 16 == 0 &&
                         (bp.V * ES) % 16 == 0;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t grid = bp.N * a.nchunks;
    const int64_t cap = (int64_t)sms * 8;  // grid-stride beyond 8 CTAs per SM
    if (grid > cap) grid = cap;
    if (grid < 1) return cudaSuccess;
    if (aligned)
        ce_bwd_vec_kernel<T, true><<<(unsigned)grid, kBwdThreads, 0, s>>>(a);
    else if (bp.vec_ok)
        ce_bwd_vec_kernel<T, false><<<(unsigned)grid, kBwdThreads, 0, s>>>(a);
    else
        ce_bwd_scalar_kernel<T><<<(unsigned)grid, kBwdThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdProblem& bp, cudaStream_t s) {
    switch (bp.dtype) {
        case CE_F32:
            return launch_bwd_typed<float>(bp, s);
        case CE_BF16:
            return launch_bwd_typed<__nv_bfloat16>(bp, s);
        default:
            return launch_bwd_typed<__half>(bp, s);
    }
}

}  // namespace gbce
