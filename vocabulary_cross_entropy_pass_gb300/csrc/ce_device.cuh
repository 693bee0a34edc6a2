// ce_device.cuh -- device helpers of the fused cross-entropy kernels (sm_103a).
//
// Thin inline-PTX wrappers (mbarrier, 1-D TMA bulk copies, cluster barriers,
// distributed shared memory), 16-byte vector traits for the three storage
// dtypes, and the (max, sum-exp, sum) partial that every level of the
// reduction combines.  The partial and its combine are the per-chunk
// statistics that mindspore/hyper-parallel #269 (section 3.1) exchanges between
// vocabulary-parallel ranks with MAX and SUM all-reduces; here they are
// exchanged between warps, CTAs of a cluster, or kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gbce {

constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;
// Bounded waits give up after this many nanoseconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 1500ull * 1000ull * 1000ull;

// ----------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on one mbarrier phase.  Returns false when the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0u && global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src and bytes must all be multiples of 16.
__device__ __forceinline__ void tma_load_1d(void* dst, const void* src, uint32_t bytes,
                                            uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t ncluster_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Whole-cluster barrier; release/acquire orders shared-memory writes made
// before it against distributed-shared-memory reads made after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Read a float4 from the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ float4 ld_dsmem_f4(const void* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(remote)
                 : "memory");
    return v;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start before the previous kernel on the stream ends;
// griddep_wait() blocks until that kernel has finished and its writes are
// visible, griddep_launch_dependents() lets the next kernel start early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint4 lds128(const void* p) {
    return *reinterpret_cast<const uint4*>(p);
}

__device__ __forceinline__ void stg128_stream(void* p, uint4 v) {
    __stcs(reinterpret_cast<uint4*>(p), v);
}

// ----------------------------------------------------------------- dtype traits
template <typename T>
struct Vec;  // one 16-byte vector of T

template <>
struct Vec<float> {
    static constexpr int kElems = 4;
    __device__ __forceinline__ static float vmax(const uint4& r) {
        return fmaxf(fmaxf(__uint_as_float(r.x), __uint_as_float(r.y)),
                     fmaxf(__uint_as_float(r.z), __uint_as_float(r.w)));
    }
    __device__ __forceinline__ static void unpack(const uint4& r, float* x) {
        x[0] = __uint_as_float(r.x);
        x[1] = __uint_as_float(r.y);
        x[2] = __uint_as_float(r.z);
        x[3] = __uint_as_float(r.w);
    }
    __device__ __forceinline__ static uint4 pack(const float* g) {
        return make_uint4(__float_as_uint(g[0]), __float_as_uint(g[1]), __float_as_uint(g[2]),
                          __float_as_uint(g[3]));
    }
    // pairs of consecutive elements, for packed f32x2 arithmetic
    __device__ __forceinline__ static void unpack2(const uint4& r, float2* x) {
        x[0] = make_float2(__uint_as_float(r.x), __uint_as_float(r.y));
        x[1] = make_float2(__uint_as_float(r.z), __uint_as_float(r.w));
    }
    __device__ __forceinline__ static uint4 pack2(const float2* g) {
        return make_uint4(__float_as_uint(g[0].x), __float_as_uint(g[0].y), __float_as_uint(g[1].x),
                          __float_as_uint(g[1].y));
    }
    // running max of a tile: kept as a float for fp32
    using Max = float;
    __device__ __forceinline__ static Max max_init() { return -INFINITY; }
    __device__ __forceinline__ static Max max_acc(Max m, const uint4& r) { return fmaxf(m, vmax(r)); }
    __device__ __forceinline__ static float max_done(Max m) { return m; }
    __device__ __forceinline__ static float load1(const void* p) {
        return *reinterpret_cast<const float*>(p);
    }
    __device__ __forceinline__ static void store1(void* p, float v) {
        *reinterpret_cast<float*>(p) = v;
    }
};

__device__ __forceinline__ __nv_bfloat162 as_bf162(uint32_t u) {
    return *reinterpret_cast<__nv_bfloat162*>(&u);
}
__device__ __forceinline__ uint32_t bf162_bits(__nv_bfloat162 v) {
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ __half2 as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }
__device__ __forceinline__ uint32_t h2_bits(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }

template <>
struct Vec<__nv_bfloat16> {
    static constexpr int kElems = 8;
    __device__ __forceinline__ static float vmax(const uint4& r) {
        // max is exact in bf16, so take it on packed pairs
        __nv_bfloat162 m = __hmax2(__hmax2(as_bf162(r.x), as_bf162(r.y)),
                                   __hmax2(as_bf162(r.z), as_bf162(r.w)));
        return fmaxf(__low2float(m), __high2float(m));
    }
    __device__ __forceinline__ static void unpack(const uint4& r, float* x) {
        // a bf16 is the upper half of an fp32
        x[0] = __uint_as_float(r.x << 16);
        x[1] = __uint_as_float(r.x & 0xffff0000u);
        x[2] = __uint_as_float(r.y << 16);
        x[3] = __uint_as_float(r.y & 0xffff0000u);
        x[4] = __uint_as_float(r.z << 16);
        x[5] = __uint_as_float(r.z & 0xffff0000u);
        x[6] = __uint_as_float(r.w << 16);
        x[7] = __uint_as_float(r.w & 0xffff0000u);
    }
    __device__ __forceinline__ static uint4 pack(const float* g) {
        return make_uint4(bf162_bits(__floats2bfloat162_rn(g[0], g[1])),
                          bf162_bits(__floats2bfloat162_rn(g[2], g[3])),
                          bf162_bits(__floats2bfloat162_rn(g[4], g[5])),
                          bf162_bits(__floats2bfloat162_rn(g[6], g[7])));
    }
    __device__ __forceinline__ static void unpack2(const uint4& r, float2* x) {
        x[0] = make_float2(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xffff0000u));
        x[1] = make_float2(__uint_as_float(r.y << 16), __uint_as_float(r.y & 0xffff0000u));
        x[2] = make_float2(__uint_as_float(r.z << 16), __uint_as_float(r.z & 0xffff0000u));
        x[3] = make_float2(__uint_as_float(r.w << 16), __uint_as_float(r.w & 0xffff0000u));
    }
    // one packed pair (4 bytes)
    __device__ __forceinline__ static float2 unpack_pair(uint32_t u) {
        return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
    }
    __device__ __forceinline__ static uint32_t pack_pair(float2 g) {
        return bf162_bits(__floats2bfloat162_rn(g.x, g.y));
    }
    __device__ __forceinline__ static uint4 pack2(const float2* g) {
        return make_uint4(bf162_bits(__floats2bfloat162_rn(g[0].x, g[0].y)),
                          bf162_bits(__floats2bfloat162_rn(g[1].x, g[1].y)),
                          bf162_bits(__floats2bfloat162_rn(g[2].x, g[2].y)),
                          bf162_bits(__floats2bfloat162_rn(g[3].x, g[3].y)));
    }
    // running max of a tile: kept packed (max is exact in bf16)
    using Max = __nv_bfloat162;
    __device__ __forceinline__ static Max max_init() { return as_bf162(0xff80ff80u); }  // -inf, -inf
    __device__ __forceinline__ static Max max_acc(Max m, const uint4& r) {
        return __hmax2(m, __hmax2(__hmax2(as_bf162(r.x), as_bf162(r.y)),
                                  __hmax2(as_bf162(r.z), as_bf162(r.w))));
    }
    __device__ __forceinline__ static float max_done(Max m) {
        return fmaxf(__low2float(m), __high2float(m));
    }
    __device__ __forceinline__ static float load1(const void* p) {
        return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
    }
    __device__ __forceinline__ static void store1(void* p, float v) {
        *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(v);
    }
};

template <>
struct Vec<__half> {
    static constexpr int kElems = 8;
    __device__ __forceinline__ static float vmax(const uint4& r) {
        __half2 m = __hmax2(__hmax2(as_h2(r.x), as_h2(r.y)), __hmax2(as_h2(r.z), as_h2(r.w)));
        return fmaxf(__low2float(m), __high2float(m));
    }
    __device__ __forceinline__ static void unpack(const uint4& r, float* x) {
        float2 a = __half22float2(as_h2(r.x));
        float2 b = __half22float2(as_h2(r.y));
        float2 c = __half22float2(as_h2(r.z));
        float2 d = __half22float2(as_h2(r.w));
        x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
        x[4] = c.x; x[5] = c.y; x[6] = d.x; x[7] = d.y;
    }
    __device__ __forceinline__ static uint4 pack(const float* g) {
        return make_uint4(h2_bits(__floats2half2_rn(g[0], g[1])), h2_bits(__floats2half2_rn(g[2], g[3])),
                          h2_bits(__floats2half2_rn(g[4], g[5])), h2_bits(__floats2half2_rn(g[6], g[7])));
    }
    __device__ __forceinline__ static void unpack2(const uint4& r, float2* x) {
        x[0] = __half22float2(as_h2(r.x));
        x[1] = __half22float2(as_h2(r.y));
        x[2] = __half22float2(as_h2(r.z));
        x[3] = __half22float2(as_h2(r.w));
    }
    __device__ __forceinline__ static float2 unpack_pair(uint32_t u) { return __half22float2(as_h2(u)); }
    __device__ __forceinline__ static uint32_t pack_pair(float2 g) { return h2_bits(__floats2half2_rn(g.x, g.y)); }
    __device__ __forceinline__ static uint4 pack2(const float2* g) {
        return make_uint4(h2_bits(__floats2half2_rn(g[0].x, g[0].y)), h2_bits(__floats2half2_rn(g[1].x, g[1].y)),
                          h2_bits(__floats2half2_rn(g[2].x, g[2].y)), h2_bits(__floats2half2_rn(g[3].x, g[3].y)));
    }
    using Max = __half2;
    __device__ __forceinline__ static Max max_init() { return as_h2(0xfc00fc00u); }  // -inf, -inf
    __device__ __forceinline__ static Max max_acc(Max m, const uint4& r) {
        return __hmax2(m, __hmax2(__hmax2(as_h2(r.x), as_h2(r.y)), __hmax2(as_h2(r.z), as_h2(r.w))));
    }
    __device__ __forceinline__ static float max_done(Max m) {
        return fmaxf(__low2float(m), __high2float(m));
    }
    __device__ __forceinline__ static float load1(const void* p) {
        return __half2float(*reinterpret_cast<const __half*>(p));
    }
    __device__ __forceinline__ static void store1(void* p, float v) {
        *reinterpret_cast<__half*>(p) = __float2half_rn(v);
    }
};

// ----------------------------------------------------------------- partials
// Statistics of a set of logits: running max m, sum-exp d relative to m, and
// the plain sum S (needed by label smoothing).  The empty set is (-inf, 0, 0).
struct Part {
    float m, d, S;
};

__device__ __forceinline__ Part part_identity() { return Part{-INFINITY, 0.f, 0.f}; }

// Commutative combine: both terms are rescaled to the common max, so
// combine(a, b) and combine(b, a) give the same bits.  This makes every lane
// of a butterfly end with identical results.
__device__ __forceinline__ Part part_combine(Part a, Part b) {
    const float m = fmaxf(a.m, b.m);
    const float da = (a.m == -INFINITY) ? 0.f : a.d * ex2_approx((a.m - m) * kLog2e);
    const float db = (b.m == -INFINITY) ? 0.f : b.d * ex2_approx((b.m - m) * kLog2e);
    return Part{m, da + db, a.S + b.S};
}

__device__ __forceinline__ Part warp_allreduce_part(Part p) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        Part q;
        q.m = __shfl_xor_sync(kFull, p.m, off);
        q.d = __shfl_xor_sync(kFull, p.d, off);
        q.S = __shfl_xor_sync(kFull, p.S, off);
        p = part_combine(p, q);
    }
    return p;
}

__device__ __forceinline__ float warp_allmax(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, off));
    return v;
}

// Max over the warp in one instruction (sm_100 family): every lane gets it.
__device__ __forceinline__ float warp_max_redux(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float warp_allsum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
    return v;
}

// The first level of the fixed-order mean, the same on every run: this
// thread's share of x[0 .. n) summed in double in a fixed order (t: the
// thread's index among T threads), eight loads in flight at a time.  On a
// 16-byte aligned x the thread takes 4-float groups t, t + T, ..., eight at a
// time, and adds the eight groups in float as a fixed tree -- each group
// (x0 + x1) + (x2 + x3), then the groups pairwise -- before one double add
// (a 32nd of the double adds, which this GPU issues slowly, and a quarter of
// the loads; the float tree's error, a few units in 2^-24 of its 32 values,
// stays far below the mean's tolerance); threads t < n % 4 take one element
// each of the last n % 4.  Otherwise single elements t, t + T, ....
__device__ __forceinline__ double strided_sum_fixed(const float* x, int64_t n, int t, int T) {
    constexpr int B = 8;
    double acc = 0.0;
    if (reinterpret_cast<uintptr_t>(x) % 16 == 0) {
        const float4* x4 = reinterpret_cast<const float4*>(x);
        const int64_t n4 = n / 4;
        for (int64_t q0 = t; q0 < n4; q0 += (int64_t)T * B) {
            float4 v[B];
#pragma unroll
            for (int u = 0; u < B; ++u) {
                const int64_t q = q0 + (int64_t)u * T;
                v[u] = q < n4 ? __ldcg(x4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float f[B];
#pragma unroll
            for (int u = 0; u < B; ++u) f[u] = (v[u].x + v[u].y) + (v[u].z + v[u].w);  // 0 past n4
            acc += (double)(((f[0] + f[1]) + (f[2] + f[3])) + ((f[4] + f[5]) + (f[6] + f[7])));
        }
        if (t < (int)(n - n4 * 4)) acc += (double)__ldcg(x + n4 * 4 + t);
        return acc;
    }
    for (int64_t r0 = t; r0 < n; r0 += (int64_t)T * B) {
        float v[B];
#pragma unroll
        for (int u = 0; u < B; ++u) {
            const int64_t r = r0 + (int64_t)u * T;
            v[u] = r < n ? __ldcg(x + r) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < B; ++u)
            if (r0 + (int64_t)u * T < n) acc += (double)v[u];
    }
    return acc;
}

}  // namespace gbce
