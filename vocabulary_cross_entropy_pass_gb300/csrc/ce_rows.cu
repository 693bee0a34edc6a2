// ce_rows.cu -- the warp-per-row fused cross-entropy kernel for short rows.
//
// When a whole row fits in one shared-memory tile (up to 16 or 32 KB: V up to
// 8192 bf16/fp16 or 4096 fp32 per 16 KB), the per-row CTA barrier and
// reduction of the stream kernel are the cost, not the bytes.  Here one warp
// owns a row from start to end:
//
//   - a producer warp copies each kept row with one 1-D TMA bulk copy into a
//     tile of the warp that will take it (rows of ignored targets are not read:
//     the producer warp writes their zero gradient itself);
//   - consumer warp w takes the kept rows w, w + NW, w + 2 NW, ... of its CTA
//     and makes three sweeps over the tile in shared memory: the row max, the
//     sum of 2^((x - m) log2e) and the plain sum (warp shuffles combine the
//     lanes: lse = m + log d, CSDN "Ascend CANN ops-nn cross-entropy fusion",
//     pitfall 1), then the gradient g (softmax - a/V) - g (1-a) [j == y]
//     (same article, "Backward", pitfall 3, smoothing over V) stored in place
//     over the row (TENPU #29 section 6) with 16-byte streaming stores.
//
// Each consumer warp owns TPW tiles of its own (TPW = stages / NW), used in
// turn, so every mbarrier phase of a tile is waited on by that one warp, in
// order: a parity wait can never mistake a later phase for an earlier one.
//
// One HBM read and one HBM write per element, two exponentials per element,
// no barrier wider than a warp after set-up.  Every wait is bounded.
#include "ce_device.cuh"
#include "ce_internal.h"

namespace gbce {
namespace {

struct RowsArgs {
    char* logits;
    int64_t s0, s1, dim1, N;
    int32_t V;
    int32_t stages;
    uint32_t row_bytes;    // V * sizeof(T), a multiple of 16, <= tile bytes
    const int64_t* targets;
    int64_t ts0, ts1, ignore_idx;
    float a, a_over_v;
    int reduce;
    const float* dloss;
    float* loss;
    float* lse_out;
    const int64_t* n_dev;
    uint32_t* err;
    uint32_t* ticket;      // CTAs done (zeroed by the count kernel)
    float* mean_out;       // reduce_loss: the last CTA to finish writes the mean here
    int flat;              // row r at r * s1, its target at r * ts1
};

__device__ __forceinline__ void mbar_arrive_rows(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

constexpr int kRowsWarps = 6;  // consumer warps per CTA

template <typename T, int NW, int TB, bool GRAD>
__global__ void __launch_bounds__(NW * 32 + 32, 1)
ce_rows_kernel(const __grid_constant__ RowsArgs p) {
    using VT = Vec<T>;
    constexpr int VEC = VT::kElems;
    constexpr int ES = sizeof(T);
    constexpr int P = VEC / 2;

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)p.stages * TB);
    uint64_t* empty = full + 16;
    double* dred = reinterpret_cast<double*>(empty + 16);   // [NW]
    volatile int* flags = reinterpret_cast<volatile int*>(dred + NW);  // abort, last

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        flags[0] = 0;
        flags[1] = 0;
        fence_barrier_init();
    }
    __syncthreads();

    auto row_target = [&](int64_t r) -> int64_t {
        if (p.flat) return __ldg(p.targets + r * p.ts1);
        const int64_t i = r / p.dim1, j = r - (r / p.dim1) * p.dim1;
        return __ldg(p.targets + i * p.ts0 + j * p.ts1);
    };
    auto row_ptr = [&](int64_t r) -> char* {
        if (p.flat) return p.logits + r * p.s1 * ES;
        const int64_t i = r / p.dim1, j = r - (r / p.dim1) * p.dim1;
        return p.logits + (i * p.s0 + j * p.s1) * ES;
    };
    auto is_loaded = [&](int64_t y) -> bool {
        return y != p.ignore_idx && y >= 0 && y < (int64_t)p.V;
    };
    const int nvec = (int)(p.row_bytes / 16);
    const int tpw = p.stages / NW;  // tiles per consumer warp

    // ------------------------------------------------------------ producer warp
    // Rows are examined 32 at a time, one per lane; a ballot gives the kept
    // ones, which lane 0 copies in order, and the warp zero-fills the others.
    if (warp == NW) {
        const uint64_t pol = l2_evict_first();
        uint32_t k = 0;         // kept rows seen
        uint32_t k_issued = 0;  // kept rows whose copy was issued (a prefix of them)
        for (int64_t q0 = 0;; q0 += 32) {
            const int64_t r = (int64_t)blockIdx.x + (q0 + lane) * (int64_t)gridDim.x;
            const bool valid = r < p.N;
            const int64_t y = valid ? row_target(r) : p.ignore_idx;
            const bool kept = valid && is_loaded(y);
            const unsigned vmask = __ballot_sync(kFull, valid);
            if (vmask == 0u) break;
            unsigned kmask = __ballot_sync(kFull, kept);
            unsigned zmask = vmask & ~kmask;
            while (zmask) {  // ignored (loss 0) or out of range (loss NaN): zero gradient, no read
                const int l = __ffs(zmask) - 1;
                zmask &= zmask - 1;
                const int64_t rl = __shfl_sync(kFull, r, l);
                const int64_t yl = __shfl_sync(kFull, y, l);
                char* row = row_ptr(rl);
                if (GRAD) {
                    const uint4 z = make_uint4(0, 0, 0, 0);
                    for (int v = lane; v < nvec; v += 32) stg128_stream(row + (size_t)v * 16, z);
                }
                if (lane == 0) {
                    p.loss[rl] = (yl == p.ignore_idx) ? 0.f : __int_as_float(0x7fc00000);
                    if (p.lse_out) p.lse_out[rl] = __int_as_float(0x7fc00000);
                }
            }
            while (kmask) {
                const int l = __ffs(kmask) - 1;
                kmask &= kmask - 1;
                const int64_t rl = __shfl_sync(kFull, r, l);
                if (lane == 0 && !flags[0]) {
                    // kept row k goes to warp k % NW, whose j-th row uses its tile j % TPW
                    const uint32_t j = k / NW;
                    const int tile = (int)(k % NW) * tpw + (int)(j % (uint32_t)tpw);
                    const uint32_t ph = (j / (uint32_t)tpw) & 1u;
                    if (!mbar_wait_bounded(&empty[tile], ph ^ 1u)) {
                        griddep_wait();  // the count kernel starts the error word
                        atomicOr(p.err, CE_DEVERR_TIMEOUT);
                        flags[0] = 1;
                    } else {
                        mbar_arrive_expect_tx(&full[tile], p.row_bytes);
                        tma_load_1d(ring + (size_t)tile * TB, row_ptr(rl), p.row_bytes, &full[tile],
                                    pol);
                        k_issued = k + 1;
                    }
                }
                ++k;
            }
        }
        __syncwarp();
        if (lane == 0 && flags[0]) {
            // let every copy already issued land before the CTA goes away: the
            // last phase issued on each tile
            for (int w = 0; w < NW; ++w) {
                const uint32_t rows_w =
                    (k_issued > (uint32_t)w) ? (k_issued - 1u - (uint32_t)w) / NW + 1u : 0u;
                for (int i = 0; i < tpw; ++i) {
                    if (rows_w > (uint32_t)i) {
                        const uint32_t uses = (rows_w - 1u - (uint32_t)i) / (uint32_t)tpw + 1u;
                        (void)mbar_wait_bounded(&full[w * tpw + i], (uses - 1u) & 1u);
                    }
                }
            }
        }
        if (p.mean_out) {
            // the producer warp's loss writes of ignored rows must precede the
            // CTA's done-ticket
            __threadfence();
            asm volatile("bar.arrive 1, %0;" ::"r"((NW + 1) * 32) : "memory");
        }
        return;
    }

    // ------------------------------------------------------------ consumer warps
    // n and the error word come from the count kernel, which may still run:
    // a warp waits for it (griddepcontrol.wait) only where it first needs
    // them -- its first gradient sweep, an error to record, or the mean --
    // so its first row's statistics overlap the count
    bool counted = false;
    float g_reduce = 1.f;
    auto need_count = [&]() {
        if (!counted) {
            griddep_wait();
            if (p.reduce) g_reduce = (p.dloss ? __ldg(p.dloss) : 1.f) / (float)(*p.n_dev);
            counted = true;
        }
    };
    uint32_t k = 0;  // kept rows seen by the whole CTA
    const float2 L2 = make_float2(kLog2e, kLog2e);
    for (int64_t q0 = 0;; q0 += 32) {
      // 32 rows at a time, one per lane; this warp takes kept rows k = warp (mod NW)
      const int64_t rq = (int64_t)blockIdx.x + (q0 + lane) * (int64_t)gridDim.x;
      const bool valid = rq < p.N;
      const int64_t yq = valid ? row_target(rq) : p.ignore_idx;
      const unsigned vmask = __ballot_sync(kFull, valid);
      if (vmask == 0u) break;
      unsigned kmask = __ballot_sync(kFull, valid && is_loaded(yq));
      while (kmask) {
        const int l = __ffs(kmask) - 1;
        kmask &= kmask - 1;
        const uint32_t mine = k++;
        if ((int)(mine % (uint32_t)NW) != warp) continue;
        const int64_t r = __shfl_sync(kFull, rq, l);
        const int64_t y = __shfl_sync(kFull, yq, l);
        const uint32_t j = mine / NW;  // this warp's j-th kept row
        const int s = warp * tpw + (int)(j % (uint32_t)tpw);
        const uint32_t ph = (j / (uint32_t)tpw) & 1u;
        if (!flags[0] && !mbar_wait_bounded(&full[s], ph)) {
            need_count();  // the count kernel starts the error word
            atomicOr(p.err, CE_DEVERR_TIMEOUT);
            flags[0] = 1;
        }
        const uint4* tile = reinterpret_cast<const uint4*>(ring + (size_t)s * TB);

        // sweep 1: row max (packed pairs), warp-wide
        typename VT::Max pm = VT::max_init();
#pragma unroll 4
        for (int v = lane; v < nvec; v += 32) pm = VT::max_acc(pm, tile[v]);
        const float m = warp_max_redux(VT::max_done(pm));
        const float nml = -m * kLog2e;
        const float2 NM = make_float2(nml, nml);

        // sweep 2: sum of 2^((x - m) log2e) and of x, packed f32x2
        float2 d2 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
#pragma unroll 4
        for (int v = lane; v < nvec; v += 32) {
            float2 x[P];
            VT::unpack2(tile[v], x);
#pragma unroll
            for (int j = 0; j < P; ++j) {
                const float2 e = __ffma2_rn(x[j], L2, NM);
                d2 = __fadd2_rn(d2, make_float2(ex2_approx(e.x), ex2_approx(e.y)));
                s2 = __fadd2_rn(s2, x[j]);
            }
        }
        const float d = warp_allsum(d2.x + d2.y);
        const float S = (p.a != 0.f) ? warp_allsum(s2.x + s2.y) : 0.f;
        const float lse = m + logf(d);
        const float xy = VT::load1(reinterpret_cast<const unsigned char*>(tile) + y * ES);
        if (lane == 0) {
            p.loss[r] = lse - (1.f - p.a) * xy - p.a_over_v * S;
            if (p.lse_out) p.lse_out[r] = lse;
        }

        // sweep 3: gradient over the row, stored in place
        if (GRAD) {
            need_count();
            const float g = p.reduce ? g_reduce : (p.dloss ? __ldg(p.dloss + r) : 1.f);
            char* rowp = row_ptr(r);
            const float nll = -lse * kLog2e;
            const float bb = g * p.a_over_v;
            const float2 NL = make_float2(nll, nll);
            const float2 G2 = make_float2(g, g);
            const float2 NB = make_float2(-bb, -bb);
            uint4* dst = reinterpret_cast<uint4*>(rowp);
#pragma unroll 4
            for (int v = lane; v < nvec; v += 32) {
                float2 x[P], o[P];
                VT::unpack2(tile[v], x);
#pragma unroll
                for (int j = 0; j < P; ++j) {
                    const float2 e = __ffma2_rn(x[j], L2, NL);
                    o[j] = __ffma2_rn(make_float2(ex2_approx(e.x), ex2_approx(e.y)), G2, NB);
                }
                stg128_stream(dst + v, VT::pack2(o));
            }
            // the target element: the lane that stored its vector rewrites it
            if (lane == (int)((y / VEC) % 32)) {
                const float e = ex2_approx(fmaf(xy, kLog2e, nll));
                VT::store1(rowp + y * ES, fmaf(e, g, -bb) - g * (1.f - p.a));
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_rows(&empty[s]);
      }
    }

    // reduce_loss: the last CTA to finish sums the per-row losses in a fixed order
    need_count();  // the mean divides by n; a warp with no gradient sweep has not waited yet
    if (p.mean_out) {
        // wait for the producer warp's loss writes, then take the ticket
        __threadfence();
        asm volatile("bar.sync 1, %0;" ::"r"((NW + 1) * 32) : "memory");
        if (tid == 0) {
            __threadfence();
            const unsigned t = atomicAdd(p.ticket, 1u);
            flags[1] = (t == gridDim.x - 1) ? 1 : 0;
        }
        asm volatile("bar.sync 2, %0;" ::"r"(NW * 32) : "memory");
        if (flags[1]) {
            __threadfence();
            double acc = strided_sum_fixed(p.loss, p.N, tid, NW * 32);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
            if (lane == 0) dred[warp] = acc;
            asm volatile("bar.sync 2, %0;" ::"r"(NW * 32) : "memory");
            if (tid == 0) {
                double tot = 0.0;
                for (int w = 0; w < NW; ++w) tot += dred[w];
                p.mean_out[0] = (float)(tot / (double)(*p.n_dev));  // 0/0 = NaN: all ignored
            }
        }
    }
}

template <typename T, int NW, int TB, bool GRAD>
cudaError_t launch_rows_one(const Problem& pb, const RowsPlan& plan, cudaStream_t s) {
    auto kern = ce_rows_kernel<T, NW, TB, GRAD>;
    RowsArgs a;
    a.logits = pb.logits;
    a.s0 = pb.s0;
    a.s1 = pb.s1;
    a.dim1 = pb.dim1;
    a.N = pb.N;
    a.V = (int32_t)pb.V;
    a.stages = plan.stages;
    a.row_bytes = (uint32_t)(pb.V * (int64_t)sizeof(T));
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
    a.ticket = pb.ticket;
    a.mean_out = pb.mean_out;
    a.flat = rows_flat(pb) ? 1 : 0;
    const size_t smem = (size_t)plan.stages * TB + 32 * sizeof(uint64_t) + NW * sizeof(double) +
                        2 * sizeof(int) + 16;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NW * 32 + 32, smem);
    if (e != cudaSuccess) return e;
    if (plan.ctas_per_sm_cap > 0 && per_sm > plan.ctas_per_sm_cap) per_sm = plan.ctas_per_sm_cap;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    int64_t grid = (int64_t)per_sm * sms;
    if (grid > pb.N) grid = pb.N;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    set_pdl_attr(&attr[0]);
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(NW * 32 + 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename T, bool GRAD>
cudaError_t launch_rows_typed(const Problem& pb, const RowsPlan& plan, cudaStream_t s) {
    if (plan.stages % kRowsWarps != 0) return cudaErrorInvalidValue;
    if (plan.tile_kb == 32) return launch_rows_one<T, kRowsWarps, 32 * 1024, GRAD>(pb, plan, s);
    return launch_rows_one<T, kRowsWarps, 16 * 1024, GRAD>(pb, plan, s);
}

}  // namespace

cudaError_t launch_rows(const Problem& p, const RowsPlan& plan, cudaStream_t s) {
    switch (p.dtype) {
        case CE_F32:
            return p.grad ? launch_rows_typed<float, true>(p, plan, s)
                          : launch_rows_typed<float, false>(p, plan, s);
        case CE_BF16:
            return p.grad ? launch_rows_typed<__nv_bfloat16, true>(p, plan, s)
                          : launch_rows_typed<__nv_bfloat16, false>(p, plan, s);
        default:
            return p.grad ? launch_rows_typed<__half, true>(p, plan, s)
                          : launch_rows_typed<__half, false>(p, plan, s);
    }
}

}  // namespace gbce
