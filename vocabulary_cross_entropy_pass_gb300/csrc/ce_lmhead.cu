// ce_lmhead.cu -- the lm_head projection on the 5th-generation tensor cores
// with the cross-entropy statistics in its epilogue.
//
// hyper-parallel #269 (background: the TorchTitan ChunkedLossWrapper) runs the
// lm_head projection and the loss a chunk of rows at a time.  Here the logits
// tiles come off the tensor cores straight into the online-softmax
// statistics.  For one chunk of rows, logits = hidden . W^T:
//
//   ce_lmhead2_kernel  (chunks of 256 rows or more) the paired-SM form below:
//              a cluster of two CTAs per 256 x 256 tile, tcgen05.mma
//              .cta_group::2, each SM loading half of each operand;
//   ce_lmhead_kernel   (smaller chunks) a persistent kernel over 128 x 256
//              output tiles, one CTA each:
//     warp 0   issues TMA tile loads (128-byte swizzle) of hidden (128 x 64)
//              and W (256 x 64) into a 4-deep ring of shared-memory stages;
//     warp 1   owns the tensor memory (two 256-column fp32 accumulators) and,
//              from one thread, issues tcgen05.mma (M 128, N 256, K 16) over
//              the ring, committing each stage back to the producer and each
//              finished accumulator to the epilogue;
//     warps 2-5  the epilogue: each thread reads its row of the accumulator
//              (tcgen05.ld, 32 columns at a time), rounds every logit to the
//              storage dtype (the logits the chunked pass works on), stores
//              them, and folds them into the tile's row partial -- running max
//              m, sum of exp(x - m), plain sum S, and the target logit when the
//              target's column lies in the tile -- written as one float4 per
//              (row, tile).  While it works, the MMA warp fills the other
//              accumulator.
//   ce_lm_combine_kernel  per row, the tiles' partials folded in a fixed
//     order -- the (m, d, x_y) combine of the vocabulary-parallel ranks of
//     hyper-parallel #269 section 3.1 -- into lse and the row's loss
//     lse - (1-a) x_y - (a/V) S (CSDN "Ascend CANN ops-nn cross-entropy
//     fusion", "Fusion scheme: log_softmax + NLL"; smoothing over V).
//
// Every wait is an mbarrier poll bounded by %globaltimer; a wait that gives up
// sets CE_DEVERR_TIMEOUT, stops the kernel's roles, lets issued copies and
// MMAs complete (bounded) and frees the tensor memory before returning.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include <mutex>

#include "ce_device.cuh"
#include "ce_internal.h"

namespace gbce {
namespace {

constexpr int kBM = 128;   // tile rows (hidden rows)
constexpr int kBN = 256;   // tile columns (vocabulary)
constexpr int kBK = 64;    // K per stage: 64 16-bit values = one 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;          // 16 KB
constexpr int kBBytes = kBN * kBK * 2;          // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;  // 48 KB
constexpr int kLmThreads = 192;                 // 6 warps
constexpr uint32_t kTmemCols = 2 * kBN;         // two fp32 accumulators
// Each epilogue warp stages 64 columns of its 32 rows (4 KB) in shared memory
// to store them a row segment of 128 bytes at a time, after the barriers.
constexpr int kStoreStageBytes = 4 * 4096;
constexpr size_t kLmSmem = (size_t)kStages * kStageBytes + 1024 /* alignment */ + 256 + kStoreStageBytes;

struct LmArgs {
    int64_t rows;             // rows of this chunk
    int64_t V;
    int64_t ldl;              // elements between logits rows in the output
    char* logits;             // out: (rows, ldl) in the storage dtype
    float4* part;             // out: [rows][ntn] {m, d, S, x_y}
    const int64_t* targets;   // [rows]
    int64_t ignore_idx;
    int mb, ntn;              // row blocks, column tiles
    int ksteps;               // ceil(H / 64)
    uint32_t* err;
};

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrives on `bar` once every tcgen05.mma this thread issued so far is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// D[tmem] (+)= A[smem] . B[smem]^T, both K-major; accumulate when acc != 0.
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
          "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
          "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand written by TMA with
// the 128-byte swizzle: 8-row atoms of 128 bytes, 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
    d |= (uint64_t)1 << 16;                              // leading offset (unused with this swizzle)
    d |= (uint64_t)(1024 >> 4) << 32;                    // stride offset: next 8-row atom
    d |= (uint64_t)1 << 46;                              // descriptor version
    d |= (uint64_t)2 << 61;                              // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B of the
// storage type (bf16 or fp16, both the same), both K-major, M 128, N 256.
template <typename T>
struct AbFormat;  // operand format code of kind::f16
template <>
struct AbFormat<__half> {
    static constexpr uint32_t kCode = 0;
};
template <>
struct AbFormat<__nv_bfloat16> {
    static constexpr uint32_t kCode = 1;
};

template <typename T>
__host__ __device__ constexpr uint32_t idesc_f16() {
    return (1u << 4) | (AbFormat<T>::kCode << 7) | (AbFormat<T>::kCode << 10) |
           ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}

// Orders the uses of 8 registers after the tcgen05.wait::ld before it: an
// empty volatile statement that takes and gives back the registers, so the
// compiler cannot move a use above the wait.
__device__ __forceinline__ void reg_fence8(uint32_t* r) {
    asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]));
}

// The epilogue's work on one accumulator row of this thread: the logits
// (row, j0 .. j0 + 255) read from TMEM (tbase: this row's lane, column j0)
// 32 columns at a time, the next 32 in flight while these are worked on;
// rounded to the storage dtype in pairs and stored (rows < p.rows); their
// statistics {m, d, S} over the columns inside the vocabulary, from the
// rounded values (what the chunk buffer holds), in packed f32x2 arithmetic.
// The target logit is read back from the stored row by the per-row combine.
// Stores: every 64 columns the warp's 32 rows x 128 bytes go through its 4 KB
// of shared memory (`stage`; 16-byte units of row r at unit u ^ (r & 7), so
// neither the writes by row nor the reads by row segment meet a bank
// conflict) and out as four rows of 128 contiguous bytes per instruction,
// instead of 32 rows of 16 bytes; where the vocabulary ends inside the 64
// columns each lane stores its own row's elements.
template <typename T>
__device__ __forceinline__ float4 epilogue_row(const LmArgs& p, uint32_t tbase, int64_t row,
                                               int64_t j0, uint4* stage, int lane) {
    using VT = Vec<T>;
    const bool live = row < p.rows;
    T* out = reinterpret_cast<T*>(p.logits) + row * p.ldl;
    const int64_t row0 = row - lane;  // the warp's first row
    uint32_t pkp[16];                 // the previous (even) chunk, rounded
    const int nvt = (int)max((int64_t)0, min((int64_t)kBN, p.V - j0));  // columns inside V
    const float2 L2 = make_float2(kLog2e, kLog2e);
    float m = -INFINITY;
    float2 d2 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
    uint32_t v[2][32];
    tmem_ld32(tbase, v[0]);
#pragma unroll
    for (int c = 0; c < kBN / 32; ++c) {
        uint32_t* u = v[c & 1];
        tmem_wait_ld();
#pragma unroll
        for (int g = 0; g < 4; ++g) reg_fence8(u + 8 * g);
        if (c + 1 < kBN / 32) tmem_ld32(tbase + (uint32_t)((c + 1) * 32), v[(c + 1) & 1]);
        // round to the storage type, two values at a time
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
            pk[e] = VT::pack_pair(make_float2(__uint_as_float(u[2 * e]), __uint_as_float(u[2 * e + 1])));
        const int nval = min(32, max(0, nvt - c * 32));
        if (nval == 32) {
            typename VT::Max tm = VT::max_init();  // max on the packed pairs: exact
#pragma unroll
            for (int q = 0; q < 4; ++q)
                tm = VT::max_acc(tm, make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]));
            const float cm = VT::max_done(tm);
            if (cm > m) {
                if (m != -INFINITY) {
                    const float r = ex2_approx((m - cm) * kLog2e);
                    d2.x *= r;
                    d2.y *= r;
                }
                m = cm;
            }
            const float nm = -m * kLog2e;
            const float2 NM = make_float2(nm, nm);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float2 x = VT::unpack_pair(pk[e]);
                const float2 a = __ffma2_rn(x, L2, NM);
                d2 = __fadd2_rn(d2, make_float2(ex2_approx(a.x), ex2_approx(a.y)));
                s2 = __fadd2_rn(s2, x);
            }
        } else if (nval > 0) {
            // the vocabulary ends inside these 32 columns (predicated,
            // unrolled: the pairs stay in registers)
            float cm = -INFINITY;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float2 x = VT::unpack_pair(pk[e]);
                if (2 * e < nval) cm = fmaxf(cm, x.x);
                if (2 * e + 1 < nval) cm = fmaxf(cm, x.y);
            }
            if (cm > m) {
                if (m != -INFINITY) {
                    const float r = ex2_approx((m - cm) * kLog2e);
                    d2.x *= r;
                    d2.y *= r;
                }
                m = cm;
            }
            const float nm = -m * kLog2e;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float2 x = VT::unpack_pair(pk[e]);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float xv = h ? x.y : x.x;
                    if (2 * e + h < nval) {
                        d2.x += ex2_approx(fmaf(xv, kLog2e, nm));
                        s2.x += xv;
                        if (live) VT::store1(out + j0 + c * 32 + 2 * e + h, xv);
                    }
                }
            }
        }
        if ((c & 1) == 0) {
#pragma unroll
            for (int e = 0; e < 16; ++e) pkp[e] = pk[e];
        } else if (nvt - (c - 1) * 32 >= 64) {
            // chunks c-1 and c, whole: through the warp's stage (nvt is the
            // same for every lane, so the whole warp takes this branch)
            __syncwarp();  // the previous pair's reads are done
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t* w = u < 4 ? pkp + 4 * u : pk + 4 * (u - 4);
                stage[lane * 8 + (u ^ (lane & 7))] = make_uint4(w[0], w[1], w[2], w[3]);
            }
            __syncwarp();
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int R = 4 * jj + (lane >> 3), k = lane & 7;
                const uint4 w = stage[R * 8 + (k ^ (R & 7))];
                if (row0 + R < p.rows)
                    *reinterpret_cast<uint4*>(reinterpret_cast<T*>(p.logits) + (row0 + R) * p.ldl + j0 +
                                              (c - 1) * 32 + k * 8) = w;
            }
        } else if (live && nvt - (c - 1) * 32 >= 32) {
            // the vocabulary ends inside chunk c: chunk c-1 is whole, stored
            // by this lane (chunk c's elements went out above)
            uint4* o4 = reinterpret_cast<uint4*>(out + j0 + (c - 1) * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) o4[q] = make_uint4(pkp[4 * q], pkp[4 * q + 1], pkp[4 * q + 2], pkp[4 * q + 3]);
        }
    }
    return make_float4(m, d2.x + d2.y, s2.x + s2.y, 0.f);
}

// ------------------------------------------------------------ the GEMM + statistics kernel
template <typename T>
__global__ void __launch_bounds__(kLmThreads, 1)
ce_lmhead_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ LmArgs p) {
    extern __shared__ uint8_t smem_raw[];
    // stages on a 1024-byte boundary: the swizzle atoms (8 rows of 128 bytes)
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (sbase - raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + (size_t)kStages * kStageBytes);
    uint64_t* empty = full + kStages;
    uint64_t* tfull = empty + kStages;  // [2] accumulator b holds a finished tile
    uint64_t* tempty = tfull + 2;       // [2] the epilogue has read accumulator b
    uint64_t* done = tempty + 2;        // every MMA issued has completed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);  // one arrival per epilogue warp
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int ntiles = p.mb * p.ntn;
    auto give_up = [&]() {
        atomicOr(p.err, CE_DEVERR_TIMEOUT);
        *abort_flag = 1;
    };

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0, issued = 0;
            for (int t = blockIdx.x; t < ntiles && !*abort_flag; t += gridDim.x) {
                const int mblk = t % p.mb, nblk = t / p.mb;
                for (int k = 0; k < p.ksteps; ++k) {
                    if (!mbar_wait_bounded(&empty[s], ph ^ 1u)) {
                        give_up();
                        break;
                    }
                    const uint32_t st = sbase + (uint32_t)(s * kStageBytes);
                    mbar_arrive_expect_tx(&full[s], (uint32_t)kStageBytes);
                    tma_load_2d(st, &tmA, k * kBK, mblk * kBM, &full[s]);
                    tma_load_2d(st + kABytes, &tmB, k * kBK, nblk * kBN, &full[s]);
                    ++issued;
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (*abort_flag) {
                // let every copy already issued land before the CTA goes away
                for (int q = 0; q < kStages; ++q)
                    if (issued > (uint32_t)q) {
                        const uint32_t last = (issued - 1u - (uint32_t)q) / (uint32_t)kStages;
                        (void)mbar_wait_bounded(&full[q], last & 1u);
                    }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16<T>();
            int s = 0;
            uint32_t ph = 0;
            int it = 0;
            for (int t = blockIdx.x; t < ntiles && !*abort_flag; t += gridDim.x, ++it) {
                const int b = it & 1;
                const uint32_t bph = (uint32_t)(it >> 1) & 1u;
                if (!mbar_wait_bounded(&tempty[b], bph ^ 1u)) {  // the epilogue drained it
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(b * kBN);
                bool ok = true;
                for (int k = 0; k < p.ksteps; ++k) {
                    if (!mbar_wait_bounded(&full[s], ph)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = sbase + (uint32_t)(s * kStageBytes);
                    const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)  // K 16 per MMA: 32 bytes along the row
                        tc_mma(d, sdesc_sw128(a_addr + kk * 32), sdesc_sw128(b_addr + kk * 32), idesc,
                               (k | kk) != 0);
                    tc_commit(&empty[s]);  // the stage is free once these MMAs are done
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(&tfull[b]);  // accumulator b is complete
            }
            tc_commit(done);
            (void)mbar_wait_bounded(done, 0);
        }
    } else {
        // ---------------------------------------------------- epilogue
        const int q = warp & 3;
        uint4* stage = reinterpret_cast<uint4*>(sm + (size_t)kStages * kStageBytes + 256) + q * 256;            // this warp's quarter of the TMEM lanes
        const int rin = q * 32 + lane;     // row within the tile
        int it = 0;
        for (int t = blockIdx.x; t < ntiles && !*abort_flag; t += gridDim.x, ++it) {
            const int b = it & 1;
            const uint32_t bph = (uint32_t)(it >> 1) & 1u;
            const int mblk = t % p.mb, nblk = t / p.mb;
            if (!__all_sync(kFull, mbar_wait_bounded(&tfull[b], bph))) {
                if (lane == 0) give_up();
                break;
            }
            tc_fence_after();
            const int64_t row = (int64_t)mblk * kBM + rin;
            const float4 pt = epilogue_row<T>(p, tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * kBN),
                                              row, (int64_t)nblk * kBN, stage, lane);
            // every read of accumulator b is done: hand it back to the MMA warp
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[b]);
            if (row < p.rows) p.part[row * p.ntn + nblk] = pt;
        }
    }

    // teardown: every role has finished (or given up); free the tensor memory
    __syncwarp();  // lane 0 of warps 0 and 1 ran their role alone
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

// ------------------------------------------------------------ the paired-SM kernel
// The two CTAs of a cluster compute one 256 x 256 tile together: CTA r loads
// rows [r*128, r*128 + 128) of the tile's hidden rows and of its W rows (half
// of each operand, 32 KB per stage), both copies completing on the leader's
// (rank 0) barrier; the leader issues tcgen05.mma.cta_group::2 (M 256, N
// 256), which reads both CTAs' stages, and commits each stage and each
// finished accumulator to the barriers of both CTAs at once; each CTA's TMEM
// holds its 128 rows of the accumulator, read by its own epilogue warps, which
// report back to the leader.  Per SM: 32 KB of operands per 512 tensor-core
// clocks instead of 48 KB, in a 6-deep ring (192 KB), beside the epilogue
// warps' 16 KB store stage (with the logits stored straight from registers,
// 32 rows of 16 bytes per instruction, a 7-deep ring had measured 1 % faster
// than 6 on the whole lm_head step).
constexpr int kStages2 = 6;
constexpr int kHalfBytes = 128 * kBK * 2;     // 16 KB: 128 rows x 64 16-bit values
constexpr int kStage2Bytes = 2 * kHalfBytes;  // per CTA: its hidden half + its W half
constexpr size_t kLmSmem2 = (size_t)kStages2 * kStage2Bytes + 1024 + 256 + kStoreStageBytes;

__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}

// The same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

template <typename T>
__global__ void __launch_bounds__(kLmThreads, 1)
ce_lmhead2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ LmArgs p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (sbase - raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + (size_t)kStages2 * kStage2Bytes);  // leader's: both CTAs' copies
    uint64_t* empty = full + kStages2;  // this CTA's stage s is free again
    uint64_t* tfull = empty + kStages2;  // [2] accumulator b holds a finished tile
    uint64_t* tempty = tfull + 2;        // [2] leader's: both CTAs' epilogues read accumulator b
    uint64_t* done = tempty + 2;         // leader: every MMA issued has completed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages2; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 8);  // one arrival per epilogue warp of either CTA
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers are initialised and their TMEM allocated
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int npairs = (int)(gridDim.x >> 1), pair = (int)(blockIdx.x >> 1);
    const int ntiles = p.mb * p.ntn;
    auto give_up = [&]() {
        atomicOr(p.err, CE_DEVERR_TIMEOUT);
        *abort_flag = 1;
    };

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer (both CTAs)
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0, issued = 0;
            for (int t = pair; t < ntiles && !*abort_flag; t += npairs) {
                const int mblk = t % p.mb, nblk = t / p.mb;
                for (int k = 0; k < p.ksteps; ++k) {
                    if (!mbar_wait_bounded(&empty[s], ph ^ 1u)) {
                        give_up();
                        break;
                    }
                    // the leader arms its barrier for both CTAs' bytes; the
                    // peer's copies may land first (the count goes below zero)
                    if (leader) mbar_arrive_expect_tx(&full[s], 2u * kStage2Bytes);
                    const uint32_t st = sbase + (uint32_t)(s * kStage2Bytes);
                    const uint32_t fb = cluster_addr(&full[s], 0);
                    tma_load_2d_pair(st, &tmA, k * kBK, mblk * 256 + (int)rank * 128, fb);
                    tma_load_2d_pair(st + kHalfBytes, &tmB, k * kBK, nblk * 256 + (int)rank * 128, fb);
                    ++issued;
                    if (++s == kStages2) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (*abort_flag && leader) {
                for (int q = 0; q < kStages2; ++q)
                    if (issued > (uint32_t)q) {
                        const uint32_t last = (issued - 1u - (uint32_t)q) / (uint32_t)kStages2;
                        (void)mbar_wait_bounded(&full[q], last & 1u);
                    }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer (leader)
        if (lane == 0 && leader) {
            constexpr uint32_t idesc = (idesc_f16<T>() & ~(31u << 24)) | ((uint32_t)(256 >> 4) << 24);
            int s = 0;
            uint32_t ph = 0;
            int it = 0;
            for (int t = pair; t < ntiles && !*abort_flag; t += npairs, ++it) {
                const int b = it & 1;
                const uint32_t bph = (uint32_t)(it >> 1) & 1u;
                if (!mbar_wait_bounded(&tempty[b], bph ^ 1u)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(b * kBN);
                bool ok = true;
                for (int k = 0; k < p.ksteps; ++k) {
                    if (!mbar_wait_bounded(&full[s], ph)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = sbase + (uint32_t)(s * kStage2Bytes);
                    const uint32_t b_addr = a_addr + kHalfBytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        asm volatile(
                            "{\n\t.reg .pred p;\n\t"
                            "setp.ne.b32 p, %4, 0;\n\t"
                            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
                            "l"(sdesc_sw128(a_addr + kk * 32)), "l"(sdesc_sw128(b_addr + kk * 32)),
                            "r"(idesc), "r"((uint32_t)((k | kk) != 0))
                            : "memory");
                    // stage s is free in both CTAs once these MMAs are done
                    asm volatile(
                        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
                        "[%0], %1;" ::"r"(smem_u32(&empty[s])),
                        "h"((uint16_t)3)
                        : "memory");
                    if (++s == kStages2) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                asm volatile(
                    "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
                    "[%0], %1;" ::"r"(smem_u32(&tfull[b])),
                    "h"((uint16_t)3)
                    : "memory");
            }
            asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                             smem_u32(done))
                         : "memory");
            (void)mbar_wait_bounded(done, 0);
        }
    } else {
        // ---------------------------------------------------- epilogue (both CTAs)
        const int q = warp & 3;
        uint4* stage = reinterpret_cast<uint4*>(sm + (size_t)kStages2 * kStage2Bytes + 256) + q * 256;
        int it = 0;
        for (int t = pair; t < ntiles && !*abort_flag; t += npairs, ++it) {
            const int b = it & 1;
            const uint32_t bph = (uint32_t)(it >> 1) & 1u;
            const int mblk = t % p.mb, nblk = t / p.mb;
            if (!__all_sync(kFull, mbar_wait_bounded(&tfull[b], bph))) {
                if (lane == 0) give_up();
                break;
            }
            tc_fence_after();
            const int64_t row = (int64_t)mblk * 256 + rank * 128 + q * 32 + lane;
            const float4 pt = epilogue_row<T>(p, tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * kBN),
                                              row, (int64_t)nblk * kBN, stage, lane);
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                                 cluster_addr(&tempty[b], 0))
                             : "memory");
            if (row < p.rows) p.part[row * p.ntn + nblk] = pt;
        }
    }

    // teardown: both CTAs have finished (or given up), so no copy, commit or
    // arrival targets either of them any more; free the tensor memory
    __syncwarp();
    tc_fence_before();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

// ------------------------------------------------------------ per-row combine of the tiles
// One warp per row: lane l folds tiles l, l + 32, ... in order, then a fixed
// butterfly; x_y is the target's logit as the chunk buffer holds it.
template <typename T>
__global__ void __launch_bounds__(256) ce_lm_combine_kernel(const float4* __restrict__ part, int ntn,
                                                            int64_t rows, int64_t V,
                                                            const T* __restrict__ logits, int64_t ldl,
                                                            const int64_t* __restrict__ targets,
                                                            int64_t ignore_idx, float a,
                                                            float* __restrict__ loss,
                                                            float* __restrict__ lse_out) {
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int64_t y = __ldg(targets + row);
    if (y == ignore_idx || y < 0 || y >= V) {  // out of range: the count kernel set the error bit
        if (lane == 0) {
            loss[row] = (y == ignore_idx) ? 0.f : __int_as_float(0x7fc00000);
            lse_out[row] = __int_as_float(0x7fc00000);
        }
        return;
    }
    const float4* pr = part + row * (int64_t)ntn;
    Part G = part_identity();
    for (int t = lane; t < ntn; t += 32) {
        const float4 v = __ldg(pr + t);
        G = part_combine(G, Part{v.x, v.y, v.z});
    }
    G = warp_allreduce_part(G);
    if (lane == 0) {
        const float xy = Vec<T>::load1(logits + row * ldl + y);
        const float l = G.m + logf(G.d);
        loss[row] = l - (1.f - a) * xy - (a / (float)V) * G.S;
        lse_out[row] = l;
    }
}

// ------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// A 2-D row-major (outer x inner) 16-bit matrix, boxes of box_outer x 64.
bool make_map(CUtensorMap* m, const void* ptr, int dtype, uint64_t inner, uint64_t outer,
              uint32_t box_outer) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, box_outer};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, dtype == CE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
              const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T>
cudaError_t launch_lmhead_typed(const LmHeadProblem& lp, cudaStream_t s) {
    // the paired-SM kernel from 256 rows on; one CTA per tile below
    const bool paired = lp.rows >= 256;
    CUtensorMap ta, tb;
    memset(&ta, 0, sizeof ta);
    memset(&tb, 0, sizeof tb);
    if (!make_map(&ta, lp.hidden, lp.dtype, (uint64_t)lp.H, (uint64_t)lp.rows, kBM) ||
        !make_map(&tb, lp.weight, lp.dtype, (uint64_t)lp.H, (uint64_t)lp.V, paired ? 128 : kBN))
        return cudaErrorInvalidValue;
    LmArgs a;
    memset(&a, 0, sizeof a);
    a.rows = lp.rows;
    a.V = lp.V;
    a.ldl = lp.ldl;
    a.logits = static_cast<char*>(lp.logits);
    a.part = lp.part;
    a.targets = lp.targets;
    a.ignore_idx = lp.ignore_idx;
    const int tile_rows = paired ? 256 : kBM;
    a.mb = (int)((lp.rows + tile_rows - 1) / tile_rows);
    a.ntn = (int)((lp.V + kBN - 1) / kBN);
    a.ksteps = (int)((lp.H + kBK - 1) / kBK);
    a.err = lp.err;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t ntiles = (int64_t)a.mb * a.ntn;
    cudaError_t e;
    if (paired) {
        auto kern = ce_lmhead2_kernel<T>;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kLmSmem2);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.blockDim = dim3(kLmThreads, 1, 1);
        cfg.dynamicSmemBytes = kLmSmem2;
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        // as many pairs as can be resident at once (one CTA per SM), at most
        // one per tile
        cfg.gridDim = dim3((unsigned)(2 * (sms / 2)), 1, 1);
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
        if (e != cudaSuccess) return e;
        if (clusters < 1) return cudaErrorInvalidConfiguration;
        if (clusters > ntiles) clusters = (int)ntiles;
        cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
        e = cudaLaunchKernelEx(&cfg, kern, ta, tb, a);
    } else {
        auto kern = ce_lmhead_kernel<T>;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kLmSmem);
        if (e != cudaSuccess) return e;
        const int grid = (int)(ntiles < sms ? ntiles : sms);
        kern<<<grid, kLmThreads, kLmSmem, s>>>(ta, tb, a);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    const int rows_per_cta = 8;
    ce_lm_combine_kernel<T><<<(unsigned)((lp.rows + rows_per_cta - 1) / rows_per_cta), 32 * rows_per_cta,
                              0, s>>>(lp.part, a.ntn, lp.rows, lp.V, static_cast<const T*>(lp.logits),
                                      lp.ldl, lp.targets, lp.ignore_idx, lp.a, lp.loss_rows, lp.lse);
    return cudaGetLastError();
}

}  // namespace

bool lmhead_supported(int dtype, int64_t H, int64_t V, const void* hidden, const void* weight) {
    if (dtype != CE_BF16 && dtype != CE_F16) return false;
    if (H % 8 || H > 0x7fffffffLL || V > 0x7fffffffLL) return false;  // 16-byte TMA row strides
    if (reinterpret_cast<uintptr_t>(hidden) % 16 || reinterpret_cast<uintptr_t>(weight) % 16) return false;
    return encode_fn() != nullptr;
}

size_t lmhead_part_bytes(int64_t rows, int64_t V) {
    return align_up((size_t)rows * (size_t)((V + kBN - 1) / kBN) * sizeof(float4), 256);
}

int64_t lmhead_ldl(int64_t V) { return (V + 7) / 8 * 8; }

cudaError_t launch_lmhead(const LmHeadProblem& lp, cudaStream_t s) {
    if (lp.rows <= 0) return cudaSuccess;
    if (lp.ldl % 8 || lp.ldl < lp.V) return cudaErrorInvalidValue;
    return lp.dtype == CE_BF16 ? launch_lmhead_typed<__nv_bfloat16>(lp, s)
                               : launch_lmhead_typed<__half>(lp, s);
}

}  // namespace gbce
