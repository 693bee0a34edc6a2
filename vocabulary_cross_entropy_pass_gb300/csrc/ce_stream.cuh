// ce_stream.cuh -- the row-streaming fused cross-entropy kernel (template;
// ce_stream.cu instantiates it for rows on the 16-byte grid and the
// class-weighted pass, ce_stream_geo.cu for rows with a scalar head and tail
// and for rows cut into vocabulary chunks).
//
// One CTA owns whole token rows, so no CTA ever waits for another: a
// persistent grid, each CTA starting on rows cta and cta + grid and then
// claiming the next unclaimed row from a counter in the workspace, so the CTAs
// finish together although ignored rows (no read) fall unevenly among them.
// The producer warp claims rows and hands them, with their targets, to the
// consumer warps through a small queue in shared memory.  Each row goes twice
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
// Class weights (torch F.cross_entropy(weight=...), the weighted NLL of
// mindspore/hyper-parallel #269): the gradient is c * softmax - g (a/V) w_j
// with c = g ((1-a) w_y + (a/V) W), so pass 1 is unchanged; in pass 2 the
// producer follows each logits tile with its fp32 weights (4/sizeof(T) times
// the tile's bytes, L2-resident, in the next ring slots), and the consumers
// also sum w_j x_j for the row's loss, (1-a) w_y (lse - x_y) + (a/V) (W lse -
// sum_j w_j x_j), written after pass 2.  Without smoothing (a = 0) no weight
// but w_y is needed.  The mean divides by the summed target weight of the
// kept rows.  (The forward-only weighted pass reads the weights in pass 1,
// with plain loads.)
//
// Row geometry (GEO):
//   kGeoAligned  rows on the 16-byte grid: the whole row goes through the
//                ring, tile k at byte k * TB;
//   kGeoEdges    rows anywhere (on a multiple of the element size): TMA copies
//                need 16-byte aligned addresses and sizes, so the ring takes the
//                row's aligned body -- whole 16-byte vectors from the first
//                16-byte boundary -- and the at most 2 (16 / sizeof(T) - 1)
//                elements before and after it (odd widths such as 50257 or
//                100277, shifted views) are one per thread, read once with a
//                plain load and kept in a register for the gradient;
//   kGeoChunks   a vocabulary split asked for: the row is cut into contiguous
//                chunks of C elements (ceil(V/K) rounded up to 16 bytes), each
//                streamed as its own run of tiles; at the end of a chunk every
//                warp reduces its (max, sum-exp, sum) to the chunk's warp
//                partial, and the CTA combine folds the warps of each chunk,
//                then the chunks in chunk order -- the (m, d, x_y) combine of
//                the vocabulary-parallel ranks of mindspore/hyper-parallel #269
//                section 3.1, inside one CTA.  The chunk partials {m, d, S, x_y}
//                are also written to the workspace.
//
// Warp specialisation: warps 0..NC/32-1 consume tiles; the last warp only
// issues copies.  `full[s]` completes when tile s has landed (TMA transaction
// count); `empty[s]` completes when every consumer warp is done with it.  Both
// waits are bounded; a wait that gives up sets CE_DEVERR_TIMEOUT and the CTA
// drains without further copies (the producer then waits, bounded, for the
// copies it already issued before the CTA exits).
#pragma once

#include "ce_device.cuh"
#include "ce_internal.h"
#include "ce_span.cuh"

#include <string.h>

namespace gbce {
namespace {

constexpr int kGeoAligned = kStreamAligned;
constexpr int kGeoEdges = kStreamEdges;
constexpr int kGeoChunks = kStreamChunks;

struct StreamArgs {
    char* logits;
    int64_t s0, s1, dim1, N;
    int32_t V;
    int32_t stages;
    uint32_t tile_bytes;   // bytes per ring tile, multiple of 16
    int32_t ntiles;        // tiles per row (kGeoEdges: per row, from where it starts)
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
    uint32_t* ticket;      // CTAs done (zeroed by the count kernel)
    float* mean_out;       // reduce_loss: the last CTA to finish writes the mean here
    const float* cw;       // class weights [V], 16-byte aligned (weighted pass) or NULL
    const double* wdenom;  // summed weight of the kept rows' targets (count kernel)
    const double* wsum;    // summed weight over the vocabulary (count kernel)
    uint32_t* row_claim;   // rows claimed past each CTA's first two, or NULL (static rows)
    uint32_t* row_done;    // CTAs done claiming
    // kGeoChunks: vocabulary chunks of chunk_elems elements (chunk_bytes, a
    // multiple of 16), tpc tiles each (the last chunk may take fewer),
    // nchunks non-empty chunks; part: per-(row, chunk) partials {m, d, S, x_y}
    // at part[row * nchunks + chunk], or NULL
    int64_t chunk_elems;
    uint32_t chunk_bytes;
    int32_t tpc;
    int32_t nchunks;
    float4* part;
    int flat;              // row r at r * s1, its target at r * ts1
};

// The part of a row that goes through the ring: `body` (16-byte aligned),
// `body_bytes` (a multiple of 16) in `ntiles` tiles; kGeoEdges: the elements
// [0, head) and [t0, V) stay outside it.
struct RowGeo {
    const char* body;
    int64_t body_bytes;
    int32_t ntiles;
    int64_t head;
    int64_t t0;
};

template <int GEO, int ES, int TB>
__device__ __forceinline__ RowGeo row_geo(const StreamArgs& p, const char* rowp) {
    RowGeo g;
    if constexpr (GEO == kGeoEdges) {
        const Span16 s = span16<ES>(rowp, 0, p.V);
        g.head = s.h1;
        g.t0 = s.t0;
        g.body = rowp + s.h1 * ES;
        g.body_bytes = s.nv * 16;
        g.ntiles = (int32_t)((g.body_bytes + TB - 1) / TB);
    } else {
        g.head = 0;
        g.t0 = p.V;
        g.body = rowp;
        g.body_bytes = (int64_t)p.V * ES;
        g.ntiles = p.ntiles;
    }
    return g;
}

// Tile k of a row: its byte offset from the body and its byte count.
template <int GEO, int TB>
__device__ __forceinline__ void tile_span(const StreamArgs& p, const RowGeo& g, int k, int64_t& off,
                                          uint32_t& bytes) {
    if constexpr (GEO == kGeoChunks) {
        const int c = k / p.tpc;
        const int j = k - c * p.tpc;
        off = (int64_t)c * p.chunk_bytes + (int64_t)j * TB;
        const int64_t cend = min((int64_t)(c + 1) * p.chunk_bytes, g.body_bytes);
        bytes = (uint32_t)min((int64_t)TB, cend - off);
    } else {
        off = (int64_t)k * TB;
        bytes = (k == g.ntiles - 1) ? (uint32_t)(g.body_bytes - off) : (uint32_t)TB;
    }
}

// The class weights of one 16-byte logits vector: VEC fp32 values, read as
// 16-byte loads (the weight vector stays in L2: V x 4 bytes).
template <typename T>
__device__ __forceinline__ void load_weights(const float* cw, int64_t e0, float2 (&w)[Vec<T>::kElems / 2]) {
    constexpr int VEC = Vec<T>::kElems;
    const float4* src = reinterpret_cast<const float4*>(cw + e0);
#pragma unroll
    for (int k = 0; k < VEC / 4; ++k) {
        const float4 f = __ldg(src + k);
        w[2 * k] = make_float2(f.x, f.y);
        w[2 * k + 1] = make_float2(f.z, f.w);
    }
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Rows handed from the producer warp to the consumer warps ahead of their tiles.
constexpr int kRowQ = 8;

// Barrier 1 over the consumer threads, returning whether any of them passed
// `v`: every consumer warp gets the same answer.
__device__ __forceinline__ bool named_bar_or(int id, int threads, bool v) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred pin, pout;\n\t"
        "setp.ne.u32 pin, %1, 0;\n\t"
        "bar.red.or.pred pout, %2, %3, pin;\n\t"
        "selp.u32 %0, 1, 0, pout;\n\t}"
        : "=r"(out)
        : "r"((uint32_t)v), "r"(id), "r"(threads)
        : "memory");
    return out != 0;
}

// One ring slot: stage index and phase parity, advanced without division.
struct Ring {
    int s = 0;
    uint32_t ph = 0;
    int n;
    __device__ explicit Ring(int stages) : n(stages) {}
    __device__ __forceinline__ void next() {
        if (++s == n) {
            s = 0;
            ph ^= 1u;
        }
    }
};

// Pass-1 work on one tile: running max, then p = 2^((x - m) log2e) summed,
// and the plain sum (WS: the class-weighted sum sum_j w_j x_j instead), in
// packed f32x2 arithmetic.  FULL: every vector valid.  e0: the row element of
// the tile's first vector (weights only).  UNI: the running max is the
// warp's (one redux per tile), so every lane's sums share it and the warp's
// partial is two plain sums.  SUM: accumulate the plain sum at all (the
// weighted gradient pass takes the weighted sum in pass 2 instead).
template <typename T, int NC, int NV, bool FULL, bool WS, bool UNI = false, bool SUM = true>
__device__ __forceinline__ void stats_tile(const uint4* tile, int tid, int nvec, float& m,
                                           float2& d2, float2& s2, const float* cw, int64_t e0) {
    using VT = Vec<T>;
    constexpr int P = VT::kElems / 2;  // float2 pairs per vector
    uint4 raw[NV];
    typename VT::Max tm = VT::max_init();
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        if (FULL || tid + i * NC < nvec) {
            raw[i] = tile[tid + i * NC];
            tm = VT::max_acc(tm, raw[i]);
        }
    }
    float tmf = VT::max_done(tm);
    if constexpr (UNI) tmf = warp_max_redux(tmf);
    if (tmf > m) {  // new running max: rescale what was summed so far
        if (m != -INFINITY) {
            const float c = ex2_approx((m - tmf) * kLog2e);
            d2.x *= c;
            d2.y *= c;
        }
        m = tmf;
    }
    const float nml = (m == -INFINITY) ? 0.f : -m * kLog2e;
    const float2 L2 = make_float2(kLog2e, kLog2e);
    const float2 NM = make_float2(nml, nml);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        if (FULL || tid + i * NC < nvec) {
            float2 x[P], w[P];
            VT::unpack2(raw[i], x);
            if constexpr (WS) load_weights<T>(cw, e0 + (int64_t)(tid + i * NC) * VT::kElems, w);
#pragma unroll
            for (int j = 0; j < P; ++j) {
                const float2 a = __ffma2_rn(x[j], L2, NM);
                d2 = __fadd2_rn(d2, make_float2(ex2_approx(a.x), ex2_approx(a.y)));
                if constexpr (WS)
                    s2 = __ffma2_rn(w[j], x[j], s2);
                else if constexpr (SUM)
                    s2 = __fadd2_rn(s2, x[j]);
            }
        }
    }
}

// Pass-2 work on one tile: c * 2^((x - lse) log2e) - b_j, rounded to T and
// stored over the logits.  Unweighted: c = g, b_j = g a/V (NB = -b).
// WT: c = g ((1-a) w_y + (a/V) W), b_j = g (a/V) w_j (NB = -g a/V), and the
// class-weighted sum sum_j w_j x_j of the loss is accumulated into sw2 here,
// so each weight is read once per row.  The tile's weights sit in WS ring
// slots after it (fp32, 4/sizeof(T) times the tile's bytes): vector v of the
// tile finds its VEC weights in slot v / (TV/WS) at vector v % (TV/WS).
template <typename T, int NC, int NV, bool FULL, bool WT>
__device__ __forceinline__ void grad_tile(const uint4* tile, uint4* dst, int tid, int nvec,
                                          float2 NL, float2 G2, float2 NB,
                                          const unsigned char* const* wslot, float2& sw2) {
    using VT = Vec<T>;
    constexpr int VEC = VT::kElems;
    constexpr int P = VEC / 2;
    constexpr int WS = 4 / (int)sizeof(T);  // weight slots per tile
    constexpr int NVS = NV / WS;            // vectors per thread whose weights share a slot
    static_assert(NV % WS == 0, "a thread's vectors split evenly over the weight slots");
    const float2 L2 = make_float2(kLog2e, kLog2e);
    uint4 raw[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i)
        if (FULL || tid + i * NC < nvec) raw[i] = tile[tid + i * NC];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        if (FULL || tid + i * NC < nvec) {
            float2 x[P], o[P], w[P];
            VT::unpack2(raw[i], x);
            if constexpr (WT) {
                const float4* ws = reinterpret_cast<const float4*>(wslot[i / NVS]) +
                                   (size_t)(tid + (i % NVS) * NC) * (VEC / 4);
#pragma unroll
                for (int k = 0; k < VEC / 4; ++k) {
                    const float4 f = ws[k];
                    w[2 * k] = make_float2(f.x, f.y);
                    w[2 * k + 1] = make_float2(f.z, f.w);
                }
            }
#pragma unroll
            for (int j = 0; j < P; ++j) {
                const float2 a = __ffma2_rn(x[j], L2, NL);
                float2 b = NB;
                if constexpr (WT) {
                    b = __fmul2_rn(w[j], NB);
                    sw2 = __ffma2_rn(w[j], x[j], sw2);
                }
                o[j] = __ffma2_rn(make_float2(ex2_approx(a.x), ex2_approx(a.y)), G2, b);
            }
            stg128_stream(dst + tid + i * NC, VT::pack2(o));
        }
    }
}

// The weighted gradient pass of 16-bit logits, in 8-byte units u = tid + j NC
// (four logits each, weights in slot j / NV at float4 tid + (j % NV) NC): a
// warp's logits loads (8 bytes a lane) and weight loads (16 bytes a lane) are
// both contiguous, so neither meets a shared-memory bank conflict (with 16-byte
// logit vectors each lane's 32 bytes of weights are two 16-byte loads 32 bytes
// apart across the warp: two-way conflicts).  Same arithmetic as grad_tile.
template <typename T, int NC, int NV, bool FULL>
__device__ __forceinline__ void grad_tile_w16(const unsigned char* tile, unsigned char* dst, int tid,
                                              int nunit, float2 NL, float2 G2, float2 NB,
                                              const unsigned char* const* wslot, float2& sw2) {
    using VT = Vec<T>;
    static_assert(sizeof(T) == 2, "8-byte units of 16-bit logits");
    constexpr int NU = 2 * NV;
    const float2 L2 = make_float2(kLog2e, kLog2e);
    uint2 raw[NU];
#pragma unroll
    for (int j = 0; j < NU; ++j)
        if (FULL || tid + j * NC < nunit) raw[j] = reinterpret_cast<const uint2*>(tile)[tid + j * NC];
#pragma unroll
    for (int j = 0; j < NU; ++j) {
        if (FULL || tid + j * NC < nunit) {
            const float4 f = reinterpret_cast<const float4*>(wslot[j / NV])[tid + (j % NV) * NC];
            const float2 x[2] = {VT::unpack_pair(raw[j].x), VT::unpack_pair(raw[j].y)};
            const float2 w[2] = {make_float2(f.x, f.y), make_float2(f.z, f.w)};
            uint32_t o[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const float2 a = __ffma2_rn(x[k], L2, NL);
                const float2 b = __fmul2_rn(w[k], NB);
                sw2 = __ffma2_rn(w[k], x[k], sw2);
                o[k] = VT::pack_pair(__ffma2_rn(make_float2(ex2_approx(a.x), ex2_approx(a.y)), G2, b));
            }
            __stcs(reinterpret_cast<uint2*>(dst) + tid + j * NC, make_uint2(o[0], o[1]));
        }
    }
}

// The 256-thread, 16 KB-tile shape is built for two CTAs per SM (96
// registers): twice the warps to hide issue latency, for rows short enough
// that two CTAs' rows between their passes still fit L2 (and for the
// weighted pass, whose gradient pass issues ~40% more instructions per
// element).  Every other shape is built for one CTA per SM.
template <typename T, int NC, int NV, bool GRAD, bool WT, int GEO>
__global__ void __launch_bounds__(NC + 32, (NC == 256 && NV * NC * 16 == 16384) ? 2 : 1)
ce_stream_kernel(const __grid_constant__ StreamArgs p) {
    using VT = Vec<T>;
    constexpr int VEC = VT::kElems;
    constexpr int ES = sizeof(T);
    constexpr int NW = NC / 32;           // consumer warps
    constexpr int TB = NC * NV * 16;      // tile bytes
    constexpr int TV = NC * NV;           // vectors per tile
    constexpr int KS = GEO == kGeoChunks ? kMaxStreamChunks : 1;  // chunk slots per row
    static_assert(!WT || GEO == kGeoAligned, "the weighted pass streams aligned rows only");

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)p.stages * TB);
    uint64_t* empty = full + 12;
    uint64_t* qfull = empty + 12;    // row queue: entry written
    uint64_t* qempty = qfull + kRowQ;  // row queue: entry read by every consumer warp
    int64_t* rowq = reinterpret_cast<int64_t*>(qempty + kRowQ);  // row index
    int64_t* yq = rowq + kRowQ;                                   // its target
    float4* red = reinterpret_cast<float4*>(yq + kRowQ);  // [2][KS][NW]
    float* xy_s = reinterpret_cast<float*>(red + 2 * KS * NW);  // [2]
    float* sw_s = xy_s + 2;                                 // [2][NW] weighted sums
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sw_s + 2 * NW);
    volatile int* last_flag = abort_flag + 1;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
        }
        for (int q = 0; q < kRowQ; ++q) {
            mbar_init(&qfull[q], 1);
            mbar_init(&qempty[q], NW);
        }
        *abort_flag = 0;
        *last_flag = 0;
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
    const int npass = GRAD ? 2 : 1;
    // weighted gradient pass with smoothing: each tile brings its class
    // weights into the next WS ring slots (without smoothing no weight is read)
    constexpr int WS = 4 / ES;
    const bool wring = WT && GRAD && p.a != 0.f;
    // Parked tiles: when pass 1 of a row ends, the ring's `stages` slots hold
    // the row's last `stages` tiles, and the ring is a queue -- so pass 2 can
    // take those tiles first, straight from shared memory (the producer
    // re-marks their slots full without a copy), then reload tiles 0 ..
    // ntiles - R - 1.  Pass-2 tile k is pass2_tile(k).  This pays for rows of
    // at least twice the ring (fewer tiles wait in L2 for pass 2: 256000 bf16
    // columns, 16 tiles, 6-deep ring, 4096 rows: 0.650 ms against 0.680 ms);
    // at 8 tiles (128000 columns) the reordered pass measured 1.3 % slower,
    // so shorter rows reload every tile.  Not with weight slots in the ring.
    // R depends on the row's tile count (kGeoEdges: on where the row starts).
    auto parked = [&](int ntiles) -> int {
        return (GRAD && !wring && ntiles >= 2 * p.stages) ? p.stages : 0;
    };
    auto pass2_tile = [](int k, int R, int ntiles) -> int { return k < R ? ntiles - R + k : k - R; };

    // ------------------------------------------------------------ producer warp
    if (warp == NW) {
        if (lane == 0) {
            const uint64_t pol_keep = p.l2_keep ? l2_evict_last_policy() : l2_evict_first_policy();
            const uint64_t pol_drop = l2_evict_first_policy();
            const uint64_t pol_wt = l2_evict_last_policy();  // every CTA reads the weights
            Ring rg(p.stages);
            Ring qr(kRowQ);
            uint32_t issued = 0;
            bool counted = false;
            // rows: the CTA's own two first rows (blockIdx.x and blockIdx.x +
            // gridDim.x), then rows claimed from the shared counter (the count
            // kernel zeroes it), or without a counter every gridDim.x-th row
            auto claim = [&](int64_t cur) -> int64_t {
                if (!p.row_claim) return cur + gridDim.x;
                if (!counted) {
                    griddep_wait();
                    counted = true;
                }
                return 2 * (int64_t)gridDim.x + (int64_t)atomicAdd(p.row_claim, 1u);
            };
            // hand a row (or the end mark -1 for any index past the last row)
            // to the consumer warps; false when the queue stays full too long
            auto publish = [&](int64_t row, int64_t y) -> bool {
                if (!mbar_wait_bounded(&qempty[qr.s], qr.ph ^ 1u)) {
                    griddep_wait();  // the count kernel starts the error word
                    atomicOr(p.err, CE_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                    return false;
                }
                rowq[qr.s] = row < p.N ? row : -1;
                yq[qr.s] = y;
                mbar_arrive(&qfull[qr.s]);
                qr.next();
                return true;
            };
            // The queue runs one row ahead of the copies: the row after this one
            // is published before this row's copies, so the consumers can read
            // it while they work on this row.  The row after that is claimed
            // before this row's copies too (on the first row, after its first
            // pass: the first claim waits for the count kernel), and its target
            // is loaded right away but first read one row later, when it is
            // published.  Each entry carries the row's target, read here once
            // for the consumer warps as well.
            int64_t r = blockIdx.x, n1 = r + gridDim.x, n2 = -1;  // this row, the next two
            int64_t yr = row_target(r), y1 = n1 < p.N ? row_target(n1) : 0, y2 = 0;
            auto claim_y = [&]() {
                n2 = claim(n1);
                y2 = n2 < p.N ? row_target(n2) : 0;
            };
            publish(r, yr);
            for (int k = 0; !*abort_flag; ++k) {
                if (!publish(n1, y1)) break;
                bool claimed = false;
                if (k > 0) {
                    claim_y();
                    claimed = true;
                }
                const bool loaded = is_loaded(yr);
                const RowGeo gr = row_geo<GEO, ES, TB>(p, row_ptr(r));
                const int R = parked(gr.ntiles);
                for (int pass = 0; loaded && pass < npass && !*abort_flag; ++pass) {
                    if (pass == 1 && !claimed) {
                        claim_y();
                        claimed = true;
                    }
                    for (int k = 0; k < gr.ntiles; ++k) {
                        if (!mbar_wait_bounded(&empty[rg.s], rg.ph ^ 1u)) {
                            griddep_wait();  // the count kernel starts the error word
                            atomicOr(p.err, CE_DEVERR_TIMEOUT);
                            *abort_flag = 1;
                            break;
                        }
                        if (pass == 1 && k < R) {
                            // a parked tile: still in this slot since pass 1
                            mbar_arrive(&full[rg.s]);
                            rg.next();
                            ++issued;
                            continue;
                        }
                        const int t = pass == 1 ? pass2_tile(k, R, gr.ntiles) : k;
                        int64_t off;
                        uint32_t bytes;
                        tile_span<GEO, TB>(p, gr, t, off, bytes);
                        // pass 1 asks L2 to keep the tiles pass 2 will reload
                        const uint64_t pol = (pass == 0 && t < gr.ntiles - R) ? pol_keep : pol_drop;
                        mbar_arrive_expect_tx(&full[rg.s], bytes);
                        tma_load_1d(ring + (size_t)rg.s * TB, gr.body + off, bytes, &full[rg.s], pol);
                        rg.next();
                        ++issued;
                        if (pass == 1 && wring) {
                            // the tile's weights: WS * bytes from cw + t * WS * TB, one
                            // slot of up to TB bytes each (a slot past the end of the
                            // weights completes with no copy)
                            const char* wsrc = reinterpret_cast<const char*>(p.cw) + (size_t)t * WS * TB;
                            const uint32_t wbytes = bytes * WS;
                            for (int h = 0; h < WS; ++h) {
                                if (!mbar_wait_bounded(&empty[rg.s], rg.ph ^ 1u)) {
                                    griddep_wait();
                                    atomicOr(p.err, CE_DEVERR_TIMEOUT);
                                    *abort_flag = 1;
                                    break;
                                }
                                const uint32_t hb = wbytes > (uint32_t)(h * TB)
                                                        ? min(wbytes - (uint32_t)(h * TB), (uint32_t)TB)
                                                        : 0u;
                                mbar_arrive_expect_tx(&full[rg.s], hb);
                                if (hb) tma_load_1d(ring + (size_t)rg.s * TB, wsrc + (size_t)h * TB, hb,
                                                    &full[rg.s], pol_wt);
                                rg.next();
                                ++issued;
                            }
                            if (*abort_flag) break;
                        }
                    }
                }
                if (!claimed) claim_y();  // a first row without a gradient pass
                r = n1;  // one CTA's rows only grow: past N, all later ones are too
                yr = y1;
                n1 = n2;
                y1 = y2;
                if (r >= p.N) break;  // its end mark is already in the queue
            }
            if (*abort_flag) {
                // let every copy already issued land before the CTA goes away
                for (int s = 0; s < p.stages; ++s) {
                    if (issued > (uint32_t)s) {
                        const uint32_t last = (issued - 1u - (uint32_t)s) / (uint32_t)p.stages;
                        (void)mbar_wait_bounded(&full[s], last & 1u);
                    }
                }
            }
        }
        return;
    }

    // ------------------------------------------------------------ consumer warps
    // The count kernel before this one may still run.  A thread waits for it
    // (griddepcontrol.wait) only where it first needs its results: the
    // gradient scale and the weight sum (after the first row's statistics
    // pass), the error word it starts, the row counters and the mean.  The
    // mean divides by the number of kept rows, or (weighted) by their summed
    // target weight.
    bool counted = false;
    float g_reduce = 1.f, wsum = 0.f;
    auto need_count = [&]() {
        if (!counted) {
            griddep_wait();
            if (p.reduce)
                g_reduce = (p.dloss ? __ldg(p.dloss) : 1.f) / (WT ? (float)(*p.wdenom) : (float)(*p.n_dev));
            if (WT) wsum = (float)(*p.wsum);
            counted = true;
        }
    };
    Ring rg(p.stages);
    int par = 0;
    auto wait_full = [&]() {
        if (!*abort_flag && !mbar_wait_bounded(&full[rg.s], rg.ph)) {
            need_count();
            atomicOr(p.err, CE_DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
    };
    auto release = [&]() {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[rg.s]);
        rg.next();
    };
    // Rows come from the producer warp's queue, one entry ahead: each row's
    // successor is read before the row's CTA combine, and that barrier (a
    // reduction) also decides for every consumer warp at once whether the
    // successor is taken -- so all of them run the same rows and barriers,
    // and rows still overlap at their boundaries.
    Ring qr(kRowQ);
    // the next entry: a row, -1 past the last row, -2 when the wait gave up;
    // yout gets the row's target
    auto next_row = [&](int64_t& yout) -> int64_t {
        int64_t v = -2;
        yout = 0;
        if (!*abort_flag) {
            const bool got = __all_sync(kFull, mbar_wait_bounded(&qfull[qr.s], qr.ph));
            if (got) {
                v = rowq[qr.s];
                yout = yq[qr.s];
                __syncwarp();
                if (lane == 0) mbar_arrive(&qempty[qr.s]);
            } else {
                need_count();
                atomicOr(p.err, CE_DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
        }
        qr.next();
        return v;
    };
    int64_t y;
    int64_t r = next_row(y);
    bool stop = named_bar_or(1, NC, r < 0 || *abort_flag);
    while (!stop) {
        char* rowp = row_ptr(r);
        const RowGeo gr = row_geo<GEO, ES, TB>(p, rowp);
        // kGeoEdges: this thread's element among the row's head and tail (or
        // -1), kept in a register from pass 1 to pass 2
        int64_t ee = -1;
        if constexpr (GEO == kGeoEdges) ee = span16_edge(Span16{gr.head, gr.body_bytes / 16, gr.t0}, 0, p.V, tid);
        if (!is_loaded(y)) {
            if (GRAD) {
                const uint4 z = make_uint4(0, 0, 0, 0);
                const int64_t nv = gr.body_bytes / 16;
                char* body = const_cast<char*>(gr.body);
                for (int64_t v = tid; v < nv; v += NC) stg128_stream(body + v * 16, z);
                if (ee >= 0) VT::store1(rowp + ee * ES, 0.f);
            }
            if (tid == 0) {
                p.loss[r] = (y == p.ignore_idx) ? 0.f : __int_as_float(0x7fc00000);
                if (p.lse_out) p.lse_out[r] = __int_as_float(0x7fc00000);
            }
            int64_t ny;
            const int64_t nx = next_row(ny);
            stop = named_bar_or(1, NC, nx < 0 || *abort_flag);
            r = nx;
            y = ny;
            continue;
        }
        const int64_t ybyte = y * ES;
        // the tile holding the target and the target's byte in that tile (-1:
        // the target is a head or tail element, outside the ring)
        int ty = -1, yoff = 0;
        if constexpr (GEO == kGeoChunks) {
            const int c = (int)(y / p.chunk_elems);
            const int64_t jb = (y - (int64_t)c * p.chunk_elems) * ES;
            const int j = (int)(jb / TB);
            ty = c * p.tpc + j;
            yoff = (int)(jb - (int64_t)j * TB);
        } else if (y >= gr.head && y < gr.t0) {
            const int64_t yb = (y - gr.head) * ES;
            ty = (int)(yb / TB);
            yoff = (int)(yb - (int64_t)ty * TB);
        }
        const int yv = yoff / 16;  // the target's vector in its tile

        // pass 1: running statistics over the tiles (and this thread's head
        // or tail element)
        float m = -INFINITY;
        float2 d2 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
        float xe = 0.f;
        if constexpr (GEO == kGeoEdges) {
            if (ee >= 0) {
                xe = VT::load1(rowp + ee * ES);
                m = xe;
                d2.x = 1.f;
                s2.x = xe;
            }
            if (ty < 0 && ee == y) xy_s[par] = xe;
        }
        for (int t = 0; t < gr.ntiles; ++t) {
            wait_full();
            int64_t off;
            uint32_t bytes;
            tile_span<GEO, TB>(p, gr, t, off, bytes);
            const uint4* tile = reinterpret_cast<const uint4*>(ring + (size_t)rg.s * TB);
            if (t == ty && tid == 0) xy_s[par] = VT::load1(ring + (size_t)rg.s * TB + yoff);
            const int64_t e0 = off / ES;
            // the weighted sum comes with pass 2 when there is one; chunked
            // rows keep the warp's running max
            constexpr bool UNI = GEO == kGeoChunks;
            constexpr bool SUM = !(WT && GRAD);
            if (bytes == (uint32_t)TB)
                stats_tile<T, NC, NV, true, WT && !GRAD, UNI, SUM>(tile, tid, TV, m, d2, s2, p.cw, e0);
            else
                stats_tile<T, NC, NV, false, WT && !GRAD, UNI, SUM>(tile, tid, (int)(bytes / 16), m, d2,
                                                                    s2, p.cw, e0);
            release();
            if constexpr (GEO == kGeoChunks) {
                // end of a chunk: the warp's partial of this chunk (its lanes
                // share the running max: two sums), then a fresh running
                // partial for the next one
                if (t == gr.ntiles - 1 || (t + 1) % p.tpc == 0) {
                    const float dw = warp_allsum(d2.x + d2.y);
                    const float sw = warp_allsum(s2.x + s2.y);
                    if (lane == 0) red[(par * KS + t / p.tpc) * NW + warp] = make_float4(m, dw, sw, 0.f);
                    m = -INFINITY;
                    d2 = make_float2(0.f, 0.f);
                    s2 = make_float2(0.f, 0.f);
                }
            }
        }

        // the successor (published before this row's copies)
        int64_t ny;
        const int64_t nx = next_row(ny);
        // CTA combine, fixed order; its barrier takes the exit decision
        if constexpr (GEO != kGeoChunks) {
            Part q = warp_allreduce_part(Part{m, d2.x + d2.y, s2.x + s2.y});
            if (lane == 0) red[par * NW + warp] = make_float4(q.m, q.d, q.S, 0.f);
        }
        stop = named_bar_or(1, NC, nx < 0 || *abort_flag);
        Part G = part_identity();
        if constexpr (GEO == kGeoChunks) {
            // lane c folds chunk c's warp partials in warp order, then every
            // lane folds the chunks in chunk order through shuffles: every
            // warp gets the same bits
            Part P = part_identity();
            if (lane < p.nchunks) {
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    const float4 v4 = red[(par * KS + lane) * NW + w];
                    P = part_combine(P, Part{v4.x, v4.y, v4.z});
                }
                if (p.part && warp == 0) {
                    const int cy = (int)(y / p.chunk_elems);
                    p.part[r * p.nchunks + lane] = make_float4(P.m, P.d, P.S, lane == cy ? xy_s[par] : 0.f);
                }
            }
            for (int c = 0; c < p.nchunks; ++c) {
                Part q;
                q.m = __shfl_sync(kFull, P.m, c);
                q.d = __shfl_sync(kFull, P.d, c);
                q.S = __shfl_sync(kFull, P.S, c);
                G = part_combine(G, q);
            }
        } else {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float4 v4 = red[par * NW + w];
                G = part_combine(G, Part{v4.x, v4.y, v4.z});
            }
        }
        need_count();
        const float g = p.reduce ? g_reduce : (p.dloss ? __ldg(p.dloss + r) : 1.f);
        const float lse = G.m + logf(G.d);
        const float xy = xy_s[par];
        const float wy = WT ? __ldg(p.cw + y) : 1.f;
        if (!(WT && GRAD) && tid == 0) {
            // weighted: (1-a) w_y (lse - x_y) + (a/V) (W lse - sum_j w_j x_j)
            p.loss[r] = WT ? (1.f - p.a) * wy * (lse - xy) + p.a_over_v * (wsum * lse - G.S)
                           : lse - (1.f - p.a) * xy - p.a_over_v * G.S;
            if (p.lse_out) p.lse_out[r] = lse;
        }

        // pass 2: gradient
        if (GRAD) {
            const float nll = -lse * kLog2e;
            const float bb = g * p.a_over_v;
            // softmax scale: g, or (weighted) g ((1-a) w_y + (a/V) W)
            const float c = WT ? g * ((1.f - p.a) * wy + p.a_over_v * wsum) : g;
            const float2 NL = make_float2(nll, nll);
            const float2 G2 = make_float2(c, c);
            const float2 NB = make_float2(-bb, -bb);
            float2 sw2 = make_float2(0.f, 0.f);
            if constexpr (GEO == kGeoEdges) {
                // this thread's head or tail element, from its register
                if (ee >= 0) {
                    const float e = ex2_approx(fmaf(xe, kLog2e, nll));
                    VT::store1(rowp + ee * ES, fmaf(e, c, -bb) - (ee == y ? g * (1.f - p.a) : 0.f));
                }
            }
            const int R = parked(gr.ntiles);
            for (int k = 0; k < gr.ntiles; ++k) {
                const int t = pass2_tile(k, R, gr.ntiles);  // the parked tiles first
                wait_full();
                int64_t off;
                uint32_t bytes;
                tile_span<GEO, TB>(p, gr, t, off, bytes);
                const int st = rg.s;
                const uint4* tile = reinterpret_cast<const uint4*>(ring + (size_t)st * TB);
                uint4* dst = reinterpret_cast<uint4*>(const_cast<char*>(gr.body) + off);
                rg.next();
                // without smoothing the weighted gradient is c * softmax -
                // c [j == y] and the loss has no sum_j w_j x_j term: no
                // per-class weight is read
                if (WT && wring) {
                    int sw[WS];
                    const unsigned char* wslot[WS];
#pragma unroll
                    for (int h = 0; h < WS; ++h) {
                        wait_full();
                        sw[h] = rg.s;
                        wslot[h] = ring + (size_t)rg.s * TB;
                        rg.next();
                    }
                    if constexpr (ES == 2) {
                        const unsigned char* tb = ring + (size_t)st * TB;
                        unsigned char* db = reinterpret_cast<unsigned char*>(dst);
                        if (bytes == (uint32_t)TB)
                            grad_tile_w16<T, NC, NV, true>(tb, db, tid, 2 * TV, NL, G2, NB, wslot, sw2);
                        else
                            grad_tile_w16<T, NC, NV, false>(tb, db, tid, (int)(bytes / 8), NL, G2, NB, wslot, sw2);
                    } else if (bytes == (uint32_t)TB) {
                        grad_tile<T, NC, NV, true, true>(tile, dst, tid, TV, NL, G2, NB, wslot, sw2);
                    } else {
                        grad_tile<T, NC, NV, false, true>(tile, dst, tid, (int)(bytes / 16), NL, G2, NB, wslot, sw2);
                    }
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&empty[st]);
#pragma unroll
                        for (int h = 0; h < WS; ++h) mbar_arrive(&empty[sw[h]]);
                    }
                } else {
                    if (bytes == (uint32_t)TB)
                        grad_tile<T, NC, NV, true, false>(tile, dst, tid, TV, NL, G2, NB, nullptr, sw2);
                    else
                        grad_tile<T, NC, NV, false, false>(tile, dst, tid, (int)(bytes / 16), NL, G2, NB, nullptr, sw2);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[st]);
                }
                // the target element: the thread that stored its vector (its
                // 8-byte unit in the weighted 16-bit pass) rewrites it with the
                // one-hot term subtracted (same thread, so the second store
                // lands after the first)
                const int yown = (WT && ES == 2 && wring) ? (yoff / 8) % NC : yv % NC;
                if (t == ty && tid == yown) {
                    const float e = ex2_approx(fmaf(xy, kLog2e, nll));
                    VT::store1(rowp + ybyte, fmaf(e, c, -bb * wy) - g * (1.f - p.a) * wy);
                }
            }
            if (WT) {
                // the weighted loss needs sum_j w_j x_j: CTA sum in a fixed order
                float sw = sw2.x + sw2.y;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) sw += __shfl_xor_sync(kFull, sw, off);
                if (lane == 0) sw_s[par * NW + warp] = sw;
                named_bar_sync(1, NC);
                if (tid == 0) {
                    float S = 0.f;
                    for (int w = 0; w < NW; ++w) S += sw_s[par * NW + w];
                    p.loss[r] = (1.f - p.a) * wy * (lse - xy) + p.a_over_v * (wsum * lse - S);
                    if (p.lse_out) p.lse_out[r] = lse;
                }
            }
        }
        par ^= 1;
        r = nx;
        y = ny;
    }

    need_count();
    // the last CTA done claiming rows zeroes the row counter for the next pass
    // (its rows were all claimed before the end mark this CTA has read)
    if (p.row_claim && tid == 0) {
        __threadfence();
        if (atomicAdd(p.row_done, 1u) == gridDim.x - 1) {
            atomicExch(p.row_claim, 0u);
            atomicExch(p.row_done, 0u);
        }
    }

    // reduce_loss: the last CTA to finish sums the per-row losses in a fixed
    // order (fixed strides per thread, butterflies, warps in order) -- the
    // mean of TENPU #29 section 1, computed on the device
    if (p.mean_out) {
        __threadfence();
        named_bar_sync(1, NC);  // every loss row of this CTA is written
        if (tid == 0) {
            __threadfence();
            const unsigned t = atomicAdd(p.ticket, 1u);
            *last_flag = (t == gridDim.x - 1) ? 1 : 0;
        }
        named_bar_sync(1, NC);
        if (*last_flag) {
            __threadfence();
            double acc = strided_sum_fixed(p.loss, p.N, tid, NC);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
            double* dred = reinterpret_cast<double*>(red);
            if (lane == 0) dred[warp] = acc;
            named_bar_sync(1, NC);
            if (tid == 0) {
                double tot = 0.0;
                for (int w = 0; w < NW; ++w) tot += dred[w];
                const double den = WT ? *p.wdenom : (double)(*p.n_dev);
                p.mean_out[0] = (float)(tot / den);  // 0/0 = NaN: all ignored
            }
        }
    }
}

template <typename T, int NC, int NV, bool GRAD, bool WT, int GEO>
cudaError_t launch_stream_one(const Problem& pb, const StreamPlan& plan, float4* parts, cudaStream_t s) {
    auto kern = ce_stream_kernel<T, NC, NV, GRAD, WT, GEO>;
    constexpr int NW = NC / 32;
    constexpr int KS = GEO == kGeoChunks ? kMaxStreamChunks : 1;
    StreamArgs a;
    memset(&a, 0, sizeof a);
    a.logits = pb.logits;
    a.s0 = pb.s0;
    a.s1 = pb.s1;
    a.dim1 = pb.dim1;
    a.N = pb.N;
    a.V = (int32_t)pb.V;
    a.stages = plan.stages;
    a.tile_bytes = (uint32_t)(NC * NV * 16);  // must match the kernel's TB
    const int64_t TB = a.tile_bytes;
    const int64_t row_bytes = pb.V * (int64_t)sizeof(T);
    if (GEO == kGeoChunks) {
        // chunks of chunk_elems elements (a multiple of the 16-byte vector),
        // tpc tiles each; the last non-empty chunk may be shorter
        const int64_t C = plan.chunk_elems;
        if (C < 1 || (C * (int64_t)sizeof(T)) % 16) return cudaErrorInvalidValue;
        const int64_t CB = C * (int64_t)sizeof(T);
        const int64_t nchunks = (pb.V + C - 1) / C;
        if (nchunks > kMaxStreamChunks || CB > 0xffffffffLL) return cudaErrorInvalidValue;
        const int64_t tpc = (CB + TB - 1) / TB;
        const int64_t last = row_bytes - (nchunks - 1) * CB;
        a.chunk_elems = C;
        a.chunk_bytes = (uint32_t)CB;
        a.tpc = (int32_t)tpc;
        a.nchunks = (int32_t)nchunks;
        a.ntiles = (int32_t)((nchunks - 1) * tpc + (last + TB - 1) / TB);
        a.part = parts;
    } else {
        // kGeoEdges computes its tiles per row, from where the row starts
        a.ntiles = (int32_t)((row_bytes + TB - 1) / TB);
    }
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
    a.ticket = pb.ticket;
    a.mean_out = pb.mean_out;
    a.cw = pb.cw;
    a.wdenom = pb.wdenom;
    a.wsum = pb.wsum;
    // rows handed out by a shared counter while row indices fit it
    a.row_claim = pb.N < (int64_t)0x7fffffff ? pb.row_claim : nullptr;
    a.row_done = pb.row_done;
    a.flat = rows_flat(pb) ? 1 : 0;
    const size_t smem = (size_t)plan.stages * a.tile_bytes + (24 + 4 * kRowQ) * sizeof(uint64_t) +
                        2 * KS * NW * sizeof(float4) + (2 + 2 * NW) * sizeof(float) + 2 * sizeof(int) +
                        16;
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
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    set_pdl_attr(&attr[0]);
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(NC + 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace
}  // namespace gbce
