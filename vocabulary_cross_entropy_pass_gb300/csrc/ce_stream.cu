// ce_stream.cu -- the row-streaming kernel (ce_stream.cuh) for rows on the
// 16-byte grid, unweighted and class-weighted.
#include "ce_stream.cuh"

namespace gbce {
namespace {

// Tiles of 16 or 32 KB, consumed by 256 or 512 threads; the weighted pass
// runs the 256-thread shapes only.
template <typename T, bool GRAD>
cudaError_t launch_stream_typed(const Problem& pb, const StreamPlan& plan, cudaStream_t s) {
    constexpr int G = kGeoAligned;
    if (pb.cw) {
        if (plan.threads != 256) return cudaErrorInvalidConfiguration;
        return plan.tile_kb == 16 ? launch_stream_one<T, 256, 4, GRAD, true, G>(pb, plan, nullptr, s)
                                  : launch_stream_one<T, 256, 8, GRAD, true, G>(pb, plan, nullptr, s);
    }
    if (plan.tile_kb == 16)
        return plan.threads == 512 ? launch_stream_one<T, 512, 2, GRAD, false, G>(pb, plan, nullptr, s)
                                   : launch_stream_one<T, 256, 4, GRAD, false, G>(pb, plan, nullptr, s);
    return plan.threads == 512 ? launch_stream_one<T, 512, 4, GRAD, false, G>(pb, plan, nullptr, s)
                               : launch_stream_one<T, 256, 8, GRAD, false, G>(pb, plan, nullptr, s);
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
