// ce_stream_geo.cu -- the row-streaming kernel (ce_stream.cuh) for rows off
// the 16-byte grid (a scalar head and tail around a TMA-copied body) and for
// rows cut into vocabulary chunks (per-chunk partials combined in chunk
// order).  256 consuming threads, 16 or 32 KB tiles; unweighted.
#include "ce_stream.cuh"

namespace gbce {
namespace {

template <typename T, bool GRAD, int G>
cudaError_t launch_geo_typed(const Problem& pb, const StreamPlan& plan, float4* parts, cudaStream_t s) {
    if (plan.threads != 256 || pb.cw) return cudaErrorInvalidConfiguration;
    return plan.tile_kb == 16 ? launch_stream_one<T, 256, 4, GRAD, false, G>(pb, plan, parts, s)
                              : launch_stream_one<T, 256, 8, GRAD, false, G>(pb, plan, parts, s);
}

template <int G>
cudaError_t launch_geo(const Problem& p, const StreamPlan& plan, float4* parts, cudaStream_t s) {
    switch (p.dtype) {
        case CE_F32:
            return p.grad ? launch_geo_typed<float, true, G>(p, plan, parts, s)
                          : launch_geo_typed<float, false, G>(p, plan, parts, s);
        case CE_BF16:
            return p.grad ? launch_geo_typed<__nv_bfloat16, true, G>(p, plan, parts, s)
                          : launch_geo_typed<__nv_bfloat16, false, G>(p, plan, parts, s);
        default:
            return p.grad ? launch_geo_typed<__half, true, G>(p, plan, parts, s)
                          : launch_geo_typed<__half, false, G>(p, plan, parts, s);
    }
}

}  // namespace

cudaError_t launch_stream_geo(const Problem& p, const StreamPlan& plan, float4* parts, cudaStream_t s) {
    if (plan.geo == kStreamEdges) return launch_geo<kGeoEdges>(p, plan, parts, s);
    if (plan.geo == kStreamChunks) return launch_geo<kGeoChunks>(p, plan, parts, s);
    return cudaErrorInvalidValue;
}

}  // namespace gbce
