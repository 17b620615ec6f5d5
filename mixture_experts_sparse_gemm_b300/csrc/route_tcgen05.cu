// Router logits on the tensor cores: not enabled yet; the CUDA-core router runs.
#include "moe_internal.cuh"

namespace moe {

bool route_tcgen05_supported(const moe_config &) { return false; }
size_t route_tcgen05_scratch_bytes(const moe_config &) { return 0; }
cudaError_t launch_route_tcgen05(const moe_config &, const void *, const void *, const float *, const float *,
                                 int32_t *, float *, float *, void *, unsigned *, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace moe
