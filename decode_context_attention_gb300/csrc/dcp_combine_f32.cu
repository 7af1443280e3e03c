// dcp_combine_f32.cu -- instantiates the merge kernels for f32 payloads (one
// translation unit per payload type so the library builds in parallel).
#include "dcp_combine.cuh"

namespace dcp {

cudaError_t launch_combine_f32(const CombineParams& p, int vb, cudaStream_t stream) {
    return launch_combine_t<float>(p, vb, stream);
}

}  // namespace dcp
