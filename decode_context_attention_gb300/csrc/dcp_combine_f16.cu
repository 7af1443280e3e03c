// dcp_combine_f16.cu -- instantiates the merge kernels for f16 payloads (one
// translation unit per payload type so the library builds in parallel).
#include "dcp_combine.cuh"

namespace dcp {

cudaError_t launch_combine_f16(const CombineParams& p, int vb, cudaStream_t stream) {
    return launch_combine_t<__half>(p, vb, stream);
}

}  // namespace dcp
