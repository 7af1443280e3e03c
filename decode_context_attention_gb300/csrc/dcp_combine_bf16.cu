// dcp_combine_bf16.cu -- instantiates the merge kernels for bf16 payloads (one
// translation unit per payload type so the library builds in parallel).
#include "dcp_combine.cuh"

namespace dcp {

cudaError_t launch_combine_bf16(const CombineParams& p, int vb, cudaStream_t stream) {
    return launch_combine_t<__nv_bfloat16>(p, vb, stream);
}

}  // namespace dcp
