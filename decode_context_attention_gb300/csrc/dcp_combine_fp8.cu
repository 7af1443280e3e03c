// dcp_combine_fp8.cu -- instantiates the merge kernels for fp8 e4m3 payloads
// (one translation unit per payload type so the library builds in parallel).
#include "dcp_combine.cuh"

namespace dcp {

cudaError_t launch_combine_fp8(const CombineParams& p, int vb, cudaStream_t stream) {
    return launch_combine_t<__nv_fp8_e4m3>(p, vb, stream);
}

}  // namespace dcp
