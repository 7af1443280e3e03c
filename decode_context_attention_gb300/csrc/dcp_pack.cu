// dcp_pack.cu -- the stride-parameterised pack (a pure bit copy).
//
// For each source row (g, b, h), with H_pr = H / N, peer p = h / H_pr and
// local head hl = h % H_pr (sglang PR #34651 report, "实现拆解" item 1):
//     dst_o  [g][p, b, hl, :] = o  [g][b, h, :]
//     dst_lse[g][p, b, hl]    = lse[g][b, h]
// One kernel serves the peer-major interleaved send buffer and the
// peer-inside split layout; only the destination strides differ.
//
// Design: HBM copy.  A group of `lpr` lanes copies one row with the widest
// vector every source and destination row start allows (16 B for the
// peer-inside layout and contiguous sources; 4 B for the interleaved rows,
// whose starts advance by D*e + 4 bytes), batching up to 8 loads per lane
// before their stores.  Lane 0 of the group copies the LSE word as raw bits.
// Rows are taken in source order so consecutive groups read consecutive
// memory.
#include "dcp_device.cuh"

namespace dcp {

template <int VB>
__global__ void __launch_bounds__(kThreads) pack_kernel(const PackParams p) {
    constexpr int KU = VB == 16 ? 4 : 8;  // loads in flight per lane
    using V = typename VecT<VB>::type;
    const LaneGroup lg = lane_group(p.lpr);
    const int nv = p.row_bytes / VB;
    for (int64_t row = lg.first; row < p.rows; row += lg.step) {
        const int64_t h = row % p.H;
        const int64_t t = row / p.H;
        const int64_t b = t % p.B;
        const int64_t g = t / p.B;
        const int64_t peer = h / p.H_pr;
        const int64_t hl = h % p.H_pr;
        if (p.copy_payload) {
            const unsigned char* src = p.o + g * p.o_sg + b * p.o_sb + h * p.o_sh;
            unsigned char* dst = p.dst_o + g * p.do_sg + peer * p.do_sn + b * p.do_sb + hl * p.do_sh;
            for (int v0 = lg.jl; v0 < nv; v0 += p.lpr * KU) {
                V x[KU];
#pragma unroll
                for (int k = 0; k < KU; ++k) {
                    const int v = v0 + k * p.lpr;
                    if (v < nv) x[k] = ld_stream<VB>(src + (int64_t)v * VB);
                }
#pragma unroll
                for (int k = 0; k < KU; ++k) {
                    const int v = v0 + k * p.lpr;
                    if (v < nv) st_vec<VB>(dst + (int64_t)v * VB, x[k]);
                }
            }
        }
        if (p.copy_lse && lg.jl == 0) {
            const unsigned bits =
                __ldg(reinterpret_cast<const unsigned*>(p.lse) + g * p.l_sg + b * p.l_sb + h * p.l_sh);
            reinterpret_cast<unsigned*>(p.dst_lse)[g * p.dl_sg + peer * p.dl_sn + b * p.dl_sb +
                                                   hl * p.dl_sh] = bits;
        }
    }
}

cudaError_t launch_pack(const PackParams& p, cudaStream_t stream) {
    const void* k;
    if (p.vb == 16) k = (const void*)pack_kernel<16>;
    else if (p.vb == 4) k = (const void*)pack_kernel<4>;
    else if (p.vb == 2) k = (const void*)pack_kernel<2>;
    else return cudaErrorInvalidValue;
    const int rows_per_cta = (kThreads / 32) * (32 / p.lpr);
    const int grid = persistent_grid(k, p.rows, rows_per_cta);
    void* args[] = {(void*)&p};
    cudaLaunchKernel(k, dim3(grid), dim3(kThreads), args, 0, stream);
    return cudaGetLastError();
}

}  // namespace dcp
