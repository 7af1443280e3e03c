// dcp_pack.cu -- the stride-parameterised pack (a pure bit copy).
//
// For each source row (g, b, h), with H_pr = H / N, peer p = h / H_pr and
// local head hl = h % H_pr (sglang PR #34651 report, "实现拆解" item 1):
//     dst_o  [g][p, b, hl, :] = o  [g][b, h, :]
//     dst_lse[g][p, b, hl]    = lse[g][b, h]
// One kernel serves the peer-major interleaved send buffer and the
// peer-inside split layout; only the destination strides differ.
//
// Design: HBM copy.  A group of `lpr` lanes owns a batch of RB consecutive
// source rows (consecutive heads of one token and peer) and issues the loads
// of the whole batch before any store, so each warp keeps 4 KiB in flight
// (8 vectors per lane of 16 bytes, or 32 of 4 bytes).
// Vectors are as wide as every source and destination row start allows
// (16 B for the peer-inside layout and contiguous sources; 4 B for the
// interleaved rows, whose starts advance by D*e + 4 bytes).  Row indices are
// advanced with carries instead of 64-bit division.  Lane k of the group
// copies the LSE word of the batch's row k as raw bits.
#include "dcp_device.cuh"

namespace dcp {

// LINEAR: the host guarantees that H_pr is a multiple of RB, so the RB rows of
// a batch share (g, b, peer) and step by one head: their addresses are one
// base plus k times the head stride.  Otherwise a batch is a single row.
// LPR > 0 fixes the lanes per row at compile time (rows of >= 2 vectors per
// lane always use whole warps), making every vector offset an immediate.
template <int VB, int VPL, bool LINEAR, int LPR>
__global__ void __launch_bounds__(kThreads) pack_kernel(const PackParams p) {
    constexpr int MAXV = VB == 16 ? 8 : 32;  // vectors held per lane per batch (<= 32 registers)
    constexpr int RB = LINEAR ? (MAXV / VPL > 0 ? MAXV / VPL : 1) : 1;  // rows per batch
    using V = typename VecT<VB>::type;
    pdl_wait();
    const int lpr = LPR > 0 ? LPR : p.lpr;
    const LaneGroup lg = lane_group(lpr);
    const int nv = p.row_bytes / VB;
    const int64_t nbatch = (p.rows + RB - 1) / RB;
    RowCursor cur;
    cur.set(lg.first * RB, p.B, p.H);
    RowStep st;
    st.set(lg.step * RB, p.B, p.H);
    for (int64_t bi = lg.first; bi < nbatch; bi += lg.step) {
        const int peer = cur.h / p.H_pr;
        const int hl = cur.h - peer * p.H_pr;
        const unsigned char* src = p.o + cur.g * p.o_sg + (int64_t)cur.b * p.o_sb + (int64_t)cur.h * p.o_sh;
        unsigned char* dst = p.dst_o + cur.g * p.do_sg + (int64_t)peer * p.do_sn +
                             (int64_t)cur.b * p.do_sb + (int64_t)hl * p.do_sh;
        if (p.copy_payload) {
            for (int v0 = lg.jl; v0 < nv; v0 += lpr * VPL) {
                V x[RB][VPL];
#pragma unroll
                for (int k = 0; k < RB; ++k)
#pragma unroll
                    for (int j = 0; j < VPL; ++j) {
                        const int v = v0 + j * lpr;
                        if (v < nv) x[k][j] = ld_stream<VB>(src + k * p.o_sh + (int64_t)v * VB);
                    }
#pragma unroll
                for (int k = 0; k < RB; ++k)
#pragma unroll
                    for (int j = 0; j < VPL; ++j) {
                        const int v = v0 + j * lpr;
                        if (v < nv) st_vec<VB>(dst + k * p.do_sh + (int64_t)v * VB, x[k][j]);
                    }
            }
        }
        if (p.copy_lse && lg.jl < RB) {
            // lane k of the group copies the LSE word of row k of the batch
            const int k = lg.jl;
            const unsigned bits = __ldg(reinterpret_cast<const unsigned*>(p.lse) + cur.g * p.l_sg +
                                        (int64_t)cur.b * p.l_sb + (int64_t)(cur.h + k) * p.l_sh);
            reinterpret_cast<unsigned*>(p.dst_lse)[cur.g * p.dl_sg + (int64_t)peer * p.dl_sn +
                                                   (int64_t)cur.b * p.dl_sb + (int64_t)(hl + k) * p.dl_sh] = bits;
        }
        cur.add(st.dg, st.db, st.dh, p.B, p.H);
    }
    pdl_trigger();
}

template <int VB, bool LINEAR>
static const void* pick_pack(int vpl) {
    if (vpl <= 1) return (const void*)pack_kernel<VB, 1, LINEAR, 0>;
    if (vpl <= 2) return (const void*)pack_kernel<VB, 2, LINEAR, 32>;
    if (vpl <= 4) return (const void*)pack_kernel<VB, 4, LINEAR, 32>;
    return (const void*)pack_kernel<VB, 8, LINEAR, 32>;
}

template <int VB>
static const void* pick_pack_linear(int vpl, bool linear) {
    return linear ? pick_pack<VB, true>(vpl) : pick_pack<VB, false>(vpl);
}

cudaError_t launch_pack(const PackParams& p, cudaStream_t stream) {
    const int nv = p.row_bytes / p.vb;
    const int vpl_need = (nv + p.lpr - 1) / p.lpr;
    const int vpl = vpl_need <= 1 ? 1 : vpl_need <= 2 ? 2 : vpl_need <= 4 ? 4 : 8;
    const int rb_linear = (p.vb == 16 ? 8 : 32) / vpl;
    const bool linear = p.H_pr % rb_linear == 0 && rb_linear <= p.lpr;
    const int rb = linear ? rb_linear : 1;
    const void* k;
    if (p.vb == 16) k = pick_pack_linear<16>(vpl, linear);
    else if (p.vb == 4) k = pick_pack_linear<4>(vpl, linear);
    else if (p.vb == 2) k = pick_pack_linear<2>(vpl, linear);
    else return cudaErrorInvalidValue;
    const int batches_per_cta = (kThreads / 32) * (32 / p.lpr);
    const int64_t nbatch = (p.rows + rb - 1) / rb;
    const int grid = grid_for(k, nbatch, batches_per_cta, kThreads, 0, false);
    void* args[] = {(void*)&p};
    return launch_pdl(k, dim3(grid), dim3(kThreads), args, 0, stream);
}

}  // namespace dcp
