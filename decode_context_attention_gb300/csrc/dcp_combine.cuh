// dcp_combine.cuh -- the LSE-weighted merge kernels (templated over the payload
// type, the vector width, the rank count and the O-sanitising flag), included
// by one translation unit per payload type.
//
// What they compute, per output row (g, b, h), over ranks r < N (sglang PR
// #34213 report, "关键源码片段", `cp_lse_ag_out_rs_mha`; sglang PR #34651
// report, "实现拆解" item 3, `dcp_lse_combine_triton`):
//     Gl  = logsumexp_r lse_r   in base e or base 2 (sglang PR #33926 report,
//           "实现拆解" item 4): any NaN -> NaN, else any +inf -> +inf, else all
//           -inf -> -inf, else max + log(sum base^(lse_r - max))
//     w_r = base^(lse_r - Gl), replaced by 0 when not finite (nan_to_num)
//     out = sum_r w_r * O_r    accumulated in fp32 in rank order, rounded once
// The weights are evaluated as base^(lse_r - max) / sum_j base^(lse_j - max),
// the same number as base^(lse_r - Gl) when Gl is finite but without the
// fp32 rounding of Gl in every weight; when Gl is not finite every weight is
// 0, as nan_to_num makes it.
//
// Design (GB300, HBM-bound: ~2N flops per 2N-4N bytes, no tensor cores):
//  * a group of `lpr` lanes (a whole warp for rows of >= 512 B) owns one row;
//    lane r of the group loads lse_r, and the max / NaN-inf class / sum of
//    exponentials are reduced with xor shuffles inside the group, then each
//    rank's weight is broadcast to the group with one shuffle;
//  * payload is streamed with 16-byte vectors when every row start is 16-byte
//    aligned; rows that start only 4-byte aligned (the interleaved receive
//    rows) are read as 16-byte-aligned chunks shifted per row when every rank
//    shares the misalignment, else with 4- (or 2-) byte vectors; 16-bit
//    elements are widened two at a time and accumulated with paired fp32 FMAs
//    (fma.rn.f32x2), about 1.5 instructions per element, fp8 e4m3 pairs
//    through the hardware e4m3x2 -> f16x2 convert, so the merge stays below
//    the HBM time;
//  * the register variants issue all ranks' loads of a chunk before the
//    weights are reduced (fixed-shape templates for the common row lengths,
//    runtime-shaped ones otherwise); a staged variant that copies the next
//    rows' rank stack into shared memory with cp.async is built only on
//    request (measured slower on GB300);
//  * persistent grid: SM count x resident CTAs, grid-stride over rows with
//    division-free row cursors.
#pragma once

#include <math.h>

#include "dcp_device.cuh"
#include "dcp_sm100.cuh"

// Tuning knobs (compile-time): use the fixed-shape merge for the common row
// lengths; use the shifted-chunk merge for 4-byte-aligned rows of those
// lengths; use the cp.async-staged merge where it applies (off: measured
// slower than the register variants on GB300), its pipeline depth (rows) and
// warps per CTA.
#ifndef DCP_COMBINE_FIXED
#define DCP_COMBINE_FIXED 1
#endif
#ifndef DCP_COMBINE_SHIFTED
#define DCP_COMBINE_SHIFTED 1
#endif

#ifndef DCP_COMBINE_STAGED
#define DCP_COMBINE_STAGED 0
#endif
#ifndef DCP_COMBINE_BULK
#define DCP_COMBINE_BULK 0  // 1: stage 16-byte-aligned rank rows with 1-D cp.async.bulk (an A/B knob)
#endif
#ifndef DCP_STAGES
#define DCP_STAGES 3
#endif
#ifndef DCP_STAGED_WARPS
#define DCP_STAGED_WARPS 4
#endif

namespace dcp {

__device__ __forceinline__ float lse_exp(float x, bool b2) { return b2 ? exp2f(x) : expf(x); }
__device__ __forceinline__ float lse_log(float x, bool b2) { return b2 ? log2f(x) : logf(x); }

// Class bits of an LSE value for the extended-real logsumexp.
constexpr unsigned kHasNaN = 1u;
constexpr unsigned kHasPosInf = 2u;

__device__ __forceinline__ float global_lse_from(unsigned cls, float m, float s, bool b2) {
    if (cls & kHasNaN) return __int_as_float(0x7fc00000);  // quiet NaN
    if (cls & kHasPosInf) return INFINITY;
    if (m == -INFINITY) return -INFINITY;
    return m + lse_log(s, b2);
}

// Shuffle logsumexp over a lane group: lane r holds lse_r (-inf for lanes
// without a rank).  Returns this lane's weight; Gl gets the global LSE.
__device__ __forceinline__ float group_weight(float l, const LaneGroup& lg, int lpr, bool b2, float& Gl) {
    unsigned cls = isnan(l) ? kHasNaN : (l == INFINITY ? kHasPosInf : 0u);
    float m = cls ? -INFINITY : l;
    for (int off = lpr >> 1; off > 0; off >>= 1) {
        m = fmaxf(m, __shfl_xor_sync(lg.mask, m, off, lpr));
        cls |= __shfl_xor_sync(lg.mask, cls, off, lpr);
    }
    float wl = 0.f, s = 0.f;
    if (cls == 0u && m != -INFINITY) {
        const float el = lse_exp(l - m, b2);  // lanes with -inf (or no rank) hold 0
        s = el;
        for (int off = lpr >> 1; off > 0; off >>= 1) s += __shfl_xor_sync(lg.mask, s, off, lpr);
        wl = el / s;
    }
    Gl = global_lse_from(cls, m, s, b2);
    return wl;
}

// Weights of ranks r < NRMAX (0 for r >= N) when a lane group is narrower than
// the rank count: every lane reduces serially.
template <int NRMAX>
__device__ __forceinline__ void serial_weights(const float* lrow, int64_t l_sn, int N, bool b2,
                                               float (&w)[NRMAX], float& Gl) {
    float l[NRMAX];
    unsigned cls = 0u;
    float m = -INFINITY;
#pragma unroll
    for (int r = 0; r < NRMAX; ++r) {
        l[r] = r < N ? __ldg(lrow + (int64_t)r * l_sn) : -INFINITY;
        if (isnan(l[r])) cls |= kHasNaN;
        else if (l[r] == INFINITY) cls |= kHasPosInf;
        else m = fmaxf(m, l[r]);
    }
    float s = 0.f;
#pragma unroll
    for (int r = 0; r < NRMAX; ++r) w[r] = 0.f;
    if (cls == 0u && m != -INFINITY) {
#pragma unroll
        for (int r = 0; r < NRMAX; ++r) {
            w[r] = lse_exp(l[r] - m, b2);  // -inf and absent ranks give 0
            s += w[r];
        }
        const float inv = 1.f / s;
#pragma unroll
        for (int r = 0; r < NRMAX; ++r) w[r] *= inv;
    }
    Gl = global_lse_from(cls, m, s, b2);
}

// ---------------------------------------------------------------------------
// Register variant.
// ---------------------------------------------------------------------------
template <typename T, int VB, int NRMAX, bool SAN>
__global__ void __launch_bounds__(kThreads, 2) combine_kernel(const CombineParams p) {
    pdl_wait();
    constexpr int EPV = VB / (int)sizeof(T);
    constexpr int RC = NRMAX < 8 ? NRMAX : 8;  // ranks per load batch
    // vectors per lane per batch: at most ~64 registers of loaded payload and
    // 32 fp32 accumulators, so two CTAs fit on an SM without spilling
    constexpr int KU_LD = 64 / (RC * (VB / 4 > 0 ? VB / 4 : 1));
    constexpr int KU_ACC = 32 / EPV;
    constexpr int KU0 = KU_LD < KU_ACC ? KU_LD : KU_ACC;
    constexpr int KU = KU0 < 1 ? 1 : (KU0 > 8 ? 8 : KU0);
    using V = typename VecT<VB>::type;

    const LaneGroup lg = lane_group(p.lpr);
    const int lpr = p.lpr;
    const bool b2 = p.base2 != 0;
    const int N = p.N;
    const int nv = p.vec_per_row;
    RowStep st;
    st.set(lg.step, p.B, p.Hc);
    RowCursor c;
    c.set(lg.first, p.B, p.Hc);
    for (int64_t row = lg.first; row < p.rows; row += lg.step, c.add(st.dg, st.db, st.dh, p.B, p.Hc)) {
        const float* lrow = p.lse + c.g * p.l_sg + (int64_t)c.b * p.l_sb + (int64_t)c.h * p.l_sh;
        const unsigned char* orow = p.o + c.g * p.o_sg + (int64_t)c.b * p.o_sb + (int64_t)c.h * p.o_sh;
        unsigned char* urow = p.out + c.g * p.u_sg + (int64_t)c.b * p.u_sb + (int64_t)c.h * p.u_sh;
        const bool shuffle = N <= lpr;
        const float l = shuffle && lg.jl < N ? __ldg(lrow + (int64_t)lg.jl * p.l_sn) : -INFINITY;
        float w[NRMAX];
        float Gl = 0.f;
        // group-uniform chunk loop (every lane runs the same iterations)
        for (int base = 0; base < nv; base += lpr * KU) {
            float acc[KU][EPV];
#pragma unroll
            for (int k = 0; k < KU; ++k)
#pragma unroll
                for (int i = 0; i < EPV; ++i) acc[k][i] = 0.f;
#pragma unroll
            for (int r0 = 0; r0 < NRMAX; r0 += RC) {
                if (r0 >= N) break;
                V x[KU][RC];
#pragma unroll
                for (int k = 0; k < KU; ++k) {
                    const int v = base + lg.jl + k * lpr;
#pragma unroll
                    for (int j = 0; j < RC; ++j)
                        if (r0 + j < N && v < nv)
                            x[k][j] = ld_stream<VB>(orow + (int64_t)(r0 + j) * p.o_sn + (int64_t)v * VB);
                }
                if (r0 == 0 && base == 0) {
                    // the weights are reduced while the first loads are in flight
                    if (shuffle) {
                        const float wl = group_weight(l, lg, lpr, b2, Gl);
#pragma unroll
                        for (int r = 0; r < NRMAX; ++r)
                            w[r] = r < N ? __shfl_sync(lg.mask, wl, r & (lpr - 1), lpr) : 0.f;
                    } else {
                        serial_weights<NRMAX>(lrow, p.l_sn, N, b2, w, Gl);
                    }
                }
#pragma unroll
                for (int k = 0; k < KU; ++k)
#pragma unroll
                    for (int j = 0; j < RC; ++j)
                        if (r0 + j < N) fma_vec<T, VB, SAN>(acc[k], x[k][j], w[r0 + j]);
            }
#pragma unroll
            for (int k = 0; k < KU; ++k) {
                const int v = base + lg.jl + k * lpr;
                if (v < nv) st_vec<VB>(urow + (int64_t)v * VB, round_vec<T, VB>(acc[k]));
            }
        }
        if (p.return_lse && lg.jl == 0) p.out_lse[c.g * p.ul_sg + (int64_t)c.b * p.ul_sb + (int64_t)c.h * p.ul_sh] = Gl;
    }
    pdl_trigger();
}

// ---------------------------------------------------------------------------
// Fixed-shape variant for the common rows: LPR lanes per row and VPL vectors
// per lane per rank are compile-time constants (row bytes = LPR * VPL * VB
// exactly), so every load and store offset is an immediate, and the fp32
// accumulators live as packed pairs for the whole row.  Needs N <= LPR (the
// shuffle reduction) and N <= NR.
// ---------------------------------------------------------------------------
template <typename T, int VB, int NR, int LPR, int VPL, bool SAN>
__global__ void __launch_bounds__(kThreads, (sizeof(T) == 1 && VB == 4) ? 3 : 2) combine_fixed_kernel(const CombineParams p) {
    pdl_wait();
    constexpr int NP = VB / (int)sizeof(T) / 2;  // fp32 pairs per vector
    // vectors per lane per rank loaded at once: <= 64 registers of payload
    // and <= 64 registers of packed fp32 accumulators
    constexpr int WPV = VB / 4;
    // payload registers per chunk: 64, or 32 for fp8 rows read in 4-byte words,
    // which run 3 CTAs per SM instead of 2 (the fp8 unpack+combine is bound by
    // latency and issue, not by bytes: 22.1 -> 20.8 us)
    constexpr int LD_REGS = (sizeof(T) == 1 && VB == 4) ? 32 : 64;
    constexpr int VCH_LD = LD_REGS / (NR * WPV) > 0 ? LD_REGS / (NR * WPV) : 1;
    constexpr int VCH_ACC = 32 / NP > 0 ? 32 / NP : 1;
    constexpr int VCH0 = VCH_LD < VCH_ACC ? VCH_LD : VCH_ACC;
    constexpr int VCH = VCH0 >= VPL ? VPL : VCH0;
    static_assert(VPL % VCH == 0, "chunks must tile the row");
    using V = typename VecT<VB>::type;

    const int lane = threadIdx.x & 31;
    LaneGroup lg;
    lg.jl = lane & (LPR - 1);
    lg.sub = lane / LPR;
    lg.mask = LPR == 32 ? 0xffffffffu : (((1u << LPR) - 1u) << (lg.sub * LPR));
    const int64_t wpc = blockDim.x / 32;
    lg.first = ((int64_t)blockIdx.x * wpc + (threadIdx.x / 32)) * (32 / LPR) + lg.sub;
    lg.step = (int64_t)gridDim.x * wpc * (32 / LPR);

    const bool b2 = p.base2 != 0;
    const int N = p.N;
    RowStep st;
    st.set(lg.step, p.B, p.Hc);
    RowCursor c;
    c.set(lg.first, p.B, p.Hc);
    const int64_t lane_off = (int64_t)lg.jl * VB;
    for (int64_t row = lg.first; row < p.rows; row += lg.step, c.add(st.dg, st.db, st.dh, p.B, p.Hc)) {
        const float* lrow = p.lse + c.g * p.l_sg + (int64_t)c.b * p.l_sb + (int64_t)c.h * p.l_sh;
        const unsigned char* orow =
            p.o + c.g * p.o_sg + (int64_t)c.b * p.o_sb + (int64_t)c.h * p.o_sh + lane_off;
        unsigned char* urow = p.out + c.g * p.u_sg + (int64_t)c.b * p.u_sb + (int64_t)c.h * p.u_sh + lane_off;
        const float l = lg.jl < N ? __ldg(lrow + (int64_t)lg.jl * p.l_sn) : -INFINITY;
        unsigned long long w2[NR];
        float Gl = 0.f;
#pragma unroll
        for (int c0 = 0; c0 < VPL; c0 += VCH) {
            V x[NR][VCH];
#pragma unroll
            for (int j = 0; j < NR; ++j)
                if (j < N) {
                    const unsigned char* rp = orow + (int64_t)j * p.o_sn;
#pragma unroll
                    for (int q = 0; q < VCH; ++q) x[j][q] = ld_stream<VB>(rp + (c0 + q) * LPR * VB);
                }
            if (c0 == 0) {
                // the weights are reduced while the first loads are in flight
                const float wl = group_weight(l, lg, LPR, b2, Gl);
#pragma unroll
                for (int j = 0; j < NR; ++j) {
                    const float wj = __shfl_sync(lg.mask, wl, j & (LPR - 1), LPR);
                    w2[j] = pack2f(wj, wj);
                }
            }
            unsigned long long acc[VCH][NP];
#pragma unroll
            for (int q = 0; q < VCH; ++q)
#pragma unroll
                for (int i = 0; i < NP; ++i) acc[q][i] = 0ull;
#pragma unroll
            for (int j = 0; j < NR; ++j)
                if (j < N)
#pragma unroll
                    for (int q = 0; q < VCH; ++q) fma_pairs<T, VB, SAN>(acc[q], x[j][q], w2[j]);
#pragma unroll
            for (int q = 0; q < VCH; ++q) st_vec<VB>(urow + (c0 + q) * LPR * VB, round_pairs<T, VB>(acc[q]));
        }
        if (p.return_lse && lg.jl == 0)
            p.out_lse[c.g * p.ul_sg + (int64_t)c.b * p.ul_sb + (int64_t)c.h * p.ul_sh] = Gl;
    }
    pdl_trigger();
}

// ---------------------------------------------------------------------------
// Shifted-chunk variant for payload rows that start on a 4-byte but not a
// 16-byte boundary (the interleaved receive rows, D*e + 4 bytes apart) when
// every rank's row of an output row has the same misalignment (rank stride a
// multiple of 16 bytes).  The lanes read the 16-byte-aligned chunks that cover
// the row -- the same chunk positions in every rank, so word k of a chunk is
// the same payload word in all of them -- merge them word by word and store
// each word at its place in the (4-byte-aligned) output row.  Chunk 0 starts
// up to 12 bytes before the row (those words are read, never used or
// written); the up to 3 payload words past the last whole chunk are merged by
// the first lanes from 4-byte loads.  Reads stay inside the aligned 16-byte
// granules that hold the row, so they never leave its pages.
// ---------------------------------------------------------------------------
template <typename T, int NR, int LPR, int VPL, bool SAN>
__global__ void __launch_bounds__(kThreads, 2) combine_shifted_kernel(const CombineParams p) {
    pdl_wait();
    constexpr int NP = 16 / (int)sizeof(T) / 2;  // fp32 pairs per chunk
    constexpr int EPW = 4 / (int)sizeof(T);      // elements per word
    constexpr int RB = LPR * VPL * 16;           // payload bytes of a row
    constexpr int VCH_LD = 64 / (NR * 4) > 0 ? 64 / (NR * 4) : 1;
    constexpr int VCH_ACC = 32 / NP > 0 ? 32 / NP : 1;
    constexpr int VCH0 = VCH_LD < VCH_ACC ? VCH_LD : VCH_ACC;
    constexpr int VCH = VCH0 >= VPL ? VPL : VCH0;
    static_assert(VPL % VCH == 0, "chunks must tile the row");

    const int lane = threadIdx.x & 31;
    LaneGroup lg;
    lg.jl = lane & (LPR - 1);
    lg.sub = lane / LPR;
    lg.mask = LPR == 32 ? 0xffffffffu : (((1u << LPR) - 1u) << (lg.sub * LPR));
    const int64_t wpc = blockDim.x / 32;
    lg.first = ((int64_t)blockIdx.x * wpc + (threadIdx.x / 32)) * (32 / LPR) + lg.sub;
    lg.step = (int64_t)gridDim.x * wpc * (32 / LPR);

    const bool b2 = p.base2 != 0;
    const int N = p.N;
    RowStep st;
    st.set(lg.step, p.B, p.Hc);
    RowCursor c;
    c.set(lg.first, p.B, p.Hc);
    for (int64_t row = lg.first; row < p.rows; row += lg.step, c.add(st.dg, st.db, st.dh, p.B, p.Hc)) {
        const float* lrow = p.lse + c.g * p.l_sg + (int64_t)c.b * p.l_sb + (int64_t)c.h * p.l_sh;
        const unsigned char* o0 = p.o + c.g * p.o_sg + (int64_t)c.b * p.o_sb + (int64_t)c.h * p.o_sh;
        unsigned char* urow = p.out + c.g * p.u_sg + (int64_t)c.b * p.u_sb + (int64_t)c.h * p.u_sh;
        const int skip = (int)((uintptr_t)o0 & 15u) >> 2;   // words of chunk 0 before the row
        const unsigned char* oal = o0 - 4 * skip + lg.jl * 16;
        const float l = lg.jl < N ? __ldg(lrow + (int64_t)lg.jl * p.l_sn) : -INFINITY;
        // payload words past the last whole chunk: lanes 0 .. skip-1, one word each
        const bool tail = lg.jl < skip;
        unsigned xt[NR];
#pragma unroll
        for (int j = 0; j < NR; ++j)
            if (j < N && tail) xt[j] = ld_stream<4>(o0 + (RB - 4 * skip) + 4 * lg.jl + (int64_t)j * p.o_sn);
        unsigned long long w2[NR];
        float Gl = 0.f;
#pragma unroll
        for (int c0 = 0; c0 < VPL; c0 += VCH) {
            uint4 x[NR][VCH];
#pragma unroll
            for (int j = 0; j < NR; ++j)
                if (j < N) {
                    const unsigned char* rp = oal + (int64_t)j * p.o_sn;
#pragma unroll
                    for (int q = 0; q < VCH; ++q) x[j][q] = ld_stream<16>(rp + (c0 + q) * LPR * 16);
                }
            if (c0 == 0) {
                const float wl = group_weight(l, lg, LPR, b2, Gl);
#pragma unroll
                for (int j = 0; j < NR; ++j) {
                    const float wj = __shfl_sync(lg.mask, wl, j & (LPR - 1), LPR);
                    w2[j] = pack2f(wj, wj);
                }
            }
            unsigned long long acc[VCH][NP];
#pragma unroll
            for (int q = 0; q < VCH; ++q)
#pragma unroll
                for (int i = 0; i < NP; ++i) acc[q][i] = 0ull;
#pragma unroll
            for (int j = 0; j < NR; ++j)
                if (j < N)
#pragma unroll
                    for (int q = 0; q < VCH; ++q) fma_pairs<T, 16, SAN>(acc[q], x[j][q], w2[j]);
#pragma unroll
            for (int q = 0; q < VCH; ++q) {
                const uint4 v = round_pairs<T, 16>(acc[q]);
                const unsigned wd[4] = {v.x, v.y, v.z, v.w};
                const int p0 = ((c0 + q) * LPR + lg.jl) * 4 - skip;   // output word of wd[0]
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (p0 + k >= 0) st_vec<4>(urow + 4 * (p0 + k), wd[k]);
            }
        }
        if (tail) {
            float at[EPW];
#pragma unroll
            for (int i = 0; i < EPW; ++i) at[i] = 0.f;
#pragma unroll
            for (int j = 0; j < NR; ++j)
                if (j < N) fma_vec<T, 4, SAN>(at, xt[j], unpack2(w2[j]).x);
            st_vec<4>(urow + (RB - 4 * skip) + 4 * lg.jl, round_vec<T, 4>(at));
        }
        if (p.return_lse && lg.jl == 0)
            p.out_lse[c.g * p.ul_sg + (int64_t)c.b * p.ul_sb + (int64_t)c.h * p.ul_sh] = Gl;
    }
    pdl_trigger();
}

// Shifted-chunk kernel for (T, NR) and this row length, or nullptr.
// Not for fp8: its rows are half as long in bytes, and the word-wise stores
// and the per-word tail cost more than the 4-byte loads they replace
// (fp8 MLA-decode unpack+combine: 25.7 us with 16 lanes x 2 chunks per row,
// 26.7 us with 32 lanes x 1 chunk, against 22.0 us for the 4-byte path).
template <typename T, int NR, bool SAN>
const void* pick_shifted(int row_bytes, int& lpr) {
    if constexpr (sizeof(T) == 1) {
        return nullptr;
    } else {
        if (row_bytes == 128 && NR <= 8) { lpr = 8; return (const void*)combine_shifted_kernel<T, NR, 8, 1, SAN>; }
        if (row_bytes == 256) { lpr = 16; return (const void*)combine_shifted_kernel<T, NR, 16, 1, SAN>; }
        if (row_bytes == 512) { lpr = 32; return (const void*)combine_shifted_kernel<T, NR, 32, 1, SAN>; }
        if (row_bytes == 1024) { lpr = 32; return (const void*)combine_shifted_kernel<T, NR, 32, 2, SAN>; }
        if (row_bytes == 2048) { lpr = 32; return (const void*)combine_shifted_kernel<T, NR, 32, 4, SAN>; }
        return nullptr;
    }
}

// Fixed-shape kernel for (T, VB, NR) and this row length, or nullptr.
template <typename T, int VB, int NR, bool SAN>
const void* pick_fixed(int row_bytes, int& lpr) {
    if constexpr (VB < 4 || (VB == 4 && sizeof(T) == 4)) {
        return nullptr;  // one element per vector: no pairs
    } else {
        if constexpr (sizeof(T) == 1) {
            // fp8 rows of 256 / 512 bytes: 32 bytes per lane and rank (as a
            // 16-bit row of the same D gets), so 4 or 2 rows share a warp and
            // twice the bytes are in flight per lane than at one vector
            constexpr int V32 = 32 / VB;
            if (row_bytes == 8 * 32 && NR <= 8) { lpr = 8; return (const void*)combine_fixed_kernel<T, VB, NR, 8, V32, SAN>; }
            if (row_bytes == 16 * 32) { lpr = 16; return (const void*)combine_fixed_kernel<T, VB, NR, 16, V32, SAN>; }
        }
        if (row_bytes == 8 * VB && NR <= 8) { lpr = 8; return (const void*)combine_fixed_kernel<T, VB, NR, 8, 1, SAN>; }
        if (row_bytes == 16 * VB) { lpr = 16; return (const void*)combine_fixed_kernel<T, VB, NR, 16, 1, SAN>; }
        if (row_bytes == 32 * VB) { lpr = 32; return (const void*)combine_fixed_kernel<T, VB, NR, 32, 1, SAN>; }
        if (row_bytes == 64 * VB) { lpr = 32; return (const void*)combine_fixed_kernel<T, VB, NR, 32, 2, SAN>; }
        if (row_bytes == 128 * VB) { lpr = 32; return (const void*)combine_fixed_kernel<T, VB, NR, 32, 4, SAN>; }
        if (row_bytes == 256 * VB) { lpr = 32; return (const void*)combine_fixed_kernel<T, VB, NR, 32, 8, SAN>; }
        return nullptr;
    }
}

// ---------------------------------------------------------------------------
// Any N (> 32): weights recomputed per batch of 8 ranks from a serial reduction.
// ---------------------------------------------------------------------------
template <typename T, int VB>
__global__ void __launch_bounds__(kThreads, 2) combine_kernel_any_n(const CombineParams p) {
    pdl_wait();
    constexpr int EPV = VB / (int)sizeof(T);
    constexpr int RC = 8;
    using V = typename VecT<VB>::type;
    const LaneGroup lg = lane_group(p.lpr);
    const bool b2 = p.base2 != 0;
    const int N = p.N;
    const int nv = p.vec_per_row;
    for (int64_t row = lg.first; row < p.rows; row += lg.step) {
        const int64_t h = row % p.Hc;
        const int64_t t = row / p.Hc;
        const int64_t b = t % p.B;
        const int64_t g = t / p.B;
        const float* lrow = p.lse + g * p.l_sg + b * p.l_sb + h * p.l_sh;
        unsigned cls = 0u;
        float m = -INFINITY;
        for (int r = 0; r < N; ++r) {
            const float l = __ldg(lrow + (int64_t)r * p.l_sn);
            if (isnan(l)) cls |= kHasNaN;
            else if (l == INFINITY) cls |= kHasPosInf;
            else m = fmaxf(m, l);
        }
        float s = 0.f;
        const bool finite_g = cls == 0u && m != -INFINITY;
        if (finite_g)
            for (int r = 0; r < N; ++r) s += lse_exp(__ldg(lrow + (int64_t)r * p.l_sn) - m, b2);
        const float Gl = global_lse_from(cls, m, s, b2);
        const float inv_s = finite_g ? 1.f / s : 0.f;

        const unsigned char* orow = p.o + g * p.o_sg + b * p.o_sb + h * p.o_sh;
        unsigned char* urow = p.out + g * p.u_sg + b * p.u_sb + h * p.u_sh;
        for (int v = lg.jl; v < nv; v += p.lpr) {
            float acc[EPV];
#pragma unroll
            for (int i = 0; i < EPV; ++i) acc[i] = 0.f;
            for (int r0 = 0; r0 < N; r0 += RC) {
                V x[RC];
                float wr[RC];
#pragma unroll
                for (int j = 0; j < RC; ++j) {
                    if (r0 + j < N) {
                        x[j] = ld_stream<VB>(orow + (int64_t)(r0 + j) * p.o_sn + (int64_t)v * VB);
                        wr[j] = finite_g ? lse_exp(__ldg(lrow + (int64_t)(r0 + j) * p.l_sn) - m, b2) * inv_s
                                         : 0.f;
                    }
                }
#pragma unroll
                for (int j = 0; j < RC; ++j) {
                    if (r0 + j < N) {
                        if (p.sanitize) fma_vec<T, VB, true>(acc, x[j], wr[j]);
                        else fma_vec<T, VB, false>(acc, x[j], wr[j]);
                    }
                }
            }
            st_vec<VB>(urow + (int64_t)v * VB, round_vec<T, VB>(acc));
        }
        if (p.return_lse && lg.jl == 0) p.out_lse[g * p.ul_sg + b * p.ul_sb + h * p.ul_sh] = Gl;
    }
    pdl_trigger();
}

// ---------------------------------------------------------------------------
// Staged variant: every lane copies its 16-byte slices of the next rows' rank
// stack into shared memory with cp.async, DCP_STAGES rows deep, while it
// merges the current row.  Nothing in flight occupies registers.  Each lane
// reads back only the slices it copied itself, so its own cp.async.wait_group
// is the only synchronisation needed (no barrier, no spin loop).  The LSE
// words of a row are loaded (lane r: rank r) when the row is issued and
// reduced with shuffles when it is merged.
// ---------------------------------------------------------------------------
constexpr int kStagedWarps = DCP_STAGED_WARPS;
constexpr int kStages = DCP_STAGES;
static_assert(kStages == 2 || kStages == 3, "pipeline depth is 2 or 3 rows");

template <int NR, int VPL>
constexpr size_t staged_smem_bytes() {
    return (size_t)kStagedWarps * kStages * NR * VPL * 32 * 16;
}

template <typename T, int NR, int VPL, bool SAN>
__global__ void __launch_bounds__(kStagedWarps * 32) combine_staged_kernel(const CombineParams p) {
    pdl_wait();
    constexpr int VPR = NR * VPL;  // 16-byte slices per lane per row
    constexpr int EPV = 16 / (int)sizeof(T);
    extern __shared__ uint4 smem[];
    const int lane = threadIdx.x & 31;
    uint4* wbuf = smem + (size_t)(threadIdx.x >> 5) * kStages * VPR * 32;

    const LaneGroup lg = lane_group(p.lpr);
    const int N = p.N;
    const int nv = p.vec_per_row;
    const int lpr = p.lpr;
    const bool b2 = p.base2 != 0;
    RowStep st;
    st.set(lg.step, p.B, p.Hc);
    RowCursor icur, ccur;  // rows being issued / merged
    icur.set(lg.first, p.B, p.Hc);
    ccur = icur;
    int64_t irow = lg.first;
    float lq[kStages];

    // issue the row at icur into stage `slot` (one commit group per row, empty
    // past the end so group counting stays uniform)
    auto issue = [&](int slot, float& lslot) {
        if (irow < p.rows) {
            const unsigned char* orow =
                p.o + icur.g * p.o_sg + (int64_t)icur.b * p.o_sb + (int64_t)icur.h * p.o_sh;
            uint4* sb = wbuf + slot * VPR * 32 + lane;
#pragma unroll
            for (int j = 0; j < NR; ++j) {
                if (j < N) {
#pragma unroll
                    for (int q = 0; q < VPL; ++q) {
                        const int v = lg.jl + q * lpr;
                        if (v < nv)
                            cp_async_16(sb + (j * VPL + q) * 32, orow + (int64_t)j * p.o_sn + (int64_t)v * 16);
                    }
                }
            }
            const float* lrow =
                p.lse + icur.g * p.l_sg + (int64_t)icur.b * p.l_sb + (int64_t)icur.h * p.l_sh;
            lslot = lg.jl < N ? __ldg(lrow + (int64_t)lg.jl * p.l_sn) : -INFINITY;
        }
        cp_async_commit();
        irow += lg.step;
        icur.add(st.dg, st.db, st.dh, p.B, p.Hc);
    };

    // merge the row at ccur from stage `slot`
    auto merge = [&](int slot, float l) {
        float Gl;
        const float wl = group_weight(l, lg, lpr, b2, Gl);
        float w[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) w[r] = __shfl_sync(lg.mask, wl, r & (lpr - 1), lpr);
        const uint4* sb = wbuf + slot * VPR * 32 + lane;
        unsigned char* urow = p.out + ccur.g * p.u_sg + (int64_t)ccur.b * p.u_sb + (int64_t)ccur.h * p.u_sh;
#pragma unroll
        for (int q = 0; q < VPL; ++q) {
            const int v = lg.jl + q * lpr;
            if (v < nv) {
                float acc[EPV];
#pragma unroll
                for (int i = 0; i < EPV; ++i) acc[i] = 0.f;
#pragma unroll
                for (int j = 0; j < NR; ++j)
                    if (j < N) fma_vec<T, 16, SAN>(acc, sb[(j * VPL + q) * 32], w[j]);
                st_vec<16>(urow + (int64_t)v * 16, round_vec<T, 16>(acc));
            }
        }
        if (p.return_lse && lg.jl == 0)
            p.out_lse[ccur.g * p.ul_sg + (int64_t)ccur.b * p.ul_sb + (int64_t)ccur.h * p.ul_sh] = Gl;
        ccur.add(st.dg, st.db, st.dh, p.B, p.Hc);
    };

    if constexpr (kStages == 3) {
        issue(0, lq[0]);
        issue(1, lq[1]);
        for (int64_t row = lg.first; row < p.rows;) {
            issue(2, lq[2]);
            cp_async_wait<2>();
            merge(0, lq[0]);
            row += lg.step;
            if (row >= p.rows) break;
            issue(0, lq[0]);
            cp_async_wait<2>();
            merge(1, lq[1]);
            row += lg.step;
            if (row >= p.rows) break;
            issue(1, lq[1]);
            cp_async_wait<2>();
            merge(2, lq[2]);
            row += lg.step;
        }
    } else {
        issue(0, lq[0]);
        for (int64_t row = lg.first; row < p.rows;) {
            issue(1, lq[1]);
            cp_async_wait<1>();
            merge(0, lq[0]);
            row += lg.step;
            if (row >= p.rows) break;
            issue(0, lq[0]);
            cp_async_wait<1>();
            merge(1, lq[1]);
            row += lg.step;
        }
    }
    cp_async_wait<0>();
    pdl_trigger();
}

// ---------------------------------------------------------------------------
// Bulk-staged variant (built with -DDCP_COMBINE_BULK=1): each warp keeps a
// ring of kBulkStages output rows in shared memory; its lane 0 fetches the N
// rank rows of each (16-byte-aligned rows of 512 x VPL bytes) with one 1-D
// cp.async.bulk per rank into this CTA's own shared memory, completing on
// the stage's mbarrier, and the warp merges from shared memory.  The copies
// occupy no registers and no load slots.  Waits are bounded as everywhere;
// a wait that runs out makes the warp stop (its rows are then left unwritten).
// ---------------------------------------------------------------------------
constexpr int kBulkStages = 3;

template <int NR, int VPL>
constexpr size_t bulk_smem_bytes() {
    return (size_t)(kThreads / 32) * (kBulkStages * NR * VPL * 512 + kBulkStages * 8) + 128;
}

template <typename T, int NR, int VPL, bool SAN>
__global__ void __launch_bounds__(kThreads, 1) combine_bulk_kernel(const CombineParams p) {
    pdl_wait();
    constexpr int ROWB = VPL * 512;
    constexpr int EPV = 16 / (int)sizeof(T);
    extern __shared__ uint8_t bsm_raw[];
    uint8_t* bsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(bsm_raw) + 127) & ~uintptr_t(127));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* ring = bsm + (size_t)warp * kBulkStages * NR * ROWB;
    uint64_t* bars = reinterpret_cast<uint64_t*>(bsm + (size_t)(kThreads / 32) * kBulkStages * NR * ROWB) +
                     warp * kBulkStages;
    if (lane == 0) {
        for (int s = 0; s < kBulkStages; ++s) sm100::mbar_init(&bars[s], 1);
        sm100::fence_mbar_init();
    }
    __syncwarp();
    int dummy_status = 0;
    volatile int stop = 0;
    const int N = p.N;
    const bool b2 = p.base2 != 0;
    const int64_t nwarps = (int64_t)gridDim.x * (kThreads / 32);
    const int64_t first = (int64_t)blockIdx.x * (kThreads / 32) + warp;
    RowStep st;
    st.set(nwarps, p.B, p.Hc);
    RowCursor icur, ccur;
    icur.set(first, p.B, p.Hc);
    ccur = icur;
    int64_t irow = first;
    float lq[kBulkStages];
    auto issue = [&](int slot) {
        if (irow < p.rows) {
            const unsigned char* orow = p.o + icur.g * p.o_sg + (int64_t)icur.b * p.o_sb + (int64_t)icur.h * p.o_sh;
            if (lane == 0) {
                sm100::mbar_arrive_expect_tx(&bars[slot], (uint32_t)(N * ROWB));
                for (int j = 0; j < N; ++j)
                    asm volatile(
                        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                            sm100::smem_u32(ring + (slot * NR + j) * ROWB)),
                        "l"(orow + (int64_t)j * p.o_sn), "r"(ROWB), "r"(sm100::smem_u32(&bars[slot]))
                        : "memory");
            }
            const float* lrow = p.lse + icur.g * p.l_sg + (int64_t)icur.b * p.l_sb + (int64_t)icur.h * p.l_sh;
            lq[slot] = lane < N ? __ldg(lrow + (int64_t)lane * p.l_sn) : -INFINITY;
        }
        irow += nwarps;
        icur.add(st.dg, st.db, st.dh, p.B, p.Hc);
    };
    const LaneGroup lg = lane_group(32);
#pragma unroll
    for (int s = 0; s < kBulkStages; ++s) issue(s);
    for (int64_t row = first, k = 0; row < p.rows; row += nwarps, ++k) {
        const int slot = (int)(k % kBulkStages);
        if (!sm100::mbar_wait(&bars[slot], (uint32_t)((k / kBulkStages) & 1), &dummy_status, 1, &stop)) break;
        float Gl;
        const float wl = group_weight(lq[slot], lg, 32, b2, Gl);
        float w[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) w[r] = __shfl_sync(0xffffffffu, wl, r);
        unsigned char* urow = p.out + ccur.g * p.u_sg + (int64_t)ccur.b * p.u_sb + (int64_t)ccur.h * p.u_sh;
#pragma unroll
        for (int q = 0; q < VPL; ++q) {
            float acc[EPV];
#pragma unroll
            for (int i = 0; i < EPV; ++i) acc[i] = 0.f;
#pragma unroll
            for (int j = 0; j < NR; ++j)
                if (j < N)
                    fma_vec<T, 16, SAN>(acc, *reinterpret_cast<const uint4*>(ring + (slot * NR + j) * ROWB +
                                                                             (q * 32 + lane) * 16),
                                        w[j]);
            st_vec<16>(urow + (int64_t)(q * 32 + lane) * 16, round_vec<T, 16>(acc));
        }
        if (p.return_lse && lane == 0)
            p.out_lse[ccur.g * p.ul_sg + (int64_t)ccur.b * p.ul_sb + (int64_t)ccur.h * p.ul_sh] = Gl;
        ccur.add(st.dg, st.db, st.dh, p.B, p.Hc);
        // the merge's reads of this stage come before the next copy into it
        sm100::fence_proxy_async_smem();
        __syncwarp();
        issue(slot);
    }
    pdl_trigger();
}

template <typename T, int NR, bool SAN>
const void* pick_staged(int vpl, size_t& smem) {
    if (vpl <= 1) {
        smem = staged_smem_bytes<NR, 1>();
        return (const void*)combine_staged_kernel<T, NR, 1, SAN>;
    }
    smem = staged_smem_bytes<NR, 2>();
    return (const void*)combine_staged_kernel<T, NR, 2, SAN>;
}

template <typename T, int VB, bool SAN>
cudaError_t launch_combine_vb(const CombineParams& p, cudaStream_t stream) {
    void* args[] = {(void*)&p};
    if constexpr (VB == 16 && DCP_COMBINE_BULK) {
        const int rb = p.vec_per_row * 16;
        if (p.N <= 8 && (rb == 512 || rb == 1024)) {
            const void* k;
            size_t smem;
            if (rb == 512) {
                k = (const void*)combine_bulk_kernel<T, 8, 1, SAN>;
                smem = bulk_smem_bytes<8, 1>();
            } else {
                k = (const void*)combine_bulk_kernel<T, 8, 2, SAN>;
                smem = bulk_smem_bytes<8, 2>();
            }
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            return launch_pdl(k, dim3(device_sm_count()), dim3(kThreads), args, smem, stream);
        }
    }
#if DCP_COMBINE_FIXED
    if constexpr (VB == 4 && DCP_COMBINE_SHIFTED) {
        // 4-byte-aligned rows whose ranks share one misalignment: 16-byte chunks
        const int rb = p.vec_per_row * VB;
        if (p.N <= 8 && p.o_sn % 16 == 0 && p.out != (unsigned char*)p.o) {
            int lpr = 0;
            const void* k = p.N <= 2 ? pick_shifted<T, 2, SAN>(rb, lpr)
                          : p.N <= 4 ? pick_shifted<T, 4, SAN>(rb, lpr)
                                     : pick_shifted<T, 8, SAN>(rb, lpr);
            if (k && p.N <= lpr) {
                CombineParams q = p;
                q.lpr = lpr;
                void* qargs[] = {(void*)&q};
                const int grid = persistent_grid(k, p.rows, (kThreads / 32) * (32 / lpr), kThreads, 0);
                return launch_pdl(k, dim3(grid), dim3(kThreads), qargs, 0, stream);
            }
        }
    }
    if (p.N <= 8) {
        int lpr = 0;
        const int rb = p.vec_per_row * VB;
        const void* k = p.N <= 2 ? pick_fixed<T, VB, 2, SAN>(rb, lpr)
                      : p.N <= 4 ? pick_fixed<T, VB, 4, SAN>(rb, lpr)
                                 : pick_fixed<T, VB, 8, SAN>(rb, lpr);
        if (k && p.N <= lpr) {
            CombineParams q = p;
            q.lpr = lpr;
            void* qargs[] = {(void*)&q};
            const int grid = persistent_grid(k, p.rows, (kThreads / 32) * (32 / lpr), kThreads, 0);
            return launch_pdl(k, dim3(grid), dim3(kThreads), qargs, 0, stream);
        }
    }
#endif
    const int rows_per_warp = 32 / p.lpr;
    if constexpr (VB == 16 && DCP_COMBINE_STAGED) {
        // staged when a lane's row holds <= 16 slices (<= 96 KiB of shared memory
        // per CTA at 3 stages); longer rows keep enough bytes in flight from
        // registers alone
        const int vpl = (p.vec_per_row + p.lpr - 1) / p.lpr;
        const int nr = p.N <= 2 ? 2 : p.N <= 4 ? 4 : 8;
        if (p.N <= 8 && vpl <= 2 && nr * vpl <= 16) {
            size_t smem = 0;
            const void* k = p.N <= 2 ? pick_staged<T, 2, SAN>(vpl, smem)
                          : p.N <= 4 ? pick_staged<T, 4, SAN>(vpl, smem)
                                     : pick_staged<T, 8, SAN>(vpl, smem);
            const int threads = kStagedWarps * 32;
            const int grid = persistent_grid(k, p.rows, kStagedWarps * rows_per_warp, threads, smem);
            return launch_pdl(k, dim3(grid), dim3(threads), args, smem, stream);
        }
    }
    const void* k;
    if (p.N <= 2) k = (const void*)combine_kernel<T, VB, 2, SAN>;
    else if (p.N <= 4) k = (const void*)combine_kernel<T, VB, 4, SAN>;
    else if (p.N <= 8) k = (const void*)combine_kernel<T, VB, 8, SAN>;
    else if (p.N <= 16) k = (const void*)combine_kernel<T, VB, 16, SAN>;
    else if (p.N <= 32) k = (const void*)combine_kernel<T, VB, 32, SAN>;
    else k = (const void*)combine_kernel_any_n<T, VB>;
    const int grid = persistent_grid(k, p.rows, (kThreads / 32) * rows_per_warp, kThreads, 0);
    return launch_pdl(k, dim3(grid), dim3(kThreads), args, 0, stream);
}

template <typename T, int VB>
cudaError_t launch_combine_san(const CombineParams& p, cudaStream_t stream) {
    return p.sanitize ? launch_combine_vb<T, VB, true>(p, stream) : launch_combine_vb<T, VB, false>(p, stream);
}

template <typename T>
cudaError_t launch_combine_t(const CombineParams& p, int vb, cudaStream_t stream) {
    if (vb == 16) return launch_combine_san<T, 16>(p, stream);
    if (vb == 4) return launch_combine_san<T, 4>(p, stream);
    if constexpr (sizeof(T) == 2) {
        if (vb == 2) return launch_combine_san<T, 2>(p, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace dcp
