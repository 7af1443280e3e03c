// dcp_combine.cuh -- the LSE-weighted merge kernel (templated over the payload
// type, the vector width and the maximum rank count), included by one
// translation unit per payload type.
//
// What it computes, per output row (g, b, h), over ranks r < N (sglang PR
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
//  * each lane streams its slice of every rank's row with 16-byte loads when
//    every row start is 16-byte aligned (4- or 2-byte otherwise), issuing all
//    ranks' loads of a chunk before any arithmetic so 8-16 KiB per warp are in
//    flight;
//  * persistent grid: SM count x resident CTAs, grid-stride over rows.
#pragma once

#include <math.h>

#include "dcp_device.cuh"

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

// Weights of ranks r < NRMAX (entries r >= N are 0) and the global LSE, for
// the row whose rank-0 LSE is at `lrow` (rank stride `l_sn` words).
template <int NRMAX>
__device__ __forceinline__ void row_weights(const float* lrow, int64_t l_sn, int N,
                                            const LaneGroup& lg, int lpr, bool b2,
                                            float (&w)[NRMAX], float& Gl) {
    if (N <= lpr) {
        // warp-shuffle logsumexp: lane r holds lse_r
        const float l = lg.jl < N ? __ldg(lrow + (int64_t)lg.jl * l_sn) : -INFINITY;
        unsigned cls = isnan(l) ? kHasNaN : (l == INFINITY ? kHasPosInf : 0u);
        float m = cls ? -INFINITY : l;
        for (int off = lpr >> 1; off > 0; off >>= 1) {
            m = fmaxf(m, __shfl_xor_sync(lg.mask, m, off, lpr));
            cls |= __shfl_xor_sync(lg.mask, cls, off, lpr);
        }
        float wl = 0.f;
        float s = 0.f;
        if (cls == 0u && m != -INFINITY) {
            const float el = lse_exp(l - m, b2);  // lanes with -inf (or no rank) hold 0
            s = el;
            for (int off = lpr >> 1; off > 0; off >>= 1) s += __shfl_xor_sync(lg.mask, s, off, lpr);
            wl = el / s;  // = base^(l - Gl) without the rounding of Gl
        }
        Gl = global_lse_from(cls, m, s, b2);
#pragma unroll
        for (int r = 0; r < NRMAX; ++r) w[r] = __shfl_sync(lg.mask, wl, r & (lpr - 1), lpr);
#pragma unroll
        for (int r = 0; r < NRMAX; ++r)
            if (r >= N || r >= lpr) w[r] = 0.f;
    } else {
        // more ranks than lanes in the group: every lane reduces serially
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
}

// Ranks per load batch: all loads of a batch are issued before its arithmetic.
template <int NRMAX>
struct RankChunk { static constexpr int value = NRMAX < 8 ? NRMAX : 8; };

template <typename T, int VB, int NRMAX>
__global__ void __launch_bounds__(kThreads, 2) combine_kernel(const CombineParams p) {
    constexpr int EPV = VB / (int)sizeof(T);
    constexpr int RC = RankChunk<NRMAX>::value;
    // vectors per lane per batch: at most ~64 registers of loaded payload and
    // 32 fp32 accumulators, so two CTAs fit on an SM without spilling
    constexpr int KU_LD = 64 / (RC * (VB / 4 > 0 ? VB / 4 : 1));
    constexpr int KU_ACC = 32 / EPV;
    constexpr int KU0 = KU_LD < KU_ACC ? KU_LD : KU_ACC;
    constexpr int KU = KU0 < 1 ? 1 : (KU0 > 8 ? 8 : KU0);
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

        float w[NRMAX];
        float Gl;
        row_weights<NRMAX>(p.lse + g * p.l_sg + b * p.l_sb + h * p.l_sh, p.l_sn, N, lg, p.lpr, b2,
                           w, Gl);

        const unsigned char* orow = p.o + g * p.o_sg + b * p.o_sb + h * p.o_sh;
        unsigned char* urow = p.out + g * p.u_sg + b * p.u_sb + h * p.u_sh;
        for (int v0 = lg.jl; v0 < nv; v0 += p.lpr * KU) {
            float acc[KU][EPV];
#pragma unroll
            for (int k = 0; k < KU; ++k)
#pragma unroll
                for (int i = 0; i < EPV; ++i) acc[k][i] = 0.f;
#pragma unroll
            for (int r0 = 0; r0 < NRMAX; r0 += RC) {
                V x[KU][RC];
#pragma unroll
                for (int k = 0; k < KU; ++k) {
                    const int v = v0 + k * p.lpr;
#pragma unroll
                    for (int j = 0; j < RC; ++j)
                        if (r0 + j < N && v < nv)
                            x[k][j] = ld_stream<VB>(orow + (int64_t)(r0 + j) * p.o_sn + (int64_t)v * VB);
                }
#pragma unroll
                for (int k = 0; k < KU; ++k) {
#pragma unroll
                    for (int j = 0; j < RC; ++j) {
                        if (r0 + j < N) {
                            float f[EPV];
                            unpack_vec<T, VB>(x[k][j], f);
#pragma unroll
                            for (int i = 0; i < EPV; ++i) {
                                const float ov = (p.sanitize && !isfinite(f[i])) ? 0.f : f[i];
                                acc[k][i] = fmaf(w[r0 + j], ov, acc[k][i]);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < KU; ++k) {
                const int v = v0 + k * p.lpr;
                if (v < nv) st_vec<VB>(urow + (int64_t)v * VB, pack_vec<T, VB>(acc[k]));
            }
        }
        if (p.return_lse && lg.jl == 0) p.out_lse[g * p.ul_sg + b * p.ul_sb + h * p.ul_sh] = Gl;
    }
}

// Any N: weights are recomputed per batch of 8 ranks from a serial reduction.
template <typename T, int VB>
__global__ void __launch_bounds__(kThreads, 2) combine_kernel_any_n(const CombineParams p) {
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
                        wr[j] = finite_g
                                    ? lse_exp(__ldg(lrow + (int64_t)(r0 + j) * p.l_sn) - m, b2) * inv_s
                                    : 0.f;
                    }
                }
#pragma unroll
                for (int j = 0; j < RC; ++j) {
                    if (r0 + j < N) {
                        float f[EPV];
                        unpack_vec<T, VB>(x[j], f);
#pragma unroll
                        for (int i = 0; i < EPV; ++i) {
                            const float ov = (p.sanitize && !isfinite(f[i])) ? 0.f : f[i];
                            acc[i] = fmaf(wr[j], ov, acc[i]);
                        }
                    }
                }
            }
            st_vec<VB>(urow + (int64_t)v * VB, pack_vec<T, VB>(acc));
        }
        if (p.return_lse && lg.jl == 0) p.out_lse[g * p.ul_sg + b * p.ul_sb + h * p.ul_sh] = Gl;
    }
}

template <typename T, int VB>
cudaError_t launch_combine_vb(const CombineParams& p, cudaStream_t stream) {
    const void* k;
    if (p.N <= 2) k = (const void*)combine_kernel<T, VB, 2>;
    else if (p.N <= 4) k = (const void*)combine_kernel<T, VB, 4>;
    else if (p.N <= 8) k = (const void*)combine_kernel<T, VB, 8>;
    else if (p.N <= 16) k = (const void*)combine_kernel<T, VB, 16>;
    else if (p.N <= 32) k = (const void*)combine_kernel<T, VB, 32>;
    else k = (const void*)combine_kernel_any_n<T, VB>;
    const int rows_per_cta = (kThreads / 32) * (32 / p.lpr);
    const int grid = persistent_grid(k, p.rows, rows_per_cta);
    void* args[] = {(void*)&p};
    cudaLaunchKernel(k, dim3(grid), dim3(kThreads), args, 0, stream);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_combine_t(const CombineParams& p, int vb, cudaStream_t stream) {
    if (vb == 16) return launch_combine_vb<T, 16>(p, stream);
    if (vb == 4) return launch_combine_vb<T, 4>(p, stream);
    if constexpr (sizeof(T) == 2) {
        if (vb == 2) return launch_combine_vb<T, 2>(p, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace dcp
