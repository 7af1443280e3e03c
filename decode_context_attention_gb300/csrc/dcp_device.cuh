// dcp_device.cuh -- device helpers shared by the DCP kernels: vector loads and
// stores of 2/4/16 bytes, payload <-> fp32 conversion, lane grouping, and a
// grid sized from the SM count and the kernel's occupancy.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dcp_internal.h"

namespace dcp {

template <int VB>
struct VecT;
template <>
struct VecT<16> { using type = uint4; };
template <>
struct VecT<4> { using type = unsigned int; };
template <>
struct VecT<2> { using type = unsigned short; };

// Streaming (evict-first) loads: every payload byte is read exactly once.
// ld.global.cs is coherent, so it is also safe on the in-place path where a
// thread later overwrites what it read.
template <int VB>
__device__ __forceinline__ typename VecT<VB>::type ld_stream(const unsigned char* p) {
    return __ldcs(reinterpret_cast<const typename VecT<VB>::type*>(p));
}

template <int VB>
__device__ __forceinline__ void st_vec(unsigned char* p, typename VecT<VB>::type v) {
    *reinterpret_cast<typename VecT<VB>::type*>(p) = v;
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// ---- paired fp32 arithmetic (sm_100+ fma.rn.f32x2: two IEEE fp32 FMAs,
// each rounded to nearest, in one instruction) ---------------------------------
__device__ __forceinline__ float2 ffma2(float w, float2 x, float2 acc) {
    float2 d;
    asm("{\n\t.reg .b64 a, b, c, d;\n\t"
        "mov.b64 a, {%2, %2};\n\t"
        "mov.b64 b, {%3, %4};\n\t"
        "mov.b64 c, {%5, %6};\n\t"
        "fma.rn.f32x2 d, a, b, c;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(w), "f"(x.x), "f"(x.y), "f"(acc.x), "f"(acc.y));
    return d;
}

__device__ __forceinline__ unsigned f32_to_pair(float2 f, __nv_bfloat16);
__device__ __forceinline__ unsigned f32_to_pair(float2 f, __half);

// fp32 pairs held in one 64-bit register (low half = first element), so the
// paired FMA needs no repacking between iterations.
__device__ __forceinline__ unsigned long long pack2(unsigned lo, unsigned hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ unsigned long long pack2f(float lo, float hi) {
    return pack2(__float_as_uint(lo), __float_as_uint(hi));
}
__device__ __forceinline__ float2 unpack2(unsigned long long r) {
    float2 f;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(r));
    return f;
}
// acc += w2 * x2, element-wise on two fp32 lanes (each an IEEE FMA, round to nearest)
__device__ __forceinline__ void ffma2_acc(unsigned long long& acc, unsigned long long w2,
                                          unsigned long long x2) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(w2), "l"(x2));
}

// One 32-bit word of payload -> its fp32 pair.  bf16 widens by placing the
// 16 bits in the upper half of an fp32; fp16 goes through the half2 convert.
template <typename T>
__device__ __forceinline__ unsigned long long word_to_pair(unsigned w);
template <>
__device__ __forceinline__ unsigned long long word_to_pair<__nv_bfloat16>(unsigned w) {
    return pack2(w << 16, w & 0xffff0000u);
}
template <>
__device__ __forceinline__ unsigned long long word_to_pair<__half>(unsigned w) {
    __half2 h;
    memcpy(&h, &w, 4);
    const float2 f = __half22float2(h);
    return pack2f(f.x, f.y);
}
__device__ __forceinline__ unsigned long long sanitize_pair(unsigned long long x2) {
    float2 f = unpack2(x2);
    f.x = isfinite(f.x) ? f.x : 0.f;
    f.y = isfinite(f.y) ? f.y : 0.f;
    return pack2f(f.x, f.y);
}

// Two fp8 e4m3 elements (16 bits, low byte first) <-> an fp32 pair.  Widening
// goes through the hardware e4m3x2 -> f16x2 convert (exact); narrowing
// rounds to nearest and saturates to the largest finite e4m3 (448).
__device__ __forceinline__ unsigned long long fp8x2_to_pair(unsigned v) {
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(v & 0xffffu), __NV_E4M3);
    __half2 h;
    memcpy(&h, &hr, 4);
    const float2 f = __half22float2(h);
    return pack2f(f.x, f.y);
}
__device__ __forceinline__ unsigned pair_to_fp8x2(float2 f) {
    return (unsigned)__nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
}

// acc[0..NP) += w2 * (payload vector x) for a VB-byte vector of T holding
// 2*NP elements (VB = 16, or VB = 4 with a 16-bit or 8-bit T).
template <typename T, int VB, bool SAN>
__device__ __forceinline__ void fma_pairs(unsigned long long (&acc)[VB / sizeof(T) / 2],
                                          const typename VecT<VB>::type& x, unsigned long long w2) {
    constexpr int NP = VB / (int)sizeof(T) / 2;
    unsigned wd[VB / 4];
    memcpy(wd, &x, VB);
#pragma unroll
    for (int k = 0; k < NP; ++k) {
        unsigned long long x2;
        if constexpr (sizeof(T) == 4) x2 = pack2(wd[2 * k], wd[2 * k + 1]);
        else if constexpr (sizeof(T) == 1) x2 = fp8x2_to_pair(wd[k >> 1] >> (16 * (k & 1)));
        else x2 = word_to_pair<T>(wd[k]);
        if (SAN) x2 = sanitize_pair(x2);
        ffma2_acc(acc[k], w2, x2);
    }
}

// Round NP fp32 pairs into one payload vector (round to nearest even).
template <typename T, int VB>
__device__ __forceinline__ typename VecT<VB>::type round_pairs(const unsigned long long (&acc)[VB / sizeof(T) / 2]) {
    constexpr int NP = VB / (int)sizeof(T) / 2;
    typename VecT<VB>::type v;
    if constexpr (sizeof(T) == 4) {
        memcpy(&v, acc, VB);
    } else if constexpr (sizeof(T) == 1) {
        unsigned wd[VB / 4];
#pragma unroll
        for (int k = 0; k < VB / 4; ++k)
            wd[k] = pair_to_fp8x2(unpack2(acc[2 * k])) | (pair_to_fp8x2(unpack2(acc[2 * k + 1])) << 16);
        memcpy(&v, wd, VB);
    } else {
        unsigned wd[VB / 4];
#pragma unroll
        for (int k = 0; k < NP; ++k) wd[k] = f32_to_pair(unpack2(acc[k]), T());
        memcpy(&v, wd, VB);
    }
    return v;
}

// Two packed 16-bit payload elements (low half first) -> two floats.
__device__ __forceinline__ float2 pair_to_f32(unsigned w, __nv_bfloat16) {
    // a bf16 is the upper half of the fp32 with the same bits
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ float2 pair_to_f32(unsigned w, __half) {
    __half2 h;
    memcpy(&h, &w, 4);
    return __half22float2(h);
}
// Two floats -> two packed 16-bit payload elements (round to nearest even).
__device__ __forceinline__ unsigned f32_to_pair(float2 f, __nv_bfloat16) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(f.x, f.y);
    unsigned w;
    memcpy(&w, &h, 4);
    return w;
}
__device__ __forceinline__ unsigned f32_to_pair(float2 f, __half) {
    const __half2 h = __floats2half2_rn(f.x, f.y);
    unsigned w;
    memcpy(&w, &h, 4);
    return w;
}

__device__ __forceinline__ float zero_if_not_finite(float x) { return isfinite(x) ? x : 0.f; }

// acc[0..EPV) += w * (payload vector x), EPV = VB / sizeof(T) elements; with
// SAN, NaN/+-inf payload elements count as 0.
template <typename T, int VB, bool SAN>
__device__ __forceinline__ void fma_vec(float (&acc)[VB / sizeof(T)], const typename VecT<VB>::type& x,
                                        float w) {
    constexpr int EPV = VB / (int)sizeof(T);
    if constexpr (sizeof(T) == 4) {
        float f[EPV];
        memcpy(f, &x, VB);
#pragma unroll
        for (int i = 0; i + 1 < EPV; i += 2) {
            float2 xf = make_float2(f[i], f[i + 1]);
            if (SAN) xf = make_float2(zero_if_not_finite(xf.x), zero_if_not_finite(xf.y));
            const float2 r = ffma2(w, xf, make_float2(acc[i], acc[i + 1]));
            acc[i] = r.x;
            acc[i + 1] = r.y;
        }
        if constexpr (EPV % 2) acc[EPV - 1] = fmaf(w, SAN ? zero_if_not_finite(f[EPV - 1]) : f[EPV - 1], acc[EPV - 1]);
    } else if constexpr (sizeof(T) == 1) {
        unsigned wd[VB / 4];
        memcpy(wd, &x, VB);
#pragma unroll
        for (int k = 0; k < EPV / 2; ++k) {
            float2 xf = unpack2(fp8x2_to_pair(wd[k >> 1] >> (16 * (k & 1))));
            if (SAN) xf = make_float2(zero_if_not_finite(xf.x), zero_if_not_finite(xf.y));
            const float2 r = ffma2(w, xf, make_float2(acc[2 * k], acc[2 * k + 1]));
            acc[2 * k] = r.x;
            acc[2 * k + 1] = r.y;
        }
    } else if constexpr (VB >= 4) {
        unsigned wd[VB / 4];
        memcpy(wd, &x, VB);
#pragma unroll
        for (int k = 0; k < VB / 4; ++k) {
            float2 xf = pair_to_f32(wd[k], T());
            if (SAN) xf = make_float2(zero_if_not_finite(xf.x), zero_if_not_finite(xf.y));
            const float2 r = ffma2(w, xf, make_float2(acc[2 * k], acc[2 * k + 1]));
            acc[2 * k] = r.x;
            acc[2 * k + 1] = r.y;
        }
    } else {
        T e;
        memcpy(&e, &x, 2);
        const float f = to_f32(e);
        acc[0] = fmaf(w, SAN ? zero_if_not_finite(f) : f, acc[0]);
    }
}

// Round EPV accumulators into one payload vector.
template <typename T, int VB>
__device__ __forceinline__ typename VecT<VB>::type round_vec(const float (&acc)[VB / sizeof(T)]) {
    typename VecT<VB>::type v;
    if constexpr (sizeof(T) == 4) {
        memcpy(&v, acc, VB);
    } else if constexpr (sizeof(T) == 1) {
        unsigned wd[VB / 4];
#pragma unroll
        for (int k = 0; k < VB / 4; ++k)
            wd[k] = pair_to_fp8x2(make_float2(acc[4 * k], acc[4 * k + 1])) |
                    (pair_to_fp8x2(make_float2(acc[4 * k + 2], acc[4 * k + 3])) << 16);
        memcpy(&v, wd, VB);
    } else if constexpr (VB >= 4) {
        unsigned wd[VB / 4];
#pragma unroll
        for (int k = 0; k < VB / 4; ++k) wd[k] = f32_to_pair(make_float2(acc[2 * k], acc[2 * k + 1]), T());
        memcpy(&v, wd, VB);
    } else {
        const T e = from_f32<T>(acc[0]);
        memcpy(&v, &e, 2);
    }
    return v;
}

// Lanes of a warp are split into groups of `lpr` consecutive lanes (a power of
// two <= 32); each group owns one row at a time.
struct LaneGroup {
    int jl;          // lane index inside the group
    int sub;         // group index inside the warp
    unsigned mask;   // the group's lanes, for *_sync shuffles
    int64_t first;   // first row of this group
    int64_t step;    // row stride of the grid-stride loop
};

__device__ __forceinline__ LaneGroup lane_group(int lpr) {
    LaneGroup lg;
    const int lane = threadIdx.x & 31;
    const int rpw = 32 / lpr;
    lg.jl = lane & (lpr - 1);
    lg.sub = lane / lpr;
    lg.mask = lpr == 32 ? 0xffffffffu : (((1u << lpr) - 1u) << (lg.sub * lpr));
    const int64_t warps_per_cta = blockDim.x / 32;
    const int64_t warp = (int64_t)blockIdx.x * warps_per_cta + (threadIdx.x / 32);
    lg.first = warp * rpw + lg.sub;
    lg.step = (int64_t)gridDim.x * warps_per_cta * rpw;
    return lg;
}

// (g, b, h) of row index r = (g * B + b) * H + h, advanced by a fixed number
// of rows without any division (the step is decomposed once per thread).
struct RowCursor {
    int64_t g;
    int b, h;
    __device__ __forceinline__ void set(int64_t r, int B, int H) {
        h = (int)(r % H);
        const int64_t t = r / H;
        b = (int)(t % B);
        g = t / B;
    }
    // add (dg, db, dh) with carries; requires db < B and dh < H
    __device__ __forceinline__ void add(int64_t dg, int db, int dh, int B, int H) {
        h += dh;
        int c = h >= H;
        if (c) h -= H;
        b += db + c;
        c = b >= B;
        if (c) b -= B;
        g += dg + c;
    }
    __device__ __forceinline__ void next(int B, int H) { add(0, 0, 1, B, H); }
};

struct RowStep {
    int64_t dg;
    int db, dh;
    __device__ __forceinline__ void set(int64_t step, int B, int H) {
        dh = (int)(step % H);
        const int64_t t = step / H;
        db = (int)(t % B);
        dg = t / B;
    }
};

// cp.async (LDGSTS): 16-byte global -> shared copies that bypass L1 and hold
// no registers while in flight; completion is tracked per thread in groups.
__device__ __forceinline__ void cp_async_16(void* smem, const void* gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Programmatic dependent launch (built with -DDCP_PDL=1).  Every kernel of
// this library is then launched with programmatic stream serialisation, so
// it may become resident while the previous kernel of its stream is still
// finishing (its launch and set-up overlap that kernel's tail).  It calls
// pdl_wait() before its first global-memory access: the wait returns once
// the previous grid has completed and its writes are visible, whatever that
// kernel was (without a previous kernel it returns at once).  pdl_trigger()
// lets the next kernel of the stream start launching; a kernel calls it when
// its CTA's work is done (that kernel still waits for this whole grid).
// Off by default: measured on GB300 it made the interleaved unpack+combine
// 13% slower (28.8 -> 32.5 us), the fp8 one 14% slower (20.9 -> 23.9 us)
// and the pack + combine step replayed as a CUDA graph no faster (60.9 ->
// 61.9 us); only the all-rank pack gained (40.8 -> 40.0 us).
#ifndef DCP_PDL
#define DCP_PDL 0
#endif
__device__ __forceinline__ void pdl_wait() {
#if DCP_PDL
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}
__device__ __forceinline__ void pdl_trigger() {
#if DCP_PDL
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

// cudaLaunchKernel with programmatic stream serialisation (see pdl_wait).
inline cudaError_t launch_pdl(const void* kernel, dim3 grid, dim3 block, void** args, size_t smem,
                              cudaStream_t stream) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = DCP_PDL ? 1 : 0;
    return cudaLaunchKernelExC(&cfg, kernel, args);
}

// Grid for a grid-stride kernel.  persistent: enough CTAs for every row,
// capped at the number resident at once (SM count x CTAs per SM), so large
// inputs run as one full wave of persistent CTAs.  Otherwise one work item per
// lane group: CTAs retire and are replaced at staggered times, which measured
// faster for the pure-copy pack.
inline int grid_for(const void* kernel, int64_t items, int items_per_cta, int threads, size_t smem,
                    bool persistent) {
    int64_t need = (items + items_per_cta - 1) / items_per_cta;
    if (need < 1) need = 1;
    if (need > 0x7fffffffll) need = 0x7fffffffll;
    if (!persistent) return (int)need;
    const int64_t cap = (int64_t)device_sm_count() * ctas_per_sm(kernel, threads, smem);
    return (int)(need < cap ? need : cap);
}
inline int persistent_grid(const void* kernel, int64_t rows, int rows_per_cta, int threads,
                           size_t smem) {
    return grid_for(kernel, rows, rows_per_cta, threads, smem, true);
}

}  // namespace dcp
