// dcp_device.cuh -- device helpers shared by the DCP kernels: vector loads and
// stores of 2/4/16 bytes, payload <-> fp32 conversion, lane grouping, and a
// grid sized from the SM count and the kernel's occupancy.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
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

// VB bytes of payload -> VB / sizeof(T) floats, and back (round to nearest even).
template <typename T, int VB>
__device__ __forceinline__ void unpack_vec(const typename VecT<VB>::type& v,
                                           float (&f)[VB / sizeof(T)]) {
    T e[VB / sizeof(T)];
    memcpy(e, &v, VB);
#pragma unroll
    for (int i = 0; i < VB / (int)sizeof(T); ++i) f[i] = to_f32(e[i]);
}

template <typename T, int VB>
__device__ __forceinline__ typename VecT<VB>::type pack_vec(const float (&f)[VB / sizeof(T)]) {
    T e[VB / sizeof(T)];
#pragma unroll
    for (int i = 0; i < VB / (int)sizeof(T); ++i) e[i] = from_f32<T>(f[i]);
    typename VecT<VB>::type v;
    memcpy(&v, e, VB);
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

// Grid for a grid-stride kernel: enough CTAs for every row, capped at the
// number that are resident at once (SM count x CTAs per SM), so large inputs
// run as one full wave of persistent CTAs.
inline int persistent_grid(const void* kernel, int64_t rows, int rows_per_cta) {
    const int64_t cap = (int64_t)device_sm_count() * ctas_per_sm(kernel);
    int64_t need = (rows + rows_per_cta - 1) / rows_per_cta;
    if (need < 1) need = 1;
    return (int)(need < cap ? need : cap);
}

}  // namespace dcp
