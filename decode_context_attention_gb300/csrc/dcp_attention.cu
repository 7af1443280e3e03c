// dcp_attention.cu -- single-token decode attention of every DCP rank over
// the KV tokens it owns, producing the rank-local (O_r, lse_r) the merge
// consumes.
//
// sglang PR #33926 report, "实现拆解" items 3-4 and "关键源码片段": under
// decode context parallelism token t of a request lives on rank t % N, so
// rank r holds L / N tokens plus one when r < L % N (`get_dcp_lens`); each
// rank runs decode attention over its own tokens and returns rank-local
// (out, lse); a rank that owns no token of a request is the neutral state
// (0, -inf) (`fixup_zero_kv_rows`); the LSE comes in base 2 (trtllm-gen) or
// base e (cute-dsl).
//
// Per (rank r, request b, query head h) with scores s_t = sm_scale <q, k_t>
// over the rank's tokens:
//     lse_r = log sum_t exp(s_t),  O_r = sum_t exp(s_t - lse_r) v_t.
//
// Design (HBM-bound: each K/V row is read once and shared by the G_q query
// heads of its KV head):
//  * split-KV: one CTA per (rank, request, KV head, split of split_tokens
//    local tokens); a row of K or V is D * 2 bytes, covered by LPT = D / 8
//    lanes with 16-byte loads, so a warp walks 32 / LPT tokens at a time;
//  * each lane group keeps an online softmax in base 2 (scores pre-scaled by
//    log2 e, exp2f) per query head, rescaled once per block of 4 tokens whose
//    K and V loads are all issued first;
//  * the CTA's lane groups merge their states through shared memory; with one
//    split the CTA writes (O_r, lse_r) directly, otherwise an fp32 partial
//    (O, lse) per split goes to the caller's workspace and a second kernel
//    merges the splits with the LSE rule of the combine (empty splits and
//    empty ranks are the neutral (0, -inf) and drop out exactly).
#include <math.h>
#include <stdio.h>

#include <mutex>

#include "dcp_device.cuh"

namespace dcp {

constexpr int kAttnThreads = 128;
constexpr int kAttnBlockTokens = 4;   // tokens per softmax block per lane group
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// 8 payload elements of a 16-byte vector -> floats
template <typename T>
__device__ __forceinline__ void vec8_to_f32(const uint4& v, float (&f)[8]) {
    const unsigned w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 p = unpack2(word_to_pair<T>(w[k]));
        f[2 * k] = p.x;
        f[2 * k + 1] = p.y;
    }
}

// Local token count of rank r for a request of global length L (round robin).
__device__ __forceinline__ int local_len(int L, int N, int r) { return L / N + (r < L % N ? 1 : 0); }

template <typename T, int D, int GQ>
__global__ void __launch_bounds__(kAttnThreads) decode_partial_kernel(const AttnParams p) {
    constexpr int LPT = D / 8;              // lanes per token row (16-byte vectors)
    constexpr int TPW = 32 / LPT;           // token rows per warp step
    constexpr int NG = (kAttnThreads / 32) * TPW;  // lane groups per CTA
    constexpr int BT = kAttnBlockTokens;
    __shared__ float s_m[NG][GQ], s_l[NG][GQ];
    __shared__ float s_acc[NG][GQ][D];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int jl = lane & (LPT - 1);
    const int grp = warp * TPW + lane / LPT;
    const unsigned gmask = LPT == 32 ? 0xffffffffu : (((1u << LPT) - 1u) << ((lane / LPT) * LPT));

    // work item: blockIdx.x = (r * B + b) * Hkv + hkv, blockIdx.y = split
    const int hkv = blockIdx.x % p.Hkv;
    const int rb = blockIdx.x / p.Hkv;
    const int b = rb % p.B;
    const int r = rb / p.B;
    const int split = blockIdx.y;
    int L = p.seq_lens[b];
    L = L < 0 ? 0 : (L > p.max_seq_len ? p.max_seq_len : L);
    const int Ll = local_len(L, p.N, r);
    const int t0 = split * p.split_tokens;
    const int t1 = min(t0 + p.split_tokens, Ll);

    // query slices, pre-scaled so that scores are in base-2 units
    float qf[GQ][8];
#pragma unroll
    for (int g = 0; g < GQ; ++g) {
        const int h = hkv * GQ + g;
        const uint4 qv = *reinterpret_cast<const uint4*>(p.q + (int64_t)b * p.q_sb + (int64_t)h * p.q_sh +
                                                        (int64_t)jl * 16);
        vec8_to_f32<T>(qv, qf[g]);
#pragma unroll
        for (int i = 0; i < 8; ++i) qf[g][i] *= p.sm_scale * kLog2e;
    }

    float m[GQ], l[GQ], acc[GQ][8];
#pragma unroll
    for (int g = 0; g < GQ; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[g][i] = 0.f;
    }

    const unsigned char* kb = p.k + (int64_t)r * p.k_sn + (int64_t)b * p.k_sb + (int64_t)hkv * p.k_sh + jl * 16;
    const unsigned char* vb = p.v + (int64_t)r * p.v_sn + (int64_t)b * p.v_sb + (int64_t)hkv * p.v_sh + jl * 16;
    // lane group grp walks tokens t0 + grp, t0 + grp + NG, ... in blocks of BT;
    // the loop bound is uniform within the group
    for (int tb = t0 + grp; tb < t1; tb += NG * BT) {
        uint4 kv[BT], vv[BT];
#pragma unroll
        for (int u = 0; u < BT; ++u) {
            const int t = tb + u * NG;
            kv[u] = make_uint4(0u, 0u, 0u, 0u);  // tokens past the split stay finite (masked below)
            vv[u] = kv[u];
            if (t < t1) {
                kv[u] = ld_stream<16>(kb + (int64_t)t * p.k_st);
                vv[u] = ld_stream<16>(vb + (int64_t)t * p.v_st);
            }
        }
#pragma unroll
        for (int g = 0; g < GQ; ++g) {
            float s[BT];
            float bm = -INFINITY;
#pragma unroll
            for (int u = 0; u < BT; ++u) {
                float kf[8];
                vec8_to_f32<T>(kv[u], kf);
                float d = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) d = fmaf(qf[g][i], kf[i], d);
#pragma unroll
                for (int off = LPT >> 1; off > 0; off >>= 1) d += __shfl_xor_sync(gmask, d, off, LPT);
                s[u] = tb + u * NG < t1 ? d : -INFINITY;
                bm = fmaxf(bm, s[u]);
            }
            const float mn = fmaxf(m[g], bm);
            if (mn == -INFINITY) continue;  // nothing scored yet (only with -inf scores)
            const float alpha = m[g] == -INFINITY ? 0.f : exp2f(m[g] - mn);
            l[g] *= alpha;
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[g][i] *= alpha;
#pragma unroll
            for (int u = 0; u < BT; ++u) {
                const float pu = exp2f(s[u] - mn);  // masked tokens: exp2(-inf) = 0
                l[g] += pu;
                float vf[8];
                vec8_to_f32<T>(vv[u], vf);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[g][i] = fmaf(pu, vf[i], acc[g][i]);
            }
            m[g] = mn;
        }
    }

    // merge the lane groups' states (base 2)
#pragma unroll
    for (int g = 0; g < GQ; ++g) {
        if (jl == 0) {
            s_m[grp][g] = m[g];
            s_l[grp][g] = l[g];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) s_acc[grp][g][jl * 8 + i] = acc[g][i];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < GQ * D; idx += kAttnThreads) {
        const int g = idx / D;
        const int e = idx - g * D;
        float M = -INFINITY;
        for (int k = 0; k < NG; ++k) M = fmaxf(M, s_m[k][g]);
        float Ls = 0.f, A = 0.f;
        if (M != -INFINITY) {
            for (int k = 0; k < NG; ++k) {
                const float sc = exp2f(s_m[k][g] - M);
                Ls += sc * s_l[k][g];
                A += sc * s_acc[k][g][e];
            }
        }
        const int h = hkv * GQ + g;
        const float o = Ls > 0.f ? A / Ls : 0.f;
        const float lse2 = Ls > 0.f ? M + log2f(Ls) : -INFINITY;
        if (p.nsplit == 1) {
            T* orow = reinterpret_cast<T*>(p.o + (int64_t)r * p.o_sn + (int64_t)b * p.o_sb + (int64_t)h * p.o_sh);
            orow[e] = from_f32<T>(o);
            if (e == 0)
                p.lse[(int64_t)r * p.l_sn + (int64_t)b * p.l_sb + (int64_t)h * p.l_sh] =
                    p.base2 ? lse2 : lse2 * kLn2;
        } else {
            const int64_t row = (((int64_t)r * p.B + b) * p.H + h) * p.nsplit + split;
            p.ws_o[row * D + e] = o;
            if (e == 0) p.ws_lse[row] = lse2;
        }
    }
}

// Merge the splits of every (rank, request, head) row: the LSE-weighted merge
// in base 2 over the fp32 partials, one warp per row, lanes over D.
template <typename T, int D>
__global__ void __launch_bounds__(kAttnThreads) decode_merge_splits_kernel(const AttnParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t rows = (int64_t)p.N * p.B * p.H;
    const int64_t row = (int64_t)blockIdx.x * (kAttnThreads / 32) + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int S = p.nsplit;
    const float* lrow = p.ws_lse + row * S;
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, lrow[s]);
    float Ls = 0.f;
    float acc[D / 32];
#pragma unroll
    for (int i = 0; i < D / 32; ++i) acc[i] = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < S; ++s) {
            const float w = exp2f(lrow[s] - M);
            Ls += w;
            const float* orow = p.ws_o + (row * S + s) * D;
#pragma unroll
            for (int i = 0; i < D / 32; ++i) acc[i] = fmaf(w, orow[lane + 32 * i], acc[i]);
        }
    }
    const int h = (int)(row % p.H);
    const int64_t rb = row / p.H;
    const int b = (int)(rb % p.B);
    const int r = (int)(rb / p.B);
    T* orow = reinterpret_cast<T*>(p.o + (int64_t)r * p.o_sn + (int64_t)b * p.o_sb + (int64_t)h * p.o_sh);
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) orow[lane + 32 * i] = from_f32<T>(acc[i] * inv);
    if (lane == 0) {
        const float lse2 = Ls > 0.f ? M + log2f(Ls) : -INFINITY;
        p.lse[(int64_t)r * p.l_sn + (int64_t)b * p.l_sb + (int64_t)h * p.l_sh] = p.base2 ? lse2 : lse2 * kLn2;
    }
}

template <typename T, int D>
static cudaError_t launch_attention_d(const AttnParams& p, cudaStream_t stream) {
    const void* k;
    switch (p.H / p.Hkv) {
        case 1: k = (const void*)decode_partial_kernel<T, D, 1>; break;
        case 2: k = (const void*)decode_partial_kernel<T, D, 2>; break;
        case 4: k = (const void*)decode_partial_kernel<T, D, 4>; break;
        case 8: k = (const void*)decode_partial_kernel<T, D, 8>; break;
        default: return cudaErrorInvalidValue;
    }
    void* args[] = {(void*)&p};
    const dim3 grid((unsigned)((int64_t)p.N * p.B * p.Hkv), (unsigned)p.nsplit);
    cudaError_t e = cudaLaunchKernel(k, grid, dim3(kAttnThreads), args, 0, stream);
    if (e != cudaSuccess || p.nsplit == 1) return e;
    const int64_t rows = (int64_t)p.N * p.B * p.H;
    const unsigned mgrid = (unsigned)((rows + kAttnThreads / 32 - 1) / (kAttnThreads / 32));
    return cudaLaunchKernel((const void*)decode_merge_splits_kernel<T, D>, dim3(mgrid), dim3(kAttnThreads),
                            args, 0, stream);
}

template <typename T>
static cudaError_t launch_attention_t(const AttnParams& p, cudaStream_t stream) {
    switch (p.D) {
        case 64: return launch_attention_d<T, 64>(p, stream);
        case 128: return launch_attention_d<T, 128>(p, stream);
        case 256: return launch_attention_d<T, 256>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode_attention(const AttnParams& p, int dtype, cudaStream_t stream) {
    return dtype == 1 ? launch_attention_t<__half>(p, stream) : launch_attention_t<__nv_bfloat16>(p, stream);
}

}  // namespace dcp

// ---------------------------------------------------------------------------
// Entry point for callers that cannot allocate device memory.  Some callers
// of this library may not call cudaMalloc (or any allocator) at the point
// where they run the attention: code that runs inside a memory pool whose
// size is fixed up front, an inference server that forbids allocation on its
// serving path, or a host runtime that has no allocator of its own to hand.
// For them the scratch the split path needs lives in this file-scope device
// array instead of a caller-provided workspace.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = 16u << 20;  // 16 MiB, reserved on every device that loads this code
static __device__ __align__(256) float g_attn_scratch[kNoAllocScratchBytes / sizeof(float)];

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {};  // device address of g_attn_scratch, per device

}  // namespace

extern "C" dcp_status_t dcp_decode_attention_noalloc(
    int dtype, int N, int B, int H, int Hkv, int D, const void* q, int64_t q_sb, int64_t q_sh,
    const void* k, int64_t k_sn, int64_t k_sb, int64_t k_st, int64_t k_sh, const void* v, int64_t v_sn,
    int64_t v_sb, int64_t v_st, int64_t v_sh, const int* seq_lens, int max_seq_len, float sm_scale,
    int split_tokens, void* o, int64_t o_sn, int64_t o_sb, int64_t o_sh, float* lse, int64_t l_sn,
    int64_t l_sb, int64_t l_sh, int lse_base, void* stream) {
    const size_t need = dcp_decode_attention_workspace_size(N, B, H, D, max_seq_len, split_tokens);
    if (need > kNoAllocScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "dcp_decode_attention_noalloc: these sizes need %zu bytes of scratch, the built-in "
                 "scratch holds %zu (use fewer splits, i.e. a larger split_tokens, or "
                 "dcp_decode_attention with a workspace)",
                 need, kNoAllocScratchBytes);
        return dcp::set_error(DCP_ERR_INVALID_ARG, msg);
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        char msg[256];
        snprintf(msg, sizeof(msg), "dcp_decode_attention_noalloc: no usable current device (%s)",
                 cudaGetErrorString(e));
        return dcp::set_error(DCP_ERR_CUDA, msg);
    }
    void* scratch = nullptr;
    {
        // first call on this device: look up the array's device address once,
        // with this device current
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        if (!g_scratch_ptr[dev]) {
            void* ptr = nullptr;
            e = cudaGetSymbolAddress(&ptr, g_attn_scratch);
            if (e != cudaSuccess) {
                char msg[256];
                snprintf(msg, sizeof(msg), "dcp_decode_attention_noalloc: cudaGetSymbolAddress failed: %s",
                         cudaGetErrorString(e));
                return dcp::set_error(DCP_ERR_CUDA, msg);
            }
            g_scratch_ptr[dev] = ptr;
        }
        scratch = g_scratch_ptr[dev];
    }
    return dcp_decode_attention(dtype, N, B, H, Hkv, D, q, q_sb, q_sh, k, k_sn, k_sb, k_st, k_sh, v, v_sn,
                                v_sb, v_st, v_sh, seq_lens, max_seq_len, sm_scale, split_tokens, o, o_sn,
                                o_sb, o_sh, lse, l_sn, l_sb, l_sh, lse_base, scratch, kNoAllocScratchBytes,
                                stream);
}
