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
//  * grouped-query heads (2..16 per KV head) instead run the score and
//    output products on the tensor cores, since their multiply-adds per byte
//    outrun the CUDA cores: at D = 128 (split_tokens a multiple of 128,
//    pages of 8 tokens or more) the tcgen05 kernel of dcp_attention_tc.cu,
//    otherwise decode_partial_mma_kernel below (warp-level mma.sync);
//  * the CTA's lane groups merge their states through shared memory; with one
//    split the CTA writes (O_r, lse_r) directly, otherwise an fp32 partial
//    (O, lse) per split goes to the caller's workspace and a second kernel
//    merges the splits with the LSE rule of the combine (empty splits and
//    empty ranks are the neutral (0, -inf) and drop out exactly).
#include <math.h>
#include <stdio.h>

#include <type_traits>

#include "dcp_device.cuh"

namespace dcp {

#ifndef DCP_ATTN_MMA
#define DCP_ATTN_MMA 1
#endif
#ifndef DCP_ATTN_PREFETCH
#define DCP_ATTN_PREFETCH 1
#endif

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

// Work item (rank, request, KV head) and split of a CTA in a 1-D grid with the
// split fastest: the splits of one item are neighbours in launch order, so a
// long request's splits start together instead of every second split
// trailing at the end of the launch (GQ = 8: 186.9 -> 181.4 us).
__device__ __forceinline__ int attn_item(int nsplit) { return (int)(blockIdx.x / (unsigned)nsplit); }
__device__ __forceinline__ int attn_split(int nsplit) { return (int)(blockIdx.x % (unsigned)nsplit); }

// Where local token t of request b on rank r lives: (page, slot) with the row
// at page * sp + slot * st.  Contiguous caches are one page of every token;
// a paged cache reads the rank's page table (sglang PR #33926 report,
// "实现拆解" item 1, `_fill_dcp_block_kv_indices`: the table covers the
// rank's round-robin slice).  An index outside the pool gives page -1 and the
// row is read as zeros, never from outside the pool.
struct KvPlace {
    int64_t page;
    int slot;
};
template <bool PAGED>
__device__ __forceinline__ KvPlace kv_place(const AttnParams& p, int r, int b, int t) {
    if constexpr (!PAGED) return {0, t};
    const int pg = __ldg(p.bt + (int64_t)r * p.bt_sn + (int64_t)b * p.bt_sb + (t >> p.page_shift));
    if ((unsigned)pg >= (unsigned)p.num_pages) return {-1, 0};
    return {(int64_t)pg, t & ((1 << p.page_shift) - 1)};
}

// Local token count of rank r for a request of global length L (round robin).
__device__ __forceinline__ int local_len(int L, int N, int r) { return L / N + (r < L % N ? 1 : 0); }

// The CTA's NG partial softmax states per query head (base 2: running max m,
// sum l, unnormalised accumulator acc) merged into (O, lse): written as the
// rank's result with one split, or as the split's fp32 partial otherwise.
template <typename T, int D, int GQ, int NG>
__device__ __forceinline__ void write_cta_result(const AttnParams& p, int r, int b, int hkv, int split,
                                                 const float (*s_m)[GQ], const float (*s_l)[GQ],
                                                 const float (*s_acc)[GQ][D]) {
    for (int idx = threadIdx.x; idx < GQ * D; idx += blockDim.x) {
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

template <typename T, int D, int GQ, bool PAGED>
__global__ void __launch_bounds__(kAttnThreads) decode_partial_kernel(const AttnParams p) {
    pdl_wait();
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

    // work item (r * B + b) * Hkv + hkv and split, from the 1-D grid
    const int item = attn_item(p.nsplit);
    const int hkv = item % p.Hkv;
    const int rb = item / p.Hkv;
    const int b = rb % p.B;
    const int r = rb / p.B;
    const int split = attn_split(p.nsplit);
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
            if constexpr (PAGED) {
                const KvPlace at = t < t1 ? kv_place<true>(p, r, b, t) : KvPlace{-1, 0};
                if (at.page >= 0) {
                    kv[u] = ld_stream<16>(kb + at.page * p.k_sp + (int64_t)at.slot * p.k_st);
                    vv[u] = ld_stream<16>(vb + at.page * p.v_sp + (int64_t)at.slot * p.v_st);
                }
            } else if (t < t1) {
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
    write_cta_result<T, D, GQ, NG>(p, r, b, hkv, split, s_m, s_l, s_acc);
    pdl_trigger();
}

// ---------------------------------------------------------------------------
// Grouped-query heads on the tensor cores.  With G_q query heads per KV head
// every K/V byte feeds 2 G_q multiply-adds (scores and output), more than the
// CUDA cores sustain at HBM speed beyond G_q = 2, so for G_q in {2, 4, 8, 16}
// the products run as warp-level mma.sync (bf16 or f16 operands, fp32
// accumulation).  One warp takes blocks of 16 tokens (8 at D = 256, where the
// registers hold no more) of its CTA's split, per 8-token half:
//   S   [16 x 8 tokens]  = Q [16 rows: the G_q heads, zero past G_q] . K^T
//   O^T [D x 8 heads]   += V^T [D x tokens] . P^T [tokens x 8 heads]
// (the output product once per block of 8 heads: twice for G_q = 16).
// K and V rows arrive by 16-byte loads; the contraction over D does not
// depend on the order of its terms, so the d positions each lane loads are
// simply the ones it feeds to the fragments (Q is read in the same order),
// and V's 8x8 tiles are transposed in registers (movmatrix) so tokens become
// the contraction index.  P goes in as two 16-bit terms (hi + lo), keeping
// ~16 significant bits of every probability instead of 8.  The online
// softmax is in base 2, per head, over the 4 lanes that hold that head's
// scores; the warps' states meet in shared memory as in the kernel above.
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ void mma_16816(float (&d)[4], const unsigned (&a)[4], unsigned b0, unsigned b1) {
    if constexpr (std::is_same<T, __half>::value)
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <typename T>
__device__ __forceinline__ void mma_1688(float (&d)[4], const unsigned (&a)[2], unsigned b0) {
    if constexpr (std::is_same<T, __half>::value)
        asm("mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
            "{%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(b0));
    else
        asm("mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
            "{%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(b0));
}

// 8x8 tile of 16-bit values, lane t holding row t/4, columns 2(t%4)..+1 ->
// the transposed tile in the same distribution.
__device__ __forceinline__ unsigned tile_transpose(unsigned x) {
    unsigned y;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}

// Two floats rounded to a T pair (the first in the low half).
template <typename T>
__device__ __forceinline__ unsigned round_pair(float lo, float hi) {
    unsigned u;
    if constexpr (std::is_same<T, __half>::value) {
        const __half2 h = __floats2half2_rn(lo, hi);
        memcpy(&u, &h, 4);
    } else {
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        memcpy(&u, &h, 4);
    }
    return u;
}

__device__ __forceinline__ unsigned word_of(const uint4& v, int w) {
    return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}

template <typename T, int D, int GQ, bool PAGED>
__global__ void __launch_bounds__(kAttnThreads) decode_partial_mma_kernel(const AttnParams p) {
    pdl_wait();
    static_assert(D % 32 == 0 && GQ >= 1 && GQ <= 16, "fragment shapes");
    constexpr int NB = GQ > 8 ? 2 : 1;    // blocks of 8 query heads (fragment rows qr and qr + 8)
    constexpr int NI = D / 32;   // 16-byte pieces per lane per token row
    constexpr int KS = D / 16;   // k-steps of the score products
    constexpr int NM = D / 16;   // output products (16 d each) per head block
    constexpr int NW = kAttnThreads / 32;
    constexpr int HB = D <= 128 ? 2 : 1;  // 8-token halves per warp block (registers bound D = 256 to one)
    constexpr int TB = 8 * HB;            // tokens per warp block
    // second register set for the next block, where the registers allow it
    constexpr bool PF = DCP_ATTN_PREFETCH && (NB == 1 ? D <= 128 : D <= 64);
    constexpr unsigned kFull = 0xffffffffu;
    __shared__ float s_m[NW][GQ], s_l[NW][GQ];
    __shared__ float s_acc[NW][GQ][D];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int qr = lane >> 2;  // fragment row (score head / token row / output d row)
    const int qc = lane & 3;   // fragment column pair

    const int item = attn_item(p.nsplit);
    const int hkv = item % p.Hkv;
    const int rb = item / p.Hkv;
    const int b = rb % p.B;
    const int r = rb / p.B;
    const int split = attn_split(p.nsplit);
    int L = p.seq_lens[b];
    L = L < 0 ? 0 : (L > p.max_seq_len ? p.max_seq_len : L);
    const int Ll = local_len(L, p.N, r);
    const int t0 = split * p.split_tokens;
    const int t1 = min(t0 + p.split_tokens, Ll);

    // Q fragments: fragment row qr + 8nb is head hkv*GQ + 8nb + qr (zero past
    // GQ); k-step ks takes d = 32(ks/2) + 8qc + 4(ks%2) + {0,1} and that + 2,
    // the positions the K fragments below carry
    bool head_ok[NB];
    unsigned qa[KS][NB][2];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        head_ok[nb] = 8 * nb + qr < GQ;
        const unsigned char* qrow =
            p.q + (int64_t)b * p.q_sb + (int64_t)(hkv * GQ + (head_ok[nb] ? 8 * nb + qr : 0)) * p.q_sh;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int d0 = 32 * (ks >> 1) + 8 * qc + 4 * (ks & 1);
            qa[ks][nb][0] = head_ok[nb] ? *reinterpret_cast<const unsigned*>(qrow + 2 * d0) : 0u;
            qa[ks][nb][1] = head_ok[nb] ? *reinterpret_cast<const unsigned*>(qrow + 2 * (d0 + 2)) : 0u;
        }
    }
    const float qscale = p.sm_scale * kLog2e;
    float m_run[NB], l_run[NB];
    float oacc[NB][NM][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        m_run[nb] = -INFINITY;
        l_run[nb] = 0.f;
#pragma unroll
        for (int j = 0; j < NM; ++j) oacc[nb][j][0] = oacc[nb][j][1] = oacc[nb][j][2] = oacc[nb][j][3] = 0.f;
    }

    const unsigned char* kb = p.k + (int64_t)r * p.k_sn + (int64_t)b * p.k_sb + (int64_t)hkv * p.k_sh + 16 * qc;
    const unsigned char* vb = p.v + (int64_t)r * p.v_sn + (int64_t)b * p.v_sb + (int64_t)hkv * p.v_sh + 16 * qc;
    // lane (qr, qc) loads token tb + 8h + qr, bytes 64i + 16qc .. +15 of its row;
    // rows past the split are zeros (never read)
    auto load_block = [&](uint4 (&kr)[HB][NI], uint4 (&vr)[HB][NI], int tb) {
#pragma unroll
        for (int h = 0; h < HB; ++h) {
            const int t = tb + 8 * h + qr;
#pragma unroll
            for (int i = 0; i < NI; ++i) {
                kr[h][i] = make_uint4(0u, 0u, 0u, 0u);
                vr[h][i] = kr[h][i];
            }
            if constexpr (PAGED) {
                const KvPlace at = t < t1 ? kv_place<true>(p, r, b, t) : KvPlace{-1, 0};
                if (at.page >= 0) {
                    const unsigned char* kp = kb + at.page * p.k_sp + (int64_t)at.slot * p.k_st;
                    const unsigned char* vp = vb + at.page * p.v_sp + (int64_t)at.slot * p.v_st;
#pragma unroll
                    for (int i = 0; i < NI; ++i) {
                        kr[h][i] = ld_stream<16>(kp + 64 * i);
                        vr[h][i] = ld_stream<16>(vp + 64 * i);
                    }
                }
            } else if (t < t1) {
#pragma unroll
                for (int i = 0; i < NI; ++i) {
                    kr[h][i] = ld_stream<16>(kb + (int64_t)t * p.k_st + 64 * i);
                    vr[h][i] = ld_stream<16>(vb + (int64_t)t * p.v_st + 64 * i);
                }
            }
        }
    };
    auto merge_block = [&](const uint4 (&kr)[HB][NI], const uint4 (&vr)[HB][NI], int tb) {
        // scores of heads qr (c0, c1) and qr + 8 (c2, c3) for tokens
        // tb + 8h + 2qc + {0,1}; the halves' products alternate, so
        // consecutive mma are independent
        float c[HB][4];
#pragma unroll
        for (int h = 0; h < HB; ++h) c[h][0] = c[h][1] = c[h][2] = c[h][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const unsigned a[4] = {qa[ks][0][0], NB > 1 ? qa[ks][NB - 1][0] : 0u, qa[ks][0][1],
                                   NB > 1 ? qa[ks][NB - 1][1] : 0u};
#pragma unroll
            for (int h = 0; h < HB; ++h) {
                const uint4& kv = kr[h][ks >> 1];
                mma_16816<T>(c[h], a, (ks & 1) ? kv.z : kv.x, (ks & 1) ? kv.w : kv.y);
            }
        }
        // online softmax (base 2) of each of the lane's heads over the quad's TB tokens
        float alpha[NB], pr[NB][HB][2];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            float sc[HB][2];
            float bm = -INFINITY;
#pragma unroll
            for (int h = 0; h < HB; ++h)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    sc[h][e] = tb + 8 * h + 2 * qc + e < t1 ? c[h][2 * nb + e] * qscale : -INFINITY;
                    bm = fmaxf(bm, sc[h][e]);
                    pr[nb][h][e] = 0.f;
                }
            bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 1));
            bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 2));
            const float mn = fmaxf(m_run[nb], bm);
            alpha[nb] = 1.f;
            if (head_ok[nb] && mn != -INFINITY) {
                alpha[nb] = m_run[nb] == -INFINITY ? 0.f : exp2f(m_run[nb] - mn);
                float ps = 0.f;
#pragma unroll
                for (int h = 0; h < HB; ++h)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        pr[nb][h][e] = exp2f(sc[h][e] - mn);  // masked: exp2(-inf) = 0
                        ps += pr[nb][h][e];
                    }
                l_run[nb] = l_run[nb] * alpha[nb] + ps;
                m_run[nb] = mn;
            }
        }
        // O^T columns of head block nb are heads 8nb + 2qc + {0,1}: their rescale
        // factors live in quads 2qc and 2qc + 1
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            const float al0 = __shfl_sync(kFull, alpha[nb], 8 * qc);
            const float al1 = __shfl_sync(kFull, alpha[nb], 8 * qc + 4);
#pragma unroll
            for (int j = 0; j < NM; ++j) {
                oacc[nb][j][0] *= al0;
                oacc[nb][j][1] *= al1;
                oacc[nb][j][2] *= al0;
                oacc[nb][j][3] *= al1;
            }
        }
        // P^T fragments: this lane's own probabilities, as hi + lo 16-bit terms
        unsigned ph[NB][HB], pl[NB][HB];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int h = 0; h < HB; ++h) {
                ph[nb][h] = round_pair<T>(pr[nb][h][0], pr[nb][h][1]);
                const float2 bh = unpack2(word_to_pair<T>(ph[nb][h]));
                pl[nb][h] = round_pair<T>(pr[nb][h][0] - bh.x, pr[nb][h][1] - bh.y);
            }
        // V^T fragments: 8x8 tiles x = 2j (rows 0-7) and 2j+1 (rows 8-15), word
        // x%4 of piece x/4, one per 8-token half; then the hi terms of every
        // (head block, d block) and the lo terms, so consecutive mma are
        // independent
        unsigned va[NM][2 * HB];
#pragma unroll
        for (int j = 0; j < NM; ++j)
#pragma unroll
            for (int h = 0; h < HB; ++h) {
                const int x0 = 2 * j, x1 = 2 * j + 1;
                va[j][2 * h] = tile_transpose(word_of(vr[h][x0 >> 2], x0 & 3));
                va[j][2 * h + 1] = tile_transpose(word_of(vr[h][x1 >> 2], x1 & 3));
            }
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int j = 0; j < NM; ++j) {
                    const unsigned* pb = t == 0 ? ph[nb] : pl[nb];
                    if constexpr (HB == 2) mma_16816<T>(oacc[nb][j], va[j], pb[0], pb[1]);
                    else mma_1688<T>(oacc[nb][j], va[j], pb[0]);
                }
    };
    const int stride = NW * TB;
    if constexpr (PF) {
        // two register sets: the next block's loads are in flight while this one merges
        uint4 ka[HB][NI], va[HB][NI], kn[HB][NI], vn[HB][NI];
        int tb = t0 + warp * TB;  // uniform across the warp
        if (tb < t1) load_block(ka, va, tb);
        while (tb < t1) {
            if (tb + stride < t1) load_block(kn, vn, tb + stride);
            merge_block(ka, va, tb);
            tb += stride;
            if (tb >= t1) break;
            if (tb + stride < t1) load_block(ka, va, tb + stride);
            merge_block(kn, vn, tb);
            tb += stride;
        }
    } else {
        for (int tb = t0 + warp * TB; tb < t1; tb += stride) {  // uniform across the warp
            uint4 kr[HB][NI], vr[HB][NI];
            load_block(kr, vr, tb);
            merge_block(kr, vr, tb);
        }
    }

    // the quad's partial sums of each head, then the warp's state to shared
    // memory: output row qr of tile x is d = 32(x/4) + 8(qr/2) + 2(x%4) + qr%2
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        l_run[nb] += __shfl_xor_sync(kFull, l_run[nb], 1);
        l_run[nb] += __shfl_xor_sync(kFull, l_run[nb], 2);
        if (head_ok[nb] && qc == 0) {
            s_m[warp][8 * nb + qr] = m_run[nb];
            s_l[warp][8 * nb + qr] = l_run[nb];
        }
#pragma unroll
        for (int j = 0; j < NM; ++j)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int x = 2 * j + half;
                const int d = 32 * (x >> 2) + 8 * (qr >> 1) + 2 * (x & 3) + (qr & 1);
                const int g0 = 8 * nb + 2 * qc;
                if (g0 < GQ) s_acc[warp][g0][d] = oacc[nb][j][2 * half];
                if (g0 + 1 < GQ) s_acc[warp][g0 + 1][d] = oacc[nb][j][2 * half + 1];
            }
    }
    __syncthreads();
    write_cta_result<T, D, GQ, NW>(p, r, b, hkv, split, s_m, s_l, s_acc);
    pdl_trigger();
}

// Merge the splits of every (rank, request, head) row: the LSE-weighted merge
// in base 2 over the fp32 partials, one warp per row, lanes over D.
template <typename T, int D>
__global__ void __launch_bounds__(kAttnThreads) decode_merge_splits_kernel(const AttnParams p) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t rows = (int64_t)p.N * p.B * p.H;
    const int64_t row = (int64_t)blockIdx.x * (kAttnThreads / 32) + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int h = (int)(row % p.H);
    const int64_t rb = row / p.H;
    const int b = (int)(rb % p.B);
    const int r = (int)(rb / p.B);
    // only the splits that hold tokens of the row (the others are (0, -inf)
    // and would drop out; the tensor-core kernel does not write them, and it
    // writes the result of a row with at most one such split itself)
    int L = p.seq_lens[b];
    L = L < 0 ? 0 : (L > p.max_seq_len ? p.max_seq_len : L);
    const int Ll = local_len(L, p.N, r);
    const int S = min(p.nsplit, (Ll + p.split_tokens - 1) / p.split_tokens);
    if (p.merge_multi_only && S <= 1) return;
    const float* lrow = p.ws_lse + row * p.nsplit;
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
            const float* orow = p.ws_o + (row * p.nsplit + s) * D;
#pragma unroll
            for (int i = 0; i < D / 32; ++i) acc[i] = fmaf(w, orow[lane + 32 * i], acc[i]);
        }
    }
    T* orow = reinterpret_cast<T*>(p.o + (int64_t)r * p.o_sn + (int64_t)b * p.o_sb + (int64_t)h * p.o_sh);
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) orow[lane + 32 * i] = from_f32<T>(acc[i] * inv);
    if (lane == 0) {
        const float lse2 = Ls > 0.f ? M + log2f(Ls) : -INFINITY;
        p.lse[(int64_t)r * p.l_sn + (int64_t)b * p.l_sb + (int64_t)h * p.l_sh] = p.base2 ? lse2 : lse2 * kLn2;
    }
    pdl_trigger();
}

template <typename T, int D>
static cudaError_t launch_split_merge(const AttnParams& p, cudaStream_t stream) {
    AttnParams q = p;
    void* args[] = {(void*)&q};
    const int64_t rows = (int64_t)p.N * p.B * p.H;
    const unsigned mgrid = (unsigned)((rows + kAttnThreads / 32 - 1) / (kAttnThreads / 32));
    return launch_pdl((const void*)decode_merge_splits_kernel<T, D>, dim3(mgrid), dim3(kAttnThreads), args, 0,
                      stream);
}

template <typename T, int D, bool PAGED>
static cudaError_t launch_attention_dp(const AttnParams& p, cudaStream_t stream) {
    const void* k;
    // grouped-query heads go to the tensor cores; one query head per KV head
    // stays on the CUDA cores, and so do two at D = 256 (measured: 1.51 ms on
    // the CUDA cores against 1.71 ms for the 8-token tensor-core blocks that
    // D = 256 is limited to by registers; from four heads up the tensor
    // cores win, 0.90 vs 1.28 ms and 0.51 vs 1.38 ms)
    if constexpr (DCP_ATTN_MMA) {
        switch (p.H / p.Hkv) {
            case 1: k = (const void*)decode_partial_kernel<T, D, 1, PAGED>; break;
            case 2:
                k = D == 256 ? (const void*)decode_partial_kernel<T, D, 2, PAGED> : (const void*)decode_partial_mma_kernel<T, D, 2, PAGED>;
                break;
            case 4: k = (const void*)decode_partial_mma_kernel<T, D, 4, PAGED>; break;
            case 8: k = (const void*)decode_partial_mma_kernel<T, D, 8, PAGED>; break;
            case 16:
                if constexpr (D <= 128) k = (const void*)decode_partial_mma_kernel<T, D, 16, PAGED>;
                else return cudaErrorInvalidValue;  // refused by the host checks
                break;
            default: return cudaErrorInvalidValue;
        }
    } else {
        switch (p.H / p.Hkv) {
            case 1: k = (const void*)decode_partial_kernel<T, D, 1, PAGED>; break;
            case 2: k = (const void*)decode_partial_kernel<T, D, 2, PAGED>; break;
            case 4: k = (const void*)decode_partial_kernel<T, D, 4, PAGED>; break;
            case 8: k = (const void*)decode_partial_kernel<T, D, 8, PAGED>; break;
            default: return cudaErrorInvalidValue;
        }
    }
    void* args[] = {(void*)&p};
    const dim3 grid((unsigned)((int64_t)p.N * p.B * p.Hkv * p.nsplit));  // split fastest
    cudaError_t e = launch_pdl(k, grid, dim3(kAttnThreads), args, 0, stream);
    if (e != cudaSuccess || p.nsplit == 1) return e;
    return launch_split_merge<T, D>(p, stream);
}

template <typename T, int D>
static cudaError_t launch_attention_d(const AttnParams& p, cudaStream_t stream) {
    // paged caches take the page-table lookup; contiguous ones compile without it
    return p.page_shift >= 0 ? launch_attention_dp<T, D, true>(p, stream) : launch_attention_dp<T, D, false>(p, stream);
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

cudaError_t launch_attention_split_merge(const AttnParams& p, int dtype, cudaStream_t stream) {
    switch (p.D) {
        case 64: return dtype == 1 ? launch_split_merge<__half, 64>(p, stream) : launch_split_merge<__nv_bfloat16, 64>(p, stream);
        case 128: return dtype == 1 ? launch_split_merge<__half, 128>(p, stream) : launch_split_merge<__nv_bfloat16, 128>(p, stream);
        case 256: return dtype == 1 ? launch_split_merge<__half, 256>(p, stream) : launch_split_merge<__nv_bfloat16, 256>(p, stream);
        default: return cudaErrorInvalidValue;
    }
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

// The array's device address belongs to the CUDA context the library's code
// is loaded into, not to the device: cudaDeviceReset destroys the primary
// context (the next runtime call loads the code again, maybe at another
// address), and a caller may make its own driver-API context current instead
// of the primary one.  So every call looks the address up in the context
// current at that call (cudaGetSymbolAddress allocates nothing; on the first
// call in a context it also loads the library's code there), and no address
// outlives the call that looked it up.
cudaError_t scratch_address(void** out) { return cudaGetSymbolAddress(out, g_attn_scratch); }

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
    void* scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof(msg), "dcp_decode_attention_noalloc: cudaGetSymbolAddress failed: %s",
                 cudaGetErrorString(e));
        return dcp::set_error(DCP_ERR_CUDA, msg);
    }
    return dcp_decode_attention(dtype, N, B, H, Hkv, D, q, q_sb, q_sh, k, k_sn, k_sb, k_st, k_sh, v, v_sn,
                                v_sb, v_st, v_sh, seq_lens, max_seq_len, sm_scale, split_tokens, o, o_sn,
                                o_sb, o_sh, lse, l_sn, l_sb, l_sh, lse_base, scratch, kNoAllocScratchBytes,
                                stream);
}
