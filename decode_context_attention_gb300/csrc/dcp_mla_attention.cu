// dcp_mla_attention.cu -- each DCP rank's decode attention over its share of
// an absorbed-MLA latent cache, on the 5th-generation tensor cores.
//
// sglang PR #33926 report, "功能与动机" and "实现拆解" items 3-4: the
// trtllm_mla decode path (DeepSeek-V3 class models on Blackwell) returns the
// rank-local (out, lse) of every rank, the LSE in base 2, and a rank that
// owns no token of a request is the neutral (0, -inf); token t of a request
// lives on rank t % N.  sglang PR #34213 report, "功能与动机": for absorbed
// MLA the output width is kv_lora_rank.
//
// Every query head h scores one shared latent row per token,
//     kv_t [576] = [ c_t (512 = kv_lora_rank) | k_rope_t (64) ],
// against its absorbed query q_h [576]; the value is the row's first 512
// elements:  s = sm_scale <q_h, kv_t>,  lse = log sum exp(s),
//            O_h = sum_t exp(s_t - lse) c_t.
//
// Design.  128 query heads x 512 output columns of fp32 accumulators are
// 256 KB: all of one SM's tensor memory, with no room left for the scores.
// So a pair of CTAs (a thread-block cluster of 2) works on one (rank,
// request, split) item at a time: CTA c owns output columns [256c, 256c +
// 256) and, for the scores, latent columns [256c, 256c + 256) plus rope
// columns [512 + 32c, 544 + 32c) -- exactly the columns it loads, so the
// pair reads every latent byte once and does every multiply-add once.  Per
// tile of 64 tokens:
//   * TMA (one thread) loads the CTA's four 64-column latent chunks of the
//     64 tokens (128-byte swizzled) and its 32 rope columns (64-byte
//     swizzled) into a 4-stage ring (36 KB a stage: the loads of a tile are
//     issued about three tiles ahead, which the memory latency under full
//     load needs);
//   * the MMA thread computes the partial scores S_c [128 heads x 64 tokens]
//     = Q_c . KV_c^T with tcgen05.mma, fp32 in tensor memory: the query's
//     256 latent columns are the A operand in tensor memory, its 32 rope
//     columns an A operand in shared memory (a TMA tile), the latent rows the
//     K-major B operand;
//   * an exchange warpgroup reads S_c as soon as it is ready, rounds it to
//     fp16 in log2 units (half the bytes of fp32 on the
//     distributed-shared-memory path), and sends it to the peer CTA with
//     st.async stores that count their bytes on the peer's mbarrier (no
//     fence) -- a 4-byte st.async credit from the peer frees each of its two
//     receive slots again -- and puts the same fp16 pairs back into tensor
//     memory for its own CTA's softmax.  Scores are double-buffered in TMEM,
//     so the exchange of tile i + 1 overlaps the softmax of tile i;
//   * two softmax warpgroups (thread (h, g) = head h = TMEM lane h, tokens
//     [32g, 32g + 32) of the tile) add the two fp16 partials with one
//     rounding to fp32 (the same bits in both CTAs: one probability for both
//     halves of the output) and run an online softmax in base 2 with a
//     lazily moved reference max (the output is rescaled only when the max
//     grows by more than 2^8, so most tiles skip it); P goes to tensor
//     memory as bf16/fp16, over its tile's consumed scores;
//   * the MMA thread accumulates O_c [128 x 256] += P . V_c with P as the
//     TMEM A operand and V_c read MN-major from the same shared-memory tile.
// With one split the softmax warps normalise O and write (O_r, lse_r);
// otherwise fp32 partials go to the workspace and a second kernel merges the
// splits with the combine's LSE rule.
//
// The pairs are persistent: as many as fit on the device at once, each
// taking its share of the items, longest first, one after the other.  The
// pipeline runs on across an item boundary -- the next item's query is
// staged (TMA into a shared-memory area, then into tensor memory) and its
// first tiles are loaded and scored while the current item's last tiles and
// its epilogue finish -- so the per-item set-up (barriers, tensor memory,
// the query, the first tile's latency) is paid once per pair, not per item.
//
// Every barrier wait is bounded (1 s): a wait that runs out records
// DCP_ERR_TIMEOUT in a device status word and the kernel winds down (its
// copies and MMAs in flight are waited for, its tensor memory freed)
// instead of hanging.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdlib.h>

#include <type_traits>

#include "dcp_device.cuh"
#include "dcp_sm100.cuh"

namespace dcp {

using namespace sm100;

namespace {

constexpr int kMlaThreads = 448;   // warps 0-7 softmax, 8-11 exchange, 12 TMA, 13 MMA
constexpr int kSoftmaxThreads = 256;
constexpr int kTileTokens = 64;    // tokens per tile (one ring stage)
constexpr int kHalf = 32;          // tokens of a tile per softmax warpgroup
#ifndef DCP_MLA_STAGES
#define DCP_MLA_STAGES 4
#endif
constexpr int kStages = DCP_MLA_STAGES;  // shared-memory ring depth
constexpr int kChunkBytes = kTileTokens * 128;      // 64 tokens x 64 columns x 2 bytes
constexpr int kRopeChunkBytes = kTileTokens * 64;   // the CTA's 32 rope columns of 64 tokens
constexpr int kStageBytes = 4 * kChunkBytes + kRopeChunkBytes;  // 4 latent chunks + the rope chunk
constexpr int kXbufBytes = kTileTokens * 128 * 2;   // fp16 partial scores of a tile (log2 units), 64 tokens x 128 heads
constexpr int kQropeBytes = 128 * 64;               // [128 heads x the CTA's 32 rope columns], 64-byte swizzled
constexpr int kQStageBytes = 2 * 128 * 128;         // half the query's latent columns: two [128 heads x 64] boxes
constexpr int kMiscBytes = 2048;                    // barriers, the warpgroups' row values, credit words
constexpr int kSeqMax = 512;                        // items a pair takes in sorted order, at most
constexpr int kSortMax = 8192;                      // items put in order (in the ring), at most
constexpr int kSortBins = 512;                      // tile counts told apart by that order
// the ring, the two receive slots, the query's rope tile, the query staging
// area, the small things, the pair's item list
constexpr int kSmemBytes =
    kStages * kStageBytes + 2 * kXbufBytes + kQropeBytes + kQStageBytes + kMiscBytes + 8 * kSeqMax + 1024 /* align */;
static_assert(kSmemBytes <= 232448, "more than a CTA's shared memory");
static_assert(kStageBytes % 1024 == 0 && kQropeBytes % 1024 == 0, "swizzled tiles stay 1024-byte aligned");
static_assert(6 * kSortMax + 4 * (kMlaThreads / 32 + 1) * kSortBins <= kStages * kStageBytes,
              "the sort's scratch lives in the ring");
// tensor-memory columns
constexpr uint32_t kColO = 0;      // O_c: 256 fp32 columns
constexpr uint32_t kColQ = 256;    // Q_c latent part: 256 16-bit elements = 128 columns
constexpr uint32_t kColSP = 384;   // two buffers of 64 columns: S_c of a tile, then its P in the first 32
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.f;  // move the reference max when it would grow by more than this
constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kLn2F = 0.6931471805599453f;

enum : int { kStatusTimeout = DCP_ERR_TIMEOUT };

__device__ int g_mla_status;  // first bounded wait that ran out (0 if none)

struct Barriers {
    uint64_t kv_full[kStages], kv_empty[kStages];
    uint64_t q_full;       // the item's latent query is in tensor memory (exchange warpgroup)
    uint64_t q_empty;      // the item's last score product has run (MMA commit)
    uint64_t qrope_full;   // the item's rope tile landed (TMA)
    uint64_t qstage_full;  // a query half landed in the staging area (TMA)
    uint64_t qstage_free;  // the staging area's half has moved to tensor memory
    uint64_t o_free;       // the item's O has been read out (softmax threads)
    uint64_t stg_free;     // the epilogue is done with the staging area (softmax warps)
    uint64_t mma_done;
    uint64_t s_full[2], own_full[2][2], p_full[2], pv_done[2];  // per score / probability buffer (own: per half)
    uint64_t xfull[2][2];  // receive slot u, token half g2: the peer's partial scores arrived (st.async bytes)
    uint64_t credit[2];  // send slot: the peer has freed its receive slot (a st.async credit)
    uint64_t red_full, red_free;  // the softmax warpgroups' per-row values: written / read
    uint32_t tmem_base;
    int abort;
    uint32_t credit_word[2];      // landing words of the peer's credits
    float red[2][128];            // per warpgroup and head: tile max, then the final row sum
};
static_assert(sizeof(Barriers) <= kMiscBytes, "misc region too small");

// Two floats to fp16 (round to nearest, values past the fp16 range to its
// largest finite, NaN kept), lo in the low half.
__device__ __forceinline__ uint32_t f16x2_satfinite(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// (a + b, c + d) with one instruction (packed fp32 add, round to nearest)
__device__ __forceinline__ float2 add_f32x2(float2 x, float2 y) {
    uint64_t a, b, d;
    memcpy(&a, &x, 8);
    memcpy(&b, &y, 8);
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    float2 r;
    memcpy(&r, &d, 8);
    return r;
}
// (a * b, c * d) with one instruction (packed fp32 multiply, round to nearest)
__device__ __forceinline__ float2 mul_f32x2(float2 x, float2 y) {
    uint64_t a, b, d;
    memcpy(&a, &x, 8);
    memcpy(&b, &y, 8);
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    float2 r;
    memcpy(&r, &d, 8);
    return r;
}
// The sums of two pairs of fp16 values (lo halves, hi halves) rounded once
// to fp32: x's halves enter the mixed-precision add as fp16, y's exactly
// widened to fp32 first.
__device__ __forceinline__ float2 add_f16x2_exact(uint32_t x, uint32_t y) {
    float2 r;
    asm("{\n .reg .b16 a0, a1, b0, b1;\n .reg .f32 f0, f1;\n mov.b32 {a0, a1}, %2;\n mov.b32 {b0, b1}, %3;\n"
        " cvt.f32.f16 f0, b0;\n cvt.f32.f16 f1, b1;\n add.rn.f32.f16 %0, a0, f0;\n add.rn.f32.f16 %1, a1, f1;\n}"
        : "=f"(r.x), "=f"(r.y)
        : "r"(x), "r"(y));
    return r;
}
// max(a, b, c) with one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// 2^x by the ex2.approx instruction (the PTX ISA puts its relative error
// near 2^-22, far below the 2^-9 / 2^-12 rounding of P to bf16 / fp16;
// results below the normal range flush to 0, 2^-inf = 0).
__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <typename T>
__device__ __forceinline__ uint32_t pack_pair(float a, float b) {
    if constexpr (std::is_same<T, __half>::value) {
        const __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t*>(&h);
    } else {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
}

// Roles, for the pair's items in turn (global tile index gi over all of
// them: score buffer and receive slot u = gi % 2, ring stage gi % 4; the
// pair's n-th item with tokens is "item n"):
//   TMA      item n's query: its two latent halves through the staging area
//            (qstage_full; the first once the area is free of item n-2's
//            epilogue and of the last half, the second once the first has
//            moved on: qstage_free), its rope tile once item n-1's last score
//            product has run (q_empty); kv_full[stage] <- each tile's 5 chunks
//   exchange item n's latent query from the staging area into tensor memory
//            once item n-1's last score product has run (q_full); then S(gi)
//            from SP[u] as fp16 pairs -> the peer's receive slot u by
//            st.async once the peer granted it (credit[u]), and into SP[u]
//            columns [32, 64) (own_full[u][half])
//   MMA      the scores run two tiles ahead of the value products, across
//            items: PV(gi) after P(gi) (pv_done[u], kv_empty[stage]; an
//            item's first once the previous item's O has been read: o_free),
//            then QK(gi + 2) into SP[u] (s_full[u]; an item's last also
//            q_empty)
//   softmax  the peer's S(gi) from slot u (xfull[u][g], one barrier per token
//            half) + the own from SP[u] (own_full[u][g]); re-arm xfull[u][*]
//            and grant the slot back to the peer;
//            P(gi) into SP[u] columns [0, 32) (p_full[u]); after an item's
//            last PV its O goes out (o_free once read) through the staging
//            area, once the next item's query has left it (stg_free after)
template <typename T>
__global__ void __launch_bounds__(kMlaThreads, 1) mla_decode_kernel(const __grid_constant__ CUtensorMap kv_map,
                                                                   const __grid_constant__ CUtensorMap kv_rope_map,
                                                                   const __grid_constant__ CUtensorMap q_map,
                                                                   const __grid_constant__ CUtensorMap q_rope_map,
                                                                   const MlaParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    uint8_t* slots = smem + kStages * kStageBytes;  // 2 x [8 token groups][128 heads] x 8 halves
    uint8_t* qrope = slots + 2 * kXbufBytes;
    uint8_t* qstage = qrope + kQropeBytes;  // half the query's latent columns, or the epilogue's rows
    Barriers* bar = reinterpret_cast<Barriers*>(qstage + kQStageBytes);
    int* seq = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(bar) + kMiscBytes);  // the pair's items
    int* spn = seq + kSeqMax;                                                           // and their tokens

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t c = cluster_ctarank();  // which half of the columns
    const uint32_t peer = c ^ 1u;
    const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
    const int nitems = p.N * p.B * p.nsplit;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bar->kv_full[s], 1);
            mbar_init(&bar->kv_empty[s], 1);
        }
        mbar_init(&bar->q_full, 128);
        mbar_init(&bar->q_empty, 1);
        mbar_init(&bar->qrope_full, 1);
        mbar_init(&bar->qstage_full, 1);
        mbar_init(&bar->qstage_free, 128);
        mbar_init(&bar->o_free, kSoftmaxThreads);
        mbar_init(&bar->stg_free, kSoftmaxThreads / 32);
        mbar_init(&bar->mma_done, 1);
        for (int u = 0; u < 2; ++u) {
            mbar_init(&bar->s_full[u], 1);
            for (int g2 = 0; g2 < 2; ++g2) mbar_init(&bar->own_full[u][g2], 4);
            mbar_init(&bar->p_full[u], 8);
            mbar_init(&bar->pv_done[u], 1);
            // the peer's bytes complete these; this CTA's expect_tx is the one
            // arrival, armed here for the first phase
            for (int g2 = 0; g2 < 2; ++g2) {
                mbar_init(&bar->xfull[u][g2], 1);
                mbar_arrive_expect_tx(&bar->xfull[u][g2], kXbufBytes / 2);
            }
            mbar_init(&bar->credit[u], 1);
            mbar_arrive_expect_tx(&bar->credit[u], 4);
        }
        mbar_init(&bar->red_full, kSoftmaxThreads);
        mbar_init(&bar->red_free, kSoftmaxThreads);
        bar->abort = 0;
        fence_mbar_init();
    }
    if (warp == 13) {
        tmem_alloc(&bar->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 12 && lane == 0) {
        tma_prefetch_map(&kv_map);
        tma_prefetch_map(&kv_rope_map);
        tma_prefetch_map(&q_map);
        tma_prefetch_map(&q_rope_map);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();  // the peer's barriers are initialised before any remote arrival
    pdl_wait();      // the set-up above overlapped the previous kernel's tail
    const uint32_t tmem = bar->tmem_base;
    volatile int* abort = &bar->abort;
    int* status = &g_mla_status;
    bool issued_any = false;  // the MMA thread issued at least one MMA
    const unsigned kAll = 0xffffffffu;

    // Item idx = (rank r, request b, split): its first local token t0, and
    // its number of local tokens (from the request's length), in tiles
    struct Item {
        int r, b, split, t0;
    };
    auto item_of = [&](int idx) {
        Item it;
        it.split = idx % p.nsplit;
        const int rb = idx / p.nsplit;
        it.b = rb % p.B;
        it.r = rb / p.B;
        it.t0 = it.split * p.split_tokens;
        return it;
    };
    auto span_of = [&](int idx) {
        const Item it = item_of(idx);
        int L = p.seq_lens[it.b];
        L = L < 0 ? 0 : (L > p.max_seq_len ? p.max_seq_len : L);
        const int Ll = L / p.N + (it.r < L % p.N ? 1 : 0);
        return max(0, min(it.t0 + p.split_tokens, Ll) - it.t0);
    };
    auto tiles_of = [](int span) { return (span + kTileTokens - 1) / kTileTokens; };
    // The pair's items.  Every CTA puts all items in order of their number of
    // tiles, most first, ties by index (a stable counting sort in the ring,
    // before any copy lands there); pair q then takes positions q, 2P - 1 -
    // q, 2P + q, 4P - 1 - q, ... (P pairs), so the longest items start first
    // and the pairs' totals come out close.  Both CTAs of a pair compute the
    // same list.  Past kSortMax items (or kSeqMax a pair), pair q takes q,
    // q + P, q + 2P, ...
    const bool sorted = nitems <= kSortMax && (nitems + npairs - 1) / npairs <= kSeqMax;
    if (sorted) {
        constexpr int kWarps = kMlaThreads / 32;
        uint16_t* bin_of = reinterpret_cast<uint16_t*>(stages);         // [item]
        int* order = reinterpret_cast<int*>(stages + 2 * kSortMax);     // [position]
        int* hist = order + kSortMax;                                   // [warp][bin]
        int* start = hist + kWarps * kSortBins;                         // [bin]
        // bin 0 holds the items with the most tiles (nbins - 1 or more)
        const int nbins = min(kSortBins, (p.split_tokens + kTileTokens - 1) / kTileTokens + 1);
        for (int i = tid; i < nitems; i += kMlaThreads)
            bin_of[i] = (uint16_t)(nbins - 1 - min(tiles_of(span_of(i)), nbins - 1));
        for (int i = tid; i < kWarps * nbins; i += kMlaThreads) hist[i] = 0;
        __syncthreads();
        // warp w takes the items [w * seg, (w + 1) * seg): first the count of
        // each bin among them
        const int seg = (nitems + kWarps - 1) / kWarps;
        const int s0 = min(warp * seg, nitems), s1 = min(s0 + seg, nitems);
        for (int i0 = s0; i0 < s1; i0 += 32) {
            const int i = i0 + lane;
            const unsigned act = __ballot_sync(kAll, i < s1);
            if (i < s1) {
                const int bn = bin_of[i];
                const unsigned peers = __match_any_sync(act, bn);
                if (lane == __ffs(peers) - 1) hist[warp * nbins + bn] += __popc(peers);
            }
            __syncwarp();
        }
        __syncthreads();
        // per bin: the items of the warps before (exclusive), and the total
        for (int bn = tid; bn < nbins; bn += kMlaThreads) {
            int run = 0;
            for (int w = 0; w < kWarps; ++w) {
                const int cnt = hist[w * nbins + bn];
                hist[w * nbins + bn] = run;
                run += cnt;
            }
            start[bn] = run;
        }
        __syncthreads();
        if (warp == 0) {  // the bins' first positions: an exclusive scan of the totals
            int carry = 0;
            for (int b0 = 0; b0 < nbins; b0 += 32) {
                const int bn = b0 + lane;
                const int tot = bn < nbins ? start[bn] : 0;
                int incl = tot;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int y = __shfl_up_sync(kAll, incl, d);
                    if (lane >= d) incl += y;
                }
                if (bn < nbins) start[bn] = carry + incl - tot;
                carry += __shfl_sync(kAll, incl, 31);
            }
        }
        __syncthreads();
        // each item's position: its bin's first, plus the bin's items in the
        // warps before, in this warp's earlier chunks and at lower lanes
        for (int i0 = s0; i0 < s1; i0 += 32) {
            const int i = i0 + lane;
            const unsigned act = __ballot_sync(kAll, i < s1);
            if (i < s1) {
                const int bn = bin_of[i];
                const unsigned peers = __match_any_sync(act, bn);
                order[start[bn] + hist[warp * nbins + bn] + __popc(peers & ((1u << lane) - 1u))] = i;
                __syncwarp(act);
                if (lane == __ffs(peers) - 1) hist[warp * nbins + bn] += __popc(peers);
            }
            __syncwarp();
        }
        __syncthreads();
        for (int k = tid; k * npairs < nitems; k += kMlaThreads) {
            const int pos = k * npairs + ((k & 1) ? npairs - 1 - pair : pair);
            const int idx = pos < nitems ? order[pos] : -1;
            seq[k] = idx;
            spn[k] = idx >= 0 ? span_of(idx) : 0;
        }
        __syncthreads();  // the ring is free for copies again
    }
    // the pair's k-th item and its local tokens (idx -1: none, -2: past the
    // list's end)
    struct Work {
        int idx, span;
    };
    auto work_at = [&](int k) -> Work {
        if (sorted) {
            if (k * npairs >= nitems) return {-2, 0};
            return {seq[k], spn[k]};
        }
        const int idx = pair + k * npairs;
        if (idx >= nitems) return {-2, 0};
        return {idx, span_of(idx)};
    };

    if (warp == 12) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            int gt = 0;      // tiles of the items before
            int nq = 0;      // items with tokens before
            int nbox = 0;    // query halves staged
            int nrope = 0;   // rope tiles loaded
            int issued = 0;  // tiles loaded
            bool ok = true;
            // half `half` of the query's latent columns [256c, 256c + 256) of
            // request b: two [128 heads x 64] boxes (heads past H read 0)
            auto stage_half = [&](int half, int b) {
                mbar_arrive_expect_tx(&bar->qstage_full, kQStageBytes);
                for (int jj = 0; jj < 2; ++jj)
                    tma_load_3d(qstage + jj * 128 * 128, &q_map, &bar->qstage_full, 256 * (int)c + 64 * (2 * half + jj),
                                0, b);
                ++nbox;
            };
            // the tile i of item `it` (global index gi) into its ring stage
            auto load_tile = [&](const Item& it, int i, int gi) -> bool {
                const int st = gi % kStages, kk = gi / kStages;
                if (kk > 0 && !mbar_wait(&bar->kv_empty[st], (kk - 1) & 1, status, kStatusTimeout, abort)) return false;
                uint8_t* dst = stages + st * kStageBytes;
                mbar_arrive_expect_tx(&bar->kv_full[st], kStageBytes);
                const int y = it.t0 + i * kTileTokens;
                for (int j = 0; j < 4; ++j)
                    tma_load_4d(dst + j * kChunkBytes, &kv_map, &bar->kv_full[st], 256 * (int)c + 64 * j, y, it.b, it.r);
                tma_load_4d(dst + 4 * kChunkBytes, &kv_rope_map, &bar->kv_full[st], 512 + 32 * (int)c, y, it.b, it.r);
                issued = gi + 1;
                return true;
            };
            for (int k = 0; ok; ++k) {
                const Work w = work_at(k);
                if (w.idx == -2) break;
                const int ntiles = tiles_of(w.span);
                if (w.idx < 0 || ntiles == 0) continue;
                const Item it = item_of(w.idx);
                // in the order they can go (every wait blocks): the query's
                // first half (once item n-2's epilogue and the last half have
                // left the staging area), the first tile, the rope tile (once
                // item n-1's last score product has run), the second half
                // (once the first has moved on), the other tiles
                ok = (nq < 2 || mbar_wait(&bar->stg_free, (nq - 2) & 1, status, kStatusTimeout, abort)) &&
                     (nbox == 0 || mbar_wait(&bar->qstage_free, (nbox - 1) & 1, status, kStatusTimeout, abort));
                if (!ok) break;
                stage_half(0, it.b);
                if (!p.stall_loads && !load_tile(it, 0, gt)) break;
                if (nq > 0 && !mbar_wait(&bar->q_empty, (nq - 1) & 1, status, kStatusTimeout, abort)) break;
                mbar_arrive_expect_tx(&bar->qrope_full, kQropeBytes);
                tma_load_3d(qrope, &q_rope_map, &bar->qrope_full, 512 + 32 * (int)c, 0, it.b);
                ++nrope;
                if (!mbar_wait(&bar->qstage_free, (nbox - 1) & 1, status, kStatusTimeout, abort)) break;
                stage_half(1, it.b);
                if (p.stall_loads) break;
                for (int i = 1; ok && i < ntiles; ++i) ok = load_tile(it, i, gt + i);
                gt += ntiles;
                ++nq;
            }
            // copies still in flight (only after an abort) land before the CTA ends
            const uint64_t t_start = global_timer_ns();
            if (nrope > 0)
                while (!mbar_try_wait(&bar->qrope_full, (nrope - 1) & 1) && global_timer_ns() - t_start < kWaitLimitNs) {
                }
            if (nbox > 0)
                while (!mbar_try_wait(&bar->qstage_full, (nbox - 1) & 1) && global_timer_ns() - t_start < kWaitLimitNs) {
                }
            for (int gi = max(0, issued - kStages); gi < issued; ++gi) {
                const uint64_t t1w = global_timer_ns();
                while (!mbar_try_wait(&bar->kv_full[gi % kStages], (gi / kStages) & 1) &&
                       global_timer_ns() - t1w < kWaitLimitNs) {
                }
            }
        }
    } else if (warp == 13) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr bool kBf16 = !std::is_same<T, __half>::value;
            const uint32_t idesc_qk = idesc_f16(128, kTileTokens, kBf16, 0, 0);
            const uint32_t idesc_pv = idesc_f16(128, 256, kBf16, 0, 1);
            const uint32_t tQ = tmem + kColQ, tO = tmem + kColO;
            const uint64_t dq = smem_desc(smem_u32(qrope), 16, 512, kSwizzle64B);
            // the score stream: the next tile whose S is computed (tile qi of
            // the pair's qk-th item, the qn-th with tokens; global tile qg)
            int qk = -1, qi = 0, qn = -1, qg = 0, qnt = 0;
            auto next_tile = [&]() -> bool {
                if (qk >= 0 && ++qi < qnt) return true;
                for (;;) {
                    const Work w = work_at(++qk);
                    if (w.idx == -2) return false;
                    qnt = w.idx >= 0 ? tiles_of(w.span) : 0;
                    if (qnt > 0) break;
                }
                qi = 0;
                ++qn;
                return true;
            };
            bool qmore = next_tile();
            // S(qg) = Q_c . KV_c(qg)^T into buffer qg % 2, then the stream
            // moves on.  The descriptor's address field is bits 0-13 in
            // 16-byte units: offsets are added to it directly.
            auto issue_qk = [&]() -> bool {
                if (qi == 0 && (!mbar_wait(&bar->q_full, qn & 1, status, kStatusTimeout, abort) ||
                                !mbar_wait(&bar->qrope_full, qn & 1, status, kStatusTimeout, abort)))
                    return false;
                const int st = qg % kStages;
                if (!mbar_wait(&bar->kv_full[st], (qg / kStages) & 1, status, kStatusTimeout, abort)) return false;
                tc_fence_after();
                const uint32_t tS = tmem + kColSP + 64 * (qg & 1);
                const uint64_t d0 = smem_desc(smem_u32(stages + st * kStageBytes), 16, 1024, kSwizzle128B);
                const uint64_t dr = smem_desc(smem_u32(stages + st * kStageBytes + 4 * kChunkBytes), 16, 512, kSwizzle64B);
#pragma unroll
                for (int s = 0; s < 16; ++s)  // latent columns: 4 chunks x 4 steps of 16, A in TMEM
                    mma_ts(tS, tQ + 8 * s, d0 + (uint64_t)(((s >> 2) * kChunkBytes + (s & 3) * 32) >> 4), idesc_qk,
                           s > 0 ? 1u : 0u);
#pragma unroll
                for (int s = 0; s < 2; ++s)  // this CTA's 32 rope columns: the 64-byte rows of both tiles
                    mma_ss(tS, dq + (uint64_t)((32 * s) >> 4), dr + (uint64_t)((32 * s) >> 4), idesc_qk, 1u);
                mma_commit(&bar->s_full[qg & 1]);
                if (qi == qnt - 1) mma_commit(&bar->q_empty);  // the item's last read of its query
                issued_any = true;
                ++qg;
                qmore = next_tile();
                return true;
            };
            bool ok = true;
            for (int j = 0; ok && qmore && j < 2; ++j) ok = issue_qk();
            int gt = 0, nq = 0;
            for (int k = 0; ok; ++k) {
                const Work w = work_at(k);
                if (w.idx == -2) break;
                const int ntiles = w.idx >= 0 ? tiles_of(w.span) : 0;
                if (ntiles == 0) continue;
                for (int i = 0; i < ntiles; ++i) {
                    // O += P(gi) . V(gi): P from TMEM (the first 32 columns of
                    // SP[gi % 2]), V read MN-major from the tile's stage
                    const int gi = gt + i, u = gi & 1;
                    if (!mbar_wait(&bar->p_full[u], (gi >> 1) & 1, status, kStatusTimeout, abort) ||
                        (i == 0 && nq > 0 && !mbar_wait(&bar->o_free, (nq - 1) & 1, status, kStatusTimeout, abort))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t dv = smem_desc(smem_u32(stages + (gi % kStages) * kStageBytes), kChunkBytes, 1024,
                                                  kSwizzle128B);
                    const uint32_t tP = tmem + kColSP + 64 * u;
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        mma_ts(tO, tP + 8 * s, dv + (uint64_t)((2048 * s) >> 4), idesc_pv, (i > 0 || s > 0) ? 1u : 0u);
                    mma_commit(&bar->pv_done[u]);
                    mma_commit(&bar->kv_empty[gi % kStages]);
                    // in issue order: QK(gi + 2) overwrites SP[u] after PV(gi) has read P(gi)
                    if (qmore && !issue_qk()) {
                        ok = false;
                        break;
                    }
                }
                gt += ntiles;
                ++nq;
            }
            if (issued_any) mma_commit(&bar->mma_done);
        }
    } else if (warp >= 8) {
        // ------------------------------------------------- exchange warpgroup
        // Thread h: row h of each item's latent query into its TMEM lane, then
        // row h of S_c of every tile to the peer's receive slot.
        const int h = tid - 256;
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        const float scale2x = p.sm_scale * kLog2eF;
        const uint32_t peer_slots = map_to_cta(slots, peer);
        const uint32_t peer_xfull = map_to_cta(&bar->xfull[0][0], peer);  // (u, g2)'s is 8 (2u + g2) bytes further
        int gt = 0, nq = 0, nbox = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const Work w = work_at(k);
            if (w.idx == -2) break;
            const int ntiles = w.idx >= 0 ? tiles_of(w.span) : 0;
            if (ntiles == 0) continue;
            // Q_c's latent columns [256c, 256c + 256) into tensor memory once
            // the previous item's last score product has read the old ones, a
            // half at a time from the staging area: two 128-byte-swizzled
            // boxes of [128 heads x 64 columns] (row h of box jj at qstage +
            // jj*16384 + h*128, 16-byte chunk k at position k ^ (h % 8)); TMEM
            // columns [16gq, 16gq + 16) are chunks 4gq .. 4gq + 3 of the row
            if (nq > 0 && !__all_sync(kAll, mbar_wait(&bar->q_empty, (nq - 1) & 1, status, kStatusTimeout, abort)))
                break;
            for (int half = 0; half < 2; ++half) {
                if (!__all_sync(kAll, mbar_wait(&bar->qstage_full, nbox & 1, status, kStatusTimeout, abort))) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t w[16];
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const uint4 x = *reinterpret_cast<const uint4*>(qstage + (j >> 1) * 128 * 128 + h * 128 +
                                                                        (((4 * (j & 1) + v) ^ (h & 7)) << 4));
                        w[4 * v] = x.x;
                        w[4 * v + 1] = x.y;
                        w[4 * v + 2] = x.z;
                        w[4 * v + 3] = x.w;
                    }
                    tmem_st16(tmem + kColQ + lane_off + 16 * (4 * half + j), w);
                }
                fence_proxy_async_smem();  // the staging reads come before the next copy into the area
                mbar_arrive(&bar->qstage_free);
                ++nbox;
            }
            if (!ok) break;
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bar->q_full);
            for (int i = 0; i < ntiles; ++i) {
                const int gi = gt + i, u = gi & 1;
                if (!__all_sync(kAll, mbar_wait(&bar->s_full[u], (gi >> 1) & 1, status, kStatusTimeout, abort))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // the row in log2 units, rounded to fp16 (saturating, NaN kept)
                // in token pairs, once for both CTAs' softmaxes: the second
                // half's loads are in flight while the first half converts and
                // goes to the peer (group q of 8 tokens to the peer's slot u at
                // offset (q * 128 + h) * 16)
                uint32_t hv[2][16];
                uint32_t ra[2][16], rb[2][16];
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) tmem_ld16(tmem + kColSP + 64 * u + lane_off + 16 * q2, ra[q2]);
                tmem_wait_ld();
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) pin(ra[q2]);
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) tmem_ld16(tmem + kColSP + 64 * u + lane_off + 32 + 16 * q2, rb[q2]);
                auto convert = [&](const uint32_t (&r)[2][16], uint32_t (&out)[16]) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float2 x = mul_f32x2(make_float2(__uint_as_float(r[j >> 3][2 * (j & 7)]),
                                                               __uint_as_float(r[j >> 3][2 * (j & 7) + 1])),
                                                   make_float2(scale2x, scale2x));
                        out[j] = f16x2_satfinite(x.x, x.y);
                    }
                };
                const uint32_t dst = peer_slots + (uint32_t)(u * kXbufBytes + h * 16);
                // token groups 4 g2 .. 4 g2 + 3: the half the peer's warpgroup g2
                // reads, counted on its own barrier
                auto send = [&](int g2) {
                    const uint32_t xb = peer_xfull + 8u * (2u * (uint32_t)u + (uint32_t)g2);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        st_async_v4(dst + (4 * g2 + q) * 128 * 16,
                                    make_float4(__uint_as_float(hv[g2][4 * q]), __uint_as_float(hv[g2][4 * q + 1]),
                                                __uint_as_float(hv[g2][4 * q + 2]), __uint_as_float(hv[g2][4 * q + 3])),
                                    xb);
                };
                convert(ra, hv[0]);
                // the peer grants slot u once it has consumed the message before
                if (!__all_sync(kAll, mbar_wait<true>(&bar->credit[u], (gi >> 1) & 1, status, kStatusTimeout, abort))) {
                    tmem_wait_ld();  // no load left in flight
                    ok = false;
                    break;
                }
                if (h == 0) mbar_arrive_expect_tx(&bar->credit[u], 4);  // arm the slot's next grant
                // pairs [16 g2, 16 g2 + 16) (tokens [32 g2, 32 g2 + 32)) into
                // SP[u] columns [32 + 16 g2, 48 + 16 g2) for this CTA's
                // warpgroup g2, over scores this thread has read
                auto keep = [&](int g2) {
                    tmem_st16(tmem + kColSP + 64 * u + 32 + 16 * g2 + lane_off, hv[g2]);
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar->own_full[u][g2]);
                };
                send(0);
                tmem_wait_ld();  // the second half is read before the first half's pairs go over it
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) pin(rb[q2]);
                keep(0);
                convert(rb, hv[1]);
                send(1);
                keep(1);
            }
            gt += ntiles;
            ++nq;
        }
    } else {
        // ------------------------------------------- softmax, two warpgroups
        // Thread (h, g): head h = TMEM lane h (warp w reaches lanes 32 (w % 4)
        // onwards), token half g = w / 4 of every tile (S columns [32g, 32g +
        // 32), P columns [16g, 16g + 16)), output columns [128g, 128g + 128).
        const int h = tid & 127, g = tid >> 7;
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t peer_credit = map_to_cta(&bar->credit[0], peer);   // slot u's is 8u bytes further
        const uint32_t peer_cword = map_to_cta(&bar->credit_word[0], peer);
        if (tid == 0) {  // both receive slots start free: grant them to the peer
            st_async_b32(peer_cword, 1u, peer_credit);
            st_async_b32(peer_cword + 4u, 1u, peer_credit + 8u);
        }
        const bool live = h < p.H;
        int nfull = 0;  // the pair's items with tokens
        for (int k = 0;; ++k) {
            const Work w = work_at(k);
            if (w.idx == -2) break;
            if (w.idx >= 0 && w.span > 0) ++nfull;
        }
        int gt = 0, gr = 0, nq = 0;  // tiles, uses of the row exchange, items with tokens: before
        // one use of the row exchange between the two warpgroups: this
        // thread's value in, the other warpgroup's for the same head out
        auto exchange_row = [&](float mine, float& other) -> bool {
            if (gr > 0 && !__all_sync(kAll, mbar_wait(&bar->red_free, (gr - 1) & 1, status, kStatusTimeout, abort)))
                return false;
            bar->red[g][h] = mine;
            mbar_arrive(&bar->red_full);
            if (!__all_sync(kAll, mbar_wait(&bar->red_full, gr & 1, status, kStatusTimeout, abort))) return false;
            other = bar->red[g ^ 1][h];
            mbar_arrive(&bar->red_free);
            ++gr;
            return true;
        };
        // tcgen05.ld / st are warp-collective: every wait's outcome is made
        // warp-uniform so that the lanes of a warp leave the loops together
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const Work w = work_at(k);
            if (w.idx == -2) break;
            if (w.idx < 0) continue;
            const int ntiles = tiles_of(w.span), span = w.span;
            const Item it = item_of(w.idx);
            if (ntiles == 0) {
                // no token of this item: a single split writes the neutral
                // (0, -inf) for its rows; with several splits the merge never
                // reads an empty split's rows
                if (p.nsplit == 1 && live) {
                    uint4* orow = reinterpret_cast<uint4*>(p.o + (int64_t)it.r * p.o_sn + (int64_t)it.b * p.o_sb +
                                                           (int64_t)h * p.o_sh + 2 * (256 * c + 128 * g));
#pragma unroll
                    for (int e = 0; e < 16; ++e) orow[e] = make_uint4(0u, 0u, 0u, 0u);
                    if (c == 0 && g == 0)
                        p.lse[(int64_t)it.r * p.l_sn + (int64_t)it.b * p.l_sb + (int64_t)h * p.l_sh] = -INFINITY;
                }
                continue;
            }
            float m_used = -INFINITY, l = 0.f;
            for (int i = 0; i < ntiles; ++i) {
                const int gi = gt + i, u = gi & 1;
                // the own partial scores of this thread's tokens, as the
                // exchange warpgroup rounded them (fp16 pairs in SP[u]
                // columns [32 + 16g, 48 + 16g)), the peer's from slot u
                if (!__all_sync(kAll, mbar_wait(&bar->own_full[u][g], (gi >> 1) & 1, status, kStatusTimeout, abort))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t own[16];
                tmem_ld16(tmem + kColSP + 64 * u + 32 + 16 * g + lane_off, own);
                tmem_wait_ld();
                pin(own);
                if (!__all_sync(kAll, mbar_wait<true>(&bar->xfull[u][g], (gi >> 1) & 1, status, kStatusTimeout, abort))) {
                    ok = false;
                    break;
                }
                // the peer's half of this thread's tokens: groups 4g .. 4g + 3 of 8
                const uint4* xin = reinterpret_cast<const uint4*>(slots + u * kXbufBytes) + 4 * g * 128;
                const int valid = span - i * kTileTokens - kHalf * g;  // tokens of this half in the split
                float s[kHalf];
#pragma unroll
                for (int q8 = 0; q8 < kHalf / 8; ++q8) {
                    const uint4 o4 = xin[q8 * 128 + h];
                    const uint32_t ow[4] = {o4.x, o4.y, o4.z, o4.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        // both partial scores in log2 units rounded to fp16
                        // alike, added with one rounding to fp32 (commutative:
                        // the same bits in both CTAs)
                        const float2 sum = add_f16x2_exact(own[4 * q8 + q], ow[q]);
                        s[8 * q8 + 2 * q] = sum.x;
                        s[8 * q8 + 2 * q + 1] = sum.y;
                    }
                }
                if (valid < kHalf) {  // the split ends inside this half
#pragma unroll
                    for (int t = 0; t < kHalf; ++t) s[t] = t < valid ? s[t] : -INFINITY;
                }
                float mt = -INFINITY;
#pragma unroll
                for (int t = 0; t < kHalf; t += 2) mt = fmax3(mt, s[t], s[t + 1]);
                // the row max of the whole tile: this thread's half and the
                // other warpgroup's
                float mt_other;
                if (!exchange_row(mt, mt_other)) {
                    ok = false;
                    break;
                }
                const float mt_all = fmaxf(mt, mt_other);
                if (tid == 0) {
                    // every softmax thread has read slot u (before its red_full
                    // arrival): re-arm it for tile gi + 2 and grant it back to the peer
                    mbar_arrive_expect_tx(&bar->xfull[u][0], kXbufBytes / 2);
                    mbar_arrive_expect_tx(&bar->xfull[u][1], kXbufBytes / 2);
                    st_async_b32(peer_cword + 4u * (uint32_t)u, 1u, peer_credit + 8u * (uint32_t)u);
                }
                const float m_new = fmaxf(m_used, mt_all);
                const bool move = m_new > m_used + kRescaleLog2 || (m_used == -INFINITY && m_new > -INFINITY);
                if (valid < kHalf) {
                    // rows past the split's last token were loaded from the cache
                    // as they are (stale values, possibly NaN): zero their value
                    // columns so that 0-probability rows add exactly 0
                    uint8_t* rows0 = stages + (gi % kStages) * kStageBytes + kHalf * g * 128;
                    const int first = valid < 0 ? 0 : valid, rows = kHalf - first;
                    for (int e = h; e < 4 * rows * 8; e += 128) {
                        const int chunk = e / (rows * 8), rem = e % (rows * 8);
                        const int row = first + rem / 8, v16 = rem % 8;
                        *reinterpret_cast<uint4*>(rows0 + chunk * kChunkBytes + row * 128 + v16 * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
                float alpha = 1.f;
                if (move) {
                    alpha = m_used == -INFINITY ? 0.f : exp2f(m_used - m_new);
                    l *= alpha;
                    m_used = m_new;
                }
                if (i > 0 && __any_sync(kAll, move)) {
                    // rescale this thread's 128 columns of O row h (alpha = 1 for
                    // rows that keep their max) once P.V of tile gi - 1 has completed
                    if (!__all_sync(kAll, mbar_wait(&bar->pv_done[u ^ 1], ((gi - 1) >> 1) & 1, status, kStatusTimeout,
                                                    abort))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int q16 = 0; q16 < 8; ++q16) {
                        uint32_t v[16];
                        tmem_ld16(tmem + kColO + 128 * g + lane_off + 16 * q16, v);
                        tmem_wait_ld();
                        pin(v);
#pragma unroll
                        for (int q = 0; q < 16; ++q) v[q] = __float_as_uint(__uint_as_float(v[q]) * alpha);
                        tmem_st16(tmem + kColO + 128 * g + lane_off + 16 * q16, v);
                    }
                }
                // P = 2^(s - m) in the payload type into SP[u] columns [16g, 16g +
                // 16), over scores the exchange warpgroup has read (own_full)
                const float msub = m_used == -INFINITY ? 0.f : m_used;
                {
                    // in pairs: s - m and the running sum two lanes wide
                    uint32_t w[16];
                    float2 l2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const float2 x = add_f32x2(make_float2(s[2 * q], s[2 * q + 1]), make_float2(-msub, -msub));
                        const float2 pp = make_float2(exp2_approx(x.x), exp2_approx(x.y));
                        l2 = add_f32x2(l2, pp);
                        w[q] = pack_pair<T>(pp.x, pp.y);
                    }
                    l += l2.x + l2.y;
                    tmem_st16(tmem + kColSP + 64 * u + 16 * g + lane_off, w);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar->p_full[u]);
            }
            if (!ok) break;
            // ------------------------------------------------------- epilogue
            // the row sum is the two warpgroups' partial sums (both relative
            // to the same reference max), added in a fixed order
            const int glast = gt + ntiles - 1;
            float l_other;
            if (!__all_sync(kAll, mbar_wait(&bar->pv_done[glast & 1], (glast >> 1) & 1, status, kStatusTimeout,
                                            abort)) ||
                !exchange_row(l, l_other))
                break;
            tc_fence_after();
            const float l_all = g == 0 ? l + l_other : l_other + l;
            // a row with no probability mass writes 0
            const bool mass = l_all > 0.f;
            const float inv = mass ? 1.f / l_all : 0.f;
            const float lse2 = mass ? m_used + log2f(l_all) : -INFINITY;
            // the staging area holds the next item's query until that has
            // moved to tensor memory
            const bool more = nq + 1 < nfull;
            if (more && !__all_sync(kAll, mbar_wait(&bar->q_full, (nq + 1) & 1, status, kStatusTimeout, abort))) break;
            // O columns [128g + 16k0, 128g + 16k0 + 32) of this thread's row
            auto load_o2 = [&](int k0, uint32_t (&v)[2][16]) {
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) tmem_ld16(tmem + kColO + 128 * g + lane_off + 16 * (k0 + q2), v[q2]);
                tmem_wait_ld();
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) pin(v[q2]);
            };
            // every column of O read: the next item's P.V may start
            auto release_o = [&]() {
                tc_fence_before();
                mbar_arrive(&bar->o_free);
            };
            // The rows go out through the staging area: a thread holds one
            // head's row, so its own stores would put each warp store across
            // 32 rows; each softmax warp instead writes 128 bytes of each of
            // its 32 rows (64 payload columns, or 32 fp32 partials) into its 4
            // KB and stores them back row by row, coalesced.  16-byte piece cc
            // of row rr sits at rr * 128 + ((cc ^ (rr % 8)) * 16).
            uint8_t* stg = qstage + warp * 4096;
            const int h0 = 32 * (warp & 3);  // the warp's first head
            // 128-byte piece x of each of the warp's rows to row0 + x * 128,
            // row0 being this lane's first row (head h0 + lane / 8), rows
            // rstride bytes apart
            auto flush = [&](unsigned char* row0, int64_t rstride, int x) {
                __syncwarp();
#pragma unroll 2
                for (int j = 0; j < 8; ++j) {  // 4 rows of 128 bytes a store
                    const int rr = 4 * j + (lane >> 3), cc = lane & 7;
                    const uint4 xv = *reinterpret_cast<const uint4*>(stg + rr * 128 + ((cc ^ (rr & 7)) << 4));
                    if (h0 + rr < p.H) *reinterpret_cast<uint4*>(row0 + 4 * j * rstride + x * 128 + 16 * cc) = xv;
                }
                __syncwarp();
            };
            if (p.nsplit == 1) {
                unsigned char* orow = p.o + (int64_t)it.r * p.o_sn + (int64_t)it.b * p.o_sb +
                                      (int64_t)(h0 + (lane >> 3)) * p.o_sh + 2 * (256 * c + 128 * g);
                for (int x = 0; x < 2; ++x) {  // 64 columns a pass, in two loads of 32
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t v[2][16];
                        load_o2(4 * x + 2 * hh, v);
                        if (x == 1 && hh == 1) release_o();
#pragma unroll
                        for (int q2 = 0; q2 < 2; ++q2) {
                            uint32_t w[8];
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                w[q] = pack_pair<T>(__uint_as_float(v[q2][2 * q]) * inv,
                                                    __uint_as_float(v[q2][2 * q + 1]) * inv);
#pragma unroll
                            for (int e = 0; e < 2; ++e)
                                *reinterpret_cast<uint4*>(stg + lane * 128 +
                                                          (((2 * (2 * hh + q2) + e) ^ (lane & 7)) << 4)) =
                                    make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
                        }
                    }
                    flush(orow, p.o_sh, x);
                }
                if (live && c == 0 && g == 0)
                    p.lse[(int64_t)it.r * p.l_sn + (int64_t)it.b * p.l_sb + (int64_t)h * p.l_sh] =
                        p.base2 ? lse2 : lse2 * kLn2F;
            } else {
                unsigned char* wrow = reinterpret_cast<unsigned char*>(
                    p.ws_o + ((((int64_t)it.r * p.B + it.b) * p.H + h0 + (lane >> 3)) * p.nsplit + it.split) * 512 +
                    256 * c + 128 * g);
                for (int x = 0; x < 4; ++x) {  // 32 fp32 columns (128 bytes) a pass
                    uint32_t v[2][16];
                    load_o2(2 * x, v);
                    if (x == 3) release_o();
#pragma unroll
                    for (int q2 = 0; q2 < 2; ++q2)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            *reinterpret_cast<float4*>(stg + lane * 128 + (((4 * q2 + e) ^ (lane & 7)) << 4)) =
                                make_float4(__uint_as_float(v[q2][4 * e]) * inv, __uint_as_float(v[q2][4 * e + 1]) * inv,
                                            __uint_as_float(v[q2][4 * e + 2]) * inv,
                                            __uint_as_float(v[q2][4 * e + 3]) * inv);
                    flush(wrow, (int64_t)p.nsplit * 512 * 4, x);
                }
                if (live && c == 0 && g == 0)
                    p.ws_lse[(((int64_t)it.r * p.B + it.b) * p.H + h) * p.nsplit + it.split] = lse2;
            }
            // the staging area is free again for the query after next
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar->stg_free);
            gt += ntiles;
            ++nq;
        }
    }

    // --------------------------------------------------------------- teardown
    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    if (warp == 13) {
        if (lane == 0 && issued_any) {
            // every MMA this CTA issued has completed before its tensor memory goes
            const uint64_t t_start = global_timer_ns();
            while (!mbar_try_wait(&bar->mma_done, 0) && global_timer_ns() - t_start < kWaitLimitNs) {
            }
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    cluster_sync();  // no CTA leaves while its peer may still write its shared memory
}

// Merge of the split partials (fp32, normalised, base-2 LSE) of every
// (rank, request, head): one warp per row, with the combine's LSE rule.  Only
// the splits that hold tokens of the rank were written; the empty ones are
// the neutral (0, -inf) and drop out, so they are not read.
template <typename T>
__global__ void __launch_bounds__(128) mla_merge_splits_kernel(const MlaParams p) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t rows = (int64_t)p.N * p.B * p.H;
    const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int h = (int)(row % p.H);
    const int64_t rbq = row / p.H;
    const int b = (int)(rbq % p.B);
    const int r = (int)(rbq / p.B);
    int L = p.seq_lens[b];
    L = L < 0 ? 0 : (L > p.max_seq_len ? p.max_seq_len : L);
    const int Ll = L / p.N + (r < L % p.N ? 1 : 0);
    const int S = min(p.nsplit, (Ll + p.split_tokens - 1) / p.split_tokens);
    const float* lrow = p.ws_lse + row * p.nsplit;
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, lrow[s]);
    float Ls = 0.f;
    float4 acc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
        for (int s = 0; s < S; ++s) {
            const float w = exp2f(lrow[s] - M);
            Ls += w;
            const float4* orow = reinterpret_cast<const float4*>(p.ws_o + (row * p.nsplit + s) * 512);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 v = orow[lane + 32 * k];
                acc[k].x = fmaf(w, v.x, acc[k].x);
                acc[k].y = fmaf(w, v.y, acc[k].y);
                acc[k].z = fmaf(w, v.z, acc[k].z);
                acc[k].w = fmaf(w, v.w, acc[k].w);
            }
        }
    }
    unsigned char* orow = p.o + (int64_t)r * p.o_sn + (int64_t)b * p.o_sb + (int64_t)h * p.o_sh;
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint2 w = make_uint2(pack_pair<T>(acc[k].x * inv, acc[k].y * inv), pack_pair<T>(acc[k].z * inv, acc[k].w * inv));
        *reinterpret_cast<uint2*>(orow + 8 * (lane + 32 * k)) = w;
    }
    if (lane == 0) {
        const float lse2 = Ls > 0.f ? M + log2f(Ls) : -INFINITY;
        p.lse[(int64_t)r * p.l_sn + (int64_t)b * p.l_sb + (int64_t)h * p.l_sh] = p.base2 ? lse2 : lse2 * kLn2F;
    }
    pdl_trigger();
}

// CTA pairs of the kernel that fit on the device at once (one per two SMs),
// per device; 0 if the occupancy query fails
template <typename T>
int resident_pairs() {
    static int cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kMlaThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (const void*)mla_decode_kernel<T>, &cfg) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        return 0;
    }
    if (dev >= 0 && dev < 64) cached[dev] = n;
    return n;
}

template <typename T>
cudaError_t launch_mla_t(const MlaParams& p, const CUtensorMap (&maps)[4], cudaStream_t stream) {
    // the shared-memory opt-in is a per-device function attribute
    const cudaError_t attr_err =
        cudaFuncSetAttribute((const void*)mla_decode_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (attr_err != cudaSuccess) return attr_err;
    const int64_t items = (int64_t)p.N * p.B * p.nsplit;
    if (items <= 0) return cudaSuccess;
    // persistent: as many CTA pairs as fit at once (each takes its share of
    // the items in turn), never more than there are items
    const int fit = resident_pairs<T>();
    if (fit <= 0) return cudaErrorLaunchOutOfResources;
    const int64_t pairs = items < fit ? items : fit;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    cfg.blockDim = dim3(kMlaThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = DCP_PDL ? 2 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, mla_decode_kernel<T>, maps[0], maps[1], maps[2], maps[3], p);
    if (e != cudaSuccess || p.nsplit == 1) return e;
    const int64_t rows = (int64_t)p.N * p.B * p.H;
    MlaParams q = p;
    void* args[] = {(void*)&q};
    return launch_pdl((const void*)mla_merge_splits_kernel<T>, dim3((unsigned)((rows + 3) / 4)), dim3(128), args, 0,
                      stream);
}

}  // namespace

cudaError_t launch_mla_decode(const MlaParams& p_in, int dtype, cudaStream_t stream) {
    MlaParams p = p_in;
    // DCP_TEST_STALL_LOADS=1 (tests of the failure path only): the kernel
    // issues none of its latent-row loads, so its first wait on them runs
    // out; it must then record DCP_ERR_TIMEOUT and end, leaving the context
    // usable.  Read per call; unset in normal use.
    const char* stall = getenv("DCP_TEST_STALL_LOADS");
    p.stall_loads = stall && stall[0] == '1';
    const EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const CUtensorMapDataType dt = dtype == DCP_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    // a dimension of extent 1 is never stepped over: give it a nominal stride
    auto stride = [](int64_t extent, int64_t bytes, int64_t nominal) -> cuuint64_t {
        return (cuuint64_t)(extent > 1 ? bytes : nominal);
    };
    // the latent cache as a 4-D tensor [N][B][Lc][576] (elements, then byte
    // strides): latent boxes of [64 tokens x 64 columns], 128-byte swizzled,
    // and rope boxes of [64 tokens x 32 columns], 64-byte swizzled
    CUtensorMap maps[4];  // latent rows, rope columns of the rows, query, rope columns of the query
    const int64_t lc = p.lcap > 0 ? p.lcap : 1;
    const cuuint64_t dims[4] = {576, (cuuint64_t)lc, (cuuint64_t)p.B, (cuuint64_t)p.N};
    const cuuint64_t strides[3] = {stride(lc, p.kv_st, 1152), stride(p.B, p.kv_sb, 1152), stride(p.N, p.kv_sn, 1152)};
    const cuuint32_t box[4] = {64, kTileTokens, 1, 1};
    const cuuint32_t rbox[4] = {32, kTileTokens, 1, 1};
    // the absorbed queries as a 3-D tensor [B][H][576]: boxes of 128 heads
    // (rows past H read 0) by 64 latent / 32 rope columns
    const cuuint64_t qdims[3] = {576, (cuuint64_t)p.H, (cuuint64_t)p.B};
    const cuuint64_t qstrides[2] = {stride(p.H, p.q_sh, 1152), stride(p.B, p.q_sb, 1152)};
    const cuuint32_t qbox[3] = {64, 128, 1};
    const cuuint32_t qrbox[3] = {32, 128, 1};
    void* kv = const_cast<unsigned char*>(p.kv);
    void* q = const_cast<unsigned char*>(p.q);
    const CUresult rc[4] = {
        enc(&maps[0], dt, 4, kv, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE),
        enc(&maps[1], dt, 4, kv, dims, strides, rbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE),
        enc(&maps[2], dt, 3, q, qdims, qstrides, qbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE),
        enc(&maps[3], dt, 3, q, qdims, qstrides, qrbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE)};
    for (const CUresult r : rc)
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    return dtype == DCP_F16 ? launch_mla_t<__half>(p, maps, stream) : launch_mla_t<__nv_bfloat16>(p, maps, stream);
}

int mla_device_status(bool clear) {
    int s = 0;
    if (cudaMemcpyFromSymbol(&s, g_mla_status, sizeof(int)) != cudaSuccess) return -1;
    if (clear && s) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_mla_status, &zero, sizeof(int)) != cudaSuccess) return -1;
    }
    return s;
}

}  // namespace dcp
