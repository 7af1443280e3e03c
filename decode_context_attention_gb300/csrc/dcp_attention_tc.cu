// dcp_attention_tc.cu -- grouped-query decode attention of every DCP rank on
// the 5th-generation tensor cores: D = 128, 2 to 16 query heads per KV head,
// contiguous or paged KV caches.
//
// sglang PR #33926 report, "实现拆解" items 1, 3-4 and "关键源码片段": token t
// of a request lives on rank t % N, so rank r holds L / N tokens plus one
// when r < L % N (`get_dcp_lens`); the page table of a rank covers its own
// round-robin slice (`_fill_dcp_block_kv_indices`); each rank returns
// rank-local (out, lse), a rank owning no token being (0, -inf)
// (`fixup_zero_kv_rows`).  Per (rank r, request b, query head h), with
// s_t = sm_scale <q_h, k_t> over the rank's tokens:
//     lse = log sum_t exp(s_t),   O_h = sum_t exp(s_t - lse) v_t.
//
// Design.  The G query heads of one KV head are too few to be the M of an
// MMA (64 or 128 rows), so both products run transposed, the tokens or the
// head dimension on M and the heads on N (zero-padded to 16 or 32):
//     S^T [128 tokens x 16]  = K_tile [128 x 128 d] . Q^T [128 d x 16]
//     O^T [128 d x 2G]      += V_tile^T [128 d x 128 tokens] . P^T [128 x 2G]
// where the 2G columns of P^T are each probability split into two 16-bit
// terms, P = P_hi + P_lo (P_hi = P rounded to the payload type, P_lo = the
// rest rounded again), so P enters the product with about 16 significant
// bits instead of 8; O = O^T[:, h] + O^T[:, G + h].  The extra columns cost
// no MMA: N = 16 holds them up to G = 8.
// One CTA per (rank, request, KV head, split), two CTAs per SM:
//   * one thread issues TMA loads of the K and V tiles (128 tokens x 128 d,
//     two 64-column boxes, 128-byte swizzled) into a ring of three slots, K
//     and V of a tile taking a slot each; a paged cache is read box by box
//     along the pages (page_size >= 8), a page index outside the pool
//     becoming an out-of-range coordinate that the copy fills with zeros;
//   * one thread issues the MMAs: K is the K-major A operand of the score
//     product, the query the K-major B operand, S^T lands in tensor memory;
//     the same V tile is the MN-major A operand of the output product, P^T
//     (written to shared memory by the softmax warps) its K-major B operand,
//     O^T accumulates in tensor memory over the split's tiles;
//   * four softmax warps, thread = token row of S^T: the tile's maximum per
//     head (a warp-wide integer max over order-preserving keys, then across
//     the four warps through shared memory), an online softmax in base 2 with
//     a lazily moved reference max (O^T is rescaled only when the max grows
//     by more than 2^8), P as P_hi + P_lo; rows past the split's end are
//     masked, and their V rows zeroed in shared memory before the product;
//   * at the end the same warps (thread = row d of O^T) normalise and write
//     (O_r, lse_r), or with several splits fp32 partials that the split merge
//     of the other attention kernels combines.
// Every barrier wait is bounded (1 s): a wait that runs out records
// DCP_ERR_TIMEOUT in a device status word and the kernel winds down (copies
// and MMAs in flight are waited for, tensor memory freed) instead of hanging.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdlib.h>

#include <type_traits>

#include "dcp_device.cuh"
#include "dcp_sm100.cuh"

#ifndef DCP_ATTN_TC
#define DCP_ATTN_TC 1
#endif

namespace dcp {

using namespace sm100;

namespace {

constexpr int kD = 128;                   // head dimension this kernel takes
constexpr int kTT = 128;                  // tokens per tile: the M of the score product
constexpr int kN = 16;                    // the MMAs' N: query heads, zero-padded
constexpr int kThreads = 192;             // warp 0 TMA, warp 1 MMA, warps 2-5 softmax
constexpr int kChunk = kTT * 128;         // one 64-column box of a tile: 128 rows x 128 bytes
constexpr int kSlotBytes = 2 * kChunk;    // a K or a V tile
#ifndef DCP_TC_SLOTS
#define DCP_TC_SLOTS 3
#endif
constexpr int kSlots = DCP_TC_SLOTS;      // 3: two CTAs per SM
constexpr int kOpBytes = 2 * kN * 128;    // Q^T: two 64-element chunks of 16 rows x 128 bytes
constexpr int kPBufBytes = 8192;          // the P^T buffers (two of 16 rows, or one of 32)
constexpr int kMiscBytes = 1024;
constexpr int kSmemBytes = kSlots * kSlotBytes + kOpBytes + kPBufBytes + kMiscBytes + 1024 /* align */;
constexpr uint32_t kColS = 0;   // two score buffers of 16 columns
constexpr uint32_t kColO = 32;  // O^T: 16 or 32 columns
constexpr uint32_t kTmemCols = 64;
constexpr float kRescaleLog2 = 8.f;
constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kLn2F = 0.6931471805599453f;

enum : int { kStatusTimeout = DCP_ERR_TIMEOUT };

__device__ int g_tc_status;  // first bounded wait that ran out (0 if none)

struct Barriers {
    uint64_t full[kSlots], empty[kSlots];  // the ring: copies landed / MMAs done reading
    uint64_t q_full;                        // Q^T (and the zero padding of P^T) written
    uint64_t s_full[2], p_full[2], pv_done[2];
    uint64_t red_full[2];                   // the softmax warps' tile maxima written
    uint64_t sum_full;                      // their final row sums written
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
    float red[2][4][kN];
    float sum[4][kN];
};
static_assert(sizeof(Barriers) <= kMiscBytes, "misc region too small");

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

// A float rounded to the payload type, as its 16 bits; and back.
template <typename T>
__device__ __forceinline__ uint32_t to_bits16(float x) {
    if constexpr (std::is_same<T, __half>::value) return __half_as_ushort(__float2half_rn(x));
    else return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
template <typename T>
__device__ __forceinline__ float from_bits16(uint32_t b) {
    if constexpr (std::is_same<T, __half>::value) return __half2float(__ushort_as_half((unsigned short)b));
    else return __bfloat162float(__ushort_as_bfloat16((unsigned short)b));
}

// An int whose signed order is the float order (for -inf and finite values):
// the warp's maximum then takes one redux instruction.
__device__ __forceinline__ int order_key(float f) {
    const int b = __float_as_int(f);
    return b ^ ((b >> 31) & 0x7fffffff);
}
__device__ __forceinline__ float from_order_key(int k) { return __int_as_float(k ^ ((k >> 31) & 0x7fffffff)); }

// Byte offset of element (row n, column k) of a K-major operand made of
// 64-column chunks of `chunk` bytes (rows x 128 bytes), 128-byte swizzled.
__device__ __forceinline__ int op_offset(int n, int k, int chunk) {
    return (k >> 6) * chunk + n * 128 + ((((k & 63) >> 3) ^ (n & 7)) << 4) + ((k & 7) << 1);
}

// The ring holds the operand tiles in the order the MMAs take them: K(0),
// then K(i + 1) and V(i) for each tile i (K runs a tile ahead of V), so the
// slot of K(i + 2) is the one V(i - 1) frees and its copy has a whole tile
// of softmax and products to land in.  Position of each in that order:
__device__ __forceinline__ int pos_k(int i) { return i == 0 ? 0 : 2 * i - 1; }
__device__ __forceinline__ int pos_v(int i, int ntiles) { return i < ntiles - 1 ? 2 * i + 2 : 2 * ntiles - 1; }

// Roles and the flow of tile i (buffer u = i % 2; the operand at ring
// position j sits in slot j % kSlots):
//   TMA      full[slot] <- K(i + 1), then V(i)
//   MMA      QK(i) -> S[u] (s_full[u], empty[K slot]); after P(i):
//            PV(i) (pv_done[u], empty[V slot]), then QK(i + 2) into S[u]
//   softmax  S(i) -> P^T (p_full[u]) once the product that last read its
//            buffer (PV(i - 2), or PV(i - 1) with one buffer) has completed
template <typename T, int GQ, bool PAGED>
__global__ void __launch_bounds__(kThreads, 2)
    gqa_decode_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                         const AttnParams p) {
    static_assert(GQ >= 2 && GQ <= kN && GQ % 2 == 0, "query heads per KV head");
    constexpr int NPV = GQ <= 8 ? 16 : 32;     // N of the output product: P_hi rows [0, G), P_lo [G, 2G)
    constexpr int PCHUNK = NPV * 128;          // one 64-token chunk of P^T
    constexpr int PBYTES = 2 * PCHUNK;         // a P^T buffer
    constexpr int NPBUF = kPBufBytes / PBYTES; // two buffers up to G = 8, one at G = 16
    static_assert(NPBUF >= 1 && NPBUF * PBYTES == kPBufBytes, "P^T buffers");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* slots = smem;
    uint8_t* qs = smem + kSlots * kSlotBytes;  // Q^T
    uint8_t* ps = qs + kOpBytes;               // the P^T buffers
    Barriers* bar = reinterpret_cast<Barriers*>(ps + kPBufBytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int item = (int)(blockIdx.x / (unsigned)p.nsplit);  // splits of one item are neighbours
    const int split = (int)(blockIdx.x % (unsigned)p.nsplit);
    const int hkv = item % p.Hkv;
    const int rb = item / p.Hkv;
    const int b = rb % p.B;
    const int r = rb / p.B;
#if !DCP_PDL
    const int Lraw = p.seq_lens[b];  // in flight during the set-up below
#endif

    if (tid == 0) {
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&bar->full[s], 1);
            mbar_init(&bar->empty[s], 1);
        }
        mbar_init(&bar->q_full, 128);
        for (int u = 0; u < 2; ++u) {
            mbar_init(&bar->s_full[u], 1);
            mbar_init(&bar->p_full[u], 4);
            mbar_init(&bar->pv_done[u], 1);
            mbar_init(&bar->red_full[u], 4);
        }
        mbar_init(&bar->sum_full, 4);
        mbar_init(&bar->mma_done, 1);
        bar->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&bar->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&kmap);
        tma_prefetch_map(&vmap);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();
#if DCP_PDL
    const int Lraw = p.seq_lens[b];
#endif
    const int L = Lraw < 0 ? 0 : (Lraw > p.max_seq_len ? p.max_seq_len : Lraw);
    const int Ll = L / p.N + (r < L % p.N ? 1 : 0);
    const int t0 = split * p.split_tokens;
    const int t1 = min(t0 + p.split_tokens, Ll);
    const int ntiles = t1 > t0 ? (t1 - t0 + kTT - 1) / kTT : 0;
    // splits of this (rank, request) that hold tokens: with at most one the
    // result goes straight to the outputs (from split 0), else fp32 partials
    // of the non-empty splits go to the workspace for the split merge
    const int nse = (Ll + p.split_tokens - 1) / p.split_tokens;
    const bool direct = p.nsplit == 1 || nse <= 1;
    const uint32_t tmem = bar->tmem_base;
    volatile int* abort = &bar->abort;
    int* status = &g_tc_status;
    bool issued_any = false;  // the MMA thread issued at least one MMA
    const unsigned kAll = 0xffffffffu;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA
        // A paged tile is read in boxes of pb rows, one per page (pb = the
        // page size up to a tile); the lanes fetch the tile's page indices.
        const int pb = PAGED ? min(1 << p.page_shift, kTT) : kTT;
        int pg_even = 0, pg_odd = 0;  // the lane's page index for the last even / odd tile whose K went
        int issued = 0;
        for (int j = 0; j < 2 * ntiles && !p.stall_loads; ++j) {
            const int s = j % kSlots, k = j / kSlots;
            // ring position j -> tile i and operand (K or V)
            const bool is_k = j == 0 || ((j & 1) && (j + 1) / 2 < ntiles);
            const int i = j == 0 ? 0 : ((j & 1) ? (is_k ? (j + 1) / 2 : ntiles - 1) : j / 2 - 1);
            const int tb = t0 + i * kTT;
            const int nseg = PAGED ? (min(kTT, t1 - tb) + pb - 1) / pb : 1;
            if constexpr (PAGED) {
                if (is_k) {  // page indices of tile i (only entries of tokens the rank holds)
                    int pg = 0;
                    if (lane < nseg) {
                        const int ts = tb + lane * pb;
                        pg = __ldg(p.bt + (int64_t)r * p.bt_sn + (int64_t)b * p.bt_sb + (ts >> p.page_shift));
                        if ((unsigned)pg >= (unsigned)p.num_pages) pg = p.num_pages;  // reads zeros
                    }
                    if (i & 1) pg_odd = pg;
                    else pg_even = pg;
                }
            }
            int go = 1;
            if (lane == 0 && k > 0) go = mbar_wait(&bar->empty[s], (k - 1) & 1, status, kStatusTimeout, abort);
            if (!__shfl_sync(kAll, go, 0)) break;
            const CUtensorMap* map = is_k ? &kmap : &vmap;
            uint8_t* dst = slots + s * kSlotBytes;
            if constexpr (!PAGED) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bar->full[s], kSlotBytes);
                    tma_load_5d(dst, map, &bar->full[s], 0, hkv, tb, b, r);
                    tma_load_5d(dst + kChunk, map, &bar->full[s], 64, hkv, tb, b, r);
                }
            } else {
                if (lane == 0) mbar_arrive_expect_tx(&bar->full[s], (uint32_t)(2 * nseg * pb * 128));
                for (int g = 0; g < nseg; ++g) {
                    const int pg = __shfl_sync(kAll, (i & 1) ? pg_odd : pg_even, g);
                    if (lane == 0) {
                        const int slot = (tb + g * pb) & ((1 << p.page_shift) - 1);
                        tma_load_5d(dst + g * pb * 128, map, &bar->full[s], 0, hkv, slot, pg, r);
                        tma_load_5d(dst + kChunk + g * pb * 128, map, &bar->full[s], 64, hkv, slot, pg, r);
                    }
                }
            }
            issued = j + 1;
        }
        // copies still in flight (only after an abort) land before the CTA ends
        if (lane == 0) {
            for (int j = max(0, issued - kSlots); j < issued; ++j) {
                const uint64_t tw = global_timer_ns();
                while (!mbar_try_wait(&bar->full[j % kSlots], (j / kSlots) & 1) &&
                       global_timer_ns() - tw < kWaitLimitNs) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr bool kBf16 = !std::is_same<T, __half>::value;
            const uint32_t idesc_qk = idesc_f16(128, kN, kBf16, 0, 0);  // K: K-major A, Q^T: K-major B
            const uint32_t idesc_pv = idesc_f16(128, NPV, kBf16, 1, 0);  // V^T: MN-major A, P^T: K-major B
            const uint32_t tO = tmem + kColO;
            const uint64_t dq = smem_desc(smem_u32(qs), 16, 1024, kSwizzle128B);
            // S^T(i) = K(i) . Q^T into buffer i % 2.  The descriptor's address
            // field is bits 0-13 in 16-byte units: offsets are added to it.
            auto issue_qk = [&](int i) -> bool {
                const int j = pos_k(i), s = j % kSlots;
                if (!mbar_wait(&bar->full[s], (j / kSlots) & 1, status, kStatusTimeout, abort)) return false;
                tc_fence_after();
                const uint32_t tS = tmem + kColS + kN * (i & 1);
                const uint64_t dk = smem_desc(smem_u32(slots + s * kSlotBytes), 16, 1024, kSwizzle128B);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {  // d in steps of 16: box kk / 4, 32 bytes a step inside it
                    const uint64_t a = dk + (uint64_t)(((kk >> 2) * kChunk + (kk & 3) * 32) >> 4);
                    const uint64_t bq = dq + (uint64_t)(((kk >> 2) * 2048 + (kk & 3) * 32) >> 4);
                    mma_ss(tS, a, bq, idesc_qk, kk > 0 ? 1u : 0u);
                }
                mma_commit(&bar->s_full[i & 1]);
                mma_commit(&bar->empty[s]);
                issued_any = true;
                return true;
            };
            bool ok = mbar_wait(&bar->q_full, 0, status, kStatusTimeout, abort);
            for (int i = 0; ok && i < ntiles && i < 2; ++i) ok = issue_qk(i);
            for (int i = 0; ok && i < ntiles; ++i) {
                // O^T += V(i)^T . P^T(i): V read MN-major from its slot (the
                // next 64 d one box further, the next 8 tokens 1024 bytes on)
                const int u = i & 1;
                const int j = pos_v(i, ntiles), s = j % kSlots;
                if (!mbar_wait(&bar->p_full[u], (i >> 1) & 1, status, kStatusTimeout, abort) ||
                    !mbar_wait(&bar->full[s], (j / kSlots) & 1, status, kStatusTimeout, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t dv = smem_desc(smem_u32(slots + s * kSlotBytes), kChunk, 1024, kSwizzle128B);
                const uint64_t dp =
                    smem_desc(smem_u32(ps + (NPBUF == 2 ? u : 0) * PBYTES), 16, 1024, kSwizzle128B);
#pragma unroll
                for (int kk = 0; kk < kTT / 16; ++kk) {  // tokens in steps of 16
                    const uint64_t a = dv + (uint64_t)((kk * 2048) >> 4);
                    const uint64_t bp = dp + (uint64_t)(((kk >> 2) * PCHUNK + (kk & 3) * 32) >> 4);
                    mma_ss(tO, a, bp, idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&bar->pv_done[u]);
                mma_commit(&bar->empty[s]);
                // in issue order: QK(i + 2) overwrites S[u], which softmax(i) has read
                if (i + 2 < ntiles && !issue_qk(i + 2)) {
                    ok = false;
                    break;
                }
            }
            if (issued_any) mma_commit(&bar->mma_done);
        }
    } else {
        // ------------------------------------------------------- softmax
        const int st = tid - 64;            // 0..127
        const int wq = warp & 3;            // TMEM lane quarter of this warp
        const int kk = 32 * wq + lane;      // token row of S^T, and row d of O^T
        const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
        // Q^T: row n = query head hkv * GQ + n (rows past GQ zero), 128-byte swizzled
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int id = st + 128 * k;  // 16-byte unit: row id / 16, unit id % 16
            const int n = id >> 4, uu = id & 15;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (n < GQ)
                v = *reinterpret_cast<const uint4*>(p.q + (int64_t)b * p.q_sb + (int64_t)(hkv * GQ + n) * p.q_sh +
                                                    16 * uu);
            *reinterpret_cast<uint4*>(qs + (uu >> 3) * 2048 + n * 128 + (((uu & 7) ^ (n & 7)) << 4)) = v;
        }
        // P^T rows past 2G stay zero in every buffer
        if constexpr (2 * GQ < NPV) {
            constexpr int pad = NPV - 2 * GQ;
            for (int id = st; id < NPBUF * 2 * pad * 8; id += 128) {
                const int unit = id & 7, row = 2 * GQ + ((id >> 3) % pad), rest = (id >> 3) / pad;
                *reinterpret_cast<uint4*>(ps + (rest >> 1) * PBYTES + (rest & 1) * PCHUNK + row * 128 + unit * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
        }
        fence_proxy_async_smem();
        mbar_arrive(&bar->q_full);

        const float qscale = p.sm_scale * kLog2eF;
        float m_run[GQ], l_part[GQ];  // reference max (the same in every thread); this token's share of the sum
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
            m_run[h] = -INFINITY;
            l_part[h] = 0.f;
        }
        bool ok = true;
        for (int i = 0; i < ntiles; ++i) {
            const int u = i & 1;
            const int tb = t0 + i * kTT;
            const bool valid = tb + kk < t1;
            if (!__all_sync(kAll, mbar_wait(&bar->s_full[u], (i >> 1) & 1, status, kStatusTimeout, abort))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t v[16];
            tmem_ld16(tmem + kColS + kN * u + lane_off, v);
            tmem_wait_ld();
            pin(v);
            // the tile's maximum of each head: over the warp, then lane h < G
            // takes head h over the four warps and hands it to every lane
            float s[GQ];
            float wmax = -INFINITY;  // lane h: this warp's maximum of head h
#pragma unroll
            for (int h = 0; h < GQ; ++h) {
                s[h] = valid ? __uint_as_float(v[h]) * qscale : -INFINITY;
                const int key = __reduce_max_sync(kAll, order_key(s[h]));
                if (lane == h) wmax = from_order_key(key);
            }
            if (lane < GQ) bar->red[u][wq][lane] = wmax;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar->red_full[u]);
            if (!__all_sync(kAll, mbar_wait(&bar->red_full[u], (i >> 1) & 1, status, kStatusTimeout, abort))) {
                ok = false;
                break;
            }
            float m4 = -INFINITY;
            if (lane < GQ)
                m4 = fmaxf(fmaxf(bar->red[u][0][lane], bar->red[u][1][lane]),
                           fmaxf(bar->red[u][2][lane], bar->red[u][3][lane]));
            float mt[GQ];
            bool grow = false;
#pragma unroll
            for (int h = 0; h < GQ; ++h) {
                mt[h] = __shfl_sync(kAll, m4, h);
                grow |= mt[h] > m_run[h] + kRescaleLog2;
            }
            if (grow) {  // every thread takes this branch together (same maxima)
                float alpha[GQ];
#pragma unroll
                for (int h = 0; h < GQ; ++h) {
                    const float mn = fmaxf(m_run[h], mt[h]);
                    alpha[h] = m_run[h] == -INFINITY ? 0.f : exp2f(m_run[h] - mn);
                    m_run[h] = mn;
                    l_part[h] *= alpha[h];
                }
                if (i > 0) {  // O^T holds P(0..i-1) . V: rescale it once PV(i - 1) has landed
                    if (!__all_sync(kAll, mbar_wait(&bar->pv_done[u ^ 1], ((i - 1) >> 1) & 1, status,
                                                    kStatusTimeout, abort))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int g = 0; g < NPV / 16; ++g) {  // column c < 2G holds head c % G (hi, then lo)
                        uint32_t o[16];
                        tmem_ld16(tmem + kColO + 16 * g + lane_off, o);
                        tmem_wait_ld();
                        pin(o);
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            if (16 * g + c < 2 * GQ)
                                o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha[(16 * g + c) % GQ]);
                        tmem_st16(tmem + kColO + 16 * g + lane_off, o);
                    }
                    tmem_wait_st();
                }
            }
            float pr[GQ];
#pragma unroll
            for (int h = 0; h < GQ; ++h) {
                pr[h] = valid && m_run[h] != -INFINITY ? exp2f(s[h] - m_run[h]) : 0.f;
                l_part[h] += pr[h];
            }
            // the P^T buffer is free once the product that last read it has completed
            const int prev = i - NPBUF;
            if (prev >= 0 && !__all_sync(kAll, mbar_wait(&bar->pv_done[prev & 1], (prev >> 1) & 1, status,
                                                          kStatusTimeout, abort))) {
                ok = false;
                break;
            }
            // this token's P^T column as 16-bit terms: row h < G is P_hi of
            // head h, row G + h its P_lo
            uint32_t t16[2 * GQ];
#pragma unroll
            for (int h = 0; h < GQ; ++h) {
                t16[h] = to_bits16<T>(pr[h]);
                t16[GQ + h] = to_bits16<T>(pr[h] - from_bits16<T>(t16[h]));
            }
            // lanes 2x and 2x + 1 hold neighbouring tokens; per store the even
            // lane writes the pair's 4 bytes of row n, the odd lane those of
            // row n ^ 4 (n ^ 1 at G = 2): under the 128-byte swizzle the two
            // rows of 32 tokens then fall in disjoint halves of the banks
            uint8_t* pbuf = ps + (NPBUF == 2 ? u : 0) * PBYTES;
            const int ke = kk & ~1;
            constexpr int kPair = GQ >= 4 ? 4 : 1;
#pragma unroll
            for (int n = 0; n < 2 * GQ; ++n) {
                if (n & kPair) continue;
                const int m = n | kPair;
                const uint32_t recv = __shfl_xor_sync(kAll, (lane & 1) ? t16[n] : t16[m], 1);
                const uint32_t w = (lane & 1) ? (recv | (t16[m] << 16)) : (t16[n] | (recv << 16));
                *reinterpret_cast<uint32_t*>(pbuf + op_offset((lane & 1) ? m : n, ke, PCHUNK)) = w;
            }
            if (tb + kTT > t1) {
                // the split's last tile: V rows past its end hold other tokens
                // (or nothing loaded) and must not reach the product as NaN/inf
                const int j = pos_v(i, ntiles), sv = j % kSlots;
                if (!__all_sync(kAll, mbar_wait(&bar->full[sv], (j / kSlots) & 1, status, kStatusTimeout, abort))) {
                    ok = false;
                    break;
                }
                if (!valid) {
                    uint8_t* row = slots + sv * kSlotBytes + kk * 128;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        reinterpret_cast<uint4*>(row)[q] = make_uint4(0u, 0u, 0u, 0u);
                        reinterpret_cast<uint4*>(row + kChunk)[q] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar->p_full[u]);
        }
        if (ok && ntiles > 0)
            ok = __all_sync(kAll, mbar_wait(&bar->pv_done[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, status,
                                            kStatusTimeout, abort));
        tc_fence_after();
        // ----------------------------------------------------------- epilogue
        // the row sums: every token's share, over the warp, then over the 4 warps
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
            float x = l_part[h];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kAll, x, o);
            if (lane == 0) bar->sum[wq][h] = x;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar->sum_full);
        // `have` is warp-uniform (it decides the warp-collective load of O^T)
        const bool have =
            ok && ntiles > 0 && __all_sync(kAll, mbar_wait(&bar->sum_full, 0, status, kStatusTimeout, abort));
        // row d of O^T: head h is column h (P_hi) plus column G + h (P_lo)
        uint32_t o[NPV];
#pragma unroll
        for (int c = 0; c < NPV; ++c) o[c] = 0u;
        if (have) {
#pragma unroll
            for (int g = 0; g < NPV / 16; ++g) {
                uint32_t w[16];
                tmem_ld16(tmem + kColO + 16 * g + lane_off, w);
                tmem_wait_ld();
                pin(w);
#pragma unroll
                for (int c = 0; c < 16; ++c) o[16 * g + c] = w[c];
            }
        }
        // lane h < G: head h's row sum, its reciprocal and base-2 LSE, then
        // handed to every lane (one reciprocal and logarithm per head)
        float inv_l = 0.f, lse2 = -INFINITY;
        int mass_l = 0;
        if (have && lane < GQ) {
            float mh = -INFINITY;
#pragma unroll
            for (int h = 0; h < GQ; ++h)
                if (lane == h) mh = m_run[h];
            const float l = bar->sum[0][lane] + bar->sum[1][lane] + bar->sum[2][lane] + bar->sum[3][lane];
            if (l > 0.f) {
                mass_l = 1;
                inv_l = 1.f / l;
                lse2 = mh + log2f(l);
            }
        }
        const int d = kk;
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
            const float inv = __shfl_sync(kAll, inv_l, h);
            const bool mass = __shfl_sync(kAll, mass_l, h) != 0;
            const float acc = __uint_as_float(o[h]) + __uint_as_float(o[GQ + h]);
            const float val = mass ? acc * inv : 0.f;
            const int head = hkv * GQ + h;
            if (direct) {
                if (split > 0) break;  // nothing to write: this split holds no token
                T* orow = reinterpret_cast<T*>(p.o + (int64_t)r * p.o_sn + (int64_t)b * p.o_sb + (int64_t)head * p.o_sh);
                orow[d] = from_f32<T>(val);
                if (st == h)
                    p.lse[(int64_t)r * p.l_sn + (int64_t)b * p.l_sb + (int64_t)head * p.l_sh] =
                        p.base2 ? lse2 : lse2 * kLn2F;
            } else {
                if (split >= nse) break;  // an empty split: the merge skips it
                const int64_t row = (((int64_t)r * p.B + b) * p.H + head) * p.nsplit + split;
                p.ws_o[row * kD + d] = val;
                if (st == h) p.ws_lse[row] = lse2;
            }
        }
    }

    // --------------------------------------------------------------- teardown
    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
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
}

template <typename T, bool PAGED>
cudaError_t launch_tc_t(const AttnParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, cudaStream_t stream) {
    const void* k;
    switch (p.H / p.Hkv) {
        case 2: k = (const void*)gqa_decode_tc_kernel<T, 2, PAGED>; break;
        case 4: k = (const void*)gqa_decode_tc_kernel<T, 4, PAGED>; break;
        case 8: k = (const void*)gqa_decode_tc_kernel<T, 8, PAGED>; break;
        case 16: k = (const void*)gqa_decode_tc_kernel<T, 16, PAGED>; break;
        default: return cudaErrorInvalidValue;
    }
    // the shared-memory opt-in is a per-device function attribute
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    AttnParams q = p;
    // DCP_TEST_STALL_LOADS=1 (tests of the failure path only): the kernel
    // issues none of its K/V loads, so its first wait on them runs out; it
    // must then record DCP_ERR_TIMEOUT and end, leaving the context usable.
    // Read per call; unset in normal use.
    const char* stall = getenv("DCP_TEST_STALL_LOADS");
    q.stall_loads = stall && stall[0] == '1';
    void* args[] = {(void*)&kmap, (void*)&vmap, (void*)&q};
    const dim3 grid((unsigned)((int64_t)p.N * p.B * p.Hkv * p.nsplit));  // split fastest
    e = launch_pdl(k, grid, dim3(kThreads), args, kSmemBytes, stream);
    return e;
}

}  // namespace

bool launch_decode_attention_tc(const AttnParams& p, int dtype, cudaStream_t stream, cudaError_t* err) {
    if (!DCP_ATTN_TC) return false;
    const int gq = p.Hkv > 0 ? p.H / p.Hkv : 0;
    if (p.D != kD || (gq != 2 && gq != 4 && gq != 8 && gq != 16)) return false;
    const bool paged = p.page_shift >= 0;
    // tiles of whole 128-token blocks (so a paged tile starts on a page
    // boundary); paged boxes of whole 8-row swizzle atoms
    if (p.split_tokens % kTT != 0 || (paged && p.page_shift < 3)) return false;
    const EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return false;
    const CUtensorMapDataType dt = dtype == DCP_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    // a dimension of extent 1 is never stepped over: give it a nominal stride
    auto stride = [](int64_t extent, int64_t bytes) -> cuuint64_t { return (cuuint64_t)(extent > 1 ? bytes : 256); };
    const int64_t lcap = ((int64_t)p.max_seq_len + p.N - 1) / p.N;
    const int64_t rows = paged ? (int64_t)1 << p.page_shift : (lcap > 0 ? lcap : 1);  // token rows of a block
    const int64_t outer = paged ? p.num_pages : p.B;                                  // blocks of a rank
    const cuuint32_t box[5] = {64, 1, (cuuint32_t)(paged ? (rows < kTT ? rows : kTT) : kTT), 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    // K and V of every rank as 5-D tensors: [N][blocks][rows][Hkv][128], the
    // blocks being requests (contiguous) or pool pages (paged); a box is 64
    // columns of one head over a tile's rows
    CUtensorMap maps[2];
    for (int m = 0; m < 2; ++m) {
        const unsigned char* base = m ? p.v : p.k;
        const int64_t st = m ? p.v_st : p.k_st, sh = m ? p.v_sh : p.k_sh, sn = m ? p.v_sn : p.k_sn;
        const int64_t sblk = paged ? (m ? p.v_sp : p.k_sp) : (m ? p.v_sb : p.k_sb);
        const cuuint64_t dims[5] = {(cuuint64_t)kD, (cuuint64_t)p.Hkv, (cuuint64_t)rows, (cuuint64_t)outer,
                                    (cuuint64_t)p.N};
        const cuuint64_t strides[4] = {stride(p.Hkv, sh), stride(rows, st), stride(outer, sblk), stride(p.N, sn)};
        if (enc(&maps[m], dt, 5, const_cast<unsigned char*>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;  // strides a tensor map cannot describe: the register-tiled kernels take it
    }
    cudaError_t e;
    if (dtype == DCP_F16)
        e = paged ? launch_tc_t<__half, true>(p, maps[0], maps[1], stream)
                  : launch_tc_t<__half, false>(p, maps[0], maps[1], stream);
    else
        e = paged ? launch_tc_t<__nv_bfloat16, true>(p, maps[0], maps[1], stream)
                  : launch_tc_t<__nv_bfloat16, false>(p, maps[0], maps[1], stream);
    if (e == cudaSuccess && p.nsplit > 1) {
        AttnParams m = p;
        m.merge_multi_only = 1;  // rows with one non-empty split were written above
        e = launch_attention_split_merge(m, dtype, stream);
    }
    *err = e;
    return true;
}

int attn_tc_device_status(bool clear) {
    int s = 0;
    if (cudaMemcpyFromSymbol(&s, g_tc_status, sizeof(int)) != cudaSuccess) return -1;
    if (clear && s) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(int)) != cudaSuccess) return -1;
    }
    return s;
}

}  // namespace dcp
