/*
 * dcp.h -- C ABI of libdcp_gb300.so: the data-parallel hot path of decode
 * context parallelism (DCP) on one GB300 (sm_103a).
 *
 * DCP splits a request's KV cache across the N ranks of a group; every rank
 * returns a partial attention output O_r [B, H, D] and its log-sum-exp
 * lse_r [B, H] (fp32), and the partials are merged with LSE weights.  This
 * library implements the three steps of that merge:
 *
 *   dcp_pack_send       scatter O and LSE into a send layout (peer-major
 *                       interleaved or peer-inside split), by strides alone;
 *   dcp_lse_combine     the LSE-weighted combine over strided views;
 *   dcp_unpack_combine  the combine reading interleaved [payload | LSE word]
 *                       receive rows in one pass;
 *   dcp_decode_attention  the step before the merge: each rank's decode
 *                       attention over its round-robin share of the KV cache
 *                       (grouped-query heads at D = 128 on the tcgen05 tensor
 *                       cores; dcp_decode_attention_mla: over an absorbed-MLA
 *                       latent cache, on the tcgen05 tensor cores).
 *
 * The cross-rank exchange itself (NCCL all-to-all, MNNVL, all-gather /
 * all-reduce) is not part of this library.  A group's N ranks can be held as
 * one stacked tensor on one device; the "received" views then address the
 * sender stack with swapped strides, or a relayout of it.
 *
 * Conventions for every entry point
 * ---------------------------------
 * - Pointers are addresses the current CUDA device can dereference: device
 *   memory, or page-locked host memory mapped at the same address (pinned
 *   allocations under unified addressing), which the kernels then read or
 *   write directly over the host link.  The caller owns every buffer.  The library allocates nothing, frees nothing, never
 *   synchronises, and enqueues its kernels on `stream` (a cudaStream_t; NULL
 *   means the legacy default stream).  Work is asynchronous: results are
 *   valid once the stream reaches that point.
 * - Strides are in ELEMENTS of the pointed-to type: payload elements (dtype)
 *   for O / dst_o / out / recv, fp32 words for every LSE pointer.  Strides
 *   must be >= 0 and <= 2^52.  The innermost (D) stride is always 1 and is
 *   not passed.
 * - Sizes: N >= 1 and D >= 1.  B, H (or Hc, Hpr) and G may be 0, in which
 *   case the call does nothing and returns DCP_OK.  N <= 4096.  A payload
 *   row (D elements) is at most 2^30 bytes, and the rows of one operand span
 *   at most 2^56 bytes from its first to its last byte (no device holds more;
 *   larger strides are refused as DCP_ERR_INVALID_ARG rather than left to
 *   wrap around in 64-bit address arithmetic).
 * - G is a batch of independent groups (for example all N destination ranks,
 *   or all N source ranks, of a group held on one device).
 * - Validation happens on the host, before any launch; a failing call
 *   launches nothing and returns a non-zero dcp_status_t.
 *   dcp_last_error_message() then describes the failure (per host thread).
 * - DCP_ERR_CUDA is returned when a launch fails (cudaGetLastError); the CUDA
 *   error string is in dcp_last_error_message().
 * - Outputs must not overlap inputs, except where an entry point says so;
 *   the rows of one output must not overlap one another.
 *
 * Payload types: DCP_F32, DCP_F16, DCP_BF16 and DCP_FP8_E4M3.  LSE values
 * are always fp32.  Merges accumulate in fp32 whatever the payload type and
 * round once into the output type.
 *
 * DCP_FP8_E4M3 is the OCP e4m3 "fn" byte format (bias 7, no infinities,
 * S.1111.111 is NaN, largest finite 448).  Its rows are moved in 4- or 16-byte
 * vectors, so with fp8 payloads D must be a multiple of 4 and every payload
 * row must start on a 4-byte boundary (DCP_ERR_MISALIGNED otherwise).  Merged
 * fp8 outputs are rounded to nearest-even, saturating at +-448; NaN stays NaN.
 * The pages leave fp8 to future work (vLLM PR #41160 report, risk list: the
 * LSE pack-dim helper rejects fp8 with a ValueError; sglang PR #34213 report,
 * risk list: the fp32-word reinterpretation needs re-reading once fp8 is
 * added); the byte layout here is the same rule carried to a 1-byte element.
 */
#ifndef DCP_GB300_DCP_H_
#define DCP_GB300_DCP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dcp_status {
    DCP_OK = 0,
    DCP_ERR_INVALID_ARG = 1,          /* bad size, NULL pointer, stride out of range, bad flag */
    DCP_ERR_UNSUPPORTED_DTYPE = 2,    /* dtype other than f32 / f16 / bf16 / fp8 e4m3 */
    DCP_ERR_HEADS_NOT_DIVISIBLE = 3,  /* H % N != 0 in the pack */
    DCP_ERR_MISALIGNED = 4,           /* D % lpd != 0, a pointer/stride not aligned to its type,
                                         or fp8 rows not on 4-byte boundaries */
    DCP_ERR_ALIAS = 5,                /* an output overlaps an input or itself */
    DCP_ERR_CUDA = 6,                 /* a CUDA call failed; see dcp_last_error_message() */
    DCP_ERR_TIMEOUT = 7               /* a kernel gave up on a bounded wait (dcp_device_status) */
} dcp_status_t;

enum { DCP_F32 = 0, DCP_F16 = 1, DCP_BF16 = 2, DCP_FP8_E4M3 = 3 };
enum { DCP_LSE_BASE_E = 0, DCP_LSE_BASE_2 = 1 };

/* Flags of dcp_lse_combine / dcp_unpack_combine. */
enum {
    /* Replace NaN/+-inf elements of O by 0 before weighting (the ag_rs merge's
     * nan_to_num_ on the partial output; sglang PR #34213 report,
     * "关键源码片段", `cp_lse_ag_out_rs_mha`). */
    DCP_SANITIZE_O = 1u,
    /* dcp_lse_combine only: `out` IS the rank-0 slice of `o` (same pointer and
     * the same G/B/H strides); each row's rank-0 partial is overwritten by the
     * merged row after all N ranks of that row were read (sglang PR #34213
     * report, "实现拆解" item 2). */
    DCP_INPLACE_RANK0 = 2u
};

/*
 * Payload elements one fp32 LSE word occupies in an interleaved row:
 * 1 for DCP_F32, 2 for DCP_F16 and DCP_BF16, 4 for DCP_FP8_E4M3, -1 for
 * anything else.  (vLLM PR #41160 report, "实现拆解" item 2,
 * `_dcp_a2a_lse_pack_dim`: fp16 -> 2, fp32 -> 1, other types rejected; bf16
 * is the other 16-bit type, and fp8 -- which that helper still rejects -- is
 * given the same 4-bytes-per-word rule.)
 */
int dcp_lse_pack_dim(int dtype);

/* Static English text for a status code (never NULL). */
const char* dcp_status_string(int status);

/* Details of the last failing call made by this host thread ("" if none). */
const char* dcp_last_error_message(void);

/*
 * dcp_pack_send -- the shared, stride-parameterised pack.
 * (sglang PR #34651 report, "实现拆解" items 1-3 and "关键源码片段",
 * `dcp_pack_a2a_send` / `_dcp_pack_a2a_send_kernel`; vLLM PR #41160 report,
 * "实现拆解" item 1, `_dcp_a2a_pack_send_kernel`.)
 *
 * For each group g < G, token b < B and head h < H, with H_pr = H / N,
 * peer p = h / H_pr and local head hl = h % H_pr:
 *     dst_o  [g][p, b, hl, 0:D] = o  [g][b, h, 0:D]     (bit copy)
 *     dst_lse[g][p, b, hl]      = lse[g][b, h]          (bit copy)
 * and no other byte is written.
 *
 *   o        [G][B, H, D]       payload, strides (o_sg, o_sb, o_sh)
 *   lse      [G][B, H]          fp32, strides (l_sg, l_sb, l_sh)
 *   dst_o    [G][N, B, H_pr, D] payload, strides (do_sg, do_sn, do_sb, do_sh)
 *   dst_lse  [G][N, B, H_pr]    fp32, strides (dl_sg, dl_sn, dl_sb, dl_sh)
 *
 * Peer-major interleaved send buffer [N, B, H_pr, D + lpd] (one flat buffer
 * split by byte offset for a single all-to-all): dst_o = buffer with strides
 * (B*H_pr*(D+lpd), H_pr*(D+lpd), D+lpd); dst_lse = (float*)buffer + D/lpd with
 * the same strides divided by lpd.  Peer-inside split layout (O [B,H_pr,N,D],
 * stats [B,H_pr,N,2]): dst_o = partial_o permuted to [N,B,H_pr,D], dst_lse =
 * stats[..., 0] permuted to [N,B,H_pr]; stats slot 1 is never touched.
 *
 * dst_lse may lie inside dst_o's buffer only as in the interleaved layout:
 * the same byte strides, starting at or after byte D*e of each row and ending
 * before the next row.  Errors: DCP_ERR_HEADS_NOT_DIVISIBLE if H % N != 0;
 * DCP_ERR_ALIAS for any other overlap; DCP_ERR_MISALIGNED for pointers not
 * aligned to their element size.
 */
dcp_status_t dcp_pack_send(int dtype, int N, int B, int H, int D, int G,
                           const void* o, int64_t o_sg, int64_t o_sb, int64_t o_sh,
                           const float* lse, int64_t l_sg, int64_t l_sb, int64_t l_sh,
                           void* dst_o, int64_t do_sg, int64_t do_sn, int64_t do_sb, int64_t do_sh,
                           float* dst_lse, int64_t dl_sg, int64_t dl_sn, int64_t dl_sb, int64_t dl_sh,
                           void* stream);

/*
 * dcp_lse_combine -- LSE-weighted merge of N rank partials over strided views.
 * (sglang PR #34213 report, "关键源码片段", `cp_lse_ag_out_rs_mha`;
 * sglang PR #34651 report, "实现拆解" item 3, `dcp_lse_combine_triton`
 * reading the non-contiguous receive views; sglang PR #33926 report,
 * "实现拆解" item 4 and "关联脉络" #34240: base-2 vs natural-log LSE.)
 *
 * For each row (g, b, h), over ranks r = 0..N-1, in the LSE base `lse_base`:
 *     Gl   = logsumexp_r lse[g][r, b, h]
 *            (any NaN -> NaN; else any +inf -> +inf; else all -inf -> -inf)
 *     w_r  = base^(lse_r - Gl), replaced by 0 when NaN or +-inf
 *     out[g][b, h, :] = sum_r w_r * O[g][r, b, h, :]   (fp32 accumulation,
 *                        rounded once to the payload type)
 *     out_lse[g][b, h] = Gl (same base as the input), when return_lse != 0.
 * With DCP_SANITIZE_O, NaN/+-inf elements of O count as 0.  N == 1 returns
 * the input unchanged (bit copy of O and LSE), as the single-rank early
 * return of `cp_lse_ag_out_rs_mha` does.
 *
 *   o        [G][N, B, Hc, D] payload, strides (o_sg, o_sn, o_sb, o_sh)
 *   lse      [G][N, B, Hc]    fp32, strides (l_sg, l_sn, l_sb, l_sh)
 *   out      [G][B, Hc, D]    payload, strides (u_sg, u_sb, u_sh)
 *   out_lse  [G][B, Hc]       fp32, strides (ul_sg, ul_sb, ul_sh); may be NULL
 *                             when return_lse == 0
 *
 * flags: DCP_SANITIZE_O | DCP_INPLACE_RANK0.  With DCP_INPLACE_RANK0, `out`
 * must equal `o` with u_sg == o_sg, u_sb == o_sb, u_sh == o_sh, and the rows
 * of `o` must not overlap one another; the caller's rank-0 partial is dead
 * after the call.  Per-rank head slices of the result (rank k keeps heads
 * [k*Hc/N, (k+1)*Hc/N)) are plain views of `out` and `out_lse`.
 */
dcp_status_t dcp_lse_combine(int dtype, int N, int B, int Hc, int D, int G,
                             const void* o, int64_t o_sg, int64_t o_sn, int64_t o_sb, int64_t o_sh,
                             const float* lse, int64_t l_sg, int64_t l_sn, int64_t l_sb, int64_t l_sh,
                             void* out, int64_t u_sg, int64_t u_sb, int64_t u_sh,
                             float* out_lse, int64_t ul_sg, int64_t ul_sb, int64_t ul_sh,
                             int lse_base, int return_lse, unsigned flags, void* stream);

/*
 * dcp_unpack_combine -- the combine reading the interleaved receive buffer.
 * (vLLM PR #41160 report, "实现拆解" item 1, `_dcp_a2a_unpack_combine_kernel`;
 * sglang PR #34651 report, "实现拆解" item 2: one flat buffer split by byte
 * offset, receive side unchanged.)
 *
 *   recv     [G][N, B, Hpr, D + lpd] payload, strides (r_sg, r_sn, r_sb, r_sh);
 *            in each row the first D elements are rank r's partial O and the
 *            fp32 word at word index D / lpd (bytes D*e .. D*e+3) is its LSE.
 *   out      [G][B, Hpr, D]  payload, strides (u_sg, u_sb, u_sh)
 *   out_lse  [G][B, Hpr]     fp32, strides (ul_sg, ul_sb, ul_sh); may be NULL
 *                            when return_lse == 0
 *
 * Same arithmetic, flags (except DCP_INPLACE_RANK0, rejected) and N == 1 rule
 * as dcp_lse_combine.  Errors: DCP_ERR_MISALIGNED if D % lpd != 0 or a row
 * start is not 4-byte aligned; DCP_ERR_ALIAS if out / out_lse overlap recv.
 *
 * Reads: rows that start on a 4- but not a 16-byte boundary (an interleaved
 * row is D*e + 4 bytes long) may be read in 16-byte chunks from the 16-byte
 * boundary at or before the row start, so up to 12 bytes before each row are
 * read and ignored.  Those bytes lie in the same 16-byte granule as the row's
 * first byte (never on another page); for every row but the first they are
 * inside recv's own extent.  The bytes before the first row count as part of
 * recv for the overlap check (an out or out_lse there is DCP_ERR_ALIAS), and
 * another stream must not be writing them during the call.
 */
dcp_status_t dcp_unpack_combine(int dtype, int N, int B, int Hpr, int D, int G,
                                const void* recv, int64_t r_sg, int64_t r_sn, int64_t r_sb, int64_t r_sh,
                                void* out, int64_t u_sg, int64_t u_sb, int64_t u_sh,
                                float* out_lse, int64_t ul_sg, int64_t ul_sb, int64_t ul_sh,
                                int lse_base, int return_lse, unsigned flags, void* stream);

/*
 * dcp_decode_attention -- each DCP rank's single-token decode attention over
 * the KV tokens it owns, producing the rank-local partials the merge takes.
 * (sglang PR #33926 report, "实现拆解" items 3-4 and "关键源码片段": token t of a
 * request lives on rank t % N, so rank r holds L / N tokens plus one when
 * r < L % N (`get_dcp_lens`); each rank returns rank-local (out, lse); a rank
 * owning no token of a request is the neutral (0, -inf) (`fixup_zero_kv_rows`);
 * trtllm-gen's LSE is base 2, cute-dsl's natural log.)
 *
 * For rank r < N, request b < B, query head h < H (KV head h / (H / Hkv)),
 * over the rank's local tokens i < L_r(b) = L_b / N + (r < L_b % N), with
 * L_b = min(seq_lens[b], max_seq_len) and scores s_i = sm_scale <q, k_i>:
 *     lse[r, b, h] = log sum_i exp(s_i)           (base e, or divided by ln 2)
 *     o  [r, b, h] = sum_i exp(s_i - lse) v_i      (0 and -inf when L_r(b) = 0)
 *
 *   q        [B, H, D]              payload, strides (q_sb, q_sh)
 *   k, v     [N][B, Lc, Hkv, D]     each rank's local cache, token i of rank r
 *                                   being global token i*N + r; Lc =
 *                                   ceil(max_seq_len / N); strides
 *                                   (k_sn, k_sb, k_st, k_sh), same for v
 *   seq_lens [B] int32 (device)     global lengths; values above max_seq_len
 *                                   count as max_seq_len
 *   o        [N, B, H, D]           payload, strides (o_sn, o_sb, o_sh)
 *   lse      [N, B, H]              fp32, strides (l_sn, l_sb, l_sh)
 *
 * dtype: DCP_F16 or DCP_BF16 (q, k, v and o); D in {64, 128, 256}; H / Hkv in
 * {1, 2, 4, 8, 16} (16 only with D <= 128); q, k and v rows start on 16-byte
 * boundaries.  Work is split into chunks of `split_tokens` local tokens;
 * with more than one chunk the partial results go through `workspace`
 * (caller-owned device memory, 16-byte aligned, at least
 * dcp_decode_attention_workspace_size(...) bytes; NULL is fine when that
 * size is 0; the size function returns 0 as well for arguments the call
 * itself refuses, such as N > 4096).  Errors: DCP_ERR_HEADS_NOT_DIVISIBLE
 * when H % Hkv != 0, DCP_ERR_INVALID_ARG for unsupported sizes or a too
 * small workspace, DCP_ERR_MISALIGNED, DCP_ERR_ALIAS for overlapping
 * operands.
 */
size_t dcp_decode_attention_workspace_size(int N, int B, int H, int D, int max_seq_len, int split_tokens);

dcp_status_t dcp_decode_attention(int dtype, int N, int B, int H, int Hkv, int D,
                                  const void* q, int64_t q_sb, int64_t q_sh,
                                  const void* k, int64_t k_sn, int64_t k_sb, int64_t k_st, int64_t k_sh,
                                  const void* v, int64_t v_sn, int64_t v_sb, int64_t v_st, int64_t v_sh,
                                  const int* seq_lens, int max_seq_len, float sm_scale, int split_tokens,
                                  void* o, int64_t o_sn, int64_t o_sb, int64_t o_sh,
                                  float* lse, int64_t l_sn, int64_t l_sb, int64_t l_sh,
                                  int lse_base, void* workspace, size_t workspace_bytes, void* stream);

/*
 * dcp_decode_attention_paged -- dcp_decode_attention over paged KV caches: the
 * same computation, outputs, workspace and errors, with each rank's tokens in
 * pages of a per-rank pool.  (sglang PR #33926 report, "实现拆解" item 1 and
 * "关键源码片段", `_fill_dcp_block_kv_indices` / `_apply_dcp_cuda_graph_metadata`:
 * under DCP the page table of a rank is built over that rank's round-robin
 * slice, from page_size and the rank-local lengths.)
 *
 *   k_pages, v_pages [N][num_pages, page_size, Hkv, D]  strides (k_sn, k_sp,
 *                    k_st, k_sh), same for v: rank, page, slot, head
 *   block_table      [N][B, max_pages] int32 (device)   strides (bt_sn, bt_sb);
 *                    local token i of request b on rank r sits in slot
 *                    i % page_size of page block_table[r][b][i / page_size]
 *
 * page_size is a power of two up to 65536; max_pages must cover the local
 * capacity, ceil(ceil(max_seq_len / N) / page_size) entries, and only the
 * entries of tokens a rank holds are read.  Page indices must lie in
 * [0, num_pages): the kernels never read outside the pool, reading a token
 * whose index does not as a zero row, which makes that result meaningless.
 */
dcp_status_t dcp_decode_attention_paged(int dtype, int N, int B, int H, int Hkv, int D,
                                        const void* q, int64_t q_sb, int64_t q_sh,
                                        const void* k_pages, int64_t k_sn, int64_t k_sp, int64_t k_st, int64_t k_sh,
                                        const void* v_pages, int64_t v_sn, int64_t v_sp, int64_t v_st, int64_t v_sh,
                                        int num_pages, int page_size,
                                        const int* block_table, int64_t bt_sn, int64_t bt_sb, int max_pages,
                                        const int* seq_lens, int max_seq_len, float sm_scale, int split_tokens,
                                        void* o, int64_t o_sn, int64_t o_sb, int64_t o_sh,
                                        float* lse, int64_t l_sn, int64_t l_sb, int64_t l_sh,
                                        int lse_base, void* workspace, size_t workspace_bytes, void* stream);

/*
 * dcp_decode_attention_noalloc -- dcp_decode_attention for callers that may
 * not allocate device memory where they run it (a fixed-size memory pool set
 * up front, a serving loop that forbids allocation, a host runtime with no
 * allocator to hand), so cannot provide a workspace.  The pages have no
 * counterpart; this is a convenience of this library.
 *
 * Same arguments, result and errors as dcp_decode_attention, without the
 * workspace: the split partials live in a 16 MiB scratch array built into the
 * library, which every device that loads the library's attention code holds
 * until the process exits.  Sizes whose scratch
 * (dcp_decode_attention_workspace_size) exceeds 16 MiB are rejected with
 * DCP_ERR_INVALID_ARG and a message giving both sizes; use a larger
 * split_tokens or dcp_decode_attention with a workspace instead.  The call
 * allocates nothing.  The scratch array's device address belongs to the
 * CUDA context the library is loaded into (the device's primary context, or
 * a driver-API context the caller made current), so every call looks it up
 * (cudaGetSymbolAddress) in the context current at that call and keeps it no
 * longer: after a cudaDeviceReset or a switch of context the next call uses
 * the array of the new context.  The first call in a context also loads the
 * library's device code there; make it before any stream capture.  All calls
 * share the one
 * array and every call writes each scratch entry before reading it (nothing
 * needs to start at zero), so calls whose work overlaps on the GPU (other
 * streams, other threads) race on the scratch: serialise them.
 */
dcp_status_t dcp_decode_attention_noalloc(int dtype, int N, int B, int H, int Hkv, int D,
                                          const void* q, int64_t q_sb, int64_t q_sh,
                                          const void* k, int64_t k_sn, int64_t k_sb, int64_t k_st, int64_t k_sh,
                                          const void* v, int64_t v_sn, int64_t v_sb, int64_t v_st, int64_t v_sh,
                                          const int* seq_lens, int max_seq_len, float sm_scale, int split_tokens,
                                          void* o, int64_t o_sn, int64_t o_sb, int64_t o_sh,
                                          float* lse, int64_t l_sn, int64_t l_sb, int64_t l_sh,
                                          int lse_base, void* stream);

/*
 * dcp_decode_attention_mla -- each DCP rank's single-token decode attention
 * over the tokens it owns of an absorbed-MLA latent cache (DeepSeek-V3
 * class: every query head scores one shared latent row per token).
 * (sglang PR #33926 report, "功能与动机" and "实现拆解" items 3-4: the
 * trtllm_mla decode path returns rank-local (out, lse), the LSE in base 2; a
 * rank owning no token of a request is the neutral (0, -inf); token t lives
 * on rank t % N.  sglang PR #34213 report, "功能与动机": for absorbed MLA the
 * output width is kv_lora_rank.)
 *
 * For rank r < N, request b < B, query head h < H, over the rank's local
 * tokens i < L_r(b) = L_b / N + (r < L_b % N), L_b = min(seq_lens[b],
 * max_seq_len), with s_i = sm_scale <q[b, h, 0:Dk], kv[r][b, i, 0:Dk]>:
 *     lse[r, b, h] = log sum_i exp(s_i)        (base e, or divided by ln 2)
 *     o  [r, b, h] = sum_i exp(s_i - lse) kv[r][b, i, 0:Dv]
 * (0 and -inf when L_r(b) = 0): the value is the first Dv elements of each
 * latent row, the score uses all Dk (kv_lora_rank, then the rope part).
 *
 *   q        [B, H, Dk]       absorbed queries (no-rope part, then rope part),
 *                             strides (q_sb, q_sh)
 *   kv       [N][B, Lc, Dk]   each rank's latent cache, Lc = ceil(max_seq_len
 *                             / N); strides (kv_sn, kv_sb, kv_st)
 *   seq_lens [B] int32 (device) global lengths
 *   o        [N, B, H, Dv]    strides (o_sn, o_sb, o_sh)
 *   lse      [N, B, H]        fp32, strides (l_sn, l_sb, l_sh)
 *
 * Supported: dtype DCP_BF16 or DCP_F16 (q, kv and o); Dk = 576 and Dv = 512;
 * 1 <= H <= 128; split_tokens a positive multiple of 64.  q and o rows start
 * on 16-byte boundaries; kv is 16-byte aligned with strides that are
 * positive multiples of 8 elements (kv_st >= Dk).  Probabilities enter the
 * value product rounded to the payload type (an 8- or 11-bit significand);
 * scores, sums and outputs accumulate in fp32.  Workspace as for
 * dcp_decode_attention, sized dcp_decode_attention_workspace_size(N, B, H,
 * Dv, max_seq_len, split_tokens).  Errors as for dcp_decode_attention; the
 * kernel's waits are bounded, and one that runs out is reported by
 * dcp_device_status().  Needs a GPU of compute capability 10.x with
 * tensor-map support in its driver (DCP_ERR_CUDA otherwise).
 */
dcp_status_t dcp_decode_attention_mla(int dtype, int N, int B, int H, int Dk, int Dv,
                                      const void* q, int64_t q_sb, int64_t q_sh,
                                      const void* kv, int64_t kv_sn, int64_t kv_sb, int64_t kv_st,
                                      const int* seq_lens, int max_seq_len, float sm_scale, int split_tokens,
                                      void* o, int64_t o_sn, int64_t o_sb, int64_t o_sh,
                                      float* lse, int64_t l_sn, int64_t l_sb, int64_t l_sh,
                                      int lse_base, void* workspace, size_t workspace_bytes, void* stream);

/*
 * dcp_device_status -- DCP_OK, or DCP_ERR_TIMEOUT when a tensor-core kernel
 * launched on the current device since the last call gave up on one of its
 * bounded waits (1 s each; its outputs are then invalid).  Synchronises with
 * the device (it reads a device status word), then clears the status.  The
 * merge kernels never wait and never set it.
 */
dcp_status_t dcp_device_status(void);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* DCP_GB300_DCP_H_ */
