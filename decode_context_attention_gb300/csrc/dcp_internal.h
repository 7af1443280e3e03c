// dcp_internal.h -- host-side launch interface between the C ABI (dcp_abi.cu)
// and the kernels (dcp_pack.cu, dcp_combine_*.cu).  Not installed; the public
// interface is include/dcp.h.
//
// All payload strides here are in BYTES and all LSE strides in fp32 WORDS; the
// ABI layer converts the caller's element strides once, after validation.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "dcp.h"

namespace dcp {

constexpr int kThreads = 256;  // threads per CTA for every kernel here

struct PackParams {
    int N, B, H, D, G, H_pr;
    int64_t rows;        // G * B * H source rows
    int row_bytes;       // D * element size
    int vb;              // vector width in bytes (16, 4 or 2)
    int lpr;             // lanes cooperating on one row (power of two <= 32)
    int copy_payload;    // 0: skip the payload (single-rank in-place combine)
    int copy_lse;        // 0: skip the LSE words (single-rank combine without return_lse)
    const unsigned char* o;
    int64_t o_sg, o_sb, o_sh;
    const float* lse;
    int64_t l_sg, l_sb, l_sh;
    unsigned char* dst_o;
    int64_t do_sg, do_sn, do_sb, do_sh;
    float* dst_lse;
    int64_t dl_sg, dl_sn, dl_sb, dl_sh;
};

struct CombineParams {
    int N, B, Hc, D, G;
    int64_t rows;        // G * B * Hc output rows
    int vec_per_row;     // D * element size / vector width
    int lpr;             // lanes cooperating on one row (power of two <= 32)
    int base2;           // LSE base: 0 = e, 1 = 2
    int return_lse;
    int sanitize;        // NaN/+-inf elements of O count as 0
    const unsigned char* o;
    int64_t o_sg, o_sn, o_sb, o_sh;
    const float* lse;
    int64_t l_sg, l_sn, l_sb, l_sh;
    unsigned char* out;
    int64_t u_sg, u_sb, u_sh;
    float* out_lse;
    int64_t ul_sg, ul_sb, ul_sh;
};

// Decode attention of every rank over its round-robin share of the KV cache.
struct AttnParams {
    int N, B, H, Hkv, D;
    int max_seq_len;   // bound on seq_lens; the local caches hold ceil(max_seq_len / N) tokens
    int split_tokens;  // local tokens per split
    int nsplit;        // splits per (rank, request, KV head)
    int base2;         // returned LSE base: 0 = e, 1 = 2
    float sm_scale;
    const unsigned char* q;
    int64_t q_sb, q_sh;                 // bytes
    const unsigned char* k;
    int64_t k_sn, k_sb, k_st, k_sh;     // bytes (k_sb = 0 for paged caches)
    const unsigned char* v;
    int64_t v_sn, v_sb, v_st, v_sh;     // bytes (v_sb = 0 for paged caches)
    // paged caches: local token i of request b on rank r sits in slot
    // i % page_size of page bt[r][b][i / page_size] (offset page * k_sp +
    // slot * k_st); page_shift < 0 for contiguous caches
    const int* bt;
    int64_t bt_sn, bt_sb;               // int32 elements
    int64_t k_sp, v_sp;                 // bytes
    int page_shift;                     // log2(page_size)
    int num_pages;                      // pages in each rank's pool
    const int* seq_lens;                // [B] global lengths
    unsigned char* o;
    int64_t o_sn, o_sb, o_sh;           // bytes
    float* lse;
    int64_t l_sn, l_sb, l_sh;           // fp32 words
    float* ws_o;                        // [N*B*H*nsplit][D] partial outputs (nsplit > 1)
    float* ws_lse;                      // [N*B*H*nsplit] partial base-2 LSEs
    int stall_loads;                    // test of the bounded waits (tensor-core path): no loads issued
    int merge_multi_only;               // split merge: only rows with two or more non-empty splits
};

// Decode attention of every rank over its share of an absorbed-MLA latent
// cache [N][B][lcap][576] (value = the first 512 elements of each row).
struct MlaParams {
    int N, B, H;
    int64_t lcap;      // local capacity: ceil(max_seq_len / N) tokens per (rank, request)
    int max_seq_len;
    int split_tokens;  // local tokens per split (a multiple of 64)
    int nsplit;
    int base2;
    float sm_scale;
    const unsigned char* q;
    int64_t q_sb, q_sh;                  // bytes
    const unsigned char* kv;
    int64_t kv_sn, kv_sb, kv_st;         // bytes
    const int* seq_lens;
    unsigned char* o;
    int64_t o_sn, o_sb, o_sh;            // bytes
    float* lse;
    int64_t l_sn, l_sb, l_sh;            // fp32 words
    float* ws_o;                         // [N*B*H*nsplit][512] (nsplit > 1)
    float* ws_lse;                       // [N*B*H*nsplit]
    int stall_loads;                     // test of the bounded waits: the loads are never issued
};

// Records `msg` as this host thread's dcp_last_error_message() and returns s.
dcp_status_t set_error(dcp_status_t s, const char* msg);

// Launchers return the launch's cudaGetLastError().
cudaError_t launch_decode_attention(const AttnParams& p, int dtype, cudaStream_t stream);
// The tensor-core (tcgen05) path of the same attention, for the shapes it
// takes (D = 128, 2 to 16 query heads per KV head, split_tokens a multiple of
// 128, pages of at least 8 tokens, strides a tensor map can describe):
// returns false without launching anything otherwise, else true with the
// launches' error in *err.  With splits it also runs the split merge.
bool launch_decode_attention_tc(const AttnParams& p, int dtype, cudaStream_t stream, cudaError_t* err);
// The merge of the fp32 split partials into (O, lse) (nsplit > 1).
cudaError_t launch_attention_split_merge(const AttnParams& p, int dtype, cudaStream_t stream);
// cudaErrorNotSupported when the driver offers no tensor-map encoder.
cudaError_t launch_mla_decode(const MlaParams& p, int dtype, cudaStream_t stream);
// The device status words of the tcgen05 kernels (the MLA attention's, the
// grouped-query attention's): 0, or the status of the first bounded wait
// that ran out; read synchronously and optionally cleared; -1 when it cannot
// be read.
int mla_device_status(bool clear);
int attn_tc_device_status(bool clear);
cudaError_t launch_pack(const PackParams& p, cudaStream_t stream);
cudaError_t launch_combine_f32(const CombineParams& p, int vb, cudaStream_t stream);
cudaError_t launch_combine_f16(const CombineParams& p, int vb, cudaStream_t stream);
cudaError_t launch_combine_bf16(const CombineParams& p, int vb, cudaStream_t stream);
cudaError_t launch_combine_fp8(const CombineParams& p, int vb, cudaStream_t stream);

// Number of SMs of the current device (cached per device).
int device_sm_count();
// Resident CTAs per SM of `kernel` at `threads` threads and `smem` bytes of
// dynamic shared memory (cached per device, kernel and shared-memory size).
int ctas_per_sm(const void* kernel, int threads, size_t smem);

}  // namespace dcp
