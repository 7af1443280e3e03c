// dcp_abi.cu -- the extern "C" entry points declared in include/dcp.h:
// argument validation on the host (sizes, pointer alignment, aliasing) and
// dispatch to the kernels.  Nothing here touches device memory: a rejected
// call launches nothing.
#include <stdarg.h>
#include <stdio.h>
#include <math.h>
#include <string.h>

#include <atomic>
#include <map>
#include <tuple>
#include <mutex>
#include <utility>

#include "dcp.h"
#include "dcp_internal.h"

namespace dcp {

int device_sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < 64) {
        const int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        n = 1;
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

int ctas_per_sm(const void* kernel, int threads, size_t smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, const void*, int, size_t>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_tuple(dev, kernel, threads, smem);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess ||
        n < 1)
        n = 1;
    cache[key] = n;
    return n;
}

}  // namespace dcp

namespace {

thread_local char g_msg[512] = "";

dcp_status_t fail(dcp_status_t s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return s;
}

dcp_status_t ok() {
    g_msg[0] = '\0';
    return DCP_OK;
}

int elem_size(int dtype) {
    switch (dtype) {
        case DCP_F32: return 4;
        case DCP_F16:
        case DCP_BF16: return 2;
        case DCP_FP8_E4M3: return 1;
        default: return 0;
    }
}

// Limits that keep every byte offset in 64 bits: a stride of at most 2^52
// elements (times at most 4 bytes), a payload row of at most 2^30 bytes (row
// and vector offsets are 32-bit in the kernels), and at most 2^56 bytes
// between the first and the last byte an operand's rows can touch.
constexpr int64_t kMaxStride = int64_t(1) << 52;
constexpr int64_t kMaxRowBytes = int64_t(1) << 30;
constexpr int64_t kMaxSpan = int64_t(1) << 56;

// A strided set of rows: `nd` outer dimensions (size, stride in BYTES) and
// `inner` contiguous bytes per row.
struct View {
    uintptr_t base = 0;
    int nd = 0;
    int64_t size[5] = {0, 0, 0, 0, 0};
    int64_t stride[5] = {0, 0, 0, 0, 0};
    int64_t inner = 0;

    View(const void* p, int64_t inner_bytes) : base((uintptr_t)p), inner(inner_bytes) {}
    View& dim(int64_t n, int64_t stride_bytes) {
        size[nd] = n;
        stride[nd] = stride_bytes;
        ++nd;
        return *this;
    }
    bool empty() const {
        for (int i = 0; i < nd; ++i)
            if (size[i] == 0) return true;
        return inner == 0;
    }
    // False when the rows would span more than kMaxSpan bytes (or the span
    // overflows): no device holds that much memory, so such strides are a
    // caller's mistake, and refusing them keeps every address computation
    // below (host and device, 64-bit) free of overflow.
    bool fits() const {
        int64_t s = inner;
        for (int i = 0; i < nd; ++i) {
            if (size[i] <= 1) continue;
            int64_t t;
            if (__builtin_mul_overflow(size[i] - 1, stride[i], &t) || __builtin_add_overflow(s, t, &s))
                return false;
        }
        return s <= kMaxSpan;
    }
    // Byte range [lo, hi) that the rows can touch.
    void extent(uintptr_t& lo, uintptr_t& hi) const {
        lo = base;
        hi = base + (uintptr_t)inner;
        for (int i = 0; i < nd; ++i)
            if (size[i] > 1) hi += (uintptr_t)((size[i] - 1) * stride[i]);
    }
    // True when distinct index tuples address disjoint byte ranges: sorted by
    // stride, every stride spans at least the block of the smaller dimensions.
    bool rows_disjoint() const { return rows_disjoint_with_inner(inner); }
    bool rows_disjoint_with_inner(int64_t row_bytes) const {
        int idx[5];
        int m = 0;
        for (int i = 0; i < nd; ++i)
            if (size[i] > 1) idx[m++] = i;
        for (int a = 1; a < m; ++a)
            for (int b = a; b > 0 && stride[idx[b]] < stride[idx[b - 1]]; --b) std::swap(idx[b], idx[b - 1]);
        int64_t span = row_bytes;
        for (int a = 0; a < m; ++a) {
            const int i = idx[a];
            if (stride[i] < span) return false;
            span = stride[i] * (size[i] - 1) + span;
        }
        return true;
    }
    // Largest power of two (<= 16) dividing every row start.
    int align() const {
        uint64_t bits = (uint64_t)base | 16u;
        for (int i = 0; i < nd; ++i)
            if (size[i] > 1) bits |= (uint64_t)stride[i];
        return (int)(bits & (~bits + 1));
    }
};

bool overlap(const View& a, const View& b) {
    if (a.empty() || b.empty()) return false;
    uintptr_t alo, ahi, blo, bhi;
    a.extent(alo, ahi);
    b.extent(blo, bhi);
    return alo < bhi && blo < ahi;
}

// A stride below 0 or above kMaxStride elements.
bool bad_stride(std::initializer_list<int64_t> s) {
    for (int64_t v : s)
        if (v < 0 || v > kMaxStride) return true;
    return false;
}

bool all_fit(std::initializer_list<const View*> views) {
    for (const View* v : views)
        if (!v->fits()) return false;
    return true;
}

// Widest vector (16, 4 or 2 bytes) that divides the row length and every row
// start of the views given by their alignments.
int pick_vb(int row_bytes, int align_a, int align_b, int e) {
    const int a = align_a < align_b ? align_a : align_b;
    if (a % 16 == 0 && row_bytes % 16 == 0) return 16;
    if (a % 4 == 0 && row_bytes % 4 == 0) return 4;
    return e == 2 ? 2 : 4;
}

// fp8 rows are moved in 4- or 16-byte vectors only: the row length and every
// row start must be multiples of 4 bytes (one e4m3 element is one byte).
bool fp8_rows_ok(int e, int D, int align_a, int align_b) {
    return e != 1 || (D % 4 == 0 && align_a >= 4 && align_b >= 4);
}

int lanes_per_row(int vectors) {
    int l = 1;
    while (l < vectors && l < 32) l <<= 1;
    return l;
}

dcp_status_t launched(cudaError_t e, const char* what) {
    if (e != cudaSuccess)
        return fail(DCP_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
    return ok();
}

constexpr int kMaxRanks = 4096;

}  // namespace

namespace dcp {
// Lets other translation units report a failure through dcp_last_error_message().
dcp_status_t set_error(dcp_status_t s, const char* msg) { return fail(s, "%s", msg); }
}  // namespace dcp

extern "C" {

int dcp_lse_pack_dim(int dtype) {
    const int e = elem_size(dtype);
    return e ? 4 / e : -1;
}

const char* dcp_status_string(int status) {
    switch (status) {
        case DCP_OK: return "success";
        case DCP_ERR_INVALID_ARG: return "invalid argument";
        case DCP_ERR_UNSUPPORTED_DTYPE: return "unsupported payload dtype (f32, f16, bf16 and fp8 e4m3 only)";
        case DCP_ERR_HEADS_NOT_DIVISIBLE: return "number of heads is not a multiple of the rank count";
        case DCP_ERR_MISALIGNED: return "misaligned pointer, stride or head dim";
        case DCP_ERR_ALIAS: return "an output overlaps an input or itself";
        case DCP_ERR_CUDA: return "CUDA error";
        case DCP_ERR_TIMEOUT: return "a kernel gave up on a bounded wait (its outputs are invalid)";
        default: return "unknown status";
    }
}

const char* dcp_last_error_message(void) { return g_msg; }

dcp_status_t dcp_pack_send(int dtype, int N, int B, int H, int D, int G,
                           const void* o, int64_t o_sg, int64_t o_sb, int64_t o_sh,
                           const float* lse, int64_t l_sg, int64_t l_sb, int64_t l_sh,
                           void* dst_o, int64_t do_sg, int64_t do_sn, int64_t do_sb, int64_t do_sh,
                           float* dst_lse, int64_t dl_sg, int64_t dl_sn, int64_t dl_sb, int64_t dl_sh,
                           void* stream) {
    const int e = elem_size(dtype);
    if (!e) return fail(DCP_ERR_UNSUPPORTED_DTYPE, "dcp_pack_send: dtype %d", dtype);
    if (N < 1 || N > kMaxRanks || D < 1 || B < 0 || H < 0 || G < 0)
        return fail(DCP_ERR_INVALID_ARG, "dcp_pack_send: sizes N=%d B=%d H=%d D=%d G=%d", N, B, H, D, G);
    if (H % N)
        return fail(DCP_ERR_HEADS_NOT_DIVISIBLE, "dcp_pack_send: H=%d is not a multiple of N=%d", H, N);
    if ((int64_t)D * e > kMaxRowBytes)
        return fail(DCP_ERR_INVALID_ARG, "dcp_pack_send: rows of D=%d elements exceed 2^30 bytes", D);
    if (G == 0 || B == 0 || H == 0) return ok();
    if (!o || !lse || !dst_o || !dst_lse)
        return fail(DCP_ERR_INVALID_ARG, "dcp_pack_send: NULL pointer");
    if (bad_stride({o_sg, o_sb, o_sh, l_sg, l_sb, l_sh, do_sg, do_sn, do_sb, do_sh, dl_sg, dl_sn,
                      dl_sb, dl_sh}))
        return fail(DCP_ERR_INVALID_ARG, "dcp_pack_send: negative stride or one above 2^52 elements");
    if ((uintptr_t)o % e || (uintptr_t)dst_o % e || (uintptr_t)lse % 4 || (uintptr_t)dst_lse % 4)
        return fail(DCP_ERR_MISALIGNED, "dcp_pack_send: pointer not aligned to its element type");
    const int H_pr = H / N;
    const int64_t rb = (int64_t)D * e;
    View vo = View(o, rb).dim(G, o_sg * e).dim(B, o_sb * e).dim(H, o_sh * e);
    View vl = View(lse, 4).dim(G, l_sg * 4).dim(B, l_sb * 4).dim(H, l_sh * 4);
    View vdo = View(dst_o, rb).dim(G, do_sg * e).dim(N, do_sn * e).dim(B, do_sb * e).dim(H_pr, do_sh * e);
    View vdl = View(dst_lse, 4).dim(G, dl_sg * 4).dim(N, dl_sn * 4).dim(B, dl_sb * 4).dim(H_pr, dl_sh * 4);
    if (!all_fit({&vo, &vl, &vdo, &vdl}))
        return fail(DCP_ERR_INVALID_ARG, "dcp_pack_send: an operand's strides span more than 2^56 bytes");
    if (overlap(vdo, vo) || overlap(vdo, vl) || overlap(vdl, vo) || overlap(vdl, vl))
        return fail(DCP_ERR_ALIAS, "dcp_pack_send: destination overlaps the source");
    if (!fp8_rows_ok(e, D, vo.align(), vdo.align()))
        return fail(DCP_ERR_MISALIGNED, "dcp_pack_send: fp8 rows need D %% 4 == 0 and 4-byte aligned row starts");
    if (!vdo.rows_disjoint() || !vdl.rows_disjoint())
        return fail(DCP_ERR_ALIAS, "dcp_pack_send: destination rows overlap one another");
    if (overlap(vdo, vdl)) {
        // only the interleaved send buffer: the LSE word sits after the payload
        // of the same row, with the same byte strides
        bool same = true;
        for (int i = 0; i < 4; ++i)
            if (vdo.size[i] > 1 && vdo.stride[i] != vdl.stride[i]) same = false;
        const int64_t off = (int64_t)((uintptr_t)dst_lse - (uintptr_t)dst_o);
        if (!same || (uintptr_t)dst_lse < (uintptr_t)dst_o || off < rb ||
            !vdo.rows_disjoint_with_inner(off + 4))
            return fail(DCP_ERR_ALIAS,
                        "dcp_pack_send: dst_lse overlaps dst_o other than as the interleaved "
                        "[payload | LSE word] row layout");
    }
    dcp::PackParams p;
    p.N = N; p.B = B; p.H = H; p.D = D; p.G = G; p.H_pr = H_pr;
    p.rows = (int64_t)G * B * H;
    p.row_bytes = (int)rb;
    p.vb = pick_vb((int)rb, vo.align(), vdo.align(), e);
    p.lpr = lanes_per_row((int)(rb / p.vb));
    p.copy_payload = 1;
    p.copy_lse = 1;
    p.o = (const unsigned char*)o; p.o_sg = o_sg * e; p.o_sb = o_sb * e; p.o_sh = o_sh * e;
    p.lse = lse; p.l_sg = l_sg; p.l_sb = l_sb; p.l_sh = l_sh;
    p.dst_o = (unsigned char*)dst_o;
    p.do_sg = do_sg * e; p.do_sn = do_sn * e; p.do_sb = do_sb * e; p.do_sh = do_sh * e;
    p.dst_lse = dst_lse; p.dl_sg = dl_sg; p.dl_sn = dl_sn; p.dl_sb = dl_sb; p.dl_sh = dl_sh;
    return launched(dcp::launch_pack(p, (cudaStream_t)stream), "dcp_pack_send");
}

// Shared tail of the two merge entry points once the views are validated.
static dcp_status_t run_merge(const char* who, int dtype, int e, int N, int B, int Hc, int D, int G,
                              const unsigned char* o, int64_t o_sg, int64_t o_sn, int64_t o_sb,
                              int64_t o_sh, const float* lse, int64_t l_sg, int64_t l_sn,
                              int64_t l_sb, int64_t l_sh, void* out, int64_t u_sg, int64_t u_sb,
                              int64_t u_sh, float* out_lse, int64_t ul_sg, int64_t ul_sb,
                              int64_t ul_sh, int lse_base, int return_lse, unsigned flags,
                              int in_align, int out_align, bool inplace, cudaStream_t stream) {
    const int64_t rb = (int64_t)D * e;
    if (N == 1) {
        // single rank: the input is returned unchanged (bit copy)
        if (inplace && !return_lse) return ok();
        dcp::PackParams p;
        p.N = 1; p.B = B; p.H = Hc; p.D = D; p.G = G; p.H_pr = Hc;
        p.rows = (int64_t)G * B * Hc;
        p.row_bytes = (int)rb;
        p.vb = pick_vb((int)rb, in_align, out_align, e);
        p.lpr = lanes_per_row((int)(rb / p.vb));
        p.copy_payload = inplace ? 0 : 1;
        p.copy_lse = return_lse ? 1 : 0;
        p.o = o; p.o_sg = o_sg; p.o_sb = o_sb; p.o_sh = o_sh;
        p.lse = lse; p.l_sg = l_sg; p.l_sb = l_sb; p.l_sh = l_sh;
        p.dst_o = (unsigned char*)out; p.do_sg = u_sg; p.do_sn = 0; p.do_sb = u_sb; p.do_sh = u_sh;
        p.dst_lse = out_lse; p.dl_sg = ul_sg; p.dl_sn = 0; p.dl_sb = ul_sb; p.dl_sh = ul_sh;
        return launched(dcp::launch_pack(p, stream), who);
    }
    dcp::CombineParams p;
    p.N = N; p.B = B; p.Hc = Hc; p.D = D; p.G = G;
    p.rows = (int64_t)G * B * Hc;
    const int vb = pick_vb((int)rb, in_align, out_align, e);
    p.vec_per_row = (int)(rb / vb);
    p.lpr = lanes_per_row(p.vec_per_row);
    p.base2 = lse_base == DCP_LSE_BASE_2;
    p.return_lse = return_lse ? 1 : 0;
    p.sanitize = (flags & DCP_SANITIZE_O) ? 1 : 0;
    p.o = o; p.o_sg = o_sg; p.o_sn = o_sn; p.o_sb = o_sb; p.o_sh = o_sh;
    p.lse = lse; p.l_sg = l_sg; p.l_sn = l_sn; p.l_sb = l_sb; p.l_sh = l_sh;
    p.out = (unsigned char*)out; p.u_sg = u_sg; p.u_sb = u_sb; p.u_sh = u_sh;
    p.out_lse = out_lse; p.ul_sg = ul_sg; p.ul_sb = ul_sb; p.ul_sh = ul_sh;
    cudaError_t err;
    switch (dtype) {
        case DCP_F32: err = dcp::launch_combine_f32(p, vb, stream); break;
        case DCP_F16: err = dcp::launch_combine_f16(p, vb, stream); break;
        case DCP_BF16: err = dcp::launch_combine_bf16(p, vb, stream); break;
        default: err = dcp::launch_combine_fp8(p, vb, stream); break;
    }
    return launched(err, who);
}

dcp_status_t dcp_lse_combine(int dtype, int N, int B, int Hc, int D, int G,
                             const void* o, int64_t o_sg, int64_t o_sn, int64_t o_sb, int64_t o_sh,
                             const float* lse, int64_t l_sg, int64_t l_sn, int64_t l_sb, int64_t l_sh,
                             void* out, int64_t u_sg, int64_t u_sb, int64_t u_sh,
                             float* out_lse, int64_t ul_sg, int64_t ul_sb, int64_t ul_sh,
                             int lse_base, int return_lse, unsigned flags, void* stream) {
    const char* who = "dcp_lse_combine";
    const int e = elem_size(dtype);
    if (!e) return fail(DCP_ERR_UNSUPPORTED_DTYPE, "%s: dtype %d", who, dtype);
    if (N < 1 || N > kMaxRanks || D < 1 || B < 0 || Hc < 0 || G < 0)
        return fail(DCP_ERR_INVALID_ARG, "%s: sizes N=%d B=%d Hc=%d D=%d G=%d", who, N, B, Hc, D, G);
    if ((int64_t)D * e > kMaxRowBytes)
        return fail(DCP_ERR_INVALID_ARG, "%s: rows of D=%d elements exceed 2^30 bytes", who, D);
    if (lse_base != DCP_LSE_BASE_E && lse_base != DCP_LSE_BASE_2)
        return fail(DCP_ERR_INVALID_ARG, "%s: lse_base %d", who, lse_base);
    if (flags & ~(unsigned)(DCP_SANITIZE_O | DCP_INPLACE_RANK0))
        return fail(DCP_ERR_INVALID_ARG, "%s: unknown flags 0x%x", who, flags);
    if (G == 0 || B == 0 || Hc == 0) return ok();
    if (!o || !lse || !out || (return_lse && !out_lse))
        return fail(DCP_ERR_INVALID_ARG, "%s: NULL pointer", who);
    if (bad_stride({o_sg, o_sn, o_sb, o_sh, l_sg, l_sn, l_sb, l_sh, u_sg, u_sb, u_sh}) ||
        (return_lse && bad_stride({ul_sg, ul_sb, ul_sh})))
        return fail(DCP_ERR_INVALID_ARG, "%s: negative stride or one above 2^52 elements", who);
    if ((uintptr_t)o % e || (uintptr_t)out % e || (uintptr_t)lse % 4 ||
        (return_lse && (uintptr_t)out_lse % 4))
        return fail(DCP_ERR_MISALIGNED, "%s: pointer not aligned to its element type", who);
    const bool inplace = (flags & DCP_INPLACE_RANK0) != 0;
    const int64_t rb = (int64_t)D * e;
    View vo = View(o, rb).dim(G, o_sg * e).dim(N, o_sn * e).dim(B, o_sb * e).dim(Hc, o_sh * e);
    View vl = View(lse, 4).dim(G, l_sg * 4).dim(N, l_sn * 4).dim(B, l_sb * 4).dim(Hc, l_sh * 4);
    View vu = View(out, rb).dim(G, u_sg * e).dim(B, u_sb * e).dim(Hc, u_sh * e);
    View vul = View(out_lse, 4).dim(G, ul_sg * 4).dim(B, ul_sb * 4).dim(Hc, ul_sh * 4);
    if (!all_fit({&vo, &vl, &vu}) || (return_lse && !vul.fits()))
        return fail(DCP_ERR_INVALID_ARG, "%s: an operand's strides span more than 2^56 bytes", who);
    if (inplace) {
        if (out != o || (G > 1 && u_sg != o_sg) || (B > 1 && u_sb != o_sb) || (Hc > 1 && u_sh != o_sh))
            return fail(DCP_ERR_INVALID_ARG,
                        "%s: DCP_INPLACE_RANK0 needs out == o with the rank-0 slice's strides", who);
        if (!vo.rows_disjoint())
            return fail(DCP_ERR_ALIAS, "%s: in-place combine over overlapping rank rows", who);
    } else if (overlap(vu, vo)) {
        return fail(DCP_ERR_ALIAS, "%s: out overlaps o (use DCP_INPLACE_RANK0 for in place)", who);
    }
    if (!fp8_rows_ok(e, D, vo.align(), vu.align()))
        return fail(DCP_ERR_MISALIGNED, "%s: fp8 rows need D %% 4 == 0 and 4-byte aligned row starts", who);
    if (overlap(vu, vl)) return fail(DCP_ERR_ALIAS, "%s: out overlaps lse", who);
    if (!vu.rows_disjoint()) return fail(DCP_ERR_ALIAS, "%s: out rows overlap one another", who);
    if (return_lse) {
        if (overlap(vul, vo) || overlap(vul, vl) || overlap(vul, vu))
            return fail(DCP_ERR_ALIAS, "%s: out_lse overlaps an input or out", who);
        if (!vul.rows_disjoint()) return fail(DCP_ERR_ALIAS, "%s: out_lse entries overlap", who);
    }
    return run_merge(who, dtype, e, N, B, Hc, D, G, (const unsigned char*)o, o_sg * e, o_sn * e,
                     o_sb * e, o_sh * e, lse, l_sg, l_sn, l_sb, l_sh, out, u_sg * e, u_sb * e,
                     u_sh * e, out_lse, ul_sg, ul_sb, ul_sh, lse_base, return_lse, flags,
                     vo.align(), vu.align(), inplace, (cudaStream_t)stream);
}

dcp_status_t dcp_unpack_combine(int dtype, int N, int B, int Hpr, int D, int G,
                                const void* recv, int64_t r_sg, int64_t r_sn, int64_t r_sb, int64_t r_sh,
                                void* out, int64_t u_sg, int64_t u_sb, int64_t u_sh,
                                float* out_lse, int64_t ul_sg, int64_t ul_sb, int64_t ul_sh,
                                int lse_base, int return_lse, unsigned flags, void* stream) {
    const char* who = "dcp_unpack_combine";
    const int e = elem_size(dtype);
    if (!e) return fail(DCP_ERR_UNSUPPORTED_DTYPE, "%s: dtype %d", who, dtype);
    if (N < 1 || N > kMaxRanks || D < 1 || B < 0 || Hpr < 0 || G < 0)
        return fail(DCP_ERR_INVALID_ARG, "%s: sizes N=%d B=%d Hpr=%d D=%d G=%d", who, N, B, Hpr, D, G);
    if ((int64_t)D * e > kMaxRowBytes)
        return fail(DCP_ERR_INVALID_ARG, "%s: rows of D=%d elements exceed 2^30 bytes", who, D);
    if (lse_base != DCP_LSE_BASE_E && lse_base != DCP_LSE_BASE_2)
        return fail(DCP_ERR_INVALID_ARG, "%s: lse_base %d", who, lse_base);
    if (flags & ~(unsigned)DCP_SANITIZE_O)
        return fail(DCP_ERR_INVALID_ARG, "%s: unsupported flags 0x%x", who, flags);
    const int lpd = 4 / e;
    if (D % lpd) return fail(DCP_ERR_MISALIGNED, "%s: D=%d is not a multiple of lpd=%d", who, D, lpd);
    if (G == 0 || B == 0 || Hpr == 0) return ok();
    if (!recv || !out || (return_lse && !out_lse))
        return fail(DCP_ERR_INVALID_ARG, "%s: NULL pointer", who);
    if (bad_stride({r_sg, r_sn, r_sb, r_sh, u_sg, u_sb, u_sh}) ||
        (return_lse && bad_stride({ul_sg, ul_sb, ul_sh})))
        return fail(DCP_ERR_INVALID_ARG, "%s: negative stride or one above 2^52 elements", who);
    if ((uintptr_t)out % e || (return_lse && (uintptr_t)out_lse % 4))
        return fail(DCP_ERR_MISALIGNED, "%s: pointer not aligned to its element type", who);
    const int64_t rb = (int64_t)D * e;
    View vr = View(recv, rb + 4).dim(G, r_sg * e).dim(N, r_sn * e).dim(B, r_sb * e).dim(Hpr, r_sh * e);
    View vu = View(out, rb).dim(G, u_sg * e).dim(B, u_sb * e).dim(Hpr, u_sh * e);
    View vul = View(out_lse, 4).dim(G, ul_sg * 4).dim(B, ul_sb * 4).dim(Hpr, ul_sh * 4);
    if (!all_fit({&vr, &vu}) || (return_lse && !vul.fits()))
        return fail(DCP_ERR_INVALID_ARG, "%s: an operand's strides span more than 2^56 bytes", who);
    if (vr.align() < 4)
        return fail(DCP_ERR_MISALIGNED, "%s: receive rows must start on 4-byte boundaries", who);
    if (!fp8_rows_ok(e, D, vr.align(), vu.align()))
        return fail(DCP_ERR_MISALIGNED, "%s: fp8 rows need 4-byte aligned row starts", who);
    // Rows that start 4 but not 16 bytes past a 16-byte boundary are read in
    // 16-byte chunks from that boundary, so up to 12 bytes before the first
    // row's start are read (and ignored): the outputs must not lie there.
    View vr_read = vr;
    vr_read.inner += (int64_t)(vr.base & 15u);
    vr_read.base &= ~(uintptr_t)15u;
    if (overlap(vu, vr_read)) return fail(DCP_ERR_ALIAS, "%s: out overlaps recv", who);
    if (!vu.rows_disjoint()) return fail(DCP_ERR_ALIAS, "%s: out rows overlap one another", who);
    if (return_lse) {
        if (overlap(vul, vr_read) || overlap(vul, vu))
            return fail(DCP_ERR_ALIAS, "%s: out_lse overlaps recv or out", who);
        if (!vul.rows_disjoint()) return fail(DCP_ERR_ALIAS, "%s: out_lse entries overlap", who);
    }
    // The LSE of each row is the fp32 word right after its payload: the same
    // rows seen as fp32 words, offset by D*e bytes.
    const unsigned char* rbase = (const unsigned char*)recv;
    const float* lse = (const float*)(rbase + rb);
    return run_merge(who, dtype, e, N, B, Hpr, D, G, rbase, r_sg * e, r_sn * e, r_sb * e, r_sh * e,
                     lse, r_sg * e / 4, r_sn * e / 4, r_sb * e / 4, r_sh * e / 4, out, u_sg * e,
                     u_sb * e, u_sh * e, out_lse, ul_sg, ul_sb, ul_sh, lse_base, return_lse, flags,
                     vr.align(), vu.align(), false, (cudaStream_t)stream);
}

// ---- decode attention per rank ------------------------------------------

static int attn_nsplit(int N, int max_seq_len, int split_tokens) {
    const int64_t lloc = ((int64_t)max_seq_len + N - 1) / N;
    const int64_t s = (lloc + split_tokens - 1) / split_tokens;
    return s < 1 ? 1 : (int)s;
}

// fp32 partial rows and their LSE words, one per (rank, request, head, split);
// SIZE_MAX when that does not fit in size_t.
static size_t attn_workspace_bytes(int N, int B, int H, int D, int nsplit) {
    if (nsplit <= 1) return 0;
    size_t rows = 1, bytes = 0;
    for (int f : {N, B, H, nsplit})
        if (__builtin_mul_overflow(rows, (size_t)f, &rows)) return SIZE_MAX;
    if (__builtin_mul_overflow(rows, (size_t)D * 4 + 4, &bytes)) return SIZE_MAX;
    return bytes;
}

size_t dcp_decode_attention_workspace_size(int N, int B, int H, int D, int max_seq_len, int split_tokens) {
    if (N < 1 || N > kMaxRanks || B < 0 || H < 1 || D < 1 || max_seq_len < 0 || split_tokens < 1) return 0;
    const size_t need = attn_workspace_bytes(N, B, H, D, attn_nsplit(N, max_seq_len, split_tokens));
    return need == SIZE_MAX ? 0 : need;
}

// Where the K/V rows live: per-request contiguous local caches, or pages of a
// per-rank pool addressed through a page table.
struct AttnKv {
    const void* k;
    int64_t k_sn, k_sb, k_st, k_sh;  // k_sb: request stride (contiguous) or page stride (paged)
    const void* v;
    int64_t v_sn, v_sb, v_st, v_sh;
    bool paged;
    int num_pages, page_size, max_pages;
    const int* bt;
    int64_t bt_sn, bt_sb;
};

static dcp_status_t run_attention(const char* who, int dtype, int N, int B, int H, int Hkv, int D,
                                  const void* q, int64_t q_sb, int64_t q_sh, const AttnKv& kv,
                                  const int* seq_lens, int max_seq_len, float sm_scale, int split_tokens,
                                  void* o, int64_t o_sn, int64_t o_sb, int64_t o_sh,
                                  float* lse, int64_t l_sn, int64_t l_sb, int64_t l_sh,
                                  int lse_base, void* workspace, size_t workspace_bytes, void* stream) {
    if (dtype != DCP_F16 && dtype != DCP_BF16)
        return fail(DCP_ERR_UNSUPPORTED_DTYPE, "%s: dtype %d (f16 or bf16 caches only)", who, dtype);
    const int e = 2;
    if (N < 1 || N > kMaxRanks || B < 0 || H < 1 || Hkv < 1 || max_seq_len < 0 || split_tokens < 1)
        return fail(DCP_ERR_INVALID_ARG, "%s: sizes N=%d B=%d H=%d Hkv=%d max_seq_len=%d split_tokens=%d",
                    who, N, B, H, Hkv, max_seq_len, split_tokens);
    if (H % Hkv) return fail(DCP_ERR_HEADS_NOT_DIVISIBLE, "%s: H=%d is not a multiple of Hkv=%d", who, H, Hkv);
    const int gq = H / Hkv;
    if (gq != 1 && gq != 2 && gq != 4 && gq != 8 && gq != 16)
        return fail(DCP_ERR_INVALID_ARG, "%s: H/Hkv=%d (1, 2, 4, 8 or 16 query heads per KV head)", who, gq);
    if (D != 64 && D != 128 && D != 256) return fail(DCP_ERR_INVALID_ARG, "%s: D=%d (64, 128 or 256)", who, D);
    if (gq == 16 && D > 128)
        return fail(DCP_ERR_INVALID_ARG, "%s: 16 query heads per KV head need D <= 128", who);
    if (!(sm_scale == sm_scale) || sm_scale == INFINITY || sm_scale == -INFINITY)
        return fail(DCP_ERR_INVALID_ARG, "%s: sm_scale is not finite", who);
    if (lse_base != DCP_LSE_BASE_E && lse_base != DCP_LSE_BASE_2)
        return fail(DCP_ERR_INVALID_ARG, "%s: lse_base %d", who, lse_base);
    const int64_t lcap = ((int64_t)max_seq_len + N - 1) / N;  // local tokens a rank may hold
    int page_shift = -1;
    if (kv.paged) {
        if (kv.page_size < 1 || kv.page_size > (1 << 16) || (kv.page_size & (kv.page_size - 1)))
            return fail(DCP_ERR_INVALID_ARG, "%s: page_size %d (a power of two up to 65536)", who, kv.page_size);
        page_shift = 0;
        while ((1 << page_shift) < kv.page_size) ++page_shift;
        if (kv.num_pages < 1) return fail(DCP_ERR_INVALID_ARG, "%s: num_pages %d", who, kv.num_pages);
        const int64_t need_pages = (lcap + kv.page_size - 1) / kv.page_size;
        if (kv.max_pages < need_pages)
            return fail(DCP_ERR_INVALID_ARG, "%s: page table rows of %d entries; %lld needed for %lld local tokens",
                        who, kv.max_pages, (long long)need_pages, (long long)lcap);
    }
    if (B == 0) return ok();
    const int nsplit = attn_nsplit(N, max_seq_len, split_tokens);
    if ((int64_t)N * B * Hkv * nsplit >= (1ll << 31))
        return fail(DCP_ERR_INVALID_ARG, "%s: too many work items (N*B*Hkv*splits >= 2^31)", who);
    if (!q || !kv.k || !kv.v || !seq_lens || !o || !lse || (kv.paged && !kv.bt))
        return fail(DCP_ERR_INVALID_ARG, "%s: NULL pointer", who);
    if (bad_stride({q_sb, q_sh, kv.k_sn, kv.k_sb, kv.k_st, kv.k_sh, kv.v_sn, kv.v_sb, kv.v_st, kv.v_sh, o_sn,
                      o_sb, o_sh, l_sn, l_sb, l_sh}) ||
        (kv.paged && bad_stride({kv.bt_sn, kv.bt_sb})))
        return fail(DCP_ERR_INVALID_ARG, "%s: negative stride or one above 2^52 elements", who);
    const int64_t rb = (int64_t)D * e;
    // K/V rows: [N][B, lcap] tokens of a contiguous cache, [N][num_pages, page_size] slots of a paged one
    const int64_t outer = kv.paged ? kv.num_pages : B;
    const int64_t inner = kv.paged ? kv.page_size : lcap;
    View vq = View(q, rb).dim(B, q_sb * e).dim(H, q_sh * e);
    View vk = View(kv.k, rb).dim(N, kv.k_sn * e).dim(outer, kv.k_sb * e).dim(inner, kv.k_st * e).dim(Hkv, kv.k_sh * e);
    View vv = View(kv.v, rb).dim(N, kv.v_sn * e).dim(outer, kv.v_sb * e).dim(inner, kv.v_st * e).dim(Hkv, kv.v_sh * e);
    View vo = View(o, rb).dim(N, o_sn * e).dim(B, o_sb * e).dim(H, o_sh * e);
    View vl = View(lse, 4).dim(N, l_sn * 4).dim(B, l_sb * 4).dim(H, l_sh * 4);
    View vs = View(seq_lens, 4).dim(B, 4);
    View vt = kv.paged ? View(kv.bt, 4).dim(N, kv.bt_sn * 4).dim(B, kv.bt_sb * 4).dim(kv.max_pages, 4)
                       : View(nullptr, 0);
    if (!all_fit({&vq, &vk, &vv, &vo, &vl, &vs, &vt}))
        return fail(DCP_ERR_INVALID_ARG, "%s: an operand's strides span more than 2^56 bytes", who);
    if (vq.align() < 16 || vk.align() < 16 || vv.align() < 16)
        return fail(DCP_ERR_MISALIGNED, "%s: q, k and v rows must start on 16-byte boundaries", who);
    if ((uintptr_t)o % e || (uintptr_t)lse % 4 || (uintptr_t)seq_lens % 4 || (uintptr_t)kv.bt % 4)
        return fail(DCP_ERR_MISALIGNED, "%s: pointer not aligned to its element type", who);
    for (const View* in : {&vq, &vk, &vv, &vs, &vt})
        if (overlap(vo, *in) || overlap(vl, *in))
            return fail(DCP_ERR_ALIAS, "%s: an output overlaps an input", who);
    if (overlap(vo, vl) || !vo.rows_disjoint() || !vl.rows_disjoint())
        return fail(DCP_ERR_ALIAS, "%s: outputs overlap", who);
    const size_t need = attn_workspace_bytes(N, B, H, D, nsplit);
    if (need) {
        if (!workspace || workspace_bytes < need)
            return fail(DCP_ERR_INVALID_ARG, "%s: workspace of %zu bytes needed (%zu given)", who, need,
                        workspace ? workspace_bytes : (size_t)0);
        if ((uintptr_t)workspace % 16) return fail(DCP_ERR_MISALIGNED, "%s: workspace not 16-byte aligned", who);
        View vw = View(workspace, (int64_t)need);
        for (const View* other : {&vq, &vk, &vv, &vs, &vt, &vo, &vl})
            if (overlap(vw, *other)) return fail(DCP_ERR_ALIAS, "%s: workspace overlaps an operand", who);
    }
    dcp::AttnParams p;
    p.N = N; p.B = B; p.H = H; p.Hkv = Hkv; p.D = D;
    p.max_seq_len = max_seq_len; p.split_tokens = split_tokens; p.nsplit = nsplit;
    p.base2 = lse_base == DCP_LSE_BASE_2;
    p.sm_scale = sm_scale;
    p.q = (const unsigned char*)q; p.q_sb = q_sb * e; p.q_sh = q_sh * e;
    p.k = (const unsigned char*)kv.k; p.k_sn = kv.k_sn * e; p.k_st = kv.k_st * e; p.k_sh = kv.k_sh * e;
    p.v = (const unsigned char*)kv.v; p.v_sn = kv.v_sn * e; p.v_st = kv.v_st * e; p.v_sh = kv.v_sh * e;
    p.k_sb = kv.paged ? 0 : kv.k_sb * e;
    p.v_sb = kv.paged ? 0 : kv.v_sb * e;
    p.k_sp = kv.paged ? kv.k_sb * e : 0;
    p.v_sp = kv.paged ? kv.v_sb * e : 0;
    p.bt = kv.bt; p.bt_sn = kv.bt_sn; p.bt_sb = kv.bt_sb;
    p.page_shift = page_shift;
    p.num_pages = kv.paged ? kv.num_pages : 0;
    p.seq_lens = seq_lens;
    p.o = (unsigned char*)o; p.o_sn = o_sn * e; p.o_sb = o_sb * e; p.o_sh = o_sh * e;
    p.lse = lse; p.l_sn = l_sn; p.l_sb = l_sb; p.l_sh = l_sh;
    const size_t rows = (size_t)N * B * H * nsplit;
    p.ws_o = need ? (float*)workspace : nullptr;
    p.ws_lse = need ? (float*)workspace + rows * D : nullptr;
    p.stall_loads = 0;
    p.merge_multi_only = 0;
    cudaError_t le;
    if (!dcp::launch_decode_attention_tc(p, dtype, (cudaStream_t)stream, &le))
        le = dcp::launch_decode_attention(p, dtype, (cudaStream_t)stream);
    return launched(le, who);
}

dcp_status_t dcp_decode_attention(int dtype, int N, int B, int H, int Hkv, int D,
                                  const void* q, int64_t q_sb, int64_t q_sh,
                                  const void* k, int64_t k_sn, int64_t k_sb, int64_t k_st, int64_t k_sh,
                                  const void* v, int64_t v_sn, int64_t v_sb, int64_t v_st, int64_t v_sh,
                                  const int* seq_lens, int max_seq_len, float sm_scale, int split_tokens,
                                  void* o, int64_t o_sn, int64_t o_sb, int64_t o_sh,
                                  float* lse, int64_t l_sn, int64_t l_sb, int64_t l_sh,
                                  int lse_base, void* workspace, size_t workspace_bytes, void* stream) {
    AttnKv kv{k, k_sn, k_sb, k_st, k_sh, v, v_sn, v_sb, v_st, v_sh, false, 0, 0, 0, nullptr, 0, 0};
    return run_attention("dcp_decode_attention", dtype, N, B, H, Hkv, D, q, q_sb, q_sh, kv, seq_lens,
                         max_seq_len, sm_scale, split_tokens, o, o_sn, o_sb, o_sh, lse, l_sn, l_sb, l_sh,
                         lse_base, workspace, workspace_bytes, stream);
}

dcp_status_t dcp_decode_attention_paged(int dtype, int N, int B, int H, int Hkv, int D,
                                        const void* q, int64_t q_sb, int64_t q_sh,
                                        const void* k_pages, int64_t k_sn, int64_t k_sp, int64_t k_st, int64_t k_sh,
                                        const void* v_pages, int64_t v_sn, int64_t v_sp, int64_t v_st, int64_t v_sh,
                                        int num_pages, int page_size,
                                        const int* block_table, int64_t bt_sn, int64_t bt_sb, int max_pages,
                                        const int* seq_lens, int max_seq_len, float sm_scale, int split_tokens,
                                        void* o, int64_t o_sn, int64_t o_sb, int64_t o_sh,
                                        float* lse, int64_t l_sn, int64_t l_sb, int64_t l_sh,
                                        int lse_base, void* workspace, size_t workspace_bytes, void* stream) {
    AttnKv kv{k_pages, k_sn, k_sp, k_st, k_sh, v_pages, v_sn, v_sp, v_st, v_sh, true,
              num_pages, page_size, max_pages, block_table, bt_sn, bt_sb};
    return run_attention("dcp_decode_attention_paged", dtype, N, B, H, Hkv, D, q, q_sb, q_sh, kv, seq_lens,
                         max_seq_len, sm_scale, split_tokens, o, o_sn, o_sb, o_sh, lse, l_sn, l_sb, l_sh,
                         lse_base, workspace, workspace_bytes, stream);
}

dcp_status_t dcp_decode_attention_mla(int dtype, int N, int B, int H, int Dk, int Dv,
                                      const void* q, int64_t q_sb, int64_t q_sh,
                                      const void* kv, int64_t kv_sn, int64_t kv_sb, int64_t kv_st,
                                      const int* seq_lens, int max_seq_len, float sm_scale, int split_tokens,
                                      void* o, int64_t o_sn, int64_t o_sb, int64_t o_sh,
                                      float* lse, int64_t l_sn, int64_t l_sb, int64_t l_sh,
                                      int lse_base, void* workspace, size_t workspace_bytes, void* stream) {
    const char* who = "dcp_decode_attention_mla";
    if (dtype != DCP_F16 && dtype != DCP_BF16)
        return fail(DCP_ERR_UNSUPPORTED_DTYPE, "%s: dtype %d (f16 or bf16 caches only)", who, dtype);
    const int e = 2;
    if (N < 1 || N > kMaxRanks || B < 0 || H < 1 || max_seq_len < 0)
        return fail(DCP_ERR_INVALID_ARG, "%s: sizes N=%d B=%d H=%d max_seq_len=%d", who, N, B, H, max_seq_len);
    if (H > 128) return fail(DCP_ERR_INVALID_ARG, "%s: H=%d query heads (at most 128)", who, H);
    if (Dk != 576 || Dv != 512)
        return fail(DCP_ERR_INVALID_ARG, "%s: Dk=%d Dv=%d (latent rows of 576 = 512 + 64 rope, value 512)", who,
                    Dk, Dv);
    if (split_tokens < 64 || split_tokens % 64)
        return fail(DCP_ERR_INVALID_ARG, "%s: split_tokens=%d (a positive multiple of 64)", who, split_tokens);
    if (!(sm_scale == sm_scale) || sm_scale == INFINITY || sm_scale == -INFINITY)
        return fail(DCP_ERR_INVALID_ARG, "%s: sm_scale is not finite", who);
    if (lse_base != DCP_LSE_BASE_E && lse_base != DCP_LSE_BASE_2)
        return fail(DCP_ERR_INVALID_ARG, "%s: lse_base %d", who, lse_base);
    if (B == 0) return ok();
    const int64_t lcap = ((int64_t)max_seq_len + N - 1) / N;
    const int nsplit = attn_nsplit(N, max_seq_len, split_tokens);
    if (2 * (int64_t)N * B * nsplit >= (1ll << 31))
        return fail(DCP_ERR_INVALID_ARG, "%s: too many work items (2*N*B*splits >= 2^31)", who);
    if (!q || !kv || !seq_lens || !o || !lse) return fail(DCP_ERR_INVALID_ARG, "%s: NULL pointer", who);
    if (bad_stride({q_sb, q_sh, kv_sn, kv_sb, kv_st, o_sn, o_sb, o_sh, l_sn, l_sb, l_sh}))
        return fail(DCP_ERR_INVALID_ARG, "%s: negative stride or one above 2^52 elements", who);
    // the cache is read by TMA as a [N][B][lcap][576] tensor: 16-byte aligned
    // base, strides that are nonzero multiples of 16 bytes below 2^40
    for (int64_t st : {kv_sn, kv_sb, kv_st})
        if (st <= 0 || st % 8 || st * e >= (int64_t(1) << 40))
            return fail(DCP_ERR_MISALIGNED, "%s: cache strides must be positive multiples of 8 elements below 2^39",
                        who);
    if (kv_st < Dk) return fail(DCP_ERR_INVALID_ARG, "%s: token stride %lld below the row of %d elements", who,
                                (long long)kv_st, Dk);
    // the queries' rope columns are read by TMA as well: byte strides below 2^40
    if (q_sb * e >= (int64_t(1) << 40) || q_sh * e >= (int64_t(1) << 40))
        return fail(DCP_ERR_INVALID_ARG, "%s: query strides must be below 2^39 elements", who);
    if ((uintptr_t)kv % 16) return fail(DCP_ERR_MISALIGNED, "%s: cache not 16-byte aligned", who);
    View vq = View(q, (int64_t)Dk * e).dim(B, q_sb * e).dim(H, q_sh * e);
    View vk = View(kv, (int64_t)Dk * e).dim(N, kv_sn * e).dim(B, kv_sb * e).dim(lcap, kv_st * e);
    View vo = View(o, (int64_t)Dv * e).dim(N, o_sn * e).dim(B, o_sb * e).dim(H, o_sh * e);
    View vl = View(lse, 4).dim(N, l_sn * 4).dim(B, l_sb * 4).dim(H, l_sh * 4);
    View vs = View(seq_lens, 4).dim(B, 4);
    if (!all_fit({&vq, &vk, &vo, &vl, &vs}))
        return fail(DCP_ERR_INVALID_ARG, "%s: an operand's strides span more than 2^56 bytes", who);
    if (vq.align() < 16 || vo.align() < 16)
        return fail(DCP_ERR_MISALIGNED, "%s: q and o rows must start on 16-byte boundaries", who);
    if ((uintptr_t)lse % 4 || (uintptr_t)seq_lens % 4)
        return fail(DCP_ERR_MISALIGNED, "%s: pointer not aligned to its element type", who);
    for (const View* in : {&vq, &vk, &vs})
        if (overlap(vo, *in) || overlap(vl, *in)) return fail(DCP_ERR_ALIAS, "%s: an output overlaps an input", who);
    if (overlap(vo, vl) || !vo.rows_disjoint() || !vl.rows_disjoint())
        return fail(DCP_ERR_ALIAS, "%s: outputs overlap", who);
    const size_t need = attn_workspace_bytes(N, B, H, Dv, nsplit);
    if (need) {
        if (!workspace || workspace_bytes < need)
            return fail(DCP_ERR_INVALID_ARG, "%s: workspace of %zu bytes needed (%zu given)", who, need,
                        workspace ? workspace_bytes : (size_t)0);
        if ((uintptr_t)workspace % 16) return fail(DCP_ERR_MISALIGNED, "%s: workspace not 16-byte aligned", who);
        View vw = View(workspace, (int64_t)need);
        for (const View* other : {&vq, &vk, &vs, &vo, &vl})
            if (overlap(vw, *other)) return fail(DCP_ERR_ALIAS, "%s: workspace overlaps an operand", who);
    }
    dcp::MlaParams p;
    p.N = N; p.B = B; p.H = H; p.lcap = lcap;
    p.max_seq_len = max_seq_len; p.split_tokens = split_tokens; p.nsplit = nsplit;
    p.base2 = lse_base == DCP_LSE_BASE_2;
    p.sm_scale = sm_scale;
    p.q = (const unsigned char*)q; p.q_sb = q_sb * e; p.q_sh = q_sh * e;
    p.kv = (const unsigned char*)kv; p.kv_sn = kv_sn * e; p.kv_sb = kv_sb * e; p.kv_st = kv_st * e;
    p.seq_lens = seq_lens;
    p.o = (unsigned char*)o; p.o_sn = o_sn * e; p.o_sb = o_sb * e; p.o_sh = o_sh * e;
    p.lse = lse; p.l_sn = l_sn; p.l_sb = l_sb; p.l_sh = l_sh;
    const size_t rows = (size_t)N * B * H * nsplit;
    p.ws_o = need ? (float*)workspace : nullptr;
    p.ws_lse = need ? (float*)workspace + rows * Dv : nullptr;
    p.stall_loads = 0;
    const cudaError_t le = dcp::launch_mla_decode(p, dtype, (cudaStream_t)stream);
    if (le == cudaErrorNotSupported)
        return fail(DCP_ERR_CUDA, "%s: the driver offers no tensor-map encoder (cuTensorMapEncodeTiled)", who);
    return launched(le, who);
}

dcp_status_t dcp_device_status(void) {
    const int s_mla = dcp::mla_device_status(true);
    const int s_gqa = dcp::attn_tc_device_status(true);
    const int s = s_mla < 0 || s_gqa < 0 ? -1 : (s_mla ? s_mla : s_gqa);
    if (s < 0) return fail(DCP_ERR_CUDA, "dcp_device_status: the device status word could not be read");
    if (s) return fail((dcp_status_t)s, "dcp_device_status: a tensor-core kernel gave up on a bounded wait");
    return ok();
}

}  // extern "C"
