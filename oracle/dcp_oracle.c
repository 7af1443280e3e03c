/*
 * dcp_oracle.c -- plain, slow, fp64 CPU oracle for the decode-context-parallel
 * (DCP) LSE merge.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file: only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or helper with the CUDA
 * library; it reads only its own arguments.
 *
 * Every function below is the plain definition of one step, written as
 * nested loops in the order the pages state it:
 *
 *   oracle_pack           sglang PR #34651 report, "实现拆解" item 1 and the
 *                         test `test_pack_serves_the_split_peer_inside_layout`
 *                         ("关键源码片段"); vLLM PR #41160 report, "实现拆解"
 *                         items 1-2 (`_dcp_a2a_pack_send_kernel`,
 *                         `_dcp_a2a_lse_pack_dim`).
 *   oracle_combine        sglang PR #34213 report, "关键源码片段"
 *                         (`cp_lse_ag_out_rs_mha`: logsumexp over the rank
 *                         stack, exp(lse - global), nan_to_num, weighted sum,
 *                         single-rank early return, in-place nan_to_num_ of O);
 *                         sglang PR #34651 report, "实现拆解" item 3
 *                         (`dcp_lse_combine_triton`, strided receive views);
 *                         sglang PR #33926 report, "实现拆解" item 4 (base-2
 *                         versus natural-log LSE).
 *   oracle_unpack_combine vLLM PR #41160 report, "实现拆解" item 1
 *                         (`_dcp_a2a_unpack_combine_kernel`): the combine
 *                         applied to rows whose LSE word follows the payload.
 *   oracle_dcp_lens       sglang PR #33926 report, "关键源码片段"
 *                         (`_get_dcp_local_max_seq_len`, `TestDcpDecodeLayout`):
 *                         round-robin KV ownership, token t on rank t % n.
 *   oracle_split_attention sglang PR #33926 report, "实现拆解" item 3
 *                         (each rank returns rank-local (out, lse); a rank
 *                         owning no KV is neutralised to (0, -inf)).
 *   oracle_split_attention_mla  the same over a latent cache (absorbed MLA,
 *                         the trtllm_mla decode path of that report): the
 *                         score uses the whole latent row, the value is its
 *                         first kv_lora_rank elements.
 *
 * Readings taken where the pages are silent (each is also listed in the
 * design notes):
 *   - logsumexp over extended reals: any NaN -> NaN; else any +inf -> +inf;
 *     else all -inf -> -inf; else finite (the semantics of the torch
 *     logsumexp the sglang #34213 code calls).
 *   - A single rank (N == 1) returns its input unchanged (sglang #34213's
 *     early return), for every entry point.
 *   - The returned LSE is in the same base as the input LSE.
 *   - O is set to 0 where it is NaN/+-inf only when the caller asks for it
 *     (flag ORACLE_SANITIZE_O; sglang #34213's nan_to_num_); otherwise
 *     out = sum_r w_r * O_r in IEEE arithmetic.
 *   - bf16 takes two output elements per LSE word, like fp16.
 *
 * Conventions: all strides are in elements of the pointed-to type (payload
 * elements for O, fp32 words for LSE); the innermost (D) stride is 1.
 * dtype codes: 0 = fp32, 1 = fp16, 2 = bf16, 3 = fp64 (fp64 payloads exist only
 * so that the self-checks can run the merge without input rounding), 4 = fp8
 * e4m3.  fp8 payloads extend the pages: vLLM PR #41160 report, "风险与影响",
 * notes that the LSE pack dimension rejects fp8 (ValueError); here an fp32
 * LSE word occupies four one-byte elements (lpd = 4).
 * base codes: 0 = e, 1 = 2.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_F16 1
#define ORACLE_BF16 2
#define ORACLE_F64 3
#define ORACLE_FP8 4
#define ORACLE_BASE_E 0
#define ORACLE_BASE_2 1
#define ORACLE_SANITIZE_O 1u

/* ln 2, the factor between base-2 and natural-log LSE values. */
static double ln2(void) { return log(2.0); }

static int elem_bytes(int dtype) {
    return dtype == ORACLE_F64 ? 8 : dtype == ORACLE_F32 ? 4 : dtype == ORACLE_FP8 ? 1 : 2;
}

/* ---- element decoding (IEEE binary16 / bfloat16 / binary32 -> double) ---- */

static double decode_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 0x1f;
    int man = h & 0x3ff;
    double v;
    if (ex == 0) {
        v = ldexp((double)man, -24); /* subnormal: man * 2^-24 */
    } else if (ex == 31) {
        v = man ? NAN : INFINITY;
    } else {
        v = ldexp((double)(man + 1024), ex - 25); /* (1.man) * 2^(ex-15) */
    }
    return sign ? -v : v;
}

/* fp8 e4m3 ("fn" variant: no infinities): 1 sign, 4 exponent bits (bias 7),
 * 3 mantissa bits; exponent and mantissa all ones is NaN. */
static double decode_fp8_e4m3(uint8_t b) {
    int sign = (b >> 7) & 1;
    int ex = (b >> 3) & 0xf;
    int man = b & 0x7;
    double v;
    if (ex == 15 && man == 7) {
        v = NAN;
    } else if (ex == 0) {
        v = ldexp((double)man, -9); /* subnormal: man * 2^-9 */
    } else {
        v = ldexp((double)(man + 8), ex - 10); /* (1.man) * 2^(ex-7) */
    }
    return sign ? -v : v;
}

static double decode_bf16(uint16_t h) {
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

static double load_elem(const void* base, int dtype, int64_t idx) {
    const unsigned char* p = (const unsigned char*)base + idx * elem_bytes(dtype);
    if (dtype == ORACLE_F64) {
        double v;
        memcpy(&v, p, 8);
        return v;
    }
    if (dtype == ORACLE_F32) {
        float f;
        memcpy(&f, p, 4);
        return (double)f;
    }
    if (dtype == ORACLE_FP8) return decode_fp8_e4m3(*p);
    uint16_t h;
    memcpy(&h, p, 2);
    return dtype == ORACLE_F16 ? decode_f16(h) : decode_bf16(h);
}

/* Public so that tests can pin the decoders against numpy's own. */
double oracle_decode_elem(int dtype, const void* base, int64_t idx) {
    return load_elem(base, dtype, idx);
}

/* ---- lse_pack_dim: payload elements one fp32 LSE word occupies ---------- */
/* vLLM #41160 "实现拆解" item 2: fp16 -> 2, fp32 -> 1, others rejected. */
int oracle_lse_pack_dim(int dtype) {
    if (dtype == ORACLE_F32) return 1;
    if (dtype == ORACLE_F16 || dtype == ORACLE_BF16) return 2;
    if (dtype == ORACLE_FP8) return 4; /* extension: four one-byte elements per word */
    return -1;
}

/* ---- pack ---------------------------------------------------------------- */
/*
 * For every source group g, token b and head h of O[g][B,H,D]:
 *   peer p = h / H_pr, local head hl = h % H_pr            (H_pr = H / N)
 *   dst_o[g][p, b, hl, 0:D]  <- the bytes of O[g][b, h, 0:D]
 *   dst_lse[g][p, b, hl]     <- the bytes of lse[g][b, h]
 * Nothing else is written.  The same strides describe both the peer-major
 * interleaved send buffer and the peer-inside split layout.
 * Returns 0, or -1 when H is not a multiple of N.
 */
int oracle_pack(int dtype, int N, int B, int H, int D, int G,
                const void* o, int64_t o_sg, int64_t o_sb, int64_t o_sh,
                const float* lse, int64_t l_sg, int64_t l_sb, int64_t l_sh,
                void* dst_o, int64_t do_sg, int64_t do_sn, int64_t do_sb, int64_t do_sh,
                float* dst_lse, int64_t dl_sg, int64_t dl_sn, int64_t dl_sb, int64_t dl_sh) {
    if (N <= 0 || H % N != 0) return -1;
    const int e = elem_bytes(dtype);
    const int H_pr = H / N;
    for (int g = 0; g < G; ++g)
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < H; ++h) {
                const int p = h / H_pr;
                const int hl = h % H_pr;
                const unsigned char* src =
                    (const unsigned char*)o + (g * o_sg + b * o_sb + h * o_sh) * e;
                unsigned char* dst = (unsigned char*)dst_o +
                                     (g * do_sg + p * do_sn + b * do_sb + hl * do_sh) * e;
                for (int d = 0; d < D; ++d)
                    for (int k = 0; k < e; ++k) dst[d * e + k] = src[d * e + k];
                memcpy(&dst_lse[g * dl_sg + p * dl_sn + b * dl_sb + hl * dl_sh],
                       &lse[g * l_sg + b * l_sb + h * l_sh], 4);
            }
    return 0;
}

/* Ranks one merge may take: as many as the library under test accepts. */
#define ORACLE_MAX_RANKS 4096

/* ---- the merge of one row ------------------------------------------------ */
/*
 * x[r]   : the N rank LSE values, already in natural-log units
 * rows[r]: pointer to rank r's payload row (dtype elements, unit stride)
 * out    : D doubles; *G_out: the global LSE in natural-log units
 *
 *   G   = logsumexp_r x[r]                       (extended reals, see header)
 *   w_r = exp(x[r] - G), set to 0 when not finite  (nan_to_num(scale, 0, 0, 0))
 *   o   = O_r[d], set to 0 when not finite if ORACLE_SANITIZE_O
 *   out[d] = sum over r = 0..N-1 of w_r * o
 */
static double logsumexp_ext(int N, const double* x) {
    int any_nan = 0, any_pinf = 0;
    double m = -INFINITY;
    for (int r = 0; r < N; ++r) {
        if (isnan(x[r])) any_nan = 1;
        else if (x[r] == INFINITY) any_pinf = 1;
        else if (x[r] > m) m = x[r];
    }
    if (any_nan) return NAN;
    if (any_pinf) return INFINITY;
    if (m == -INFINITY) return -INFINITY;
    double s = 0.0;
    for (int r = 0; r < N; ++r) s += exp(x[r] - m);
    return m + log(s);
}

static void merge_row(int dtype, int N, int D, const double* x, const void* const* rows,
                      unsigned flags, double* out, double* G_out) {
    double w[ORACLE_MAX_RANKS];
    const double G = logsumexp_ext(N, x);
    for (int r = 0; r < N; ++r) {
        w[r] = exp(x[r] - G);
        if (!isfinite(w[r])) w[r] = 0.0;
    }
    for (int d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int r = 0; r < N; ++r) {
            double o = load_elem(rows[r], dtype, d);
            if ((flags & ORACLE_SANITIZE_O) && !isfinite(o)) o = 0.0;
            acc += w[r] * o;
        }
        out[d] = acc;
    }
    *G_out = G;
}

/* Base-2 LSE values are converted to natural-log units on the way in
 * (x = l * ln 2) and the global LSE is converted back (G / ln 2). */
static double to_nat(double l, int base) { return base == ORACLE_BASE_2 ? l * ln2() : l; }
static double from_nat(double G, int base) { return base == ORACLE_BASE_2 ? G / ln2() : G; }

/* ---- combine over strided O and LSE views -------------------------------- */
/*
 * O viewed as [G][N, B, Hc, D], LSE as [G][N, B, Hc] (fp32 words).
 * out: contiguous double [G, B, Hc, D]; out_lse: contiguous double [G, B, Hc].
 * N == 1 returns O and lse unchanged (converted to double), for every row.
 * Returns 0, or -1 for N outside 1..ORACLE_MAX_RANKS.
 */
int oracle_combine(int dtype, int N, int B, int Hc, int D, int G,
                   const void* o, int64_t o_sg, int64_t o_sn, int64_t o_sb, int64_t o_sh,
                   const float* lse, int64_t l_sg, int64_t l_sn, int64_t l_sb, int64_t l_sh,
                   double* out, double* out_lse, int base, unsigned flags) {
    if (N <= 0 || N > ORACLE_MAX_RANKS) return -1;
    const int e = elem_bytes(dtype);
    double x[ORACLE_MAX_RANKS];
    const void* rows[ORACLE_MAX_RANKS];
    for (int g = 0; g < G; ++g)
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < Hc; ++h) {
                const int64_t row = ((int64_t)g * B + b) * Hc + h;
                double* orow = out + row * D;
                if (N == 1) {
                    const void* src = (const unsigned char*)o + (g * o_sg + b * o_sb + h * o_sh) * e;
                    for (int d = 0; d < D; ++d) orow[d] = load_elem(src, dtype, d);
                    out_lse[row] = (double)lse[g * l_sg + b * l_sb + h * l_sh];
                    continue;
                }
                for (int r = 0; r < N; ++r) {
                    x[r] = to_nat((double)lse[g * l_sg + r * l_sn + b * l_sb + h * l_sh], base);
                    rows[r] = (const unsigned char*)o + (g * o_sg + r * o_sn + b * o_sb + h * o_sh) * e;
                }
                double Gn;
                merge_row(dtype, N, D, x, rows, flags, orow, &Gn);
                out_lse[row] = from_nat(Gn, base);
            }
    return 0;
}

/* ---- fused unpack + combine over the interleaved receive buffer ---------- */
/*
 * recv viewed as [G][N, B, Hpr, D + lpd] (payload elements).  In each row the
 * first D elements are rank r's partial O and the fp32 word at word index
 * D / lpd (bytes D*e .. D*e+3 from the row start) is its LSE.
 * Returns 0, -1 for bad N, -2 when D is not a multiple of lpd.
 */
int oracle_unpack_combine(int dtype, int N, int B, int Hpr, int D, int G,
                          const void* recv, int64_t r_sg, int64_t r_sn, int64_t r_sb, int64_t r_sh,
                          double* out, double* out_lse, int base, unsigned flags) {
    if (N <= 0 || N > ORACLE_MAX_RANKS) return -1;
    const int lpd = oracle_lse_pack_dim(dtype);
    if (lpd <= 0 || D % lpd != 0) return -2;
    const int e = elem_bytes(dtype);
    double x[ORACLE_MAX_RANKS];
    const void* rows[ORACLE_MAX_RANKS];
    for (int g = 0; g < G; ++g)
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < Hpr; ++h) {
                const int64_t row = ((int64_t)g * B + b) * Hpr + h;
                double* orow = out + row * D;
                for (int r = 0; r < N; ++r) {
                    const unsigned char* rp =
                        (const unsigned char*)recv + (g * r_sg + r * r_sn + b * r_sb + h * r_sh) * e;
                    float lw;
                    memcpy(&lw, rp + (int64_t)D * e, 4);
                    x[r] = (double)lw;
                    rows[r] = rp;
                }
                if (N == 1) {
                    for (int d = 0; d < D; ++d) orow[d] = load_elem(rows[0], dtype, d);
                    out_lse[row] = x[0];
                    continue;
                }
                for (int r = 0; r < N; ++r) x[r] = to_nat(x[r], base);
                double Gn;
                merge_row(dtype, N, D, x, rows, flags, orow, &Gn);
                out_lse[row] = from_nat(Gn, base);
            }
    return 0;
}

/* ---- round-robin KV ownership ------------------------------------------- */
/* Token t of a length-L sequence lives on rank t % n, so rank r holds
 * L / n tokens, plus one when r < L % n. */
int64_t oracle_dcp_lens(int64_t L, int n, int r) {
    return L / n + (r < L % n ? 1 : 0);
}

/* ---- split single-query attention (brute force, for self-checks) -------- */
/*
 * q [D], K [L, D], V [L, D] (double).  Rank r attends over the tokens it owns
 * (t % n == r) with scores s_t = scale * <q, K_t>:
 *   lse_r = log sum_t exp(s_t)          (natural log; base 2: lse_r / ln 2)
 *   O_r   = sum_t exp(s_t - lse_r) V_t
 * A rank that owns no token returns (O = 0, lse = -inf).
 * O: [n, D]; lse: [n].
 */
void oracle_split_attention(int L, int D, int n, double scale, const double* q,
                            const double* K, const double* V, int base, double* O,
                            double* lse) {
    for (int r = 0; r < n; ++r) {
        double m = -INFINITY;
        int owned = 0;
        for (int t = r; t < L; t += n) {
            double s = 0.0;
            for (int d = 0; d < D; ++d) s += q[d] * K[(int64_t)t * D + d];
            s *= scale;
            if (s > m) m = s;
            owned = 1;
        }
        for (int d = 0; d < D; ++d) O[(int64_t)r * D + d] = 0.0;
        if (!owned) {
            lse[r] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int t = r; t < L; t += n) {
            double s = 0.0;
            for (int d = 0; d < D; ++d) s += q[d] * K[(int64_t)t * D + d];
            sum += exp(s * scale - m);
        }
        const double l = m + log(sum);
        for (int t = r; t < L; t += n) {
            double s = 0.0;
            for (int d = 0; d < D; ++d) s += q[d] * K[(int64_t)t * D + d];
            const double p = exp(s * scale - l);
            for (int d = 0; d < D; ++d) O[(int64_t)r * D + d] += p * V[(int64_t)t * D + d];
        }
        lse[r] = base == ORACLE_BASE_2 ? l / ln2() : l;
    }
}

/* ---- split single-query attention over a latent cache (absorbed MLA) ---- */
/*
 * sglang PR #33926 report, "功能与动机" and "实现拆解" items 3-4: the trtllm_mla
 * decode path (absorbed multi-head latent attention, DeepSeek-V3 class) returns
 * rank-local (out, lse) under the round-robin owner rule; sglang PR #34213
 * report, "功能与动机": for absorbed MLA the output width is kv_lora_rank.
 * Every query head scores one shared latent row per token,
 *   KV_t [Dk] = [ c_t (Dv elements, kv_lora_rank) | k_rope_t (Dk - Dv elements) ],
 * against its absorbed query q [Dk] (the query's rope part concatenated after
 * its absorbed no-rope part), and the value is the row's first Dv elements:
 *   s_t   = scale <q, KV_t>                         (all Dk elements)
 *   lse_r = log sum_{t owned by r} exp(s_t)         (base 2: lse_r / ln 2)
 *   O_r   = sum_{t owned by r} exp(s_t - lse_r) KV_t[0:Dv]
 * A rank that owns no token returns (O = 0, lse = -inf).
 * q [Dk], KV [L, Dk] (double); O: [n, Dv]; lse: [n].
 */
/* <q, KV_t> over the whole latent row. */
static double latent_dot(const double* q, const double* row, int Dk) {
    double acc = 0.0;
    for (int d = 0; d < Dk; ++d) acc += q[d] * row[d];
    return acc;
}

void oracle_split_attention_mla(int L, int Dk, int Dv, int n, double scale, const double* q,
                                const double* KV, int base, double* O, double* lse) {
    for (int r = 0; r < n; ++r) {
        double* Or = O + (int64_t)r * Dv;
        for (int d = 0; d < Dv; ++d) Or[d] = 0.0;
        lse[r] = -INFINITY; /* the neutral pair, kept when rank r owns no token (none when r >= L) */
        if (r >= L) continue;
        double smax = -INFINITY;
        for (int t = r; t < L; t += n) smax = fmax(smax, scale * latent_dot(q, KV + (int64_t)t * Dk, Dk));
        double z = 0.0;
        for (int t = r; t < L; t += n) z += exp(scale * latent_dot(q, KV + (int64_t)t * Dk, Dk) - smax);
        const double lse_nat = smax + log(z);
        for (int t = r; t < L; t += n) {
            const double* row = KV + (int64_t)t * Dk;
            const double prob = exp(scale * latent_dot(q, row, Dk) - lse_nat);
            for (int d = 0; d < Dv; ++d) Or[d] += prob * row[d]; /* value: the row's first Dv elements */
        }
        lse[r] = base == ORACLE_BASE_2 ? lse_nat / ln2() : lse_nat;
    }
}
