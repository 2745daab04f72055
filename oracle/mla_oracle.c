/*
 * TEST INFRASTRUCTURE ONLY.  Plain fp64 CPU oracle for absorbed-MLA decode
 * over a paged latent KV cache.  Nothing in the product path may call it;
 * it shares no code, header or constant with the CUDA library.
 *
 * What it computes (the definition, written out with no online softmax,
 * no tiling and no reordering):
 *
 *   Absorbed MLA decode is multi-query attention with one shared KV head
 *   ("Benchmarking MLA", FlashInfer issue #700: the fused-rope MQA
 *   observation and the note that for the matrix-absorbed decode kernel
 *   qk_head_dim = 512 + 64 and v_head_dim = 512):
 *     key   k_t = [ckv_t (512) | kpe_t (64)]
 *     value v_t =  ckv_t (512)           -- ckv serves as both K and V
 *   For request b with page list kv_indices[kv_indptr[b] .. kv_indptr[b+1])
 *   and n_b pages, L_b = (n_b - 1) * page_size + kv_last_page_len[b] tokens;
 *   token t lives in page kv_indices[kv_indptr[b] + t / page_size], slot
 *   t % page_size (the paged ckv/kpe buffers of "perf: MLA decode kernel
 *   implemented by CuTe targeted to SM80", FlashInfer PR #844).
 *   For every head h:
 *     x_t   = sm_scale * (q_nope[b,h,:] . ckv_t + q_pe[b,h,:] . kpe_t)
 *     m     = max_t x_t,   e_t = exp(x_t - m),   l = sum_t e_t
 *     out   = (sum_t e_t * v_t) / l
 *     lse   = m + ln(l)          (natural log, in units of the scaled logits)
 *   L_b = 0 gives out = 0 and lse = -inf.
 *
 *   Splitting the token range and merging the partial (out_i, lse_i) by
 *     M = max_i lse_i, w_i = exp(lse_i - M),
 *     out = sum_i w_i out_i / sum_i w_i,  lse = M + ln(sum_i w_i)
 *   reproduces the unsplit result (the split-KV + combine of FlashMLA
 *   PR #233, "balanced scheduler, deterministic combine").
 *
 *   8-bit cache (FlashMLA PR #233, "FP8 e4m3 ... with one scale per token
 *   (644 instead of 1152 bytes per token), dequantized inside the kernel"):
 *   ckv_t[i] = scale_t * e4m3(code_t[i]) in exact fp64, used for both the key
 *   and the value; kpe stays bf16.  The same page's INT8 variant ("FP8 e4m3 or
 *   INT8 with one scale per token") reads ckv_t[i] = scale_t * code_t[i] with the
 *   code a two's-complement signed byte.  E4M3 follows the OCP 8-bit floating
 *   point definition: 1 sign, 4 exponent (bias 7), 3 mantissa bits,
 *   subnormals at exponent field 0, no infinities, S.1111.111 is NaN,
 *   largest finite magnitude 448.
 *
 *   fp16 inputs ("bf16 / fp16" inputs of the decode kernel, FlashMLA PR #233): q_nope,
 *   q_pe, ckv and kpe all hold IEEE binary16 values (1 sign, 5 exponent bits with bias
 *   15, 10 mantissa bits, subnormals at exponent field 0, all-ones exponent for infinities
 *   and NaN) instead of bfloat16.
 *
 * bf16 and fp16 inputs are decoded exactly to double; all arithmetic is fp64.
 * Requests run in parallel with OpenMP; the order of every sum is fixed.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_D_CKV 512
#define ORACLE_D_KPE 64

/* Mistakes planted on purpose, compiled only into throw-away copies by the
 * test that checks the pins catch them.  0 = the real oracle. */
#ifndef ORACLE_PLANT
#define ORACLE_PLANT 0
#endif

static double bf16_bits_to_double(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16 bits -> double, exactly. */
double oracle_f16_decode(uint16_t h) {
    int s = h >> 15;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0x1F) {
        v = m ? NAN : INFINITY;
    } else if (e == 0) {
        v = ldexp((double)m, -24);            /* (m / 1024) * 2^(1 - 15) */
    } else {
        v = ldexp(1024.0 + (double)m, e - 25); /* (1 + m / 1024) * 2^(e - 15) */
    }
    return s ? -v : v;
}

double oracle_e4m3_decode(uint8_t code) {
    int s = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);           /* (m / 8) * 2^(1 - 7) */
    else
        v = ldexp(8.0 + (double)m, e - 10); /* (1 + m / 8) * 2^(e - 7) */
    return s ? -v : v;
}

/* Round-to-nearest-even onto the finite e4m3 grid, magnitudes saturated at
 * 448 (the harness clamps to +-448 before encoding).  Written as a search
 * over the 127 non-negative finite codes, which are monotone in value. */
uint8_t oracle_e4m3_encode(double x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0) return sign | 0x7E;
    int best = 0;
    double best_err = a;
    for (int c = 1; c <= 0x7E; ++c) {
        double err = fabs(a - oracle_e4m3_decode((uint8_t)c));
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return sign | (uint8_t)best;
}

/* The cache as the oracle sees it: one token's ckv and kpe rows in fp64.  ckv_is_fp8 is the
 * cache kind: 0 bf16, 1 e4m3 codes, 2 int8 codes, 3 fp16 (then q and kpe are fp16 too). */
typedef struct {
    int page_size, ckv_is_fp8;
    const void* ckv;
    const float* ckv_scale;
    const uint16_t* kpe;
} cache_view;

/* A 16-bit input value (q or kpe, or a 16-bit ckv) in the cache's format. */
static double in16(const cache_view* c, uint16_t bits) {
#if ORACLE_PLANT == 5
    (void)c;
    return bf16_bits_to_double(bits);   /* planted: fp16 inputs read as bfloat16 */
#else
    return c->ckv_is_fp8 == 3 ? oracle_f16_decode(bits) : bf16_bits_to_double(bits);
#endif
}

static void load_token(const cache_view* c, int page, int slot, double* ckv_row, double* kpe_row) {
    size_t tok = (size_t)page * (size_t)c->page_size + (size_t)slot;
    if (c->ckv_is_fp8 == 1) {
        const uint8_t* codes = (const uint8_t*)c->ckv + tok * ORACLE_D_CKV;
        double s = (double)c->ckv_scale[tok];
        for (int i = 0; i < ORACLE_D_CKV; ++i) ckv_row[i] = s * oracle_e4m3_decode(codes[i]);
    } else if (c->ckv_is_fp8 == 2) {
#if ORACLE_PLANT == 4
        const uint8_t* codes = (const uint8_t*)c->ckv + tok * ORACLE_D_CKV;   /* planted: codes read unsigned */
#else
        const int8_t* codes = (const int8_t*)c->ckv + tok * ORACLE_D_CKV;
#endif
        double s = (double)c->ckv_scale[tok];
        for (int i = 0; i < ORACLE_D_CKV; ++i) ckv_row[i] = s * (double)codes[i];
    } else {
        const uint16_t* row = (const uint16_t*)c->ckv + tok * ORACLE_D_CKV;
        for (int i = 0; i < ORACLE_D_CKV; ++i) ckv_row[i] = in16(c, row[i]);
    }
    const uint16_t* krow = c->kpe + tok * ORACLE_D_KPE;
    for (int j = 0; j < ORACLE_D_KPE; ++j) kpe_row[j] = in16(c, krow[j]);
}

/* Token t of a request: its page and slot (standard paged layout). */
static void token_place(const cache_view* c, const int32_t* pages_b, int tok, int* page, int* slot) {
    *page = pages_b[tok / c->page_size];
#if ORACLE_PLANT == 3
    *slot = c->page_size - 1 - tok % c->page_size;   /* planted: slots reversed */
#else
    *slot = tok % c->page_size;
#endif
}

/* Attention of all H heads of request b over its tokens [t_begin, t_end).
 * out_bh: [H, 512], lse_h: [H].  Scratch is allocated per call. */
static int attend_range(int H, const cache_view* c,
                        const uint16_t* q_nope_b, const uint16_t* q_pe_b,
                        const int32_t* pages_b, int t_begin, int t_end, double sm_scale,
                        double* out_bh, double* lse_h) {
    const int DQ = ORACLE_D_CKV + ORACLE_D_KPE;
    int L = t_end - t_begin;
    for (int i = 0; i < H * ORACLE_D_CKV; ++i) out_bh[i] = 0.0;
    if (L <= 0) {
        for (int h = 0; h < H; ++h) lse_h[h] = -INFINITY;
        return 0;
    }
    double* q = (double*)malloc(sizeof(double) * (size_t)H * DQ);
    double* x = (double*)malloc(sizeof(double) * (size_t)L * H);   /* scores, then weights */
    double* l = (double*)malloc(sizeof(double) * (size_t)H);
    double* ckv_row = (double*)malloc(sizeof(double) * ORACLE_D_CKV);
    double* kpe_row = (double*)malloc(sizeof(double) * ORACLE_D_KPE);
    int err = !q || !x || !l || !ckv_row || !kpe_row;
    if (!err) {
        for (int h = 0; h < H; ++h) {
            for (int i = 0; i < ORACLE_D_CKV; ++i)
                q[(size_t)h * DQ + i] = in16(c, q_nope_b[(size_t)h * ORACLE_D_CKV + i]);
            for (int j = 0; j < ORACLE_D_KPE; ++j)
                q[(size_t)h * DQ + ORACLE_D_CKV + j] = in16(c, q_pe_b[(size_t)h * ORACLE_D_KPE + j]);
        }
        /* x[t,h] = sm_scale * (q_nope . ckv_t + q_pe . kpe_t) */
        for (int t = 0; t < L; ++t) {
            int page, slot;
            token_place(c, pages_b, t_begin + t, &page, &slot);
            load_token(c, page, slot, ckv_row, kpe_row);
            for (int h = 0; h < H; ++h) {
                const double* qh = q + (size_t)h * DQ;
                double dot = 0.0;
                for (int i = 0; i < ORACLE_D_CKV; ++i) dot += qh[i] * ckv_row[i];
#if ORACLE_PLANT != 1
                for (int j = 0; j < ORACLE_D_KPE; ++j) dot += qh[ORACLE_D_CKV + j] * kpe_row[j];
#endif
                x[(size_t)t * H + h] = sm_scale * dot;
            }
        }
        /* m = max_t x_t, e_t = exp(x_t - m), l = sum_t e_t, lse = m + ln l */
        for (int h = 0; h < H; ++h) {
            double m = -INFINITY;
            for (int t = 0; t < L; ++t) {
                double v = x[(size_t)t * H + h];
#if ORACLE_PLANT == 2
                if (m == -INFINITY || v < m) m = v;   /* planted: min instead of max */
#else
                if (v > m) m = v;
#endif
            }
            double s = 0.0;
            for (int t = 0; t < L; ++t) {
                double e = exp(x[(size_t)t * H + h] - m);
                x[(size_t)t * H + h] = e;
                s += e;
            }
            l[h] = s;
            lse_h[h] = m + log(s);
        }
        /* out = (sum_t e_t v_t) / l, with v_t = ckv_t */
        for (int t = 0; t < L; ++t) {
            int page, slot;
            token_place(c, pages_b, t_begin + t, &page, &slot);
            load_token(c, page, slot, ckv_row, kpe_row);
            for (int h = 0; h < H; ++h) {
                double e = x[(size_t)t * H + h];
                double* o = out_bh + (size_t)h * ORACLE_D_CKV;
                for (int i = 0; i < ORACLE_D_CKV; ++i) o[i] += e * ckv_row[i];
            }
        }
        for (int h = 0; h < H; ++h) {
            double* o = out_bh + (size_t)h * ORACLE_D_CKV;
            for (int i = 0; i < ORACLE_D_CKV; ++i) o[i] /= l[h];
        }
    }
    free(q); free(x); free(l); free(ckv_row); free(kpe_row);
    return err;
}

static int request_len(int b, int P, const int32_t* kv_indptr, const int32_t* kv_last_page_len) {
    int n = kv_indptr[b + 1] - kv_indptr[b];
    return n > 0 ? (n - 1) * P + kv_last_page_len[b] : 0;
}

/* Full decode.  q_nope [B,H,512] bf16 bits, q_pe [B,H,64] bf16 bits,
 * ckv [num_pages,P,512] (bf16 bits; e4m3 codes when ckv_is_fp8 == 1, int8 codes when 2; when 3
 * fp16 bits, and q_nope, q_pe and kpe are fp16 bits too),
 * ckv_scale [num_pages,P] fp32 (8-bit cache only, else NULL),
 * kpe [num_pages,P,64] bf16 bits.  out [B,H,512], lse [B,H] in fp64.
 * threads <= 0 uses the OpenMP default.  Returns 0 on success. */
int oracle_mla_decode(int B, int H, int P,
                      const uint16_t* q_nope, const uint16_t* q_pe,
                      const void* ckv, int ckv_is_fp8, const float* ckv_scale, const uint16_t* kpe,
                      const int32_t* kv_indices, const int32_t* kv_indptr, const int32_t* kv_last_page_len,
                      double sm_scale, double* out, double* lse, int threads) {
    cache_view c = {P, ckv_is_fp8, ckv, ckv_scale, kpe};
    int err = 0;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int b = 0; b < B; ++b) {
        int L = request_len(b, P, kv_indptr, kv_last_page_len);
        err |= attend_range(H, &c, q_nope + (size_t)b * H * ORACLE_D_CKV, q_pe + (size_t)b * H * ORACLE_D_KPE,
                            kv_indices + kv_indptr[b], 0, L, sm_scale,
                            out + (size_t)b * H * ORACLE_D_CKV, lse + (size_t)b * H);
    }
    return err;
}

/* One request, token range [t_begin, t_end) only: the partial (out, lse) a
 * split-KV piece would produce.  out_bh [H,512], lse_h [H]. */
int oracle_mla_decode_range(int H, int P, int b,
                            const uint16_t* q_nope, const uint16_t* q_pe,
                            const void* ckv, int ckv_is_fp8, const float* ckv_scale, const uint16_t* kpe,
                            const int32_t* kv_indices, const int32_t* kv_indptr,
                            int t_begin, int t_end, double sm_scale, double* out_bh, double* lse_h) {
    cache_view c = {P, ckv_is_fp8, ckv, ckv_scale, kpe};
    return attend_range(H, &c, q_nope + (size_t)b * H * ORACLE_D_CKV, q_pe + (size_t)b * H * ORACLE_D_KPE,
                        kv_indices + kv_indptr[b], t_begin, t_end, sm_scale, out_bh, lse_h);
}

/* Merge k partials in the fixed order 0..k-1.  o_parts [k,H,D], lse_parts [k,H]. */
void oracle_merge(int k, int H, int D, const double* o_parts, const double* lse_parts,
                  double* out, double* lse) {
    for (int h = 0; h < H; ++h) {
        double M = -INFINITY;
        for (int i = 0; i < k; ++i)
            if (lse_parts[(size_t)i * H + h] > M) M = lse_parts[(size_t)i * H + h];
        double* o = out + (size_t)h * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (M == -INFINITY) {
            lse[h] = -INFINITY;
            continue;
        }
        double wsum = 0.0;
        for (int i = 0; i < k; ++i) {
            double w = exp(lse_parts[(size_t)i * H + h] - M);
            wsum += w;
            const double* oi = o_parts + ((size_t)i * H + h) * D;
            for (int d = 0; d < D; ++d) o[d] += w * oi[d];
        }
        for (int d = 0; d < D; ++d) o[d] /= wsum;
        lse[h] = M + log(wsum);
    }
}
