/*
 * fd_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU restatement of what the split-KV decode
 * attention library computes.  Only the test suite, the package's smoke check
 * and the benchmark's CPU-baseline leg may load this code; the product path
 * never does.  It shares no code, header, table or constant with the CUDA
 * library.
 *
 * Arithmetic: attention is evaluated in IEEE binary64 from the exact values of
 * the bf16 inputs.  The key quantizer is an *encoding* and is therefore
 * evaluated in IEEE binary32 with a fixed operation order (the file must be
 * compiled with -ffp-contract=off and without fast-math), so that its codes
 * and fp16 scales are reproducible bit for bit.
 *
 * Sources restated here:
 *   "Flash Decoding" tutorial (aiqz.cc/article/flash-decoding.html):
 *     section 1 (standard attention, steps 1-4), section 2 (two-stage max
 *     merge equation and its steps 1-4), section 3 (paged KV cache).
 *   Benchmarking blog on a hosted 1M-context model (xxmr.cn), section 1:
 *     an 8-bit-or-narrower ("FP4") KV cache as the lever on decode bytes
 *     (the fp8 and fp4 cache encodings below are this library's definitions).
 *   "Faster Than Flash / Faster Flash Decoding" summary (PaperDaily):
 *     section 3 (top-delta rule s >= m - delta), section 4 (pseudo-max from
 *     attention-sink and local-window anchors), section 5 (2-bit body scan,
 *     8-bit residual correction of the candidates), Fig. 2 (pipeline order).
 *
 * Every public function returns 0 on success and a negative value on a bad
 * argument.  Threads: n_threads <= 0 means "all OpenMP threads".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static float bf16_value_f(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* IEEE binary16 -> binary32, exact (normals, subnormals, inf, nan). */
static float half_value(uint16_t h) {
    uint32_t sign = (uint32_t)(h >> 15) << 31;
    uint32_t expo = (h >> 10) & 0x1f;
    uint32_t mant = h & 0x3ff;
    float f;
    if (expo == 0) {
        /* zero or subnormal: mant * 2^-24, exact in binary32 */
        f = (float)mant * 0x1p-24f;
        if (sign) f = -f;
        return f;
    }
    uint32_t u;
    if (expo == 31) {
        u = sign | 0x7f800000u | (mant << 13);
    } else {
        u = sign | ((expo - 15 + 127) << 23) | (mant << 13);
    }
    memcpy(&f, &u, sizeof f);
    return f;
}

/* IEEE binary32 -> binary16, round to nearest, ties to even; overflow to inf.
 * Written from the binary16 format definition: 1 sign bit, 5 exponent bits
 * (bias 15), 10 fraction bits, subnormals below 2^-14. */
uint16_t oracle_float_to_half(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t expo = (u >> 23) & 0xff;
    uint32_t mant = u & 0x7fffffu;
    if (expo == 0xff) {                       /* inf / nan */
        if (mant) return (uint16_t)(sign | 0x7e00u);
        return (uint16_t)(sign | 0x7c00u);
    }
    int e = (int)expo - 127;                  /* unbiased exponent */
    if (expo == 0) return sign;               /* binary32 subnormal -> signed zero */
    uint32_t sig = mant | 0x800000u;          /* 24-bit significand, value sig * 2^(e-23) */
    int shift;
    uint32_t hexp;
    if (e >= -14) {
        /* normal binary16 candidate: keep 11 significant bits */
        shift = 13;
        hexp = (uint32_t)(e + 15);
    } else {
        /* subnormal binary16: value = m * 2^-24, m = sig * 2^(e-23+24) */
        shift = 13 + (-14 - e);
        hexp = 0;
        if (shift > 24) return sign;          /* below half of the smallest subnormal */
    }
    uint32_t kept = sig >> shift;
    uint32_t rem = sig & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (kept & 1u))) kept += 1;
    if (hexp == 0) {
        /* subnormal result (may round up into the smallest normal: kept == 0x400) */
        return (uint16_t)(sign | kept);
    }
    /* kept has the implicit bit at position 10; a carry can move it to 11 */
    if (kept & 0x800u) { kept >>= 1; hexp += 1; }
    if (hexp >= 31) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (hexp << 10) | (kept & 0x3ffu));
}

float oracle_half_to_float(uint16_t h) { return half_value(h); }

static int pick_threads(int n_threads) {
#ifdef _OPENMP
    return n_threads > 0 ? n_threads : omp_get_max_threads();
#else
    (void)n_threads;
    return 1;
#endif
}

int oracle_max_threads(void) { return pick_threads(0); }

/* ------------------------------------------------------------------------ */
/* Dense decode attention (definition)                                      */
/* ------------------------------------------------------------------------ */

/* One query row against one key/value sequence of length L, all in binary64.
 * Standard attention, Flash Decoding tutorial section 1, steps 1-4:
 *   s_j = scale * <q, k_j>,  w_j = exp(s_j) / sum_i exp(s_i),  o = sum_j w_j v_j.
 * The maximum is subtracted before exponentiating (same value, no overflow).
 * LSE = log(sum_j exp(s_j)) in scaled-score units; L == 0 gives o = 0 and
 * LSE = -inf.  `sc` is scratch for L scores. */
static void attend_row(const double* q, const double* K, const double* V,
                       int L, int d, double scale, double* sc,
                       double* out, double* lse) {
    for (int c = 0; c < d; ++c) out[c] = 0.0;
    if (L <= 0) { *lse = -INFINITY; return; }
    double m = -INFINITY;
    for (int j = 0; j < L; ++j) {
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += q[c] * K[(size_t)j * d + c];
        sc[j] = scale * dot;
        if (sc[j] > m) m = sc[j];
    }
    double Z = 0.0;
    for (int j = 0; j < L; ++j) {
        double w = exp(sc[j] - m);
        Z += w;
        for (int c = 0; c < d; ++c) out[c] += w * V[(size_t)j * d + c];
    }
    for (int c = 0; c < d; ++c) out[c] /= Z;
    *lse = m + log(Z);
}

/* Dense decode with binary64 inputs.
 * q: [B, Hq, d]; K, V: [B, Hkv, L_max, d]; seq_lens: [B] or NULL (= L_max).
 * Query head hq reads KV head hq / (Hq / Hkv).
 * out: [B, Hq, d]; lse: [B, Hq]. */
int oracle_decode_dense_f64(const double* q, const double* K, const double* V,
                            const int32_t* seq_lens, int B, int Hq, int Hkv,
                            int L_max, int d, double scale,
                            double* out, double* lse, int n_threads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || L_max < 0 || d <= 0) return -1;
    if (seq_lens) for (int b = 0; b < B; ++b) if (seq_lens[b] < 0 || seq_lens[b] > L_max) return -2;
    int G = Hq / Hkv;
    int nt = pick_threads(n_threads);
    int rows = B * Hq;
    int bad = 0;
    #pragma omp parallel num_threads(nt)
    {
        double* sc = (double*)malloc(sizeof(double) * (size_t)(L_max > 0 ? L_max : 1));
        int ok = sc != NULL;
        if (!ok) {
            #pragma omp atomic write
            bad = 1;
        }
        {
            #pragma omp for schedule(dynamic, 1)
            for (int r = 0; r < rows; ++r) {
                if (!ok) continue;
                int b = r / Hq, hq = r % Hq, h = hq / G;
                int L = seq_lens ? seq_lens[b] : L_max;
                size_t kv = ((size_t)b * Hkv + h) * (size_t)L_max * d;
                attend_row(q + (size_t)r * d, K + kv, V + kv, L, d, scale, sc,
                           out + (size_t)r * d, lse + r);
            }
            free(sc);
        }
    }
    return bad ? -3 : 0;
}

/* Widen bf16 rows to binary64. */
static void widen_rows(const uint16_t* src, size_t n, double* dst) {
    for (size_t i = 0; i < n; ++i) dst[i] = bf16_value(src[i]);
}

/* attend_row with bf16 K and V rows, widened exactly as they are read. */
static void attend_row_bf16(const double* q, const uint16_t* K, const uint16_t* V,
                            int L, int d, double scale, double* sc,
                            double* out, double* lse) {
    for (int c = 0; c < d; ++c) out[c] = 0.0;
    if (L <= 0) { *lse = -INFINITY; return; }
    double m = -INFINITY;
    for (int j = 0; j < L; ++j) {
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += q[c] * bf16_value(K[(size_t)j * d + c]);
        sc[j] = scale * dot;
        if (sc[j] > m) m = sc[j];
    }
    double Z = 0.0;
    for (int j = 0; j < L; ++j) {
        double w = exp(sc[j] - m);
        Z += w;
        for (int c = 0; c < d; ++c) out[c] += w * bf16_value(V[(size_t)j * d + c]);
    }
    for (int c = 0; c < d; ++c) out[c] /= Z;
    *lse = m + log(Z);
}

/* Dense decode with bf16 inputs (the library's contiguous-cache problem).
 * Same layouts as oracle_decode_dense_f64, values given as bf16 bit patterns. */
int oracle_decode_dense(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        const int32_t* seq_lens, int B, int Hq, int Hkv,
                        int L_max, int d, double scale,
                        double* out, double* lse, int n_threads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || L_max < 0 || d <= 0) return -1;
    if (seq_lens) for (int b = 0; b < B; ++b) if (seq_lens[b] < 0 || seq_lens[b] > L_max) return -2;
    int G = Hq / Hkv;
    int nt = pick_threads(n_threads);
    int rows = B * Hq;
    int bad = 0;
    #pragma omp parallel num_threads(nt)
    {
        double* sc = (double*)malloc(sizeof(double) * (size_t)(L_max > 0 ? L_max : 1));
        double* qd = (double*)malloc(sizeof(double) * (size_t)d);
        int ok = sc && qd;
        if (!ok) {
            #pragma omp atomic write
            bad = 1;
        }
        {
            #pragma omp for schedule(dynamic, 1)
            for (int r = 0; r < rows; ++r) {
                if (!ok) continue;
                int b = r / Hq, hq = r % Hq, h = hq / G;
                int L = seq_lens ? seq_lens[b] : L_max;
                size_t kv = ((size_t)b * Hkv + h) * (size_t)L_max * d;
                widen_rows(q + (size_t)r * d, (size_t)d, qd);
                attend_row_bf16(qd, k + kv, v + kv, L, d, scale, sc, out + (size_t)r * d, lse + r);
            }
        }
        free(sc); free(qd);
    }
    return bad ? -3 : 0;
}

/* ------------------------------------------------------------------------ */
/* Split form: per-chunk statistics and the exact merge                      */
/* ------------------------------------------------------------------------ */

/* Flash Decoding tutorial, section 2.  The cache of one sequence is cut into
 * S chunks along the sequence.  Chunk i covers [i*c, min(L, (i+1)*c)) with
 * c = ceil(L / S), so every token is covered (the tutorial's demo uses
 * L // S and drops the remainder; that is not followed).  For a non-empty
 * chunk:
 *   m_i = max_j s_j,  l_i = sum_j exp(s_j - m_i),
 *   O_i = sum_j exp(s_j - m_i) v_j / l_i      (locally normalised)
 * and the merge is the section-2 equation
 *   m = max_i m_i,  w_i = exp(m_i - m) * l_i,  O = sum_i w_i O_i / sum_i w_i.
 * The merge equation multiplies O_i by l_i, which is only right for the
 * locally normalised O_i; that reading is the one taken.  An empty chunk has
 * m_i = -inf, l_i = 0, O_i = 0 and takes no part in the merge.
 * LSE = m + log(sum_i w_i).
 * part_m, part_l: [B, Hq, S]; part_o: [B, Hq, S, d] (each may be NULL). */
int oracle_decode_split(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        const int32_t* seq_lens, int B, int Hq, int Hkv,
                        int L_max, int d, double scale, int S,
                        double* out, double* lse,
                        double* part_m, double* part_l, double* part_o,
                        int n_threads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || L_max < 0 || d <= 0 || S <= 0) return -1;
    if (seq_lens) for (int b = 0; b < B; ++b) if (seq_lens[b] < 0 || seq_lens[b] > L_max) return -2;
    int G = Hq / Hkv;
    int nt = pick_threads(n_threads);
    int rows = B * Hq;
    int bad = 0;
    #pragma omp parallel num_threads(nt)
    {
        size_t cap = (size_t)(L_max > 0 ? L_max : 1);
        double* Kd = (double*)malloc(sizeof(double) * cap * d);
        double* Vd = (double*)malloc(sizeof(double) * cap * d);
        double* sc = (double*)malloc(sizeof(double) * cap);
        double* qd = (double*)malloc(sizeof(double) * (size_t)d);
        double* mi = (double*)malloc(sizeof(double) * (size_t)S);
        double* li = (double*)malloc(sizeof(double) * (size_t)S);
        double* Oi = (double*)malloc(sizeof(double) * (size_t)S * d);
        int ok = Kd && Vd && sc && qd && mi && li && Oi;
        if (!ok) {
            #pragma omp atomic write
            bad = 1;
        }
        {
            #pragma omp for schedule(dynamic, 1)
            for (int r = 0; r < rows; ++r) {
                if (!ok) continue;
                int b = r / Hq, hq = r % Hq, h = hq / G;
                int L = seq_lens ? seq_lens[b] : L_max;
                size_t kv = ((size_t)b * Hkv + h) * (size_t)L_max * d;
                widen_rows(k + kv, (size_t)L * d, Kd);
                widen_rows(v + kv, (size_t)L * d, Vd);
                widen_rows(q + (size_t)r * d, (size_t)d, qd);
                int chunk = (L + S - 1) / S;
                /* step 1: per-chunk local statistics */
                for (int i = 0; i < S; ++i) {
                    int j0 = i * chunk, j1 = (i + 1) * chunk;
                    if (j1 > L) j1 = L;
                    double* O = Oi + (size_t)i * d;
                    for (int c = 0; c < d; ++c) O[c] = 0.0;
                    if (chunk == 0 || j0 >= j1) { mi[i] = -INFINITY; li[i] = 0.0; continue; }
                    double m = -INFINITY;
                    for (int j = j0; j < j1; ++j) {
                        double dot = 0.0;
                        for (int c = 0; c < d; ++c) dot += qd[c] * Kd[(size_t)j * d + c];
                        sc[j] = scale * dot;
                        if (sc[j] > m) m = sc[j];
                    }
                    double l = 0.0;
                    for (int j = j0; j < j1; ++j) {
                        double w = exp(sc[j] - m);
                        l += w;
                        for (int c = 0; c < d; ++c) O[c] += w * Vd[(size_t)j * d + c];
                    }
                    for (int c = 0; c < d; ++c) O[c] /= l;
                    mi[i] = m;
                    li[i] = l;
                }
                /* steps 2-4: global max, rescale, normalised merge */
                double M = -INFINITY;
                for (int i = 0; i < S; ++i) if (li[i] > 0.0 && mi[i] > M) M = mi[i];
                double* o = out + (size_t)r * d;
                for (int c = 0; c < d; ++c) o[c] = 0.0;
                if (M == -INFINITY) {
                    lse[r] = -INFINITY;
                } else {
                    double W = 0.0;
                    for (int i = 0; i < S; ++i) {
                        if (li[i] <= 0.0) continue;
                        double w = exp(mi[i] - M) * li[i];
                        W += w;
                        for (int c = 0; c < d; ++c) o[c] += w * Oi[(size_t)i * d + c];
                    }
                    for (int c = 0; c < d; ++c) o[c] /= W;
                    lse[r] = M + log(W);
                }
                if (part_m) for (int i = 0; i < S; ++i) part_m[(size_t)r * S + i] = mi[i];
                if (part_l) for (int i = 0; i < S; ++i) part_l[(size_t)r * S + i] = li[i];
                if (part_o) memcpy(part_o + (size_t)r * S * d, Oi, sizeof(double) * (size_t)S * d);
            }
        }
        free(Kd); free(Vd); free(sc); free(qd); free(mi); free(li); free(Oi);
    }
    return bad ? -3 : 0;
}

/* ------------------------------------------------------------------------ */
/* Paged cache: gather, then the dense definition                            */
/* ------------------------------------------------------------------------ */

/* Flash Decoding tutorial, section 3: the cache is cut into fixed-size pages.
 * Pools: [num_pages, Hkv, page_size, d]; token t of sequence b lives in page
 * page_table[b * max_pages + t / page_size] at row t % page_size.  This route
 * first copies each sequence's pages into a contiguous [L_b, d] slab and then
 * applies the dense definition; it does not share the kernel's indirection.
 * Returns -4 when a referenced page id lies outside [0, num_pages). */
int oracle_decode_paged(const uint16_t* q, const uint16_t* k_pages, const uint16_t* v_pages,
                        const int32_t* page_table, int max_pages, int num_pages,
                        const int32_t* seq_lens, int page_size,
                        int B, int Hq, int Hkv, int d, double scale,
                        double* out, double* lse, int n_threads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || page_size <= 0 || !seq_lens) return -1;
    for (int b = 0; b < B; ++b) {
        if (seq_lens[b] < 0 || seq_lens[b] > (long long)max_pages * page_size) return -2;
        int np = (seq_lens[b] + page_size - 1) / page_size;
        for (int p = 0; p < np; ++p) {
            int id = page_table[(size_t)b * max_pages + p];
            if (id < 0 || id >= num_pages) return -4;
        }
    }
    int G = Hq / Hkv;
    int nt = pick_threads(n_threads);
    int units = B * Hkv;
    int Lcap = 1;
    for (int b = 0; b < B; ++b) if (seq_lens[b] > Lcap) Lcap = seq_lens[b];
    int bad = 0;
    #pragma omp parallel num_threads(nt)
    {
        uint16_t* Kg = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)Lcap * d);
        uint16_t* Vg = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)Lcap * d);
        double* sc = (double*)malloc(sizeof(double) * (size_t)Lcap);
        double* qd = (double*)malloc(sizeof(double) * (size_t)d);
        int ok = Kg && Vg && sc && qd;
        if (!ok) {
            #pragma omp atomic write
            bad = 1;
        }
        {
            #pragma omp for schedule(dynamic, 1)
            for (int u = 0; u < units; ++u) {
                if (!ok) continue;
                int b = u / Hkv, h = u % Hkv;
                int L = seq_lens[b];
                for (int t = 0; t < L; ++t) {
                    int id = page_table[(size_t)b * max_pages + t / page_size];
                    size_t row = (((size_t)id * Hkv + h) * page_size + (t % page_size)) * d;
                    memcpy(Kg + (size_t)t * d, k_pages + row, sizeof(uint16_t) * (size_t)d);
                    memcpy(Vg + (size_t)t * d, v_pages + row, sizeof(uint16_t) * (size_t)d);
                }
                for (int g = 0; g < G; ++g) {
                    int r = b * Hq + h * G + g;
                    widen_rows(q + (size_t)r * d, (size_t)d, qd);
                    attend_row_bf16(qd, Kg, Vg, L, d, scale, sc, out + (size_t)r * d, lse + r);
                }
            }
        }
        free(Kg); free(Vg); free(sc); free(qd);
    }
    return bad ? -3 : 0;
}

/* ------------------------------------------------------------------------ */
/* Key quantizer: 2-bit body + 8-bit residual (an encoding; binary32)        */
/* ------------------------------------------------------------------------ */

/* Faster Flash Decoding summary, section 5: every key is split into a 2-bit
 * body (read for the full scan) and an 8-bit residual (read only for the
 * candidates).  The page gives no formulas; the encoding below is the one
 * this library defines, per token and per group of 32 channels:
 *   mn  = min x,  mx = max x                       (exact bf16 values; a zero
 *                                                   extreme is taken as +0)
 *   mn16 = half(mn),  s16 = half((mx - mn) / 3)    (binary32 ops, then RNE to fp16)
 *   code = clamp(rint((x - mn16) / s16), 0, 3)     (all codes 0 when s16 == 0)
 *   deq2 = mn16 + code * s16                       (binary32, two roundings)
 *   r    = x - deq2
 *   rs16 = half(max|r| / 127)
 *   rq   = clamp(rint(r / rs16), -127, 127)        (all 0 when rs16 == 0)
 * rint rounds to nearest, ties to even.  Outputs for tokens t >= seq_lens[b]
 * are left unwritten.
 * Layouts (row = (b * Hkv + h) * L_max + t):
 *   codes     [row, d/4]  u8, channel c in byte c/4 at bits 2*(c%4)..+1
 *   mn_scale  [row, d/32, 2] fp16 bits (mn16, s16)
 *   res       [row, d]    int8
 *   res_scale [row, d/32] fp16 bits (rs16)                                  */
int oracle_quantize_keys(const uint16_t* k, const int32_t* seq_lens,
                         int B, int Hkv, int L_max, int d,
                         uint8_t* codes, uint16_t* mn_scale, int8_t* res,
                         uint16_t* res_scale, int n_threads) {
    if (B < 0 || Hkv <= 0 || L_max < 0 || d <= 0 || d % 32) return -1;
    if (seq_lens) for (int b = 0; b < B; ++b) if (seq_lens[b] < 0 || seq_lens[b] > L_max) return -2;
    int nt = pick_threads(n_threads);
    long long rows = (long long)B * Hkv * L_max;
    int ng = d / 32;
    #pragma omp parallel for num_threads(nt) schedule(static)
    for (long long row = 0; row < rows; ++row) {
        int b = (int)(row / ((long long)Hkv * L_max));
        int t = (int)(row % L_max);
        int L = seq_lens ? seq_lens[b] : L_max;
        if (t >= L) continue;
        const uint16_t* x = k + (size_t)row * d;
        uint8_t* cd = codes + (size_t)row * (d / 4);
        for (int i = 0; i < d / 4; ++i) cd[i] = 0;
        for (int g = 0; g < ng; ++g) {
            float xv[32];
            for (int c = 0; c < 32; ++c) xv[c] = bf16_value_f(x[g * 32 + c]);
            float mn = xv[0], mx = xv[0];
            for (int c = 1; c < 32; ++c) {
                if (xv[c] < mn) mn = xv[c];
                if (xv[c] > mx) mx = xv[c];
            }
            /* min and max are values: a zero extreme is +0 whatever its sign */
            mn = mn + 0.0f;
            mx = mx + 0.0f;
            float diff = mx - mn;
            float third = diff / 3.0f;
            uint16_t mn16 = oracle_float_to_half(mn);
            uint16_t s16 = oracle_float_to_half(third);
            float mnf = half_value(mn16);
            float sf = half_value(s16);
            float deq2[32];
            int code[32];
            for (int c = 0; c < 32; ++c) {
                int q2 = 0;
                if (sf != 0.0f) {
                    float num = xv[c] - mnf;
                    float ratio = num / sf;
                    float rr = nearbyintf(ratio);
                    if (rr < 0.0f) rr = 0.0f;
                    if (rr > 3.0f) rr = 3.0f;
                    q2 = (int)rr;
                }
                code[c] = q2;
                volatile float cs = (float)q2 * sf;   /* rounded on its own: no fused multiply-add */
                deq2[c] = mnf + cs;
            }
            float r[32];
            float amax = 0.0f;
            for (int c = 0; c < 32; ++c) {
                float rv = xv[c] - deq2[c];
                r[c] = rv;
                float a = fabsf(rv);
                if (a > amax) amax = a;
            }
            float rsv = amax / 127.0f;
            uint16_t rs16 = oracle_float_to_half(rsv);
            float rsf = half_value(rs16);
            for (int c = 0; c < 32; ++c) {
                int q8 = 0;
                if (rsf != 0.0f) {
                    float ratio = r[c] / rsf;
                    float rr = nearbyintf(ratio);
                    if (rr < -127.0f) rr = -127.0f;
                    if (rr > 127.0f) rr = 127.0f;
                    q8 = (int)rr;
                }
                res[(size_t)row * d + g * 32 + c] = (int8_t)q8;
                int ch = g * 32 + c;
                cd[ch / 4] = (uint8_t)(cd[ch / 4] | (code[c] << (2 * (ch % 4))));
            }
            mn_scale[((size_t)row * ng + g) * 2 + 0] = mn16;
            mn_scale[((size_t)row * ng + g) * 2 + 1] = s16;
            res_scale[(size_t)row * ng + g] = rs16;
        }
    }
    return 0;
}

/* Dequantized key values of one token row, as binary32 per the encoding:
 * deq2 = mn16 + code * s16 and deq8 = rq * rs16 (both exact binary32 ops in
 * the order given).  Written to binary64 arrays. */
static void dequant_row(const uint8_t* cd, const uint16_t* ms, const int8_t* rq,
                        const uint16_t* rs, int d, double* deq2, double* deq8) {
    for (int c = 0; c < d; ++c) {
        int g = c / 32;
        int code = (cd[c / 4] >> (2 * (c % 4))) & 3;
        float mnf = half_value(ms[2 * g + 0]);
        float sf = half_value(ms[2 * g + 1]);
        volatile float cs = (float)code * sf;  /* rounded on its own: no fused multiply-add */
        float dq = mnf + cs;
        deq2[c] = (double)dq;
        if (deq8) {
            float r8 = (float)rq[c] * half_value(rs[g]);
            deq8[c] = (double)r8;
        }
    }
}

/* Materialise the dequantized keys k~ = deq2 + deq8 as binary64 [B,Hkv,L_max,d]
 * (tokens past seq_lens[b] are set to 0).  Used to reduce the top-delta path
 * with delta = +inf to the dense definition. */
int oracle_dequantize_keys(const uint8_t* codes, const uint16_t* mn_scale,
                           const int8_t* res, const uint16_t* res_scale,
                           const int32_t* seq_lens, int B, int Hkv, int L_max, int d,
                           int with_residual, double* k_tilde) {
    if (B < 0 || Hkv <= 0 || L_max < 0 || d <= 0 || d % 32) return -1;
    int ng = d / 32;
    double* tmp = (double*)malloc(sizeof(double) * (size_t)d);
    if (!tmp) return -3;
    for (long long row = 0; row < (long long)B * Hkv * L_max; ++row) {
        int b = (int)(row / ((long long)Hkv * L_max));
        int t = (int)(row % L_max);
        int L = seq_lens ? seq_lens[b] : L_max;
        double* kt = k_tilde + (size_t)row * d;
        if (t >= L) { for (int c = 0; c < d; ++c) kt[c] = 0.0; continue; }
        dequant_row(codes + (size_t)row * (d / 4), mn_scale + (size_t)row * ng * 2,
                    res + (size_t)row * d, res_scale + (size_t)row * ng, d, kt,
                    with_residual ? tmp : NULL);
        if (with_residual) for (int c = 0; c < d; ++c) kt[c] += tmp[c];
    }
    free(tmp);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Top-delta decode (Faster Flash Decoding), step by step                   */
/* ------------------------------------------------------------------------ */

/* For every (b, query head), in the order of the summary's Fig. 2:
 *  1. approximate scores from the 2-bit body only:
 *       s~_j = scale * <q, deq2_j>                      (section 5)
 *  2. pseudo-max over the anchors, i.e. the attention-sink tokens at the
 *     start and the local window at the end (section 4):
 *       A = {0 .. n_sink-1} U {L-window .. L-1}  (clipped to [0, L)),
 *       m^ = max_{j in A} s~_j
 *  3. top-delta candidate set, an inclusive element-wise test (section 3):
 *       Sel = { j < L : s~_j >= m^ - delta }     (delta = +inf keeps all)
 *  4. residual correction of the candidates (section 5):
 *       k~_j = deq2_j + deq8_j,  s_j = scale * <q, k~_j>
 *  5. exact softmax attention over Sel only, with bf16 V:
 *       out = sum_{j in Sel} exp(s_j) v_j / sum_{j in Sel} exp(s_j),
 *       LSE = log sum_{j in Sel} exp(s_j).
 * Selection is per query head (the rule is stated per query i).  L == 0
 * gives out = 0, LSE = -inf, m^ = -inf and an empty set.
 * Optional outputs: sel_mask [B, Hq, ceil(L_max/32)] (bit j%32 of word j/32),
 * sel_count [B, Hq], m_hat [B, Hq], s_tilde [B, Hq, L_max] (unwritten past L). */
int oracle_decode_topdelta(const uint16_t* q, const uint8_t* codes, const uint16_t* mn_scale,
                           const int8_t* res, const uint16_t* res_scale, const uint16_t* v,
                           const int32_t* seq_lens, int B, int Hq, int Hkv, int L_max, int d,
                           double scale, double delta, int n_sink, int window,
                           double* out, double* lse, uint32_t* sel_mask, int32_t* sel_count,
                           double* m_hat, double* s_tilde, int n_threads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || L_max < 0 || d <= 0 || d % 32) return -1;
    if (n_sink < 0 || window < 0 || !(delta >= 0.0)) return -1;
    if (seq_lens) for (int b = 0; b < B; ++b) if (seq_lens[b] < 0 || seq_lens[b] > L_max) return -2;
    int G = Hq / Hkv;
    int ng = d / 32;
    int words = (L_max + 31) / 32;
    int nt = pick_threads(n_threads);
    int rows = B * Hq;
    int bad = 0;
    #pragma omp parallel num_threads(nt)
    {
        size_t cap = (size_t)(L_max > 0 ? L_max : 1);
        double* st = (double*)malloc(sizeof(double) * cap);
        double* sx = (double*)malloc(sizeof(double) * cap);
        unsigned char* sel = (unsigned char*)malloc(cap);
        double* qd = (double*)malloc(sizeof(double) * (size_t)d);
        double* d2 = (double*)malloc(sizeof(double) * (size_t)d);
        double* d8 = (double*)malloc(sizeof(double) * (size_t)d);
        int ok = st && sx && sel && qd && d2 && d8;
        if (!ok) {
            #pragma omp atomic write
            bad = 1;
        }
        {
            #pragma omp for schedule(dynamic, 1)
            for (int r = 0; r < rows; ++r) {
                if (!ok) continue;
                int b = r / Hq, hq = r % Hq, h = hq / G;
                int L = seq_lens ? seq_lens[b] : L_max;
                size_t base = ((size_t)b * Hkv + h) * (size_t)L_max;
                widen_rows(q + (size_t)r * d, (size_t)d, qd);
                double* o = out + (size_t)r * d;
                for (int c = 0; c < d; ++c) o[c] = 0.0;
                if (sel_mask) for (int w = 0; w < words; ++w) sel_mask[(size_t)r * words + w] = 0u;
                /* 1. scan on the 2-bit body */
                for (int j = 0; j < L; ++j) {
                    size_t row = base + j;
                    dequant_row(codes + row * (d / 4), mn_scale + row * ng * 2, NULL, NULL, d, d2, NULL);
                    double dot = 0.0;
                    for (int c = 0; c < d; ++c) dot += qd[c] * d2[c];
                    st[j] = scale * dot;
                    if (s_tilde) s_tilde[(size_t)r * L_max + j] = st[j];
                }
                /* 2. pseudo-max over sinks and window */
                double mh = -INFINITY;
                for (int j = 0; j < L; ++j) {
                    int anchor = (j < n_sink) || (j >= L - window);
                    if (anchor && st[j] > mh) mh = st[j];
                }
                if (m_hat) m_hat[r] = mh;
                /* 3. candidates */
                double thr = mh - delta;
                int cnt = 0;
                for (int j = 0; j < L; ++j) {
                    sel[j] = (unsigned char)(st[j] >= thr);
                    if (sel[j]) {
                        ++cnt;
                        if (sel_mask) sel_mask[(size_t)r * words + j / 32] |= (1u << (j % 32));
                    }
                }
                if (sel_count) sel_count[r] = cnt;
                if (cnt == 0) { lse[r] = -INFINITY; continue; }
                /* 4. residual-corrected scores of the candidates */
                double m = -INFINITY;
                for (int j = 0; j < L; ++j) {
                    if (!sel[j]) continue;
                    size_t row = base + j;
                    dequant_row(codes + row * (d / 4), mn_scale + row * ng * 2, res + row * d,
                                res_scale + row * ng, d, d2, d8);
                    double dot = 0.0;
                    for (int c = 0; c < d; ++c) dot += qd[c] * (d2[c] + d8[c]);
                    sx[j] = scale * dot;
                    if (sx[j] > m) m = sx[j];
                }
                /* 5. exact softmax over the candidates, bf16 V */
                double Z = 0.0;
                for (int j = 0; j < L; ++j) {
                    if (!sel[j]) continue;
                    double w = exp(sx[j] - m);
                    Z += w;
                    const uint16_t* vr = v + (base + j) * d;
                    for (int c = 0; c < d; ++c) o[c] += w * bf16_value(vr[c]);
                }
                for (int c = 0; c < d; ++c) o[c] /= Z;
                lse[r] = m + log(Z);
            }
        }
        free(st); free(sx); free(sel); free(qd); free(d2); free(d8);
    }
    return bad ? -3 : 0;
}

/* ------------------------------------------------------------------------ */
/* fp8 (e4m3) KV cache encoding                                             */
/* ------------------------------------------------------------------------ */

/* IEEE-style e4m3 ("fn" variant: 1 sign, 4 exponent bits with bias 7, 3
 * mantissa bits, subnormals m * 2^-9, largest finite 448 = 0x7E, 0x7F NaN, no
 * infinity).  Round to nearest, ties to even; magnitudes beyond 448 saturate
 * to 448.  Written from that format definition. */
uint8_t oracle_float_to_e4m3(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint8_t sign = (uint8_t)((u >> 24) & 0x80u);
    float a = fabsf(f);
    if (a != a) return (uint8_t)(sign | 0x7f);           /* NaN */
    if (a >= 448.0f) return (uint8_t)(sign | 0x7e);      /* saturate */
    /* the representable magnitudes are k * 2^(e-3) for normals (e >= -6) and
     * k * 2^-9 for subnormals; pick the quantum of a's binade and round */
    int e;
    (void)frexpf(a, &e);                                  /* a = m * 2^e, m in [0.5, 1) */
    int ex = e - 1;                                       /* a in [2^ex, 2^(ex+1)) */
    if (ex < -6) ex = -6;                                 /* subnormal quantum 2^-9 */
    float quantum = ldexpf(1.0f, ex - 3);
    float k = a / quantum;                                /* exact: power-of-two scaling */
    float kr = nearbyintf(k);                             /* ties to even */
    float r = kr * quantum;
    if (r >= 448.0f) r = 448.0f;
    /* encode r */
    if (r == 0.0f) return sign;
    int er;
    (void)frexpf(r, &er);
    int eb = er - 1;                                      /* r in [2^eb, 2^(eb+1)) */
    if (eb < -6) {                                        /* subnormal: r = m * 2^-9 */
        int m = (int)(r * 512.0f);
        return (uint8_t)(sign | m);
    }
    int mant = (int)(r / ldexpf(1.0f, eb - 3)) - 8;       /* 3-bit fraction */
    return (uint8_t)(sign | ((eb + 7) << 3) | mant);
}

/* Exact value of an e4m3 code. */
double oracle_e4m3_value(uint8_t c) {
    int sign = c & 0x80;
    int ex = (c >> 3) & 0xf;
    int m = c & 7;
    double v;
    if (ex == 0xf && m == 7) return NAN;
    if (ex == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, ex - 7);
    return sign ? -v : v;
}

/* Per row (token, head) of a bf16 cache [B, H, L_max, d]:
 *   a = max_c |x_c|,  s = a / 448          (binary32 division)
 *   code_c = e4m3(x_c / s)                  (binary32 division, RNE, saturating; 0 when s == 0)
 * codes [B, H, L_max, d] u8, scales [B, H, L_max] binary32.  Rows past
 * seq_lens[b] are not written.  The dequantized value is e4m3(code) * s. */
int oracle_quantize_kv_fp8(const uint16_t* x, const int32_t* seq_lens, int B, int H, int L_max, int d,
                           uint8_t* codes, float* scales, int n_threads) {
    if (B < 0 || H <= 0 || L_max < 0 || d <= 0) return -1;
    if (seq_lens) for (int b = 0; b < B; ++b) if (seq_lens[b] < 0 || seq_lens[b] > L_max) return -2;
    int nt = pick_threads(n_threads);
    long long rows = (long long)B * H * L_max;
    #pragma omp parallel for num_threads(nt) schedule(static)
    for (long long row = 0; row < rows; ++row) {
        int b = (int)(row / ((long long)H * L_max));
        int t = (int)(row % L_max);
        int L = seq_lens ? seq_lens[b] : L_max;
        if (t >= L) continue;
        const uint16_t* xr = x + (size_t)row * d;
        float a = 0.0f;
        for (int c = 0; c < d; ++c) {
            float v = fabsf(bf16_value_f(xr[c]));
            if (v > a) a = v;
        }
        float sc = a / 448.0f;
        scales[row] = sc;
        for (int c = 0; c < d; ++c) {
            uint8_t code = 0;
            if (sc != 0.0f) {
                float y = bf16_value_f(xr[c]) / sc;
                code = oracle_float_to_e4m3(y);
            }
            codes[(size_t)row * d + c] = code;
        }
    }
    return 0;
}

/* Dequantized cache as binary64 (exact products e4m3(code) * s); rows past
 * seq_lens[b] are 0. */
int oracle_dequantize_kv_fp8(const uint8_t* codes, const float* scales, const int32_t* seq_lens,
                             int B, int H, int L_max, int d, double* out) {
    if (B < 0 || H <= 0 || L_max < 0 || d <= 0) return -1;
    for (long long row = 0; row < (long long)B * H * L_max; ++row) {
        int b = (int)(row / ((long long)H * L_max));
        int t = (int)(row % L_max);
        int L = seq_lens ? seq_lens[b] : L_max;
        for (int c = 0; c < d; ++c)
            out[(size_t)row * d + c] = t < L ? oracle_e4m3_value(codes[(size_t)row * d + c]) * (double)scales[row] : 0.0;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* fp4 (e2m1) KV cache encoding with power-of-two block scales               */
/* ------------------------------------------------------------------------ */

/* e2m1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit; magnitudes
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6 for codes 0..7, no infinity or NaN. */
double oracle_e2m1_value(uint8_t c) {
    int e = (c >> 1) & 3, m = c & 1;
    double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return (c & 8) ? -v : v;
}

/* Nearest e2m1 code to y (ties to the even code, i.e. mantissa bit 0),
 * magnitudes above 6 saturating to 6.  Written as a search over the eight
 * magnitudes so that it can be checked against the table by eye. */
uint8_t oracle_double_to_e2m1(double y) {
    uint8_t sign = signbit(y) ? 8 : 0;
    double a = fabs(y);
    if (a >= 6.0) return (uint8_t)(sign | 7);
    int best = 0;
    double bd = a;  /* distance to code 0 */
    for (int k = 1; k < 8; ++k) {
        double dk = fabs(a - oracle_e2m1_value((uint8_t)k));
        if (dk < bd || (dk == bd && (k & 1) == 0 && (best & 1) == 1)) {
            best = k;
            bd = dk;
        }
    }
    return (uint8_t)(sign | best);
}

/* Block scale exponent: the smallest e in [-126, 127] with 6 * 2^e >= amax. */
int oracle_fp4_block_exponent(double amax) {
    int e = -126;
    while (e < 127 && 6.0 * ldexp(1.0, e) < amax) ++e;
    return e;
}

/* Per cache row (token, head) of a bf16 cache [B, H, L_max, d] and per
 * 32-channel block b of it:
 *   e_b  = oracle_fp4_block_exponent(max over the block of |x_c|)
 *   code = e2m1(x_c * 2^-e_b)                       (exact product, RNE)
 * codes [B, H, L_max, d/2] u8: channel c in byte c/2, the low nibble for even
 * c; scales [B, H, L_max, d/32] u8: e_b + 127.  Rows past seq_lens[b] are
 * not written.  The decoded value is e2m1(code) * 2^e_b. */
int oracle_quantize_kv_fp4(const uint16_t* x, const int32_t* seq_lens, int B, int H, int L_max, int d,
                           uint8_t* codes, uint8_t* scales, int n_threads) {
    if (B < 0 || H <= 0 || L_max < 0 || d <= 0 || d % 32 != 0) return -1;
    if (seq_lens) for (int b = 0; b < B; ++b) if (seq_lens[b] < 0 || seq_lens[b] > L_max) return -2;
    int nt = pick_threads(n_threads);
    long long rows = (long long)B * H * L_max;
    #pragma omp parallel for num_threads(nt) schedule(static)
    for (long long row = 0; row < rows; ++row) {
        int b = (int)(row / ((long long)H * L_max));
        int t = (int)(row % L_max);
        int L = seq_lens ? seq_lens[b] : L_max;
        if (t >= L) continue;
        const uint16_t* xr = x + (size_t)row * d;
        for (int blk = 0; blk < d / 32; ++blk) {
            double amax = 0.0;
            for (int c = 32 * blk; c < 32 * blk + 32; ++c) {
                double v = fabs(bf16_value(xr[c]));
                if (v > amax) amax = v;
            }
            int e = oracle_fp4_block_exponent(amax);
            scales[(size_t)row * (d / 32) + blk] = (uint8_t)(e + 127);
            for (int c = 32 * blk; c < 32 * blk + 32; c += 2) {
                uint8_t lo = oracle_double_to_e2m1(bf16_value(xr[c]) * ldexp(1.0, -e));
                uint8_t hi = oracle_double_to_e2m1(bf16_value(xr[c + 1]) * ldexp(1.0, -e));
                codes[(size_t)row * (d / 2) + c / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
    return 0;
}

/* Decoded cache as binary64 (exact); rows past seq_lens[b] are 0. */
int oracle_dequantize_kv_fp4(const uint8_t* codes, const uint8_t* scales, const int32_t* seq_lens,
                             int B, int H, int L_max, int d, double* out) {
    if (B < 0 || H <= 0 || L_max < 0 || d <= 0 || d % 32 != 0) return -1;
    for (long long row = 0; row < (long long)B * H * L_max; ++row) {
        int b = (int)(row / ((long long)H * L_max));
        int t = (int)(row % L_max);
        int L = seq_lens ? seq_lens[b] : L_max;
        for (int c = 0; c < d; ++c) {
            double v = 0.0;
            if (t < L) {
                uint8_t byte = codes[(size_t)row * (d / 2) + c / 2];
                uint8_t code = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
                int e = (int)scales[(size_t)row * (d / 32) + c / 32] - 127;
                v = oracle_e2m1_value(code) * ldexp(1.0, e);
            }
            out[(size_t)row * d + c] = v;
        }
    }
    return 0;
}
