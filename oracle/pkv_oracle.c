/*
 * CPU oracle for paged KV-cache decode — TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg load this library. The product path (libpkv) never calls it, links it
 * or shares a line of code with it.
 *
 * It is the plain definition of what the paged decode step computes, written
 * for a reader to check by eye, in fp64, with no blocking, fusion or
 * reordering:
 *
 *   oracle_decode      For each sequence, walk its block table to assemble a
 *                      contiguous K and V (per kv head), then run dense
 *                      softmax attention for every query head.
 *                      - Block table: logical block i holds tokens i*B ..
 *                        i*B+B-1 and maps to a physical block of the pool
 *                        ("PagedAttention — Math + Memory Model", section
 *                        "PagedAttention: blocks and the block table";
 *                        "KV-cache paging in vLLM", section "PagedAttention:
 *                        Paging for KV-Caches").
 *                      - The kernel gathers keys and values through the table
 *                        for QK^T and the value-weighted sum (same page,
 *                        section "PagedAttention: blocks and the block table";
 *                        "KV-cache paging in vLLM", section "The Attention
 *                        Kernel Change"). Paging changes where the bytes live,
 *                        not the result, so this is dense attention on the
 *                        gathered rows.
 *                      - Grouped queries: q head h reads kv head h / (Hq/Hk)
 *                        (the pages give only n_kv_heads in the per-token byte
 *                        count, "PagedAttention — Math + Memory Model",
 *                        section "The KV cache is big, and it grows"; the
 *                        contiguous grouping is this library's reading).
 *   oracle_append      Write each new token's K/V row into its slot,
 *                      slot = physical_block * B + offset ("KV-Cache
 *                      Optimization & PagedAttention for Long-Context Agents",
 *                      section "Key KV-Cache Optimization Principles", item 1:
 *                      blocks are filled as the model generates).
 *   oracle_block_copy  Copy a whole physical block (K and V, all heads) to a
 *                      fresh block ("PagedAttention — Math + Memory Model",
 *                      section "Copy-on-write").
 *   oracle_append_quant, oracle_decode_quant
 *                      The same append and decode over an 8-bit quantized
 *                      cache (see "quantized KV" below).
 *   oracle_decode_flat The same attention over K/V that sit in one flat span
 *                      per sequence instead of blocks: the alternative that
 *                      keeps each sequence's cache contiguous in virtual
 *                      memory and commits physical pages on demand
 *                      ("Contiguous vs Paged KV Cache on RDNA4", section "Why
 *                      the single-user verdict flipped", on vAttention).
 *
 * Element decoding (fp16 / bf16 / fp32 -> double) follows the IEEE-754
 * binary16 and bfloat16 bit layouts directly; it does not use any library
 * conversion.
 *
 * Layouts: q [S][Hq][D]; pools [NB][Hk][B][D]; tables [S][M] int32;
 * lens [S] int32; out [S][Hq][D] double. dtype codes: 0 f32, 1 f16, 2 bf16.
 *
 * Return codes: 0 ok, -1 invalid argument, -2 a block id or slot out of range.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_F32 0
#define OR_F16 1
#define OR_BF16 2

static size_t elem_size(int dtype) {
    return dtype == OR_F32 ? 4 : 2;
}

/* IEEE-754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);              /* subnormal: f * 2^(1-15-10) */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(f + 1024), e - 25);   /* (1.f) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE-754 binary32. */
static double decode_bf16(uint16_t h) {
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

static double decode_f32(uint32_t bits) {
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

static double load_elem(const void *base, int dtype, size_t idx) {
    if (dtype == OR_F32) {
        uint32_t b;
        memcpy(&b, (const char *)base + idx * 4, 4);
        return decode_f32(b);
    }
    uint16_t h;
    memcpy(&h, (const char *)base + idx * 2, 2);
    return dtype == OR_F16 ? decode_f16(h) : decode_bf16(h);
}

/* Exposed so the tests can check the decoders against every bit pattern. */
double oracle_decode_elem(int dtype, uint32_t bits) {
    if (dtype == OR_F32) return decode_f32(bits);
    if (dtype == OR_F16) return decode_f16((uint16_t)bits);
    return decode_bf16((uint16_t)bits);
}

/* Dense softmax attention of the G q heads of kv head g of sequence s over
 * L contiguous rows Kc, Vc [L][D] (fp64):
 *   z_t = scale * <q_h, k_t>,  w = softmax(z),  out_h = sum_t w_t v_t. */
static int attend(const void *q, int dtype, int Hq, int Hk, int D, int L, const double *Kc,
                  const double *Vc, double scale, int s, int g, double *out) {
    int G = Hq / Hk;
    double *z = (double *)malloc(sizeof(double) * (size_t)L);
    double *qh = (double *)malloc(sizeof(double) * (size_t)D);
    if (!z || !qh) { free(z); free(qh); return -1; }
    for (int j = 0; j < G; ++j) {
        int h = g * G + j;
        size_t qrow = ((size_t)s * Hq + h) * D;
        for (int d = 0; d < D; ++d) qh[d] = load_elem(q, dtype, qrow + d);
        /* scores z_t = scale * <q_h, k_t> */
        double m = -INFINITY;
        for (int t = 0; t < L; ++t) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += qh[d] * Kc[(size_t)t * D + d];
            z[t] = scale * acc;
            if (z[t] > m) m = z[t];
        }
        /* softmax weights w_t = exp(z_t - m) / sum exp(z - m) */
        double sum = 0.0;
        for (int t = 0; t < L; ++t) {
            z[t] = exp(z[t] - m);
            sum += z[t];
        }
        /* out = sum_t w_t v_t */
        for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int t = 0; t < L; ++t) acc += z[t] * Vc[(size_t)t * D + d];
            out[qrow + d] = acc / sum;
        }
    }
    free(z);
    free(qh);
    return 0;
}

/* Zero output rows for a sequence with no context. */
static void zero_rows(int Hq, int Hk, int D, int s, int g, double *out) {
    int G = Hq / Hk;
    for (int j = 0; j < G; ++j)
        for (int d = 0; d < D; ++d)
            out[((size_t)s * Hq + g * G + j) * D + d] = 0.0;
}

/* Attention for one (sequence, kv head): assemble contiguous K/V rows by
 * walking the block table, then dense softmax attention for each q head of
 * the group. */
static int decode_one(const void *q, int dtype, int Hq, int Hk, int B, int D,
                      const void *k_pool, const void *v_pool, int NB,
                      const int32_t *table_row, int M, int L, double scale,
                      int s, int g, double *out) {
    if (L == 0) {
        zero_rows(Hq, Hk, D, s, g, out);
        return 0;
    }
    if (L < 0 || (L + B - 1) / B > M) return -1;

    double *Kc = (double *)malloc(sizeof(double) * (size_t)L * D);
    double *Vc = (double *)malloc(sizeof(double) * (size_t)L * D);
    if (!Kc || !Vc) { free(Kc); free(Vc); return -1; }

    /* gather: token t lives at offset t % B of physical block table[t / B] */
    for (int t = 0; t < L; ++t) {
        int32_t phys = table_row[t / B];
        if (phys < 0 || phys >= NB) { free(Kc); free(Vc); return -2; }
        size_t row = (((size_t)phys * Hk + g) * B + (t % B)) * D;
        for (int d = 0; d < D; ++d) {
            Kc[(size_t)t * D + d] = load_elem(k_pool, dtype, row + d);
            Vc[(size_t)t * D + d] = load_elem(v_pool, dtype, row + d);
        }
    }
    int rc = attend(q, dtype, Hq, Hk, D, L, Kc, Vc, scale, s, g, out);
    free(Kc);
    free(Vc);
    return rc;
}

int oracle_decode(const void *q, int dtype, int S, int Hq, int Hk, int D, int B,
                  const void *k_pool, const void *v_pool, int NB,
                  const int32_t *block_tables, int M, const int32_t *context_lens,
                  double scale, double *out) {
    if (!q || !k_pool || !v_pool || !block_tables || !context_lens || !out) return -1;
    if (S < 0 || Hq <= 0 || Hk <= 0 || Hq % Hk != 0 || D <= 0 || B <= 0 || M <= 0) return -1;
    if (dtype < 0 || dtype > 2) return -1;
    int status = 0;
    long units = (long)S * Hk;
#pragma omp parallel for schedule(dynamic, 1)
    for (long u = 0; u < units; ++u) {
        int s = (int)(u / Hk), g = (int)(u % Hk);
        int rc = decode_one(q, dtype, Hq, Hk, B, D, k_pool, v_pool, NB,
                            block_tables + (size_t)s * M, M, context_lens[s], scale, s, g, out);
        if (rc != 0) {
#pragma omp critical
            status = rc;
        }
    }
    return status;
}

int oracle_append(const void *k_new, const void *v_new, const int64_t *slot_mapping, int N,
                  void *k_pool, void *v_pool, int dtype, int NB, int Hk, int B, int D) {
    if (!k_new || !v_new || !slot_mapping || !k_pool || !v_pool) return -1;
    if (dtype < 0 || dtype > 2 || N < 0 || NB <= 0 || Hk <= 0 || B <= 0 || D <= 0) return -1;
    size_t row_bytes = (size_t)D * elem_size(dtype);
    for (int i = 0; i < N; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0) continue;                 /* negative slot: no write */
        int64_t blk = slot / B, off = slot % B;
        if (blk >= NB) return -2;
        for (int g = 0; g < Hk; ++g) {
            size_t dst = ((size_t)(blk * Hk + g) * B + (size_t)off) * row_bytes;
            size_t src = ((size_t)i * Hk + g) * row_bytes;
            memcpy((char *)k_pool + dst, (const char *)k_new + src, row_bytes);
            memcpy((char *)v_pool + dst, (const char *)v_new + src, row_bytes);
        }
    }
    return 0;
}

int oracle_block_copy(const int64_t *pairs, int n, void *k_pool, void *v_pool,
                      int dtype, int NB, int Hk, int B, int D) {
    if (!pairs || !k_pool || !v_pool) return -1;
    if (dtype < 0 || dtype > 2 || n < 0) return -1;
    size_t blk_bytes = (size_t)Hk * B * D * elem_size(dtype);
    for (int i = 0; i < n; ++i) {
        int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= NB || dst < 0 || dst >= NB) return -2;
        memcpy((char *)k_pool + dst * blk_bytes, (const char *)k_pool + src * blk_bytes, blk_bytes);
        memcpy((char *)v_pool + dst * blk_bytes, (const char *)v_pool + src * blk_bytes, blk_bytes);
    }
    return 0;
}

/* ------------------------------------------------------------ quantized KV
 *
 * The pages name an 8-bit KV cache as the lever that halves the bytes each
 * decode step reads ("Contiguous vs Paged KV Cache on RDNA4", section "The
 * order of the memory levers": Q8 KV halves each agent's private read;
 * "KV-Cache Optimization & PagedAttention for Long-Context Agents",
 * introduction: PagedAttention together with KV-cache quantization). They fix
 * no code format and no scale granularity. This oracle follows the plainest
 * reading:
 *   - one 8-bit code per element, pools [NB][Hk][B][D] as for 16-bit data:
 *       kind 1 = int8, two's complement, codes -127 .. 127;
 *       kind 2 = fp8 E4M3 (the OCP 8-bit floating-point E4M3 format: 1 sign
 *       bit, 4 exponent bits with bias 7, 3 mantissa bits, subnormals, no
 *       infinities, S.1111.111 is NaN, largest finite magnitude 448);
 *   - one fp32 scale per (token, kv head) row, pools [NB][Hk][B], for K and
 *     for V;
 *   - a row x[0..D) (the fp16/bf16 activation, exact in fp32) becomes
 *       a = max_i |x_i|,  s = a / Qmax   (fp32 division, nearest even),
 *       Qmax = 127 (int8) or 448 (E4M3),
 *       code_i = x_i / s (fp32 division) rounded to the nearest int8 / E4M3
 *       value, ties to even, saturated to +-Qmax;
 *     a = 0 gives s = 0 and every code 0;
 *   - attention sees the value s * value(code), formed exactly in fp64.
 */
#define OR_Q_INT8 1
#define OR_Q_E4M3 2

/* E4M3 code -> value. */
static double e4m3_value(uint8_t b) {
    int sign = b >> 7, e = (b >> 3) & 0xf, m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);            /* subnormal: m/8 * 2^(1-7) */
    else v = ldexp(1.0 + m / 8.0, e - 7);           /* (1.m) * 2^(e-7) */
    return sign ? -v : v;
}

/* fp32 value -> nearest E4M3 code, ties to the even mantissa, saturating
 * finite values to +-448 (the midpoint between 448 and the next step, 480,
 * rounds to 448, so everything from 464 up saturates). */
static uint8_t e4m3_code(float xf) {
    if (isnan(xf)) return 0x7f;
    uint8_t sign = signbit(xf) ? 0x80 : 0;
    double a = fabs((double)xf);
    if (a >= 464.0) return sign | 0x7e;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: multiples of 2^-9; 8 * 2^-9 is the smallest normal,
         * whose code is 0x08, so the count is the code */
        return sign | (uint8_t)nearbyint(a * 512.0);
    }
    int e2;
    frexp(a, &e2);                                /* a in [2^(e2-1), 2^e2) */
    int E = e2 - 1;
    double m = nearbyint((ldexp(a, -E) - 1.0) * 8.0);  /* 0 .. 8 */
    if (m == 8.0) { m = 0.0; E += 1; }
    return sign | (uint8_t)(((E + 7) << 3) | (int)m);
}

/* Exposed so the tests can check the codec against a library conversion. */
double oracle_e4m3_decode(int code) { return e4m3_value((uint8_t)code); }
int oracle_e4m3_encode(float x) { return e4m3_code(x); }

static double code_value(int kind, uint8_t c) {
    return kind == OR_Q_INT8 ? (double)(int8_t)c : e4m3_value(c);
}

/* Quantize one row of D activations (decoded exactly to fp32). */
static void quantize_row(int kind, const float *x, int D, uint8_t *codes, float *scale) {
    float a = 0.0f;
    for (int d = 0; d < D; ++d) {
        float ax = fabsf(x[d]);
        if (ax > a) a = ax;
    }
    const float qmax = kind == OR_Q_INT8 ? 127.0f : 448.0f;
    float s = a / qmax;
    *scale = s;
    for (int d = 0; d < D; ++d) {
        if (a == 0.0f) { codes[d] = 0; continue; }
        float v = x[d] / s;
        if (kind == OR_Q_INT8) {
            float r = nearbyintf(v);
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
            codes[d] = (uint8_t)(int8_t)r;
        } else {
            codes[d] = e4m3_code(v);
        }
    }
}

/* Quantized append: each new token's K and V rows are quantized and written
 * with their scales at slot = block * B + offset; negative slots are skipped.
 * k_new / v_new [N][Hk][D] in act_dtype (f16 or bf16). */
int oracle_append_quant(int kind, int act_dtype, const void *k_new, const void *v_new,
                        const int64_t *slot_mapping, int N, uint8_t *k_codes, uint8_t *v_codes,
                        float *k_scales, float *v_scales, int NB, int Hk, int B, int D) {
    if (!k_new || !v_new || !slot_mapping || !k_codes || !v_codes || !k_scales || !v_scales)
        return -1;
    if ((kind != OR_Q_INT8 && kind != OR_Q_E4M3) || (act_dtype != OR_F16 && act_dtype != OR_BF16))
        return -1;
    if (N < 0 || NB <= 0 || Hk <= 0 || B <= 0 || D <= 0) return -1;
    float *x = (float *)malloc(sizeof(float) * (size_t)D);
    if (!x) return -1;
    for (int i = 0; i < N; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        int64_t blk = slot / B, off = slot % B;
        if (blk >= NB) { free(x); return -2; }
        for (int g = 0; g < Hk; ++g) {
            size_t row = (size_t)(blk * Hk + g) * B + (size_t)off;   /* row of the pool */
            size_t src = ((size_t)i * Hk + g) * D;
            for (int d = 0; d < D; ++d) x[d] = (float)load_elem(k_new, act_dtype, src + d);
            quantize_row(kind, x, D, k_codes + row * D, k_scales + row);
            for (int d = 0; d < D; ++d) x[d] = (float)load_elem(v_new, act_dtype, src + d);
            quantize_row(kind, x, D, v_codes + row * D, v_scales + row);
        }
    }
    free(x);
    return 0;
}

/* Quantized decode: gather through the block table as oracle_decode does,
 * forming each cache value as scale * value(code) in fp64, then the same
 * dense attention. q [S][Hq][D] in act_dtype. */
static int decode_one_quant(const void *q, int act_dtype, int Hq, int Hk, int B, int D, int kind,
                            const uint8_t *k_codes, const uint8_t *v_codes,
                            const float *k_scales, const float *v_scales, int NB,
                            const int32_t *table_row, int M, int L, double scale, int s, int g,
                            double *out) {
    if (L == 0) {
        zero_rows(Hq, Hk, D, s, g, out);
        return 0;
    }
    if (L < 0 || (L + B - 1) / B > M) return -1;
    double *Kc = (double *)malloc(sizeof(double) * (size_t)L * D);
    double *Vc = (double *)malloc(sizeof(double) * (size_t)L * D);
    if (!Kc || !Vc) { free(Kc); free(Vc); return -1; }
    for (int t = 0; t < L; ++t) {
        int32_t phys = table_row[t / B];
        if (phys < 0 || phys >= NB) { free(Kc); free(Vc); return -2; }
        size_t row = ((size_t)phys * Hk + g) * B + (t % B);
        double sk = k_scales[row], sv = v_scales[row];
        for (int d = 0; d < D; ++d) {
            Kc[(size_t)t * D + d] = sk * code_value(kind, k_codes[row * D + d]);
            Vc[(size_t)t * D + d] = sv * code_value(kind, v_codes[row * D + d]);
        }
    }
    int rc = attend(q, act_dtype, Hq, Hk, D, L, Kc, Vc, scale, s, g, out);
    free(Kc);
    free(Vc);
    return rc;
}

int oracle_decode_quant(const void *q, int act_dtype, int S, int Hq, int Hk, int D, int B,
                        int kind, const uint8_t *k_codes, const uint8_t *v_codes,
                        const float *k_scales, const float *v_scales, int NB,
                        const int32_t *block_tables, int M, const int32_t *context_lens,
                        double scale, double *out) {
    if (!q || !k_codes || !v_codes || !k_scales || !v_scales || !block_tables || !context_lens ||
        !out)
        return -1;
    if (S < 0 || Hq <= 0 || Hk <= 0 || Hq % Hk != 0 || D <= 0 || B <= 0 || M <= 0) return -1;
    if ((kind != OR_Q_INT8 && kind != OR_Q_E4M3) || (act_dtype != OR_F16 && act_dtype != OR_BF16))
        return -1;
    int status = 0;
    long units = (long)S * Hk;
#pragma omp parallel for schedule(dynamic, 1)
    for (long u = 0; u < units; ++u) {
        int s = (int)(u / Hk), g = (int)(u % Hk);
        int rc = decode_one_quant(q, act_dtype, Hq, Hk, B, D, kind, k_codes, v_codes, k_scales,
                                  v_scales, NB, block_tables + (size_t)s * M, M, context_lens[s],
                                  scale, s, g, out);
        if (rc != 0) {
#pragma omp critical
            status = rc;
        }
    }
    return status;
}

/* ------------------------------------------------------------- flat spans
 * Sequence s's cache is one span [capacity][Hk][D] (token-major: the rows of
 * all kv heads of token t are adjacent) at slot slots[s] of k_flat / v_flat
 * [num_slots][capacity][Hk][D]. Token t of kv head g is row (t * Hk + g) of
 * the span; no block table is involved. */
int oracle_decode_flat(const void *q, int dtype, int S, int Hq, int Hk, int D,
                       const void *k_flat, const void *v_flat, int num_slots, int capacity,
                       const int32_t *slots, const int32_t *context_lens, double scale,
                       double *out) {
    if (!q || !k_flat || !v_flat || !slots || !context_lens || !out) return -1;
    if (S < 0 || Hq <= 0 || Hk <= 0 || Hq % Hk != 0 || D <= 0 || capacity <= 0) return -1;
    if (dtype < 0 || dtype > 2) return -1;
    int status = 0;
    long units = (long)S * Hk;
#pragma omp parallel for schedule(dynamic, 1)
    for (long u = 0; u < units; ++u) {
        int s = (int)(u / Hk), g = (int)(u % Hk);
        int L = context_lens[s], slot = slots[s];
        int rc = 0;
        if (slot < 0 || slot >= num_slots || L < 0 || L > capacity) {
            rc = -2;
        } else if (L == 0) {
            zero_rows(Hq, Hk, D, s, g, out);
        } else {
            double *Kc = (double *)malloc(sizeof(double) * (size_t)L * D);
            double *Vc = (double *)malloc(sizeof(double) * (size_t)L * D);
            if (!Kc || !Vc) {
                rc = -1;
            } else {
                for (int t = 0; t < L; ++t) {
                    size_t row = (((size_t)slot * capacity + t) * Hk + g) * D;
                    for (int d = 0; d < D; ++d) {
                        Kc[(size_t)t * D + d] = load_elem(k_flat, dtype, row + d);
                        Vc[(size_t)t * D + d] = load_elem(v_flat, dtype, row + d);
                    }
                }
                rc = attend(q, dtype, Hq, Hk, D, L, Kc, Vc, scale, s, g, out);
            }
            free(Kc);
            free(Vc);
        }
        if (rc != 0) {
#pragma omp critical
            status = rc;
        }
    }
    return status;
}

/* Number of threads OpenMP uses (1 when built without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Set the number of threads later calls use (n >= 1); no effect without OpenMP. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
