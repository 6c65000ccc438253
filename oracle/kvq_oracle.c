/*
 * kvq oracle: a plain, slow, obviously correct CPU restatement of the quantized
 * KV-cache hot path (quantize-on-write, single-token decode attention, and
 * causal attention of a chunk of new queries over the cache).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may build, load or call this file.  It shares no
 * code, header, table or constant with the CUDA library: every table below is
 * generated here from the format definitions.
 *
 * Sources (web pages; cited by title and section):
 *  [TGI]  "Accelerating Inference with FP8 KV Cache" (text-generation-inference
 *         docs): intro (KV stored in FP8, computation in FP16); section
 *         "FP8 Formats: E4M3 and E5M2" (bit layouts, per-tensor fp32 scale);
 *         section "FP8 E4M3 KV Cache" (default scale 1.0).
 *  [LMD]  "[Feature] TurboMind support W8A8 or FP8 KV Cache" (lmdeploy issue
 *         1463): online KV-cache INT8 (quant-policy 8); the maintainers' reply
 *         names the INT8 and INT4 implementations side by side.
 *  OCP 8-bit floating point (named by [TGI]): E4M3 bias 7, no infinities,
 *  NaN = S.1111.111, max 448; E5M2 bias 15, IEEE-like Inf/NaN, max 57344.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - quantize divides by the scale, dequantize multiplies by it;
 *  - fp32 -> FP8 rounds to nearest, ties to even, and saturates to +-max
 *    (Inf included); NaN encodes to 0x7F;
 *  - INT8 is symmetric, one fp32 scale per (token, kv-head) row:
 *    s = fl32(amax / 127), q = clamp(rint(fl32(x / s)), -127, 127); amax == 0
 *    gives s = 0 and all-zero codes;
 *  - INT4 is the same with 4 bits: s = fl32(amax / 7), q in [-7, 7], two codes
 *    per byte (channel 2i in the low nibble, 2i+1 in the high nibble, 4-bit
 *    two's complement), so a cached row is D / 2 bytes;
 *  - per-group INT8 / INT4 (group quantization, named on the QQQ page "Scale
 *    factors and benchmarks" for a 4-bit KV cache): the row is cut into D / g
 *    groups of g consecutive channels, and each group is quantized exactly as a
 *    row is above (its own amax and fp32 scale); g = 0 or D is the per-row
 *    format.  Scales are stored [NB][Hkv][BS][D / g];
 *  - attention: logits l_t = sm_scale * <q, k_t> over all t < context_len,
 *    softmax, out = sum_t w_t v_t; q-head h reads kv-head h / (Hq / Hkv);
 *    context_len 0 gives zeros;
 *  - a chunk of n new queries of a sequence with context_len tokens (the
 *    chunk's own K/V already appended) holds positions context_len - n ...
 *    context_len - 1; query i attends causally to every t <= its position,
 *    i.e. it is the decode attention above with context_len - n + i + 1.
 *
 * Floating point: compile without fast-math and with -ffp-contract=off; every
 * fp32 step below is one IEEE operation in fp32, everything else is fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_E4M3 1
#define ORC_E5M2 2
#define ORC_INT8 3
#define ORC_INT4 4

/* ---------------------------------------------------------------- fp16 ---- */

/* IEEE binary16 bits -> value (1 sign, 5 exponent bits with bias 15, 10
 * mantissa bits).  Every binary16 value is exact in fp32 and fp64. */
static double half_bits_to_double(uint16_t h) {
    int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);               /* subnormal: m/1024 * 2^-14 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp(1024.0 + (double)m, e - 25);   /* (1 + m/1024) * 2^(e-15) */
    return s ? -v : v;
}

double oracle_half_to_double(uint16_t h) { return half_bits_to_double(h); }

/* ----------------------------------------------------------------- FP8 ---- */

/* [TGI] section "FP8 Formats": E4M3 = 1 sign, 4 biased exponent, 3 mantissa
 * bits; E5M2 = 1 sign, 5 biased exponent, 2 mantissa bits.  Values from the OCP
 * definitions named there. */
double oracle_fp8_decode(int fmt, uint8_t c) {
    int s = c >> 7;
    double v;
    if (fmt == ORC_E4M3) {
        int e = (c >> 3) & 15, m = c & 7;
        if (e == 15 && m == 7) return NAN;       /* the only NaN pattern; no Inf */
        v = (e == 0) ? ldexp((double)m, -9)      /* m/8 * 2^-6 */
                     : ldexp(8.0 + m, e - 10);   /* (1 + m/8) * 2^(e-7) */
    } else if (fmt == ORC_E5M2) {
        int e = (c >> 2) & 31, m = c & 3;
        if (e == 31) return m ? NAN : (s ? -INFINITY : INFINITY);
        v = (e == 0) ? ldexp((double)m, -16)     /* m/4 * 2^-14 */
                     : ldexp(4.0 + m, e - 17);   /* (1 + m/4) * 2^(e-15) */
    } else {
        return NAN;
    }
    return s ? -v : v;
}

/* Positive finite values of a format, sorted ascending, with their codes.
 * Built by decoding all 128 sign-0 codes and sorting by value; nothing assumes
 * that code order equals value order. */
typedef struct { double v; uint8_t code; } fp8_entry;
static fp8_entry g_tab[3][128];
static int g_ntab[3];

static int cmp_entry(const void* a, const void* b) {
    double x = ((const fp8_entry*)a)->v, y = ((const fp8_entry*)b)->v;
    return (x > y) - (x < y);
}

static const fp8_entry* fp8_table(int fmt, int* n) {
    int i = fmt - 1;
    if (g_ntab[i] == 0) {
        int k = 0;
        for (int c = 0; c < 128; ++c) {
            double v = oracle_fp8_decode(fmt, (uint8_t)c);
            if (isfinite(v)) { g_tab[i][k].v = v; g_tab[i][k].code = (uint8_t)c; ++k; }
        }
        qsort(g_tab[i], (size_t)k, sizeof(fp8_entry), cmp_entry);
        g_ntab[i] = k;
    }
    *n = g_ntab[i];
    return g_tab[i];
}

/* Must be called once before any parallel use of the encoder. */
void oracle_init(void) {
    int n;
    fp8_table(ORC_E4M3, &n);
    fp8_table(ORC_E5M2, &n);
}

/* fp32 -> FP8 code: nearest representable value, ties to the code with an even
 * mantissa LSB, saturating to +-max (Inf too); signed zero for values that round
 * to zero; NaN -> 0x7F. */
uint8_t oracle_fp8_encode(int fmt, float y) {
    if (isnan(y)) return 0x7F;
    int n;
    const fp8_entry* t = fp8_table(fmt, &n);
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs((double)y);
    if (a >= t[n - 1].v) return sign | t[n - 1].code;
    /* binary search: largest i with t[i].v <= a  (t[0].v == 0 <= a) */
    int lo = 0, hi = n - 1;                   /* invariant: t[lo].v <= a < t[hi].v */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (t[mid].v <= a) lo = mid; else hi = mid;
    }
    double midpoint = 0.5 * (t[lo].v + t[hi].v);   /* exact: dyadic, few bits */
    uint8_t code;
    if (a < midpoint) code = t[lo].code;
    else if (a > midpoint) code = t[hi].code;
    else code = (t[lo].code & 1) ? t[hi].code : t[lo].code;
    return sign | code;
}

void oracle_fp8_encode_array(int fmt, const float* y, uint8_t* out, int64_t n) {
    oracle_init();
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_fp8_encode(fmt, y[i]);
}

/* ---------------------------------------------------------------- INT8 ---- */

/* [LMD] online KV INT8, symmetric reading: one fp32 scale per row of D values.
 * x: D fp32 values; writes D codes and returns the scale. */
static float int8_quant_row(const float* x, int D, int8_t* q) {
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) {
        float ax = fabsf(x[d]);
        if (ax > amax) amax = ax;
    }
    float s = amax / 127.0f;
    for (int d = 0; d < D; ++d) {
        if (s == 0.0f) { q[d] = 0; continue; }
        float y = x[d] / s;
        float r = rintf(y);                      /* ties to even (default mode) */
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q[d] = (int8_t)r;
    }
    return s;
}

float oracle_int8_quant_row(const float* x, int D, int8_t* q) { return int8_quant_row(x, D, q); }

/* ---------------------------------------------------------------- INT4 ---- */

/* The INT4 reading: one fp32 scale per row, s = fl32(amax / 7), codes
 * clamp(rint(fl32(x / s)), -7, 7) packed two per byte (channel 2i low nibble,
 * 2i+1 high nibble).  x: D fp32 values (D even); writes D / 2 bytes and returns
 * the scale. */
static float int4_quant_row(const float* x, int D, uint8_t* packed) {
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) {
        float ax = fabsf(x[d]);
        if (ax > amax) amax = ax;
    }
    float s = amax / 7.0f;
    for (int i = 0; i < D / 2; ++i) {
        int q2[2];
        for (int z = 0; z < 2; ++z) {
            float r = 0.0f;
            if (s != 0.0f) {
                r = rintf(x[2 * i + z] / s);         /* ties to even (default mode) */
                if (r > 7.0f) r = 7.0f;
                if (r < -7.0f) r = -7.0f;
            }
            q2[z] = (int)r;
        }
        packed[i] = (uint8_t)((q2[0] & 0xF) | ((q2[1] & 0xF) << 4));
    }
    return s;
}

float oracle_int4_quant_row(const float* x, int D, uint8_t* packed) { return int4_quant_row(x, D, packed); }

/* The signed 4-bit code of channel d of a packed row. */
static int int4_code(const uint8_t* row, int d) {
    int nib = (row[d >> 1] >> ((d & 1) * 4)) & 0xF;
    return nib >= 8 ? nib - 16 : nib;
}

/* Bytes of one cached (token, kv-head) row. */
static int row_bytes(int fmt, int D) { return fmt == ORC_INT4 ? D / 2 : D; }

/* Formats that carry fp32 scales per (token, kv-head) row (one, or one per group). */
static int row_scaled(int fmt) { return fmt == ORC_INT8 || fmt == ORC_INT4; }

/* Channels per scale of a row-scaled format: group (0 = the whole row). */
static int group_channels(int D, int group) { return group > 0 ? group : D; }

/* A valid group for the format and head_dim: 0, or a divisor of D (even for INT4). */
static int group_ok(int fmt, int D, int group) {
    if (group == 0) return 1;
    if (!row_scaled(fmt) || group < 0 || D % group != 0) return 0;
    return fmt != ORC_INT4 || group % 2 == 0;
}

/* The scale of channel d of cached row `row`: the per-tensor scale for FP8,
 * else the row's scale of the group holding d. */
static float scale_of(int fmt, const float* scales, size_t row, int D, int group, int d, float scale) {
    if (!row_scaled(fmt)) return scale;
    const int gc = group_channels(D, group);
    return scales[row * (size_t)(D / gc) + (size_t)(d / gc)];
}

/* -------------------------------------------------------------- append ---- */

/* Quantize-on-write.  k, v: fp16 bits [T][Hkv][D].  The paged cache holds codes
 * [NB][Hkv][BS][D] (u8 FP8 / i8 INT8; [D / 2] packed bytes for INT4) and, for
 * INT8 and INT4, scales [NB][Hkv][BS][D / g] (g = group channels, the whole
 * row when group is 0).
 * Token t goes to block slot[t] / BS, row slot[t] % BS; slot -1 is skipped.
 * scale: per-tensor fp32 scale (FP8 only; [TGI] default 1.0 applies when the
 * caller passes none).  Returns 0, -1 on a slot outside the cache, -2 on a
 * group the format and D do not allow. */
int oracle_append(const uint16_t* k, const uint16_t* v, int64_t T, int Hkv, int D,
                  const int64_t* slot_mapping, uint8_t* k_codes, uint8_t* v_codes,
                  float* k_scales, float* v_scales, int64_t NB, int BS, int fmt, int group,
                  float scale) {
    oracle_init();
    if (!group_ok(fmt, D, group)) return -2;
    const int gc = group_channels(D, group), ng = D / gc;
    int bad = 0;
    float* x = (float*)malloc(sizeof(float) * (size_t)D);
    for (int64_t t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot == -1) continue;
        if (slot < 0 || slot >= NB * BS) { bad = 1; continue; }
        int64_t blk = slot / BS, off = slot % BS;
        for (int h = 0; h < Hkv; ++h) {
            for (int which = 0; which < 2; ++which) {
                const uint16_t* src = (which ? v : k) + ((size_t)t * Hkv + h) * D;
                uint8_t* dst = (which ? v_codes : k_codes) + (((size_t)blk * Hkv + h) * BS + off) * row_bytes(fmt, D);
                for (int d = 0; d < D; ++d) x[d] = (float)half_bits_to_double(src[d]);
                float* sc = (which ? v_scales : k_scales) + (((size_t)blk * Hkv + h) * BS + off) * ng;
                if (fmt == ORC_INT8) {
                    for (int j = 0; j < ng; ++j) sc[j] = int8_quant_row(x + j * gc, gc, (int8_t*)dst + j * gc);
                } else if (fmt == ORC_INT4) {
                    for (int j = 0; j < ng; ++j) sc[j] = int4_quant_row(x + j * gc, gc, dst + j * gc / 2);
                } else {
                    for (int d = 0; d < D; ++d) dst[d] = oracle_fp8_encode(fmt, x[d] / scale);
                }
            }
        }
    }
    free(x);
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------- dequant ---- */

/* Dequantize-on-read of one cached value: FP8 fl32(decode(c) * s) with the
 * per-tensor scale, INT8 fl32(q * s_row). */
static float dequant_value(int fmt, uint8_t c, float s) {
    if (fmt == ORC_INT8) return (float)(int8_t)c * s;
    return (float)oracle_fp8_decode(fmt, c) * s;
}

/* Channel d of a cached row (row = its first byte), dequantized: INT4
 * fl32(q * s_row), else as dequant_value. */
static float cached_value(int fmt, const uint8_t* row, int d, float s) {
    if (fmt == ORC_INT4) return (float)int4_code(row, d) * s;
    return dequant_value(fmt, row[d], s);
}

/* Gather + dequantize rows at the given slots: out [n][Hkv][D] fp32 (K and V). */
int oracle_dequant(const uint8_t* k_codes, const uint8_t* v_codes, const float* k_scales,
                   const float* v_scales, int64_t NB, int BS, int Hkv, int D, int fmt, int group,
                   const int64_t* slots, int64_t n, float scale, float* out_k, float* out_v) {
    if (!group_ok(fmt, D, group)) return -2;
    const size_t rb = (size_t)row_bytes(fmt, D);
    for (int64_t i = 0; i < n; ++i) {
        int64_t slot = slots[i];
        if (slot < 0 || slot >= NB * BS) return -1;
        int64_t blk = slot / BS, off = slot % BS;
        for (int h = 0; h < Hkv; ++h) {
            size_t row = ((size_t)blk * Hkv + h) * BS + off;
            for (int d = 0; d < D; ++d) {
                float sk = scale_of(fmt, k_scales, row, D, group, d, scale);
                float sv = scale_of(fmt, v_scales, row, D, group, d, scale);
                out_k[((size_t)i * Hkv + h) * D + d] = cached_value(fmt, k_codes + row * rb, d, sk);
                out_v[((size_t)i * Hkv + h) * D + d] = cached_value(fmt, v_codes + row * rb, d, sv);
            }
        }
    }
    return 0;
}

/* ---------------------------------------------------------- attention ---- */

/* Single-token decode attention over the paged quantized cache, in fp64 on the
 * fp32-dequantized values.  q: fp16 bits [B][Hq][D], D <= 512.  block_tables int32
 * [B][max_blocks]; context_lens int32 [B].  out: fp64 [B][Hq][D].  weights
 * (optional, may be NULL): fp64 [B][Hq][w_stride], the softmax weights.
 * Returns 0, or -1 on a block id / context length outside the cache or table. */
int oracle_decode_attention(const uint16_t* q, int B, int Hq, int D,
                            const uint8_t* k_codes, const uint8_t* v_codes,
                            const float* k_scales, const float* v_scales,
                            int64_t NB, int BS, int Hkv, int fmt, int group,
                            const int32_t* block_tables, int max_blocks,
                            const int32_t* context_lens, float scale, double sm_scale,
                            double* out, double* weights, int64_t w_stride) {
    if (!group_ok(fmt, D, group)) return -2;
    int G = Hq / Hkv;
    const size_t rb = (size_t)row_bytes(fmt, D);
    int bad = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) reduction(| : bad)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < Hq; ++h) {
            int kvh = h / G;
            int ctx = context_lens[b];
            double* o = out + ((size_t)b * Hq + h) * D;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            if (ctx <= 0) continue;
            if ((int64_t)ctx > (int64_t)max_blocks * BS) { bad = 1; continue; }
            double qv[512];
            for (int d = 0; d < D; ++d) qv[d] = half_bits_to_double(q[((size_t)b * Hq + h) * D + d]);
            double* logit = (double*)malloc(sizeof(double) * (size_t)ctx);
            int ok = 1;
            for (int t = 0; t < ctx && ok; ++t) {
                int32_t blk = block_tables[(size_t)b * max_blocks + t / BS];
                if (blk < 0 || blk >= NB) { ok = 0; break; }
                size_t row = ((size_t)blk * Hkv + kvh) * BS + t % BS;
                double acc = 0.0;
                for (int d = 0; d < D; ++d)
                    acc += qv[d] * (double)cached_value(fmt, k_codes + row * rb, d,
                                                        scale_of(fmt, k_scales, row, D, group, d, scale));
                logit[t] = sm_scale * acc;
            }
            if (!ok) { bad = 1; free(logit); continue; }
            double m = -INFINITY;
            for (int t = 0; t < ctx; ++t) if (logit[t] > m) m = logit[t];
            double denom = 0.0;
            for (int t = 0; t < ctx; ++t) { logit[t] = exp(logit[t] - m); denom += logit[t]; }
            for (int t = 0; t < ctx; ++t) {
                double w = logit[t] / denom;
                if (weights) weights[((size_t)b * Hq + h) * w_stride + t] = w;
                int32_t blk = block_tables[(size_t)b * max_blocks + t / BS];
                size_t row = ((size_t)blk * Hkv + kvh) * BS + t % BS;
                for (int d = 0; d < D; ++d)
                    o[d] += w * (double)cached_value(fmt, v_codes + row * rb, d,
                                                     scale_of(fmt, v_scales, row, D, group, d, scale));
            }
            free(logit);
        }
    }
    return bad ? -1 : 0;
}

/* Causal attention of chunks of new queries over the paged quantized cache,
 * fp64 on the fp32-dequantized values.  q: fp16 bits [Tq][Hq][D], D <= 512, the
 * rows of sequence b at query_start[b] .. query_start[b+1]-1 (n_b of them, in
 * position order); context_lens[b] counts every cached token of b, the chunk's
 * own included.  Query i of sequence b sits at p = context_lens[b] - n_b + i
 * and attends to t = 0 .. p:  l_t = sm_scale <q, k_t>, w = softmax(l),
 * out = sum_t w_t v_t.  out: fp64 [Tq][Hq][D].  Returns 0, or -1 on a chunk
 * longer than its context or a block id / context outside the cache or table. */
int oracle_prefill_attention(const uint16_t* q, int64_t Tq, int B, int Hq, int D,
                             const uint8_t* k_codes, const uint8_t* v_codes,
                             const float* k_scales, const float* v_scales,
                             int64_t NB, int BS, int Hkv, int fmt, int group,
                             const int32_t* block_tables, int max_blocks,
                             const int32_t* context_lens, const int32_t* query_start,
                             float scale, double sm_scale, double* out) {
    if (!group_ok(fmt, D, group)) return -2;
    int G = Hq / Hkv;
    const size_t rb = (size_t)row_bytes(fmt, D);
    int bad = 0;
    for (int64_t r = 0; r < Tq * Hq * D; ++r) out[r] = 0.0;
    for (int b = 0; b < B; ++b) {
        int n = query_start[b + 1] - query_start[b];
        if (n < 0 || n > context_lens[b] || query_start[b] < 0 || query_start[b + 1] > Tq) bad = 1;
        if ((int64_t)context_lens[b] > (int64_t)max_blocks * BS) bad = 1;
    }
    if (bad) return -1;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t row = 0; row < Tq; ++row) {
        int b = 0;
        while (b < B && !(row >= query_start[b] && row < query_start[b + 1])) ++b;
        if (b == B) continue;                       /* a row no chunk covers stays zero */
        int n = query_start[b + 1] - query_start[b];
        int pos = context_lens[b] - n + (int)(row - query_start[b]);
        int len = pos + 1;                          /* tokens 0 .. pos attend */
        double* logit = (double*)malloc(sizeof(double) * (size_t)len);
        double qv[512];
        for (int h = 0; h < Hq; ++h) {
            int kvh = h / G;
            double* o = out + ((size_t)row * Hq + h) * D;
            for (int d = 0; d < D; ++d) qv[d] = half_bits_to_double(q[((size_t)row * Hq + h) * D + d]);
            int ok = 1;
            for (int t = 0; t < len; ++t) {
                int32_t blk = block_tables[(size_t)b * max_blocks + t / BS];
                if (blk < 0 || blk >= NB) { ok = 0; break; }
                size_t kr = ((size_t)blk * Hkv + kvh) * BS + t % BS;
                double acc = 0.0;
                for (int d = 0; d < D; ++d)
                    acc += qv[d] * (double)cached_value(fmt, k_codes + kr * rb, d,
                                                        scale_of(fmt, k_scales, kr, D, group, d, scale));
                logit[t] = sm_scale * acc;
            }
            if (!ok) { bad = 1; break; }
            double m = -INFINITY;
            for (int t = 0; t < len; ++t) if (logit[t] > m) m = logit[t];
            double denom = 0.0;
            for (int t = 0; t < len; ++t) { logit[t] = exp(logit[t] - m); denom += logit[t]; }
            for (int t = 0; t < len; ++t) {
                double w = logit[t] / denom;
                int32_t blk = block_tables[(size_t)b * max_blocks + t / BS];
                size_t vr = ((size_t)blk * Hkv + kvh) * BS + t % BS;
                for (int d = 0; d < D; ++d)
                    o[d] += w * (double)cached_value(fmt, v_codes + vr * rb, d,
                                                     scale_of(fmt, v_scales, vr, D, group, d, scale));
            }
        }
        free(logit);
    }
    return bad ? -1 : 0;
}

int oracle_num_threads(void) {
    int n = 1;
#ifdef _OPENMP
#pragma omp parallel
    {
#pragma omp single
        n = omp_get_num_threads();
    }
#endif
    return n;
}
