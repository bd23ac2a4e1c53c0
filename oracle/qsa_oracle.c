/*
 * Packed QSA decode oracle: plain FP64 CPU reference.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or
 * calls this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg do. It shares no code, header, table or
 * constant with the CUDA implementation.
 *
 * What it computes (sglang PR #36845 "fix(qsa): restore SM121 correctness",
 * sections "Changes" and "Optimized kernel"; sglang PR #37798 "quantized KV
 * pools with dequant-on-gather", section "Modifications"):
 *
 *   for every sequence b with L = cu[b+1] - cu[b] selected slots
 *   I_j = sel[cu[b] + j] (order and duplicates kept, 1Cat-vLLM PR #523,
 *   "Purpose"), and every query head h with KV head g = h / (Hq / Hkv):
 *
 *     s_j = softmax_scale * sum_d q[b,h,d] * Khat[I_j, g, d]
 *     o_d = sum_j exp(s_j - max s) Vhat[I_j, g, d] / sum_j exp(s_j - max s)
 *     L == 0  ->  o = 0
 *
 * Dequantisation is exact in FP64 and follows the pool formats:
 *   bf16    : the stored value
 *   fp8     : e4m3fn(byte) * s_tensor            (one fp32 scale per pool)
 *   int8    : int8 * s[slot, g]                  (fp32 per (slot, KV head))
 *   int4    : sext4(nibble) * s[slot, g]; two per byte, element 2i in the
 *             low nibble (two's-complement nibbles)
 *   int8_g64: int8 * s16[slot, g, d / 64]       (IEEE binary16 per 64-channel
 *             group; group 0 holds the rotary dims)
 *   int4_g32: (nibble - 8) * s16[slot, g, d / 32] (offset-binary nibbles, element
 *             2i in the low nibble; binary16 per 32-channel group)
 * (the grouped formats: sglang PR #37798, "Modifications", the int8 and int4
 * KV pool modules)
 *   int8ring_int4: a row (slot, g) reads the int8_g64 ring row
 *             (slot & (R - 1), g) when owner[slot & (R - 1)] == slot (hot),
 *             else the int4_g32 pool row (slot, g) (cold)  (same PR, the
 *             tiered KV pool module: every token is written to both)
 *
 * Every step is written as the definition states it: no tiling, no
 * online softmax, no split, no merge. The scores use one exact max
 * subtraction, as the textbook softmax does.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_BF16 = 0, ORC_FP8_E4M3 = 1, ORC_INT8 = 2, ORC_INT4 = 3, ORC_INT8_G64 = 4, ORC_INT4_G32 = 5,
       ORC_INT8RING_INT4 = 6 };

/* Channels per scale group: 64 / 32 for the grouped formats, 0 otherwise. */
static int group_size(int format) {
    return format == ORC_INT8_G64 ? 64 : format == ORC_INT4_G32 ? 32 : 0;
}

/* Pool rows hold D / 2 bytes (two 4-bit codes per byte). */
static int is_nibble_format(int format) {
    return format == ORC_INT4 || format == ORC_INT4_G32 || format == ORC_INT8RING_INT4;
}

/* bf16 -> double: a bf16 is the upper half of an IEEE binary32. */
double orc_bf16_to_double(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3 ("fn": no infinities, S.1111.111 is NaN, max 448): 1 sign,
 * 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 encodes
 * subnormals m/8 * 2^-6. */
double orc_e4m3fn_to_double(uint8_t b) {
    int sign = b >> 7;
    int e = (b >> 3) & 0xF;
    int m = b & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* IEEE 754 binary16: 1 sign, 5 exponent bits with bias 15, 10 fraction bits;
 * exponent field 0 encodes subnormals f/1024 * 2^-14, field 31 inf / NaN. */
double orc_fp16_to_double(uint16_t h) {
    int sign = h >> 15;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0x1F) v = f ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)f / 1024.0, -14);
    else v = ldexp(1.0 + (double)f / 1024.0, e - 15);
    return sign ? -v : v;
}

/* Round a binary32 value to the nearest binary16 (ties to even), returning its
 * bits; magnitudes that round beyond 65504 give infinity. */
uint16_t orc_round_fp16(float x) {
    if (isnan(x)) return 0x7E00;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs((double)x);
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | 0x7C00;
    int e2;
    frexp(a, &e2);
    int E = e2 - 1;              /* floor(log2 a) */
    if (E < -14) E = -14;        /* subnormal quantum is 2^-24 */
    double quantum = ldexp(1.0, E - 10);
    double r = nearbyint(a / quantum) * quantum; /* ties to even */
    if (r > 65504.0) return sign | 0x7C00;
    if (r < ldexp(1.0, -14)) return sign | (uint16_t)(r / ldexp(1.0, -24));
    frexp(r, &e2);
    E = e2 - 1;
    uint16_t frac = (uint16_t)((r / ldexp(1.0, E) - 1.0) * 1024.0);
    return sign | (uint16_t)((E + 15) << 10) | frac;
}

/* Offset-binary 4-bit value held in bits [4*hi, 4*hi+3] of `byte`: u - 8. */
int orc_int4_offset_value(uint8_t byte, int hi) {
    int n = hi ? (byte >> 4) & 0xF : byte & 0xF;
    return n - 8;
}

/* Two's-complement 4-bit value held in bits [4*hi, 4*hi+3] of `byte`. */
int orc_int4_value(uint8_t byte, int hi) {
    int n = hi ? (byte >> 4) & 0xF : byte & 0xF;
    return n >= 8 ? n - 16 : n;
}

/* Round a double to the nearest bf16 (ties to even), returning its bits.
 * bf16 keeps 8 significant bits and the binary32 exponent range. */
uint16_t orc_round_bf16(double x) {
    if (isnan(x)) return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | 0x7F80;
    int e2;
    frexp(a, &e2);                 /* a = m * 2^e2, m in [0.5, 1) */
    int E = e2 - 1;                /* floor(log2 a) */
    if (E < -126) E = -126;        /* subnormal quantum is 2^-133 */
    double quantum = ldexp(1.0, E - 7);
    double r = nearbyint(a / quantum) * quantum; /* default mode: ties to even */
    if (r > 3.3895313892515355e38) return sign | 0x7F80; /* beyond max bf16 */
    float f = (float)r;            /* exact: r is a bf16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

/* Element-wise orc_round_bf16 over n doubles. */
void orc_round_bf16_array(const double* x, uint16_t* bits, int64_t n) {
    for (int64_t i = 0; i < n; ++i) bits[i] = orc_round_bf16(x[i]);
}

typedef struct {
    const void* pool;
    int format;
    int Hkv;
    int D;
    const void* scale; /* fp8: float [1]; int8/int4: float [num_slots * Hkv];
                          grouped: binary16 bits [num_slots * Hkv * D / group]; bf16: unused */
    /* int8ring_int4 only: the hot ring (int8_g64 rows [R, Hkv, D] and binary16
     * scales [R, Hkv, D / 64]) and its owner table [R]; pool / scale above are
     * the int4_g32 rows and scales of every slot */
    const int8_t* ring;
    const uint16_t* ring_scale;
    const int32_t* owner;
    int64_t R;
} orc_pool;

/* Dequantised element d of pool row (slot, g), exactly in FP64. */
static double pool_elem(const orc_pool* p, int64_t slot, int g, int d) {
    int64_t row = slot * p->Hkv + g;
    if (p->format == ORC_INT8RING_INT4) {
        const int64_t pos = slot & (p->R - 1);
        if ((int64_t)p->owner[pos] == slot) { /* hot: the ring row */
            orc_pool hot = {p->ring, ORC_INT8_G64, p->Hkv, p->D, p->ring_scale, 0, 0, 0, 0};
            return pool_elem(&hot, pos, g, d);
        }
        orc_pool cold = {p->pool, ORC_INT4_G32, p->Hkv, p->D, p->scale, 0, 0, 0, 0};
        return pool_elem(&cold, slot, g, d);
    }
    switch (p->format) {
    case ORC_BF16:
        return orc_bf16_to_double(((const uint16_t*)p->pool)[row * p->D + d]);
    case ORC_FP8_E4M3:
        return orc_e4m3fn_to_double(((const uint8_t*)p->pool)[row * p->D + d]) *
               (double)((const float*)p->scale)[0];
    case ORC_INT8:
        return (double)((const int8_t*)p->pool)[row * p->D + d] * (double)((const float*)p->scale)[row];
    case ORC_INT4: {
        uint8_t byte = ((const uint8_t*)p->pool)[row * (p->D / 2) + d / 2];
        return (double)orc_int4_value(byte, d & 1) * (double)((const float*)p->scale)[row];
    }
    case ORC_INT8_G64: {
        const int groups = p->D / 64;
        const uint16_t s16 = ((const uint16_t*)p->scale)[row * groups + d / 64];
        return (double)((const int8_t*)p->pool)[row * p->D + d] * orc_fp16_to_double(s16);
    }
    case ORC_INT4_G32: {
        const int groups = p->D / 32;
        const uint16_t s16 = ((const uint16_t*)p->scale)[row * groups + d / 32];
        uint8_t byte = ((const uint8_t*)p->pool)[row * (p->D / 2) + d / 2];
        return (double)orc_int4_offset_value(byte, d & 1) * orc_fp16_to_double(s16);
    }
    }
    return NAN;
}

/* Dequantise one pool row into `dst` (D doubles). */
void orc_dequant_row(const void* pool, int format, int Hkv, int D, const void* scale,
                     int64_t slot, int g, double* dst) {
    orc_pool p = {pool, format, Hkv, D, scale, 0, 0, 0, 0};
    for (int d = 0; d < D; ++d) dst[d] = pool_elem(&p, slot, g, d);
}

/*
 * Full decode. Returns 0 on success and a negative value when the input
 * breaks the contract the pages define (the oracle refuses such inputs
 * instead of guessing an answer):
 *   -1  bad geometry (Hq not a multiple of Hkv, D odd for int4, D not a
 *       multiple of the scale group, unknown format)
 *   -2  cu_seqlens not monotone, negative, or beyond the index buffer
 *   -3  a selected slot outside [0, num_slots)
 *
 * q       : bf16 bits, element (b, h, d) at q[b*q_sb + h*q_sh + d]
 * rows    : optional subset of sequences to compute (NULL: all bs rows);
 *           output row i holds sequence rows[i]
 * out     : double [n_rows][Hq][D]
 */
static int decode_impl(const uint16_t* q, int64_t q_sb, int64_t q_sh, orc_pool kp, orc_pool vp,
                       int64_t num_slots, double softmax_scale, const int32_t* sel, int64_t n_sel,
                       const int32_t* cu, int bs, int Hq, const int32_t* rows, int n_rows,
                       double* out, int nthreads);

int orc_decode(const uint16_t* q, int64_t q_sb, int64_t q_sh,
               const void* k_pool, const void* v_pool, int format,
               int64_t num_slots, int Hkv, int D,
               const void* k_scale, const void* v_scale, double softmax_scale,
               const int32_t* sel, int64_t n_sel, const int32_t* cu, int bs, int Hq,
               const int32_t* rows, int n_rows, double* out, int nthreads) {
    if (Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0 || D <= 0) return -1;
    if (format < ORC_BF16 || format > ORC_INT4_G32) return -1;
    if (is_nibble_format(format) && (D & 1)) return -1;
    if (group_size(format) && D % group_size(format)) return -1;
    orc_pool kp = {k_pool, format, Hkv, D, k_scale, 0, 0, 0, 0};
    orc_pool vp = {v_pool, format, Hkv, D, v_scale, 0, 0, 0, 0};
    return decode_impl(q, q_sb, q_sh, kp, vp, num_slots, softmax_scale, sel, n_sel, cu, bs, Hq,
                       rows, n_rows, out, nthreads);
}

/* Decode over a tiered pool: int4_g32 rows + scales of every slot (k_pool,
 * k_scale, ...), the int8_g64 ring [R, Hkv, D] with binary16 scales
 * [R, Hkv, D / 64], and the owner table [R] (R a power of two). Same return
 * codes as orc_decode. */
int orc_decode_tiered(const uint16_t* q, int64_t q_sb, int64_t q_sh,
                      const void* k_pool, const void* v_pool, int64_t num_slots, int Hkv, int D,
                      const void* k_scale, const void* v_scale,
                      const int8_t* k_ring, const int8_t* v_ring,
                      const uint16_t* k_ring_scale, const uint16_t* v_ring_scale,
                      const int32_t* owner, int64_t R, double softmax_scale,
                      const int32_t* sel, int64_t n_sel, const int32_t* cu, int bs, int Hq,
                      const int32_t* rows, int n_rows, double* out, int nthreads) {
    if (Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0 || D <= 0 || D % 64) return -1;
    if (R <= 0 || (R & (R - 1))) return -1;
    orc_pool kp = {k_pool, ORC_INT8RING_INT4, Hkv, D, k_scale, k_ring, k_ring_scale, owner, R};
    orc_pool vp = {v_pool, ORC_INT8RING_INT4, Hkv, D, v_scale, v_ring, v_ring_scale, owner, R};
    return decode_impl(q, q_sb, q_sh, kp, vp, num_slots, softmax_scale, sel, n_sel, cu, bs, Hq,
                       rows, n_rows, out, nthreads);
}

static int decode_impl(const uint16_t* q, int64_t q_sb, int64_t q_sh, orc_pool kp, orc_pool vp,
                       int64_t num_slots, double softmax_scale, const int32_t* sel, int64_t n_sel,
                       const int32_t* cu, int bs, int Hq, const int32_t* rows, int n_rows,
                       double* out, int nthreads) {
    const int Hkv = kp.Hkv, D = kp.D;
    if (rows == NULL) n_rows = bs;
    for (int i = 0; i < n_rows; ++i) {
        int b = rows ? rows[i] : i;
        if (b < 0 || b >= bs) return -1;
        int64_t start = cu[b], stop = cu[b + 1];
        if (start < 0 || stop < start || stop > n_sel) return -2;
        for (int64_t t = start; t < stop; ++t)
            if (sel[t] < 0 || (int64_t)sel[t] >= num_slots) return -3;
    }
    const int group = Hq / Hkv;
    const int64_t tasks = (int64_t)n_rows * Hq;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t task = 0; task < tasks; ++task) {
        int i = (int)(task / Hq);
        int h = (int)(task % Hq);
        int b = rows ? rows[i] : i;
        int g = h / group;
        int64_t L = (int64_t)cu[b + 1] - cu[b];
        const int32_t* idx = sel + cu[b];
        double* o = out + ((int64_t)i * Hq + h) * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (L == 0) continue;

        double* qd = (double*)malloc(sizeof(double) * D);
        double* s = (double*)malloc(sizeof(double) * L);
        for (int d = 0; d < D; ++d) qd[d] = orc_bf16_to_double(q[b * q_sb + h * q_sh + d]);

        /* scores */
        for (int64_t j = 0; j < L; ++j) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += qd[d] * pool_elem(&kp, idx[j], g, d);
            s[j] = softmax_scale * acc;
        }
        /* softmax weights with one max subtraction */
        double smax = s[0];
        for (int64_t j = 1; j < L; ++j)
            if (s[j] > smax) smax = s[j];
        double z = 0.0;
        for (int64_t j = 0; j < L; ++j) {
            s[j] = exp(s[j] - smax);
            z += s[j];
        }
        /* weighted sum of the selected V rows */
        for (int64_t j = 0; j < L; ++j)
            for (int d = 0; d < D; ++d) o[d] += s[j] * pool_elem(&vp, idx[j], g, d);
        for (int d = 0; d < D; ++d) o[d] /= z;
        free(qd);
        free(s);
    }
    return 0;
}

/* ------------------------------------------------------------------ KV write
 *
 * The quantising write that fills the pools (sglang PR #37798, "Modifications":
 * one fused quantise + scatter per write; part 1, mem_cache/memory_pool.py: the
 * fp8 write saturates to +-448 before the e4m3 cast). Everything here is
 * binary32 arithmetic, as the write path computes it, so a code decided by
 * rounding is decided the same way on both sides.
 */

/* e4m3fn encoding of a binary32 value: round to nearest, ties to even, values
 * of magnitude >= 448 (and infinities) saturate to +-448; NaN -> 0x7F. */
uint8_t orc_e4m3fn_encode(float v) {
    if (isnan(v)) return 0x7F;
    const uint8_t sign = signbit(v) ? 0x80 : 0x00;
    const double a = fabs((double)v);
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        /* subnormals m * 2^-9, m = 0..7; m = 8 is the smallest normal 0x08 */
        const double m = nearbyint(a / ldexp(1.0, -9));
        return sign | (uint8_t)m;
    }
    int e2;
    frexp(a, &e2);
    int E = e2 - 1; /* a in [2^E, 2^(E+1)) */
    double m = nearbyint((a / ldexp(1.0, E) - 1.0) * 8.0);
    if (m == 8.0) {
        m = 0.0;
        E += 1;
    }
    return sign | (uint8_t)(((E + 7) << 3) | (int)m);
}

/* Quantise n rows of D bf16 values:
 *   bf16 (0): codes are the input bits (2 bytes per value)
 *   fp8  (1): codes[d] = e4m3fn(x[d] / s), s = fp8_scale (one per pool)
 *   int8 (2): s = absmax / 127, codes[d] = clamp(rint(x[d] / s), -127, 127)
 *   int4 (3): s = absmax / 7,   codes[d] = clamp(rint(x[d] / s), -8, 7), two per
 *             byte, channel 2i in the low nibble
 *   int8_g64 (4), int4_g32 (5): per group of 64 / 32 channels, the binary32
 *             absmax / 127 (/ 7) clamped to 65504 and rounded to binary16 is
 *             the group's scale s16; codes[d] = clamp(rint(x[d] / s16), -q, q)
 *             with q = 127 (7); int4_g32 stores nibbles q + 8 (offset binary),
 *             channel 2i in the low nibble. The codes divide by the stored
 *             binary16 scale, the one the reader multiplies by.
 * An all-zero row or group (or a scale that rounds to 0) gets s = 0 and zero
 * codes (offset-binary 8 for int4_g32). rint is round-half-to-even. codes: n * D
 * bytes (2n * D for bf16, n * D / 2 for the 4-bit formats); scales: n floats
 * (int8 / int4) or n * D / group binary16 bits (grouped). Returns 0, or -1 for a
 * bad format or a D the format cannot hold. */
static void put_code(uint8_t* codes, int64_t r, int D, int format, int d, int q) {
    if (format == ORC_INT8 || format == ORC_INT8_G64) {
        codes[r * D + d] = (uint8_t)(int8_t)q;
        return;
    }
    const int u = format == ORC_INT4_G32 ? q + 8 : q & 0xF;
    uint8_t* byte = codes + r * (D / 2) + d / 2;
    if ((d & 1) == 0)
        *byte = (uint8_t)u;
    else
        *byte |= (uint8_t)(u << 4);
}

int orc_quantize_rows(const uint16_t* x, int64_t n, int D, int format, float fp8_scale,
                      uint8_t* codes, void* scales) {
    if (format < ORC_BF16 || format > ORC_INT4_G32 || D <= 0 ||
        (is_nibble_format(format) && (D & 1)) ||
        (group_size(format) && D % group_size(format)))
        return -1;
    for (int64_t r = 0; r < n; ++r) {
        const uint16_t* xr = x + r * D;
        if (format == ORC_BF16) {
            memcpy(codes + r * D * 2, xr, (size_t)D * 2);
            continue;
        }
        if (format == ORC_FP8_E4M3) {
            for (int d = 0; d < D; ++d) {
                const float xf = (float)orc_bf16_to_double(xr[d]);
                const float y = xf / fp8_scale;
                codes[r * D + d] = orc_e4m3fn_encode(y);
            }
            continue;
        }
        const int grouped = group_size(format) != 0;
        const int gs = grouped ? group_size(format) : D;
        const float qmax = (format == ORC_INT8 || format == ORC_INT8_G64) ? 127.0f : 7.0f;
        const float qmin = format == ORC_INT4 ? -8.0f : -qmax;
        for (int k = 0; k < D / gs; ++k) {
            float amax = 0.0f;
            for (int d = k * gs; d < (k + 1) * gs; ++d) {
                const float a = fabsf((float)orc_bf16_to_double(xr[d]));
                if (a > amax) amax = a;
            }
            float s = amax / qmax;
            if (grouped) {
                if (s > 65504.0f) s = 65504.0f;
                const uint16_t s16 = orc_round_fp16(s);
                ((uint16_t*)scales)[r * (D / gs) + k] = s16;
                s = (float)orc_fp16_to_double(s16);
            } else {
                ((float*)scales)[r] = s;
            }
            for (int d = k * gs; d < (k + 1) * gs; ++d) {
                int q = 0;
                if (s > 0.0f) {
                    const float y = (float)orc_bf16_to_double(xr[d]) / s;
                    float qf = rintf(y);
                    if (qf > qmax) qf = qmax;
                    if (qf < qmin) qf = qmin;
                    q = (int)qf;
                }
                put_code(codes, r, D, format, d, q);
            }
        }
    }
    return 0;
}

/* Threads the OpenMP runtime would use (1 without OpenMP). */
int orc_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
