// Fused quantise + scatter write of new K/V rows into the paged pools.
//
// What it computes (sglang PR #37798 "quantized KV pools with
// dequant-on-gather", "Modifications": writing is one fused quantise + scatter
// launch; part 1, "mem_cache/memory_pool.py": the fp8 write saturates to +-448
// before the e4m3 cast, whose result would otherwise be NaN). For every new
// token i and KV head g the 256 bf16 values x go to pool row slot[i] * Hkv + g:
//   bf16 : stored as they are
//   fp8  : e4m3fn(x / s), s the pool's fp32 scale, nearest-even, saturating
//   int8 : s = absmax(x) / 127 -> scale[row]; codes clamp(rint(x / s), -127, 127)
//   int4 : s = absmax(x) / 7   -> scale[row]; codes clamp(rint(x / s), -8, 7),
//          two per byte, channel 2i in the low nibble
//   int8_g64 / int4_g32 (the int8 and int4 KV pool modules of the same PR):
//          per 64 / 32-channel group s16 = binary16(min(absmax / q, 65504)),
//          q = 127 / 7, -> scale[row][group]; codes clamp(rint(x / s16), -q, q);
//          int4_g32 stores offset-binary nibbles code + 8
//   int8ring_int4 (the tiered KV pool module): the int4_g32 row of the slot, and
//          the int8_g64 row of ring position slot & (R - 1) with owner = slot when
//          the token owns that position (the last token of the write that maps
//          there, claimed by a first kernel)
// all in binary32 with IEEE division; an all-zero row gets s = 0 and zero codes.
//
// One warp per (token, head, K-or-V) row: a 16-byte load per lane covers the
// row, the absmax is a warp reduction, and each lane stores its codes with one
// 16/8/4-byte store, so a row is one coalesced read and one coalesced write.
// Each warp issues the loads of its RPW rows before converting any of them.

#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <initializer_list>

#include "qsa.h"

void qsa_detail_set_error(const char* msg);

namespace qsakv {

constexpr int D = 256;
constexpr int WARPS = 8; // warps per CTA
constexpr int RPW = 4;   // rows per warp

struct Params {
    const __nv_bfloat16* kx;
    const __nv_bfloat16* vx;
    long long k_st, k_sh, v_st, v_sh;
    const int* slots;
    int n, Hkv;
    uint8_t* kpool;
    uint8_t* vpool;
    long long num_slots;
    void* kscale; // fp32 (fp8: [1]; int8/int4: [slots * Hkv]) or binary16 [slots * Hkv * groups]
    void* vscale;
    int* err;
    // tiered: int8_g64 ring rows [R, Hkv, 256], binary16 scales [R, Hkv, 4], owner [R]
    uint8_t* kring;
    uint8_t* vring;
    __half* kring_scale;
    __half* vring_scale;
    int* owner;
    int ring_mask;
};

// Two binary32 values -> two e4m3fn codes (lo in the low byte), nearest-even,
// saturating to the largest finite magnitude.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Codes are defined on q = fl(x / s), the correctly rounded binary32 quotient.
//
// fp8 (s is any pool scale): with r = fl(1 / s), r_lo = fl(r * (1 - 2^-20)) and
// r_hi = fl(r * (1 + 2^-20)), fl(x * r_lo) and fl(x * r_hi) lie on either side
// of q (each is at least |x / s| * 2^-21 away from x / s, q at most
// |x / s| * 2^-24). The conversion is monotone, so where both give the same code
// that is the code of q; pairs where they differ divide.
//
// int8 / int4 (s = fl(a / qmax), a = absmax, a bf16 value; the grouped formats
// round s to binary16 first, s16 = fl16(fl(a / qmax))): q comes from
// Markstein's correction (P. Markstein, "Computation of elementary functions on
// the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990):
// q0 = fl(x * r), e = fma(-q0, s, x), q = fma(e, r, q0) with r = fl(1 / s). For
// a in [1, 2) it was checked against exact rational arithmetic for every bf16
// x with 2^-11 a <= |x| <= a and every a (smaller |x| gives code 0 either way);
// the steps commute with scaling by 2^E while all terms stay normal, which holds
// for a >= 2^-60. s and r for a = m * 2^E are those of m (a 128-entry table of
// the bf16 mantissas) with the exponent moved by E. The same check holds for the
// binary16 scales s16 of every mantissa, which scale the same way while
// fl(a / qmax) is a normal binary16 value (2^-14 .. 65504).

// x + 1.5 * 2^23 rounds once, to an integer (the spacing of binary32 in
// [2^23, 2^24)), ties to even: its bit pattern is 0x4B400000 + rint(x) for
// |x| < 2^22, so the low byte is the two's complement byte of rint(x).
constexpr float RINT_MAGIC = 12582912.0f;
constexpr float FAST_MIN_ABSMAX = 0x1p-60f;

__device__ __forceinline__ uint32_t rint_bits(float q) { return __float_as_uint(__fadd_rn(q, RINT_MAGIC)); }

// Low bytes of four words packed into one (a in the lowest byte).
__device__ __forceinline__ uint32_t low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

// Low nibbles of the four bytes of w, in order, as 16 bits.
__device__ __forceinline__ uint32_t low_nibbles(uint32_t w) {
    const uint32_t t = (w & 0x0F0F0F0Fu) | ((w >> 4) & 0xF0F0F0F0u); // bytes 0 and 2 hold pairs
    return __byte_perm(t, 0u, 0x4420);
}

__device__ __forceinline__ void unpack(const uint4 raw, float x[8]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        x[2 * k] = __uint_as_float(w[k] << 16);
        x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint8_t* row_ptr(const Params& p, bool isv, long long row, int row_bytes) {
    return (isv ? p.vpool : p.kpool) + row * row_bytes;
}

// POW2: the scale is a power of two, so x * (1 / s) is the exact quotient and
// its code needs no bracket (fr_lo = fr_hi = 1 / s).
template <bool POW2>
__device__ __forceinline__ void store_fp8(const Params& p, const uint4 raw, long long row, bool isv,
                                          int lane, float fr_lo, float fr_hi) {
    float x[8];
    unpack(raw, x);
    uint32_t c[4];
    if constexpr (POW2) {
#pragma unroll
        for (int k = 0; k < 4; ++k) c[k] = e4m3x2(x[2 * k] * fr_lo, x[2 * k + 1] * fr_lo);
    } else {
        uint32_t d[4];
        bool same = true;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            c[k] = e4m3x2(x[2 * k] * fr_lo, x[2 * k + 1] * fr_lo);
            d[k] = e4m3x2(x[2 * k] * fr_hi, x[2 * k + 1] * fr_hi);
            same &= c[k] == d[k];
        }
        if (!same) {
            const float s = __ldg(static_cast<const float*>(isv ? p.vscale : p.kscale));
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (c[k] != d[k]) c[k] = e4m3x2(x[2 * k] / s, x[2 * k + 1] / s);
        }
    }
    reinterpret_cast<uint2*>(row_ptr(p, isv, row, D))[lane] =
        make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

template <int FMT> __device__ __forceinline__ void codes_divide(const float x[8], float s, uint32_t z[8]);
template <int FMT>
__device__ __forceinline__ void codes_markstein(const float x[8], float s, float r, uint32_t z[8]);

// One lane's 8 values of a grouped row (GFMT int8_g64 or int4_g32): the group's
// absmax over its lanes, the binary16 scale, the codes; the group leaders store
// the scales (one 8- / 16-byte block per row). tab: (s, s16) pairs per mantissa
// then fl(1 / s16) per mantissa.
template <int GFMT>
__device__ __forceinline__ void store_grouped(const float x[8], const uint32_t* tab, uint8_t* codes,
                                              __half* scales, int lane) {
    constexpr int GS = GFMT == QSA_KV_INT8_G64 ? 64 : 32; // channels per scale
    constexpr int LPG = GS / 8;                            // lanes per group
    constexpr float qmax = GFMT == QSA_KV_INT8_G64 ? 127.0f : 7.0f;
    float a = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) a = fmaxf(a, fabsf(x[k]));
#pragma unroll
    for (int off = 1; off < LPG; off <<= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, off));
    // a = (1 + t / 128) * 2^E: fl(a / qmax) from the table, exponent moved by E
    const uint32_t ab = __float_as_uint(a);
    const int t = (ab >> 16) & 0x7F;
    const uint32_t e = (ab & 0x7F800000u) - (127u << 23);
    const float s32 = __uint_as_float(tab[2 * t] + e);
    uint32_t z[8];
    float sc;
    if (a >= FAST_MIN_ABSMAX && s32 >= 0x1p-14f && s32 <= 65504.0f) { // uniform per group
        sc = __uint_as_float(tab[2 * t + 1] + e);
        codes_markstein<GFMT>(x, sc, __uint_as_float(tab[256 + t] - e), z);
    } else {
        sc = __half2float(__float2half_rn(fminf(__fdiv_rn(a, qmax), 65504.0f)));
        codes_divide<GFMT>(x, sc, z);
    }
    const uint32_t b0 = low_bytes(z[0], z[1], z[2], z[3]);
    const uint32_t b1 = low_bytes(z[4], z[5], z[6], z[7]);
    if constexpr (GFMT == QSA_KV_INT8_G64)
        reinterpret_cast<uint2*>(codes)[lane] = make_uint2(b0, b1);
    else // offset binary: code + 8 is code ^ 8 on a two's-complement nibble
        reinterpret_cast<uint32_t*>(codes)[lane] = (low_nibbles(b0) | (low_nibbles(b1) << 16)) ^ 0x88888888u;
    if (lane % LPG == 0) scales[lane / LPG] = __float2half_rn(sc);
}

// Codes of one lane's 8 values, as low bytes of z (int8: -127..127, int4: -8..7).
template <int FMT>
__device__ __forceinline__ void codes_markstein(const float x[8], float s, float r, uint32_t z[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float q0 = __fmul_rn(x[k], r);
        const float e = __fmaf_rn(-q0, s, x[k]);
        z[k] = rint_bits(__fmaf_rn(e, r, q0));
    }
}

// The definition as it stands, for absmax below 2^-60 (subnormal or zero scales).
template <int FMT>
__device__ __forceinline__ void codes_divide(const float x[8], float s, uint32_t z[8]) {
    constexpr float qmax = (FMT == QSA_KV_INT8 || FMT == QSA_KV_INT8_G64) ? 127.0f : 7.0f;
    constexpr float qmin = FMT == QSA_KV_INT4 ? -8.0f : -qmax;
#pragma unroll
    for (int k = 0; k < 8; ++k)
        z[k] = static_cast<uint32_t>(s > 0.0f ? static_cast<int>(fminf(fmaxf(rintf(x[k] / s), qmin), qmax)) : 0);
}

template <int FMT>
__device__ __forceinline__ void store_codes(const Params& p, long long row, bool isv, int lane, float s,
                                            const uint32_t z[8]) {
    const uint32_t b0 = low_bytes(z[0], z[1], z[2], z[3]);
    const uint32_t b1 = low_bytes(z[4], z[5], z[6], z[7]);
    if constexpr (FMT == QSA_KV_INT8)
        reinterpret_cast<uint2*>(row_ptr(p, isv, row, D))[lane] = make_uint2(b0, b1);
    else
        reinterpret_cast<uint32_t*>(row_ptr(p, isv, row, D / 2))[lane] = low_nibbles(b0) | (low_nibbles(b1) << 16);
    if (lane == 0) static_cast<float*>(isv ? p.vscale : p.kscale)[row] = s;
}

// One row's conversion and store; rows are resolved from the task index
// t in [0, 2 n Hkv): K rows first, token-major, then V rows.
template <int FMT> struct Converter {
    float k_lo, k_hi, v_lo, v_hi;     // fp8: 1 / pool scale times 1 -+ 2^-20 (or 1)
    const uint32_t* s_tab;            // int8/int4: s and 1 / s for a = 1 + t / 128;
    const uint32_t* r_tab;            // grouped: the store_grouped table (s_tab), tiered: the
                                      // int4_g32 one (s_tab) and the int8_g64 one (r_tab)

    // row = slot * Hkv + g of token `tok`
    __device__ __forceinline__ void operator()(const Params& p, const uint4 raw, long long row, bool isv,
                                               int lane, int tok, int slot) const {
        if constexpr (FMT == QSA_KV_BF16) {
            reinterpret_cast<uint4*>(row_ptr(p, isv, row, 2 * D))[lane] = raw;
        } else if constexpr (FMT == QSA_KV_FP8_E4M3) {
            const float lo = isv ? v_lo : k_lo, hi = isv ? v_hi : k_hi;
            if (lo == hi) // uniform across the grid
                store_fp8<true>(p, raw, row, isv, lane, lo, hi);
            else
                store_fp8<false>(p, raw, row, isv, lane, lo, hi);
        } else if constexpr (FMT == QSA_KV_INT8_G64 || FMT == QSA_KV_INT4_G32) {
            constexpr int G = FMT == QSA_KV_INT8_G64 ? 4 : 8; // scales per row
            float x[8];
            unpack(raw, x);
            store_grouped<FMT>(x, s_tab, row_ptr(p, isv, row, FMT == QSA_KV_INT8_G64 ? D : D / 2),
                               static_cast<__half*>(isv ? p.vscale : p.kscale) + row * G, lane);
        } else if constexpr (FMT == QSA_KV_INT8RING_INT4) {
            float x[8];
            unpack(raw, x);
            store_grouped<QSA_KV_INT4_G32>(x, s_tab, row_ptr(p, isv, row, D / 2),
                                           static_cast<__half*>(isv ? p.vscale : p.kscale) + row * 8, lane);
            // the ring row: only the token that owns the position (its claim mark, or
            // its slot once one of its rows has stamped it) writes it; with distinct
            // slots no other token can match either value
            const int pos = slot & p.ring_mask;
            const int own = *reinterpret_cast<volatile const int*>(p.owner + pos);
            if (own == -2 - tok || own == slot) {
                const long long rrow = (long long)pos * p.Hkv + (row - (long long)slot * p.Hkv);
                store_grouped<QSA_KV_INT8_G64>(x, r_tab, (isv ? p.vring : p.kring) + rrow * D,
                                               (isv ? p.vring_scale : p.kring_scale) + rrow * 4, lane);
                __syncwarp();
                if (lane == 0) p.owner[pos] = slot;
            }
        } else {
            constexpr float qmax = FMT == QSA_KV_INT8 ? 127.0f : 7.0f;
            float x[8];
            unpack(raw, x);
            float m = 0.0f;
#pragma unroll
            for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(x[k]));
            // m >= 0, so its bit pattern orders like its value
            const float a = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(m)));
            uint32_t z[8];
            float sc;
            if (a >= FAST_MIN_ABSMAX) { // uniform across the warp
                // a = (1 + t / 128) * 2^E exactly: move the table entries' exponents by E
                const uint32_t ab = __float_as_uint(a);
                const int t = (ab >> 16) & 0x7F;
                const uint32_t e = (ab & 0x7F800000u) - (127u << 23);
                sc = __uint_as_float(s_tab[t] + e);
                codes_markstein<FMT>(x, sc, __uint_as_float(r_tab[t] - e), z);
            } else {
                sc = __fdiv_rn(a, qmax);
                codes_divide<FMT>(x, sc, z);
            }
            store_codes<FMT>(p, row, isv, lane, sc, z);
        }
    }
};

// Task t -> source row and destination pool row; false for t past the end or a
// slot outside the pool (then *bad).
__device__ __forceinline__ bool resolve(const Params& p, int rows, int t, const __nv_bfloat16** src,
                                        long long* dst, bool* isv, bool* bad, int* tok, int* slot_out) {
    *bad = false;
    if (t >= 2 * rows) return false;
    *isv = t >= rows;
    const int r = *isv ? t - rows : t;
    const int i = p.Hkv == 2 ? r >> 1 : r, g = p.Hkv == 2 ? r & 1 : 0;
    const int slot = __ldg(p.slots + i);
    *tok = i;
    *slot_out = slot;
    if (slot < 0 || (long long)slot >= p.num_slots) {
        *bad = true;
        return false;
    }
    *src = *isv ? p.vx + i * p.v_st + g * p.v_sh : p.kx + i * p.k_st + g * p.k_sh;
    *dst = (long long)slot * p.Hkv + g;
    return true;
}

// Bracket factors for an fp8 pool scale s: both 1 / s when s is a power of two
// (then x / s = x * (1 / s) exactly), else 1 / s times 1 -+ 2^-20.
__device__ __forceinline__ void fp8_factors(float s, float* lo, float* hi) {
    const float r = __frcp_rn(s);
    const bool pow2 = (__float_as_uint(s) & 0x007FFFFFu) == 0 && s > 0x1p-126f && s < 0x1p126f;
    *lo = pow2 ? r : r * (1.0f - 0x1p-20f);
    *hi = pow2 ? r : r * (1.0f + 0x1p-20f);
}

// The grouped-format table of store_grouped for one qmax: per bf16 mantissa t,
// (fl((1 + t / 128) / qmax), its binary16 rounding) pairs, then fl(1 / s16).
__device__ __forceinline__ void fill_grouped_table(uint32_t* tab, float qmax) {
    if (threadIdx.x < 128) {
        const float s0 = __fdiv_rn(1.0f + threadIdx.x * 0x1p-7f, qmax);
        const float s16 = __half2float(__float2half_rn(s0));
        tab[2 * threadIdx.x] = __float_as_uint(s0);
        tab[2 * threadIdx.x + 1] = __float_as_uint(s16);
        tab[256 + threadIdx.x] = __float_as_uint(__frcp_rn(s16));
    }
}

// Programmatic dependent launch: wait until the grids this launch depends on
// have completed and their memory is visible (a no-op for an ordinary launch);
// let the next dependent launch be scheduled.
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <int FMT>
__global__ void __launch_bounds__(WARPS * 32, 5) kv_write_kernel(const Params p) {
    constexpr bool GROUPED = FMT == QSA_KV_INT8_G64 || FMT == QSA_KV_INT4_G32;
    constexpr bool TIERED = FMT == QSA_KV_INT8RING_INT4;
    constexpr bool INTQ = FMT == QSA_KV_INT8 || FMT == QSA_KV_INT4;
    constexpr float qmax = (FMT == QSA_KV_INT8 || FMT == QSA_KV_INT8_G64) ? 127.0f : 7.0f;
    // int8/int4: per bf16 mantissa t, s = fl((1 + t / 128) / qmax) and fl(1 / s);
    // grouped: one store_grouped table; tiered: the int4_g32 and int8_g64 tables
    constexpr int TAB = INTQ ? 128 : (GROUPED || TIERED) ? 384 : 1;
    __shared__ uint32_t s_tab[TAB], r_tab[INTQ ? 128 : TIERED ? 384 : 1];
    Converter<FMT> conv{0.0f, 0.0f, 0.0f, 0.0f, s_tab, r_tab};
    if constexpr (INTQ) {
        if (threadIdx.x < 128) {
            const float s0 = __fdiv_rn(1.0f + threadIdx.x * 0x1p-7f, qmax);
            s_tab[threadIdx.x] = __float_as_uint(s0);
            r_tab[threadIdx.x] = __float_as_uint(__frcp_rn(s0));
        }
        __syncthreads();
    } else if constexpr (GROUPED) {
        fill_grouped_table(s_tab, qmax);
        __syncthreads();
    } else if constexpr (TIERED) {
        fill_grouped_table(s_tab, 7.0f);
        fill_grouped_table(r_tab, 127.0f);
        __syncthreads();
    }
    // the tables above are shared memory only; global memory from here on
    griddep_wait();
    griddep_launch_dependents();
    if constexpr (FMT == QSA_KV_FP8_E4M3) {
        fp8_factors(__ldg(static_cast<const float*>(p.kscale)), &conv.k_lo, &conv.k_hi);
        fp8_factors(__ldg(static_cast<const float*>(p.vscale)), &conv.v_lo, &conv.v_hi);
    }
    const int lane = threadIdx.x & 31;
    const int rows = p.n * p.Hkv; // n <= 2^28 and Hkv <= 2: every task index fits in 32 bits
    const int first = (blockIdx.x * WARPS + (threadIdx.x >> 5)) * RPW;
    uint4 raw[RPW];
    long long dst[RPW];
    bool isv[RPW];
    int tok[RPW], slot[RPW];
#pragma unroll
    for (int u = 0; u < RPW; ++u) {
        const __nv_bfloat16* src;
        bool bad;
        dst[u] = -1;
        raw[u] = make_uint4(0u, 0u, 0u, 0u);
        if (resolve(p, rows, first + u, &src, &dst[u], &isv[u], &bad, &tok[u], &slot[u]))
            raw[u] = __ldg(reinterpret_cast<const uint4*>(src) + lane); // dims 8 lane .. 8 lane + 7
        else if (bad && lane == 0 && p.err)
            atomicOr(p.err, QSA_DEVERR_SLOT_RANGE);
    }
#pragma unroll
    for (int u = 0; u < RPW; ++u)
        if (dst[u] >= 0) conv(p, raw[u], dst[u], isv[u], lane, tok[u], slot[u]);
}

// Tiered write, first kernel: every token marks its ring position with -2 - i;
// the minimum, i.e. the last token of the write mapping there, remains.
__global__ void ring_claim_kernel(const int* slots, int n, long long num_slots, int* owner, int mask) {
    griddep_wait();
    griddep_launch_dependents();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const int slot = __ldg(slots + i);
        if (slot < 0 || (long long)slot >= num_slots) continue;
        atomicMin(owner + (slot & mask), -2 - i);
    }
}

namespace {

int fail(int code, const char* fmt, ...) {
    char msg[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(msg, sizeof msg, fmt, ap);
    va_end(ap);
    qsa_detail_set_error(msg);
    return code;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// Launch with programmatic stream serialization: the kernels wait for the
// previous grid themselves (griddepcontrol.wait) before touching global memory.
template <typename... Args>
cudaError_t launch_pdl(void (*kernel)(Args...), unsigned grid, unsigned block, cudaStream_t st,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

template <int FMT> int launch(const Params& prm, cudaStream_t st) {
    const long long tasks = 2LL * prm.n * prm.Hkv;
    const long long blocks = (tasks + WARPS * RPW - 1) / (WARPS * RPW);
    const cudaError_t e = launch_pdl(kv_write_kernel<FMT>, static_cast<unsigned>(blocks), WARPS * 32, st, prm);
    if (e != cudaSuccess) return fail(QSA_ERR_CUDA, "kv write launch: %s", cudaGetErrorString(e));
    return QSA_OK;
}

} // namespace
} // namespace qsakv

namespace qsakv {
namespace {

// Validate a write of `format` rows and fill the parameters (nothing enqueued).
int prepare(int32_t format, const qsa_tensor* k_new, const qsa_tensor* v_new, const qsa_tensor* slots,
            const qsa_tensor* k_pool, const qsa_tensor* v_pool, void* k_scale, void* v_scale,
            int32_t* device_error, Params* prm) {
    if (!k_new || !v_new || !slots || !k_pool || !v_pool)
        return fail(QSA_ERR_INVALID_ARGUMENT, "a descriptor pointer is NULL");
    if (format < QSA_KV_BF16 || format > QSA_KV_INT4_G32)
        return fail(QSA_ERR_UNSUPPORTED, "unknown K/V pool format %d", format);
    if (k_new->ndim != 3 || v_new->ndim != 3)
        return fail(QSA_ERR_INVALID_ARGUMENT, "k_new and v_new must be [n, Hkv, 256]");
    const long long n = k_new->shape[0], hkv = k_new->shape[1];
    if (hkv != 1 && hkv != 2)
        return fail(QSA_ERR_UNSUPPORTED, "%lld KV heads: the decode contract has 1 or 2", hkv);
    for (const qsa_tensor* t : {k_new, v_new}) {
        const char* nm = t == k_new ? "k_new" : "v_new";
        if (t->dtype != QSA_DTYPE_BF16)
            return fail(QSA_ERR_INVALID_ARGUMENT, "%s must be bf16", nm);
        if (t->shape[0] != n || t->shape[1] != hkv || t->shape[2] != D)
            return fail(QSA_ERR_INVALID_ARGUMENT, "%s must be [n=%lld, Hkv=%lld, 256]", nm, n, hkv);
        if (t->stride[2] != 1 || t->stride[0] % 8 || t->stride[1] % 8 || t->stride[0] < 0 ||
            t->stride[1] < 0)
            return fail(QSA_ERR_MISALIGNED,
                        "%s must be contiguous along the head dimension with strides that are "
                        "non-negative multiples of 8", nm);
        if (n > 0 && (t->data == nullptr || !aligned16(t->data)))
            return fail(QSA_ERR_MISALIGNED, "%s must be a non-NULL 16-byte aligned pointer", nm);
    }
    if (slots->dtype != QSA_DTYPE_INT32 || slots->ndim != 1 || slots->shape[0] != n ||
        (n > 1 && slots->stride[0] != 1) || (n > 0 && slots->data == nullptr))
        return fail(QSA_ERR_INVALID_ARGUMENT, "slots must be a contiguous int32 [n]");
    const int want_dtype = format == QSA_KV_BF16                                    ? QSA_DTYPE_BF16
                           : (format == QSA_KV_INT8 || format == QSA_KV_INT8_G64) ? QSA_DTYPE_INT8
                                                                                  : QSA_DTYPE_UINT8;
    const long long row_elems = (format == QSA_KV_INT4 || format == QSA_KV_INT4_G32) ? D / 2 : D;
    for (const qsa_tensor* pool : {k_pool, v_pool}) {
        const char* nm = pool == k_pool ? "k_pool" : "v_pool";
        if (pool->dtype != want_dtype)
            return fail(QSA_ERR_INVALID_ARGUMENT, "%s dtype %d does not match pool format %d", nm,
                        pool->dtype, format);
        if (pool->ndim != 3 || pool->shape[1] != hkv || pool->shape[2] != row_elems ||
            pool->shape[0] < 1 || pool->stride[2] != 1 || pool->stride[1] != row_elems ||
            pool->stride[0] != hkv * row_elems)
            return fail(QSA_ERR_INVALID_ARGUMENT, "%s must be a contiguous [num_slots, Hkv=%lld, %lld]",
                        nm, hkv, row_elems);
        if (pool->data == nullptr || !aligned16(pool->data))
            return fail(QSA_ERR_MISALIGNED, "%s must be a non-NULL 16-byte aligned pointer", nm);
    }
    if (k_pool->shape[0] != v_pool->shape[0])
        return fail(QSA_ERR_INVALID_ARGUMENT, "k_pool and v_pool hold different slot counts");
    if (format != QSA_KV_BF16) {
        if (k_scale == nullptr || v_scale == nullptr)
            return fail(QSA_ERR_INVALID_ARGUMENT, "quantised pools need k_scale and v_scale");
        // the alignment qsa_decode reads these scales with
        const uintptr_t al = format == QSA_KV_INT8_G64 ? 8 : format == QSA_KV_INT4_G32 ? 16 : 4;
        if ((reinterpret_cast<uintptr_t>(k_scale) & (al - 1)) ||
            (reinterpret_cast<uintptr_t>(v_scale) & (al - 1)))
            return fail(QSA_ERR_MISALIGNED, "scales must be %d-byte aligned for this format", (int)al);
    }
    if (n > (1LL << 28)) return fail(QSA_ERR_UNSUPPORTED, "more than 2^28 new tokens in one call");
    prm->kx = static_cast<const __nv_bfloat16*>(k_new->data);
    prm->vx = static_cast<const __nv_bfloat16*>(v_new->data);
    prm->k_st = k_new->stride[0];
    prm->k_sh = k_new->stride[1];
    prm->v_st = v_new->stride[0];
    prm->v_sh = v_new->stride[1];
    prm->slots = static_cast<const int*>(slots->data);
    prm->n = static_cast<int>(n);
    prm->Hkv = static_cast<int>(hkv);
    prm->kpool = static_cast<uint8_t*>(k_pool->data);
    prm->vpool = static_cast<uint8_t*>(v_pool->data);
    prm->num_slots = k_pool->shape[0];
    prm->kscale = k_scale;
    prm->vscale = v_scale;
    prm->err = device_error;
    prm->kring = prm->vring = nullptr;
    prm->kring_scale = prm->vring_scale = nullptr;
    prm->owner = nullptr;
    prm->ring_mask = 0;
    return QSA_OK;
}

} // namespace
} // namespace qsakv

extern "C" int qsa_kv_write(int32_t format, const qsa_tensor* k_new, const qsa_tensor* v_new,
                            const qsa_tensor* slots, const qsa_tensor* k_pool,
                            const qsa_tensor* v_pool, void* k_scale, void* v_scale,
                            int32_t* device_error, void* stream) {
    using namespace qsakv;
    Params prm;
    const int rc = prepare(format, k_new, v_new, slots, k_pool, v_pool, k_scale, v_scale,
                           device_error, &prm);
    if (rc != QSA_OK) return rc;
    qsa_detail_set_error("");
    if (prm.n == 0) return QSA_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (format) {
    case QSA_KV_BF16: return launch<QSA_KV_BF16>(prm, st);
    case QSA_KV_FP8_E4M3: return launch<QSA_KV_FP8_E4M3>(prm, st);
    case QSA_KV_INT8: return launch<QSA_KV_INT8>(prm, st);
    case QSA_KV_INT4: return launch<QSA_KV_INT4>(prm, st);
    case QSA_KV_INT8_G64: return launch<QSA_KV_INT8_G64>(prm, st);
    default: return launch<QSA_KV_INT4_G32>(prm, st);
    }
}

extern "C" int qsa_kv_write_tiered(const qsa_tensor* k_new, const qsa_tensor* v_new,
                                   const qsa_tensor* slots, const qsa_tensor* k_pool,
                                   const qsa_tensor* v_pool, void* k_scale, void* v_scale,
                                   const qsa_kv_tier* tier, int32_t* device_error, void* stream) {
    using namespace qsakv;
    Params prm;
    const int rc = prepare(QSA_KV_INT4_G32, k_new, v_new, slots, k_pool, v_pool, k_scale, v_scale,
                           device_error, &prm);
    if (rc != QSA_OK) return rc;
    if (tier == nullptr) return fail(QSA_ERR_INVALID_ARGUMENT, "tier is NULL");
    const int R = tier->ring_slots;
    if (R < 1 || R > (1 << 30) || (R & (R - 1)))
        return fail(QSA_ERR_INVALID_ARGUMENT, "ring_slots %d is not a power of two in 1..2^30", R);
    if (!tier->k_ring || !tier->v_ring || !tier->k_ring_scale || !tier->v_ring_scale || !tier->owner)
        return fail(QSA_ERR_INVALID_ARGUMENT, "a tier pointer is NULL");
    if (!aligned16(tier->k_ring) || !aligned16(tier->v_ring) ||
        (reinterpret_cast<uintptr_t>(tier->k_ring_scale) & 7u) ||
        (reinterpret_cast<uintptr_t>(tier->v_ring_scale) & 7u) ||
        (reinterpret_cast<uintptr_t>(tier->owner) & 3u))
        return fail(QSA_ERR_MISALIGNED,
                    "ring rows must be 16-byte, ring scales 8-byte and owner 4-byte aligned");
    prm.kring = static_cast<uint8_t*>(tier->k_ring);
    prm.vring = static_cast<uint8_t*>(tier->v_ring);
    prm.kring_scale = static_cast<__half*>(tier->k_ring_scale);
    prm.vring_scale = static_cast<__half*>(tier->v_ring_scale);
    prm.owner = tier->owner;
    prm.ring_mask = R - 1;
    qsa_detail_set_error("");
    if (prm.n == 0) return QSA_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int threads = 256;
    const long long want = (prm.n + threads - 1) / threads;
    const cudaError_t e = launch_pdl(ring_claim_kernel, static_cast<unsigned>(want < 4096 ? want : 4096),
                                     threads, st, prm.slots, prm.n, prm.num_slots, prm.owner,
                                     prm.ring_mask);
    if (e != cudaSuccess) return fail(QSA_ERR_CUDA, "ring claim launch: %s", cudaGetErrorString(e));
    return launch<QSA_KV_INT8RING_INT4>(prm, st);
}
