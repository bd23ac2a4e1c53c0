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
// all in binary32 with IEEE division; an all-zero row gets s = 0 and zero codes.
//
// One warp per (token, head, K-or-V) row: a 16-byte load per lane covers the
// row, the absmax is a warp reduction, and each lane stores its codes with one
// 16/8/4-byte store, so a row is one coalesced read and one coalesced write.

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
    float* kscale;
    float* vscale;
    int* err;
};

// Two binary32 values -> two e4m3fn codes (lo in the low byte), nearest-even,
// saturating to the largest finite magnitude.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Codes are defined on fl(x / s), the correctly rounded binary32 quotient. With
// r = fl(1 / s), r_lo = fl(r * (1 - 2^-20)) and r_hi = fl(r * (1 + 2^-20)), the
// exact products x * r_lo and x * r_hi lie on either side of fl(x / s) (their
// distance from x / s is at least |x / s| * 2^-21, the rounding of fl(x / s)
// and r at most |x / s| * 2^-23). Rounding is monotone, so where the codes of
// both products agree that is the code of fl(x / s); only the rare lane where
// they differ divides.

// fma(x, c, 1.5 * 2^23) rounds x * c + 1.5 * 2^23 once, to an integer (the
// spacing of binary32 in [2^23, 2^24)), ties to even: its bit pattern is
// 0x4B400000 + rint(x * c) for |x * c| < 2^22, so the low byte is the two's
// complement byte of rint(x * c).
constexpr float RINT_MAGIC = 12582912.0f;

__device__ __forceinline__ uint32_t rint_bits(float x, float c) {
    return __float_as_uint(__fmaf_rn(x, c, RINT_MAGIC));
}

// Low bytes of four words packed into one (a in the lowest byte).
__device__ __forceinline__ uint32_t low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

// Low nibbles of the four bytes of w, in order, as 16 bits.
__device__ __forceinline__ uint32_t low_nibbles(uint32_t w) {
    const uint32_t t = (w & 0x0F0F0F0Fu) | ((w >> 4) & 0xF0F0F0F0u); // bytes 0 and 2 hold pairs
    return __byte_perm(t, 0u, 0x4420);
}

template <int FMT>
__device__ __forceinline__ void write_row(const Params& p, const uint4 raw, long long row, bool isv,
                                          int lane, float fr_lo, float fr_hi) {
    uint8_t* const pool = isv ? p.vpool : p.kpool;
    if constexpr (FMT == QSA_KV_BF16) {
        reinterpret_cast<uint4*>(pool + row * (D * 2))[lane] = raw;
    } else {
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
        float x[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x[2 * k] = __uint_as_float(w[k] << 16);
            x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
        }
        if constexpr (FMT == QSA_KV_FP8_E4M3) {
            uint32_t c[4];
            bool same = true;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t lo = e4m3x2(x[2 * k] * fr_lo, x[2 * k + 1] * fr_lo);
                const uint32_t hi = e4m3x2(x[2 * k] * fr_hi, x[2 * k + 1] * fr_hi);
                same &= lo == hi;
                c[k] = lo;
            }
            if (!same) {
                const float s = __ldg(isv ? p.vscale : p.kscale);
#pragma unroll
                for (int k = 0; k < 4; ++k) c[k] = e4m3x2(x[2 * k] / s, x[2 * k + 1] / s);
            }
            reinterpret_cast<uint2*>(pool + row * D)[lane] =
                make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
        } else {
            constexpr float qmax = FMT == QSA_KV_INT8 ? 127.0f : 7.0f;
            constexpr float qmin = FMT == QSA_KV_INT8 ? -127.0f : -8.0f;
            float a = 0.0f;
#pragma unroll
            for (int k = 0; k < 8; ++k) a = fmaxf(a, fabsf(x[k]));
            // a >= 0, so its bit pattern orders like its value
            a = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(a)));
            const float s = __fdiv_rn(a, qmax);
            uint32_t b0, b1;
            bool same = false;
            // Below 2^-100 the scale or its reciprocal leaves the normal range (and
            // codes can need the clamp); above, |x / s| <= qmax * (1 + 2^-19).
            if (a >= 0x1p-100f) {
                const float r = __frcp_rn(s);
                const float r_lo = r * (1.0f - 0x1p-20f), r_hi = r * (1.0f + 0x1p-20f);
                uint32_t lo[8], hi[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    lo[k] = rint_bits(x[k], r_lo);
                    hi[k] = rint_bits(x[k], r_hi);
                }
                b0 = low_bytes(lo[0], lo[1], lo[2], lo[3]);
                b1 = low_bytes(lo[4], lo[5], lo[6], lo[7]);
                same = b0 == low_bytes(hi[0], hi[1], hi[2], hi[3]) &&
                       b1 == low_bytes(hi[4], hi[5], hi[6], hi[7]);
            }
            if (!same) {
                int q[8];
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    q[k] = s > 0.0f ? static_cast<int>(fminf(fmaxf(rintf(x[k] / s), qmin), qmax)) : 0;
                b0 = low_bytes(q[0], q[1], q[2], q[3]);
                b1 = low_bytes(q[4], q[5], q[6], q[7]);
            }
            if constexpr (FMT == QSA_KV_INT8) {
                reinterpret_cast<uint2*>(pool + row * D)[lane] = make_uint2(b0, b1);
            } else {
                reinterpret_cast<uint32_t*>(pool + row * (D / 2))[lane] =
                    low_nibbles(b0) | (low_nibbles(b1) << 16);
            }
            if (lane == 0) (isv ? p.vscale : p.kscale)[row] = s;
        }
    }
}

// Each warp takes RPW consecutive (token, head, K-or-V) rows and issues all their
// loads before converting any, so a warp keeps RPW row reads in flight.
template <int FMT>
__global__ void __launch_bounds__(WARPS * 32) kv_write_kernel(const Params p) {
    const int lane = threadIdx.x & 31;
    const int rows = p.n * p.Hkv; // n <= 2^28 and Hkv <= 2: every task index fits in 32 bits
    const int first = (blockIdx.x * WARPS + (threadIdx.x >> 5)) * RPW;
    float kr_lo = 0.0f, kr_hi = 0.0f, vr_lo = 0.0f, vr_hi = 0.0f;
    if constexpr (FMT == QSA_KV_FP8_E4M3) {
        const float kr = __frcp_rn(__ldg(p.kscale)), vr = __frcp_rn(__ldg(p.vscale));
        kr_lo = kr * (1.0f - 0x1p-20f);
        kr_hi = kr * (1.0f + 0x1p-20f);
        vr_lo = vr * (1.0f - 0x1p-20f);
        vr_hi = vr * (1.0f + 0x1p-20f);
    }
    uint4 raw[RPW];
    long long dst[RPW];
#pragma unroll
    for (int u = 0; u < RPW; ++u) {
        const int task = first + u;
        dst[u] = -1;
        raw[u] = make_uint4(0u, 0u, 0u, 0u);
        if (task >= 2 * rows) continue;
        const bool isv = task >= rows;
        const int r = isv ? task - rows : task;
        const int i = p.Hkv == 2 ? r >> 1 : r, g = p.Hkv == 2 ? r & 1 : 0;
        const int slot = __ldg(p.slots + i);
        if (slot < 0 || (long long)slot >= p.num_slots) {
            if (lane == 0 && p.err) atomicOr(p.err, QSA_DEVERR_SLOT_RANGE);
            continue;
        }
        const __nv_bfloat16* src =
            isv ? p.vx + i * p.v_st + g * p.v_sh : p.kx + i * p.k_st + g * p.k_sh;
        raw[u] = __ldg(reinterpret_cast<const uint4*>(src) + lane); // dims 8*lane .. +7
        dst[u] = (long long)slot * p.Hkv + g;
    }
#pragma unroll
    for (int u = 0; u < RPW; ++u) {
        const bool isv = first + u >= rows;
        if (dst[u] >= 0)
            write_row<FMT>(p, raw[u], dst[u], isv, lane, isv ? vr_lo : kr_lo, isv ? vr_hi : kr_hi);
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

template <int FMT> int launch(const Params& prm, cudaStream_t st) {
    const long long tasks = 2LL * prm.n * prm.Hkv;
    const long long blocks = (tasks + WARPS * RPW - 1) / (WARPS * RPW);
    kv_write_kernel<FMT><<<static_cast<unsigned>(blocks), WARPS * 32, 0, st>>>(prm);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(QSA_ERR_CUDA, "kv write launch: %s", cudaGetErrorString(e));
    return QSA_OK;
}

} // namespace
} // namespace qsakv

extern "C" int qsa_kv_write(int32_t format, const qsa_tensor* k_new, const qsa_tensor* v_new,
                            const qsa_tensor* slots, const qsa_tensor* k_pool,
                            const qsa_tensor* v_pool, float* k_scale, float* v_scale,
                            int32_t* device_error, void* stream) {
    using namespace qsakv;
    if (!k_new || !v_new || !slots || !k_pool || !v_pool)
        return fail(QSA_ERR_INVALID_ARGUMENT, "a descriptor pointer is NULL");
    if (format < QSA_KV_BF16 || format > QSA_KV_INT4)
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
    const int want_dtype = format == QSA_KV_BF16   ? QSA_DTYPE_BF16
                           : format == QSA_KV_INT8 ? QSA_DTYPE_INT8
                                                   : QSA_DTYPE_UINT8;
    const long long row_elems = format == QSA_KV_INT4 ? D / 2 : D;
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
        if ((reinterpret_cast<uintptr_t>(k_scale) & 3u) || (reinterpret_cast<uintptr_t>(v_scale) & 3u))
            return fail(QSA_ERR_MISALIGNED, "scales must be 4-byte aligned");
    }
    if (n > (1LL << 28)) return fail(QSA_ERR_UNSUPPORTED, "more than 2^28 new tokens in one call");
    qsa_detail_set_error("");
    if (n == 0) return QSA_OK;

    Params prm;
    prm.kx = static_cast<const __nv_bfloat16*>(k_new->data);
    prm.vx = static_cast<const __nv_bfloat16*>(v_new->data);
    prm.k_st = k_new->stride[0];
    prm.k_sh = k_new->stride[1];
    prm.v_st = v_new->stride[0];
    prm.v_sh = v_new->stride[1];
    prm.slots = static_cast<const int*>(slots->data);
    prm.n = static_cast<int>(n);
    prm.Hkv = static_cast<int>(hkv);
    prm.kpool = static_cast<uint8_t*>(k_pool->data);
    prm.vpool = static_cast<uint8_t*>(v_pool->data);
    prm.num_slots = k_pool->shape[0];
    prm.kscale = k_scale;
    prm.vscale = v_scale;
    prm.err = device_error;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (format) {
    case QSA_KV_BF16: return launch<QSA_KV_BF16>(prm, st);
    case QSA_KV_FP8_E4M3: return launch<QSA_KV_FP8_E4M3>(prm, st);
    case QSA_KV_INT8: return launch<QSA_KV_INT8>(prm, st);
    default: return launch<QSA_KV_INT4>(prm, st);
    }
}
