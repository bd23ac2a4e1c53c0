// Exact top-k over compressed-block scores and index expansion: the step that
// produces qsa_decode's selected slots and their cu_seqlens, on the device.
//
// What it computes (1Cat-vLLM PR #523, "Follow-up: device-planned MQA and QSA
// quality attribution": exact top-k + index expansion at a fixed 256K capacity,
// compress ratios 4 / 8 / 16; sglang PR #37798, "Decode routing": the index-row
// width token_topk + compress_ratio - 1 = 2051, 64-token pages). Per sequence b
// with context length T (tokens) and compress ratio r:
//   * block i covers tokens [i r, (i + 1) r); the nb = floor(T / r) complete
//     blocks each carry one caller-given float32 score; the last T mod r tokens
//     are not yet in a block;
//   * k = token_topk / r blocks are kept: all when nb <= k, else the k ranked
//     first -- higher score first, equal scores by lower block index, NaN below
//     every number, -0.0 equal to +0.0 (an exact selection, no approximation);
//   * the row lists the kept blocks' tokens in ascending position, then the tail
//     tokens; a page table maps position p to slot pt[p / page] * page + p % page;
//   * rows are packed in sequence order; cu_seqlens[b] is where row b starts.
//
// GB300 design: one CTA of 1024 threads per sequence, no scratch memory.
//  * Scores become order-preserving 32-bit keys (sign-flipped IEEE bits, NaN ->
//    0, -0.0 -> +0.0), so ranking is unsigned integer comparison.
//  * Radix select, four 8-bit digits from the top: each pass histograms the
//    digit of the keys that still match the chosen prefix (warp-aggregated
//    shared-memory atomics: __match_any_sync groups equal digits), and a
//    256-thread descending scan picks the digit holding the k-th key. After
//    four passes the k-th key (the threshold) and the number of blocks equal to
//    it that are kept (the lowest-indexed ones) are exact.
//  * Compaction in index order: chunks of 4096 blocks, each warp 4 rounds of 32;
//    ballots give every block its rank among the threshold ties and among the
//    kept blocks, warp totals a block-wide prefix. A kept block's r token slots
//    go straight to its place in the packed row.
//  * Each CTA computes its row's offset from the context lengths of the rows
//    before it, so the whole step is one launch with no host readback, and a
//    captured graph stays valid when the lengths and scores change.

#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>

#include "qsa.h"

void qsa_detail_set_error(const char* msg);

namespace qsatk {

constexpr int THREADS = 1024;
constexpr int WARPS = THREADS / 32;
constexpr int ROUNDS = 4;                      // 32-block rounds per warp per chunk
constexpr int CHUNK = THREADS * ROUNDS;        // blocks per compaction chunk
constexpr int MAX_BS = 128;
constexpr int MAX_CAPACITY = 262144;           // the pages' fixed 256K context capacity
constexpr int MAX_ROW = 2055;                  // the decode's selected-KV capacity
constexpr unsigned FULL = 0xFFFFFFFFu;

struct Params {
    const float* scores;
    long long s_stride;
    const int* ctx;
    const int* pt;          // page table, or nullptr
    long long pt_stride;
    int page_shift;         // log2(page size)
    int* sel;
    int* cu;
    int* err;               // optional device error word
    int ratio, kb, capacity;
};

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Unsigned key with the order of the ranking: +x above -x, larger above smaller,
// -0.0 == +0.0, every NaN (key 0) below -inf (key 0x007FFFFF).
__device__ __forceinline__ uint32_t order_key(float x) {
    uint32_t u = __float_as_uint(x);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0u;
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int clamp_len(int T, int cap) { return T < 0 ? 0 : (T > cap ? cap : T); }

__device__ __forceinline__ int row_len(int T, int r, int kb) {
    const int nb = T / r;
    return r * (nb < kb ? nb : kb) + (T - nb * r);
}

// Slot of logical position pos of a row; flags (and returns -1 for) a page
// entry that puts the slot outside [0, 2^31).
__device__ __forceinline__ int slot_of(const Params& p, const int* ptrow, int pos, bool& bad) {
    if (ptrow == nullptr) return pos;
    const long long page = 1LL << p.page_shift;
    const long long s = (long long)__ldg(ptrow + (pos >> p.page_shift)) * page + (pos & (page - 1));
    if (s < 0 || s > 0x7FFFFFFFLL) {
        bad = true;
        return -1;
    }
    return static_cast<int>(s);
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__global__ void __launch_bounds__(THREADS, 1) topk_expand_kernel(const Params p) {
    __shared__ uint32_t hist[256];
    __shared__ int wsum[WARPS];
    __shared__ int sh_digit, sh_before, sh_off;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x;
    griddep_wait();
    griddep_launch_dependents();

    // ---------------------------------------------------------------- the row's place
    const int r = p.ratio, kb = p.kb;
    {
        int before = tid < b ? row_len(clamp_len(p.ctx[tid], p.capacity), r, kb) : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(FULL, before, o);
        if (lane == 0 && warp < MAX_BS / 32) wsum[warp] = before;
        __syncthreads();
        if (tid == 0) sh_off = wsum[0] + wsum[1] + wsum[2] + wsum[3];
    }
    const int Traw = p.ctx[b];
    if (tid == 0 && p.err != nullptr && (Traw < 0 || Traw > p.capacity))
        atomicOr(p.err, QSA_DEVERR_CTX_LEN);
    const int T = clamp_len(Traw, p.capacity);
    const int nb = T / r, tail = T - nb * r;
    __syncthreads();
    const int off = sh_off;
    if (tid == 0) {
        p.cu[b + 1] = off + row_len(T, r, kb);
        if (b == 0) p.cu[0] = 0;
    }
    int* const out = p.sel + off;
    const int* const ptrow = p.pt ? p.pt + (long long)b * p.pt_stride : nullptr;
    bool bad = false;

    if (nb <= kb) { // every block kept: the row is positions 0 .. T - 1
        for (int j = tid; j < T; j += THREADS) out[j] = slot_of(p, ptrow, j, bad);
        if (bad && p.err != nullptr) atomicOr(p.err, QSA_DEVERR_SLOT_RANGE);
        return;
    }
    const float* const srow = p.scores + (long long)b * p.s_stride;

    // ---------------------------------------------------------------- radix select
    uint32_t prefix = 0u, mask = 0u;
    int need = kb; // rank of the wanted key among the keys matching the prefix
#pragma unroll 1
    for (int shift = 24; shift >= 0; shift -= 8) {
        if (tid < 256) hist[tid] = 0u;
        __syncthreads();
#pragma unroll 1
        for (int base = 0; base < nb; base += THREADS) {
            const int i = base + tid;
            const uint32_t key = i < nb ? order_key(srow[i]) : 0u;
            const bool cand = i < nb && (key & mask) == prefix;
            const unsigned act = __ballot_sync(FULL, cand);
            if (cand) {
                const uint32_t dig = (key >> shift) & 255u;
                const unsigned peers = __match_any_sync(act, dig);
                if (lane == __ffs(peers) - 1) atomicAdd(&hist[dig], static_cast<uint32_t>(__popc(peers)));
            }
        }
        __syncthreads();
        // digits from the top: the one whose bin holds the need-th key
        int incl = 0, c = 0;
        if (tid < 256) {
            c = static_cast<int>(hist[255 - tid]);
            incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(FULL, incl, o);
                if (lane >= o) incl += v;
            }
            if (lane == 31) wsum[warp] = incl;
        }
        __syncthreads();
        if (tid < 256) {
            for (int w = 0; w < warp; ++w) incl += wsum[w];
            const int excl = incl - c;
            if (excl < need && need <= incl) {
                sh_digit = 255 - tid;
                sh_before = excl;
            }
        }
        __syncthreads();
        prefix |= static_cast<uint32_t>(sh_digit) << shift;
        mask |= 255u << shift;
        need -= sh_before;
    }
    const uint32_t thr = prefix; // the k-th key; `need` blocks equal to it are kept

    // ---------------------------------------------------------------- compaction
    int eq_carry = 0, sel_carry = 0;
    const uint32_t lt = lanemask_lt();
#pragma unroll 1
    for (int base = 0; base < nb; base += CHUNK) {
        const int wbase = base + warp * 32 * ROUNDS;
        uint32_t eqm[ROUNDS], gtm[ROUNDS];
        int weq = 0;
#pragma unroll
        for (int e = 0; e < ROUNDS; ++e) {
            const int i = wbase + e * 32 + lane;
            const uint32_t key = i < nb ? order_key(srow[i]) : 0u;
            eqm[e] = __ballot_sync(FULL, i < nb && key == thr);
            gtm[e] = __ballot_sync(FULL, i < nb && key > thr);
            weq += __popc(eqm[e]);
        }
        __syncthreads(); // wsum free (previous chunk's readers are done)
        if (lane == 0) wsum[warp] = weq;
        __syncthreads();
        int eq_before = eq_carry, eq_total = 0;
        for (int w = 0; w < WARPS; ++w) {
            const int v = wsum[w];
            if (w < warp) eq_before += v;
            eq_total += v;
        }
        uint32_t selm[ROUNDS];
        int wsel = 0;
#pragma unroll
        for (int e = 0; e < ROUNDS; ++e) {
            const bool eq = (eqm[e] >> lane) & 1u;
            const bool sel = ((gtm[e] >> lane) & 1u) || (eq && eq_before + __popc(eqm[e] & lt) < need);
            eq_before += __popc(eqm[e]);
            selm[e] = __ballot_sync(FULL, sel);
            wsel += __popc(selm[e]);
        }
        __syncthreads();
        if (lane == 0) wsum[warp] = wsel;
        __syncthreads();
        int rank = sel_carry, sel_total = 0;
        for (int w = 0; w < WARPS; ++w) {
            const int v = wsum[w];
            if (w < warp) rank += v;
            sel_total += v;
        }
#pragma unroll
        for (int e = 0; e < ROUNDS; ++e) {
            const int j = rank + __popc(selm[e] & lt);
            if (((selm[e] >> lane) & 1u) && j < kb) { // exactly kb are kept; the bound guards the row
                const int i = wbase + e * 32 + lane;
                int* const dst = out + j * r;
                for (int t = 0; t < r; ++t) dst[t] = slot_of(p, ptrow, i * r + t, bad);
            }
            rank += __popc(selm[e]);
        }
        eq_carry += eq_total;
        sel_carry += sel_total;
    }
    // the tail tokens, after the k kept blocks
    for (int t = tid; t < tail; t += THREADS) out[kb * r + t] = slot_of(p, ptrow, nb * r + t, bad);
    if (bad && p.err != nullptr) atomicOr(p.err, QSA_DEVERR_SLOT_RANGE);
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

bool contiguous_i32(const qsa_tensor* t, long long n) {
    return t != nullptr && t->dtype == QSA_DTYPE_INT32 && t->ndim == 1 && t->shape[0] == n &&
           (n <= 1 || t->stride[0] == 1) && t->data != nullptr;
}

} // namespace
} // namespace qsatk

extern "C" int qsa_topk_expand(const qsa_tensor* scores, const qsa_tensor* ctx_lens,
                               const qsa_tensor* page_table, const qsa_topk_params* params,
                               const qsa_tensor* sel_indices, const qsa_tensor* cu_seqlens,
                               int32_t* device_error, void* stream) {
    using namespace qsatk;
    if (!scores || !ctx_lens || !params || !sel_indices || !cu_seqlens)
        return fail(QSA_ERR_INVALID_ARGUMENT, "a descriptor pointer is NULL");
    const int r = params->compress_ratio, K = params->token_topk, cap = params->capacity;
    if (r < 1 || r > 64)
        return fail(QSA_ERR_UNSUPPORTED, "compress ratio %d outside 1..64", r);
    if (K < r || K % r != 0)
        return fail(QSA_ERR_UNSUPPORTED, "token_topk %d is not a positive multiple of the compress ratio %d",
                    K, r);
    const long long width = (long long)K + r - 1;
    if (width > MAX_ROW)
        return fail(QSA_ERR_UNSUPPORTED,
                    "token_topk + compress_ratio - 1 = %lld exceeds the decode's selected-KV capacity %d",
                    width, MAX_ROW);
    if (cap < 1 || cap > MAX_CAPACITY)
        return fail(QSA_ERR_UNSUPPORTED, "context capacity %d outside 1..%d", cap, MAX_CAPACITY);
    if (ctx_lens->ndim != 1 || ctx_lens->shape[0] < 1 || ctx_lens->shape[0] > MAX_BS)
        return fail(QSA_ERR_UNSUPPORTED, "ctx_lens must be int32 [bs], 1 <= bs <= %d", MAX_BS);
    const long long bs = ctx_lens->shape[0];
    if (!contiguous_i32(ctx_lens, bs))
        return fail(QSA_ERR_INVALID_ARGUMENT, "ctx_lens must be a contiguous int32 [bs]");
    const long long nbmax = cap / r;
    if (scores->dtype != QSA_DTYPE_FLOAT32 || scores->ndim != 2 || scores->shape[0] != bs ||
        scores->shape[1] < nbmax || scores->stride[1] != 1 || scores->stride[0] < scores->shape[1] ||
        scores->data == nullptr)
        return fail(QSA_ERR_INVALID_ARGUMENT,
                    "scores must be float32 [bs, >= capacity / compress_ratio = %lld], unit stride "
                    "along the blocks", nbmax);
    const int ps = params->page_size;
    int shift = 0;
    const int* pt = nullptr;
    long long pt_stride = 0;
    if (ps != 0) {
        if (ps < 1 || ps > 65536 || (ps & (ps - 1)))
            return fail(QSA_ERR_UNSUPPORTED, "page size %d is not a power of two in 1..65536", ps);
        while ((1 << shift) < ps) ++shift;
        const long long pages = (cap + ps - 1) / ps;
        if (page_table == nullptr || page_table->dtype != QSA_DTYPE_INT32 || page_table->ndim != 2 ||
            page_table->shape[0] != bs || page_table->shape[1] < pages || page_table->stride[1] != 1 ||
            page_table->stride[0] < page_table->shape[1] || page_table->data == nullptr)
            return fail(QSA_ERR_INVALID_ARGUMENT,
                        "page_table must be int32 [bs, >= ceil(capacity / page_size) = %lld], unit "
                        "stride along the pages", pages);
        pt = static_cast<const int*>(page_table->data);
        pt_stride = page_table->stride[0];
    }
    if (sel_indices->dtype != QSA_DTYPE_INT32 || sel_indices->ndim != 1 ||
        sel_indices->shape[0] < bs * width || sel_indices->stride[0] != 1 || sel_indices->data == nullptr)
        return fail(QSA_ERR_INVALID_ARGUMENT,
                    "sel_indices must be a contiguous int32 vector of at least bs * (token_topk + "
                    "compress_ratio - 1) = %lld entries", bs * width);
    if (!contiguous_i32(cu_seqlens, bs + 1))
        return fail(QSA_ERR_INVALID_ARGUMENT, "cu_seqlens must be a contiguous int32 [bs + 1]");

    Params p;
    p.scores = static_cast<const float*>(scores->data);
    p.s_stride = scores->stride[0];
    p.ctx = static_cast<const int*>(ctx_lens->data);
    p.pt = pt;
    p.pt_stride = pt_stride;
    p.page_shift = shift;
    p.sel = static_cast<int*>(sel_indices->data);
    p.cu = static_cast<int*>(cu_seqlens->data);
    p.err = device_error;
    p.ratio = r;
    p.kb = K / r;
    p.capacity = cap;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(bs));
    cfg.blockDim = dim3(THREADS);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, topk_expand_kernel, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(QSA_ERR_CUDA, "top-k launch: %s", cudaGetErrorString(e));
    qsa_detail_set_error("");
    return QSA_OK;
}
