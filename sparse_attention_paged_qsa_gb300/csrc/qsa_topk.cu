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
// GB300 design: one CTA of 512 threads per sequence (a cluster of them for small
// batches of long rows, below), no global scratch.
//  * Scores become order-preserving 32-bit keys (sign-flipped IEEE bits, NaN ->
//    0, -0.0 -> +0.0), so ranking is unsigned integer comparison.
//  * The score row streams into shared memory in 16 KB pieces by bulk copies
//    (cp.async.bulk, the TMA engine) into a two-slot ring completed on
//    mbarriers, so a whole piece is in flight per slot instead of one load per
//    thread. Every wait is bounded.
//  * Radix select with digits of 11, 11 and 10 bits from the top: a histogram
//    of the digit (shared-memory atomics) and a descending scan over its bins
//    give the digit that holds the k-th key. A row of at most KEYS_CAP blocks is
//    kept as keys in shared memory after the first streaming pass, and the
//    other passes and the compaction run there. A longer row of up to 65,536
//    blocks (the 256K context at ratio 4) keeps each key's top 16 bits in shared
//    memory during its one streaming pass; from those, the blocks whose top
//    digit is the k-th key's or above (about k + one bin) are gathered in index
//    order and only their scores are read again. Rows where those are too many,
//    or longer rows, stream again to gather the k-th key's bin, and rows whose
//    bin is too large stream every pass.
//  * Compaction in index order. Over keys in shared memory each warp takes one
//    contiguous run, a lane 4 keys per 16-byte load: one pass counts the keys
//    above the threshold and the ties, one block-wide prefix, one pass emits.
//    Over streamed pieces, per 4096-block piece each warp takes 8 rounds of 32;
//    ballots give every block its rank among the ties (or the gathered bin) and
//    among the kept blocks, warp totals a block-wide prefix. The kept blocks'
//    r token slots are written after the selection, all blocks at once.
//  * Small batches of long rows (at least 32,768 blocks; as many CTAs as fit the
//    SMs, up to 8 per row) take a thread-block cluster per row: each CTA streams
//    and counts its own part, the parts' histograms are reduced over distributed
//    shared memory (each CTA sums one slice of the bins, then every CTA reads the
//    slice that holds the k-th key), each part's candidates go to the leader CTA
//    at their offset in index order, and the leader selects and writes the row.
//    Every CTA reaches every cluster barrier; when the candidates do not fit the
//    leader, it takes the whole row alone.
//  * Each CTA computes its row's offset from the context lengths of the rows
//    before it, so the whole step is one launch with no host readback, and a
//    captured graph stays valid when the lengths and scores change.

#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "qsa.h"

void qsa_detail_set_error(const char* msg);

namespace qsatk {

constexpr int THREADS = 512;
constexpr int WARPS = THREADS / 32;
constexpr int ROUNDS = 8;                      // 32-block rounds per warp per piece
constexpr int PIECE = THREADS * ROUNDS;        // blocks per piece (4096 = 16 KB of scores)
constexpr int KEYS_CAP = 44 * 1024;            // keys kept in shared memory (176 KB)
constexpr int MAX_BS = 128;
constexpr int MAX_CAPACITY = 262144;           // the pages' fixed 256K context capacity
constexpr int MAX_ROW = 2055;                  // the decode's selected-KV capacity
constexpr unsigned FULL = 0xFFFFFFFFu;
constexpr int NBINS = 2048;                    // bins of an 11-bit digit
constexpr int P16_CAP = 65536;                 // blocks whose 16-bit key prefixes fit the key area
constexpr int CAND_CAP = KEYS_CAP - P16_CAP / 2; // gathered block indices kept next to those prefixes
constexpr int CCAP = CAND_CAP / 2;             // cluster rows: candidates the leader holds (indices, keys)
constexpr int MAX_CLUSTER = 8;                 // CTAs per row for small batches (portable cluster size)
constexpr long long WAIT_NS = 2000000000LL;    // bounded-wait limit (2 s)
constexpr uint32_t KEPT = 0xFFFFFFFFu;         // not a key: order_key maps every NaN to 0
// dynamic shared memory: the two ring slots, the keys, the histogram
constexpr int OFF_RING = 0;
constexpr int OFF_KEYS = OFF_RING + 2 * PIECE * 4;
constexpr int OFF_HIST = OFF_KEYS + KEYS_CAP * 4;
constexpr int OFF_KEPT = OFF_HIST + NBINS * 4;           // kept block index by rank
constexpr int SMEM_BYTES = OFF_KEPT + (MAX_ROW + 1) * 4;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(NBINS % THREADS == 0 && NBINS / THREADS <= 4, "digit scan");
static_assert(CCAP % 4 == 0 && (P16_CAP / 2 + CCAP) % 4 == 0, "cluster candidate lists stay 16-byte aligned");
static_assert(ROUNDS % 4 == 0 && PIECE % 4096 == 0, "16-byte first-pass accesses stay aligned");
static_assert(CAND_CAP > 0 && P16_CAP % 2 == 0, "prefix and candidate areas");
static_assert(P16_CAP / 32 <= MAX_ROW + 1 && P16_CAP <= 128 * THREADS, "prefix bitmap in the kept-list area");

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
__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for the phase with `parity` of an mbarrier for at most WAIT_NS.
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 63 && globaltimer() - t0 > (unsigned long long)WAIT_NS) return false;
    }
}
// The timer is read only when the first try does not see the phase complete.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    return mbar_try_wait(bar, parity) || mbar_wait_slow(bar, parity);
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Thread-block clusters: this CTA's rank and the cluster's size, another CTA's
// shared-memory address (distributed shared memory), and a barrier of every
// thread of every CTA of the cluster (release / acquire).
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ uint32_t ld_dsmem(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_dsmem(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
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

// Exclusive prefix over the warps of one value per warp; returns (before, total).
// Bracketed by barriers, so `wsum` may be reused right after.
__device__ __forceinline__ int2 block_prefix(int v, int* wsum) {
    const int warp = threadIdx.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) wsum[warp] = v;
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
        const int x = wsum[w];
        before += w < warp ? x : 0;
        total += x;
    }
    return make_int2(before, total);
}

// The digit (of a `bins`-bin histogram, taken from the top) whose bin holds the
// need-th key, and the number of keys in the bins above it.
__device__ __forceinline__ int2 find_digit(const uint32_t* hist, int bins, int need, int* wsum, int* sh) {
    const int tid = threadIdx.x, lane = tid & 31, per = bins / THREADS;
    int c[4] = {0, 0, 0, 0}, s = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q)
        if (q < per) {
            c[q] = static_cast<int>(hist[bins - 1 - (tid * per + q)]);
            s += c[q];
        }
    int incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += v;
    }
    const int2 pw = block_prefix(__shfl_sync(FULL, incl, 31), wsum);
    int excl = pw.x + incl - s;
#pragma unroll
    for (int q = 0; q < 4; ++q)
        if (q < per) {
            if (excl < need && need <= excl + c[q]) {
                sh[0] = bins - 1 - (tid * per + q);
                sh[1] = excl;
            }
            excl += c[q];
        }
    __syncthreads();
    return make_int2(sh[0], sh[1]);
}

// One piece of an index-ordered scan: n <= PIECE keys key_at(0 .. n-1), global
// positions base + j. Each key gets its rank among the keys with is_a() (counted
// from `carry_a`), decide(key, is_a, rank_a) says whether it is kept, and
// emit(j, rank) receives every kept key with its rank among the kept ones
// (counted from `carry_s`). The carries advance by the piece's totals.
template <class KeyAt, class IsA, class Decide, class Emit>
__device__ __forceinline__ void scan_piece(int n, KeyAt key_at, IsA is_a, Decide decide, Emit emit,
                                           int& carry_a, int& carry_s, int* wsum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t lt = lanemask_lt();
    const int wbase = warp * 32 * ROUNDS;
    uint32_t am[ROUNDS];
    int wa = 0;
#pragma unroll
    for (int e = 0; e < ROUNDS; ++e) {
        const int j = wbase + e * 32 + lane;
        am[e] = __ballot_sync(FULL, j < n && is_a(key_at(j)));
        wa += __popc(am[e]);
    }
    const int2 pa = block_prefix(wa, wsum);
    int ra = carry_a + pa.x;
    uint32_t sm[ROUNDS];
    int ws = 0;
#pragma unroll
    for (int e = 0; e < ROUNDS; ++e) {
        const int j = wbase + e * 32 + lane;
        const bool isa = (am[e] >> lane) & 1u;
        const bool sel = j < n && decide(key_at(j), isa, ra + __popc(am[e] & lt));
        ra += __popc(am[e]);
        sm[e] = __ballot_sync(FULL, sel);
        ws += __popc(sm[e]);
    }
    const int2 ps = block_prefix(ws, wsum);
    int rs = carry_s + ps.x;
#pragma unroll
    for (int e = 0; e < ROUNDS; ++e) {
        if ((sm[e] >> lane) & 1u) emit(wbase + e * 32 + lane, rs + __popc(sm[e] & lt));
        rs += __popc(sm[e]);
    }
    carry_a += pa.y;
    carry_s += ps.y;
}

// Index-ordered compaction of n keys in shared memory: every key above thr and
// the first need_t keys equal to thr go to emit(i, rank), rank counted among the
// emitted keys in index order. Each warp takes one contiguous run of 4-key
// chunks, a lane one chunk per 16-byte load, so the whole array takes a single
// block-wide prefix of the warps' counts, packed as (above << 16) | equal: fewer
// than k <= 2048 keys lie above thr, and n < 65536.
template <class Emit>
__device__ __forceinline__ void compact_keys(const uint32_t* kk, int n, uint32_t thr, int need_t, Emit emit,
                                             int* wsum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int chunks = (n + 3) >> 2;
    const int per = (((chunks + WARPS - 1) / WARPS) + 31) & ~31;
    const int c0 = min(chunks, warp * per), c1 = min(chunks, c0 + per);
    const uint4* const kv = reinterpret_cast<const uint4*>(kk);
    auto count = [&](const uint4& v, int i) {
        const uint32_t k[4] = {v.x, v.y, v.z, v.w};
        int s = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (i + q < n) s += k[q] > thr ? 0x10000 : (k[q] == thr ? 1 : 0);
        return s;
    };
    int cnt = 0;
#pragma unroll 4
    for (int c = c0 + lane; c < c1; c += 32) cnt += count(kv[c], 4 * c);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(FULL, cnt, o);
    int before = block_prefix(cnt, wsum).x;
    for (int cb = c0; cb < c1; cb += 32) { // warp-uniform bounds
        const int c = cb + lane;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        int my = 0;
        if (c < c1) {
            v = kv[c];
            my = count(v, 4 * c);
        }
        int incl = my;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(FULL, incl, o);
            if (lane >= o) incl += t;
        }
        if (my != 0) {
            const int at0 = before + incl - my;
            int above = at0 >> 16, at = at0 & 0xFFFF;
            const uint32_t k[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int i = 4 * c + q;
                if (i < n && k[q] > thr) {
                    emit(i, above + min(at, need_t));
                    ++above;
                } else if (i < n && k[q] == thr) {
                    if (at < need_t) emit(i, above + at);
                    ++at;
                }
            }
        }
        before += __shfl_sync(FULL, incl, 31);
    }
}

// A bitmap of the n <= 128 * THREADS 16-bit key prefixes in shared memory that
// are >= t, in index order: bit b of bm[w] for prefix 32w + b. A thread takes
// 8 adjacent prefixes per 16-byte load (units tid, tid + THREADS, ... , 4 in
// flight) and stores their 8 bits as one byte (bits past n are zero through the
// end of the last word). Ends with a barrier.
__device__ __forceinline__ void bitmap_ge16(const uint16_t* p16, int n, uint32_t t, uint32_t* bm) {
    const int tid = threadIdx.x;
    const int units = (n + 7) >> 3, nbytes = ((n + 31) >> 5) * 4; // whole words, zero past n
    const uint4* const pv = reinterpret_cast<const uint4*>(p16);
    uint8_t* const bb = reinterpret_cast<uint8_t*>(bm);
    const uint32_t T = t << 16; // a word is >= T when its upper prefix is >= t
    auto bits2 = [&](uint32_t w) { // the word's lower prefix in bit 0, upper in bit 1
        return static_cast<uint32_t>((w << 16) >= T) | (static_cast<uint32_t>(w >= T) << 1);
    };
#pragma unroll 4
    for (int u = tid; u < nbytes; u += THREADS) {
        uint32_t m = 0u;
        if (u < units) {
            const uint4 v = pv[u];
            m = bits2(v.x) | (bits2(v.y) << 2) | (bits2(v.z) << 4) | (bits2(v.w) << 6);
            const int left = n - 8 * u; // prefixes of this unit inside the row (>= 1)
            if (left < 8) m &= (1u << left) - 1u;
        }
        bb[u] = static_cast<uint8_t>(m);
    }
    __syncthreads();
}

// The same bitmap of the n <= 128 * THREADS 32-bit keys in shared memory that
// are >= t, a thread taking 4 adjacent keys per 16-byte load and storing their 4
// bits in one half of a byte; two threads' halves share a byte, so the pair
// combine theirs by shuffle and the even one stores it (bits past n are zero
// through the end of the last word). Ends with a barrier.
__device__ __forceinline__ void bitmap_ge32(const uint32_t* kk, int n, uint32_t t, uint32_t* bm) {
    const int tid = threadIdx.x, lane = tid & 31;
    const int quads = (n + 3) >> 2, nquads = ((n + 31) >> 5) * 8; // whole words, zero past n
    const int rounds = (nquads + THREADS - 1) / THREADS;
    const uint4* const kv = reinterpret_cast<const uint4*>(kk);
    uint8_t* const bb = reinterpret_cast<uint8_t*>(bm);
#pragma unroll 4
    for (int r = 0; r < rounds; ++r) { // uniform trip count: the shuffle sees the whole warp
        const int u = r * THREADS + tid;
        uint32_t m = 0u;
        if (u < quads) {
            const uint4 v = kv[u];
            m = static_cast<uint32_t>(v.x >= t) | (static_cast<uint32_t>(v.y >= t) << 1) |
                (static_cast<uint32_t>(v.z >= t) << 2) | (static_cast<uint32_t>(v.w >= t) << 3);
            const int left = n - 4 * u;
            if (left < 4) m &= (1u << left) - 1u;
        }
        const uint32_t hi = __shfl_down_sync(FULL, m, 1);
        if ((lane & 1) == 0 && u < nquads) bb[u >> 1] = static_cast<uint8_t>(m | (hi << 4));
    }
    __syncthreads();
}

// The set bits of a bitmap over n <= 128 * THREADS positions, in index order:
// each thread takes up to 4 consecutive words, their popcounts take one
// block-wide prefix, and when the total lies in [lo, cap] each set position goes
// to out[rank]. Returns the total.
__device__ __forceinline__ int emit_bitmap(const uint32_t* bm, int n, int lo, int cap, uint32_t* out,
                                           int* wsum) {
    const int tid = threadIdx.x, lane = tid & 31;
    const int words = (n + 31) >> 5, per = (words + THREADS - 1) / THREADS;
    const int w0 = min(words, tid * per), w1 = min(words, w0 + per);
    int cnt = 0;
    for (int w = w0; w < w1; ++w) cnt += __popc(bm[w]);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += x;
    }
    const int2 pw = block_prefix(__shfl_sync(FULL, incl, 31), wsum);
    if (pw.y >= lo && pw.y <= cap) {
        int rank = pw.x + incl - cnt;
        for (int w = w0; w < w1; ++w) {
            uint32_t m = bm[w];
            while (m != 0u) {
                const int bit = __ffs(m) - 1;
                m &= m - 1u;
                out[rank++] = static_cast<uint32_t>(w * 32 + bit);
            }
        }
    }
    return pw.y;
}

// The same walk as emit_bitmap in two steps, for a caller that places the set
// bits at an offset known only after the total: bitmap_ranks gives this thread's
// first rank and the block's total; bitmap_emit calls emit(i, rank) for this
// thread's set positions, ranks counted from `start`.
__device__ __forceinline__ int2 bitmap_ranks(const uint32_t* bm, int n, int* wsum) {
    const int tid = threadIdx.x, lane = tid & 31;
    const int words = (n + 31) >> 5, per = (words + THREADS - 1) / THREADS;
    const int w0 = min(words, tid * per), w1 = min(words, w0 + per);
    int cnt = 0;
    for (int w = w0; w < w1; ++w) cnt += __popc(bm[w]);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += x;
    }
    const int2 pw = block_prefix(__shfl_sync(FULL, incl, 31), wsum);
    return make_int2(pw.x + incl - cnt, pw.y);
}
template <class Emit>
__device__ __forceinline__ void bitmap_emit(const uint32_t* bm, int n, int start, Emit emit) {
    const int tid = threadIdx.x;
    const int words = (n + 31) >> 5, per = (words + THREADS - 1) / THREADS;
    const int w0 = min(words, tid * per), w1 = min(words, w0 + per);
    int rank = start;
    for (int w = w0; w < w1; ++w) {
        uint32_t m = bm[w];
        while (m != 0u) {
            const int bit = __ffs(m) - 1;
            m &= m - 1u;
            emit(w * 32 + bit, rank++);
        }
    }
}

// Index-ordered gather of the prefixes >= t (see bitmap_ge16 and emit_bitmap).
__device__ __forceinline__ int gather_ge16(const uint16_t* p16, int n, uint32_t t, uint32_t* bm, uint32_t* out,
                                           int cap, int* wsum) {
    bitmap_ge16(p16, n, t, bm);
    return emit_bitmap(bm, n, 0, cap, out, wsum);
}

// Streams the first nb scores of a row through the two-slot ring, one PIECE at a
// time, calling fn(piece, base, n) with the piece in shared memory (n floats at
// row positions base .. base + n - 1). Thread 0 keeps the next piece in flight.
// `seq` counts pieces across passes (ring slot and mbarrier parity). Returns
// false (uniformly) when a wait ran out; copies in flight have then landed or
// been waited for, with a limit.
template <class Fn>
__device__ bool stream_row(const float* srow, int nb, float* ring, uint32_t bar0, uint32_t& seq, Fn fn) {
    const int tid = threadIdx.x;
    const int pieces = (nb + PIECE - 1) / PIECE;
    auto issue = [&](int c) { // thread 0: piece c into slot (seq + c) & 1
        const int n = min(PIECE, nb - c * PIECE), al = n & ~3;
        const uint32_t slot = (seq + c) & 1u, bar = bar0 + 8u * slot;
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(al * 4));
        if (al > 0) bulk_g2s(smem_u32(ring + slot * PIECE), srow + (long long)c * PIECE, al * 4, bar);
    };
    if (tid == 0) {
        fence_proxy_async(); // earlier generic accesses of the ring before the copies
        issue(0);
        if (pieces > 1) issue(1);
    }
    bool ok = true;
    int c = 0;
    for (; c < pieces; ++c) {
        const uint32_t slot = (seq + c) & 1u;
        const bool landed = mbar_wait(bar0 + 8u * slot, ((seq + c) >> 1) & 1u);
        if (__syncthreads_or(!landed)) {
            ok = false;
            break;
        }
        float* const piece = ring + slot * PIECE;
        const int n = min(PIECE, nb - c * PIECE), al = n & ~3;
        if (n != al) { // the unaligned end (uniform)
            if (tid < n - al) piece[al + tid] = srow[(long long)c * PIECE + al + tid];
            __syncthreads();
        }
        fn(piece, c * PIECE, n);
        __syncthreads(); // the slot's readers are done
        if (tid == 0 && c + 2 < pieces) {
            fence_proxy_async();
            issue(c + 2);
        }
    }
    if (!ok && tid == 0) { // let the copies still in flight land before the CTA leaves
        for (int k = c; k < pieces && k < c + 2; ++k)
            mbar_wait(bar0 + 8u * ((seq + k) & 1u), ((seq + k) >> 1) & 1u);
    }
    seq += static_cast<uint32_t>(pieces);
    return ok;
}

// One row's top-k and expansion. CL: the row belongs to a thread-block cluster of
// C CTAs (small batches): each streams and counts its own part of the row, the
// parts' histograms are summed over distributed shared memory, each part's
// candidates go to the leader (rank 0) in index order, and the leader finishes
// the row; without CL, or when the candidates do not fit the leader, one CTA
// takes the whole row.
template <bool CL>
__device__ __forceinline__ void topk_row(const Params& p) {
    extern __shared__ __align__(128) uint8_t smem[];
    float* const ring = reinterpret_cast<float*>(smem + OFF_RING);
    uint32_t* const keys = reinterpret_cast<uint32_t*>(smem + OFF_KEYS);
    uint32_t* const hist = reinterpret_cast<uint32_t*>(smem + OFF_HIST);
    int* const kept = reinterpret_cast<int*>(smem + OFF_KEPT);
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ int wsum[WARPS];
    __shared__ int sh[4];
    __shared__ uint32_t few[32]; // the last radix pass's keys, when at most 32
    __shared__ int nfew;
    __shared__ int ccount[MAX_CLUSTER]; // cluster rows, in the leader: each part's candidate count
    __shared__ int stot[MAX_CLUSTER];   // cluster rows: each CTA's histogram-slice total
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int crank = CL ? static_cast<int>(cluster_ctarank()) : 0;
    const int csize = CL ? static_cast<int>(cluster_nctarank()) : 1;
    const bool leader = crank == 0;
    const int b = CL ? static_cast<int>(blockIdx.x) / csize : static_cast<int>(blockIdx.x);
    const uint32_t bar0 = smem_u32(bars);
    if (tid == 0) {
        mbar_init(bar0, 1);
        mbar_init(bar0 + 8, 1);
        fence_mbarrier_init();
        sh[0] = sh[1] = 0;
    }
    griddep_wait();
    griddep_launch_dependents();

    // ---------------------------------------------------------------- the row's place
    const int r = p.ratio, kb = p.kb;
    int before = 0;
    for (int j = tid; j < b; j += THREADS) before += row_len(clamp_len(p.ctx[j], p.capacity), r, kb);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(FULL, before, o);
    const int off = block_prefix(before, wsum).y;
    const int Traw = p.ctx[b];
    if (tid == 0 && p.err != nullptr && (Traw < 0 || Traw > p.capacity))
        atomicOr(p.err, QSA_DEVERR_CTX_LEN);
    const int T = clamp_len(Traw, p.capacity);
    const int nb = T / r, tail = T - nb * r;
    if (tid == 0 && leader) {
        p.cu[b + 1] = off + row_len(T, r, kb);
        if (b == 0) p.cu[0] = 0;
    }
    int* const out = p.sel + off;
    const int* const ptrow = p.pt ? p.pt + (long long)b * p.pt_stride : nullptr;
    bool bad = false;

    if (nb <= kb) { // every block kept: the row is positions 0 .. T - 1
        if (!leader) return;
        for (int j = tid; j < T; j += THREADS) out[j] = slot_of(p, ptrow, j, bad);
        if (bad && p.err != nullptr) atomicOr(p.err, QSA_DEVERR_SLOT_RANGE);
        return;
    }
    const float* const srow = p.scores + (long long)b * p.s_stride;
    uint32_t seq = 0;
    auto timed_out = [&]() {
        if (tid == 0 && p.err != nullptr) atomicOr(p.err, QSA_DEVERR_TIMEOUT);
    };
    auto clear_hist = [&]() {
        for (int i = tid; i < NBINS; i += THREADS) hist[i] = 0u;
        __syncthreads();
    };
    // a kept block at its rank; its r token slots are written after the scan by
    // write_kept, all blocks at once, so the page-table reads overlap
    auto put_block = [&](int i, int j) {
        if (j < kb) kept[j] = i; // exactly kb are kept; the bound guards the row
    };
    auto write_kept = [&]() {
        __syncthreads();
        for (int j = tid; j < kb; j += THREADS) {
            int* const dst = out + j * r;
            const int pos0 = kept[j] * r;
            if (ptrow != nullptr && (pos0 >> p.page_shift) == ((pos0 + r - 1) >> p.page_shift)) {
                // the block's r tokens lie in one page: one page-table read for all
                const long long page = 1LL << p.page_shift;
                const long long s0 = (long long)__ldg(ptrow + (pos0 >> p.page_shift)) * page + (pos0 & (page - 1));
                for (int t = 0; t < r; ++t) { // the same range check as slot_of, per token
                    const long long st = s0 + t;
                    const bool out_of_range = st < 0 || st > 0x7FFFFFFFLL;
                    bad |= out_of_range;
                    dst[t] = out_of_range ? -1 : static_cast<int>(st);
                }
            } else {
                for (int t = 0; t < r; ++t) dst[t] = slot_of(p, ptrow, pos0 + t, bad);
            }
        }
    };
    // radix passes 1 and 2 (digits of 11 and 10 bits) over keys in shared memory
    // radix passes 1 and 2 (digits of 11 and 10 bits) over keys in shared memory.
    // When at most 32 keys are left for pass 2 (usually one or two), they are
    // collected instead and one warp ranks them: the need-th largest is the key
    // with fewer than need keys above it and at least need at or above it.
    auto select_in_smem = [&](const uint32_t* kk, int n, uint32_t& prefix, uint32_t& mask, int& need) {
        for (int pass = 1; pass < 3; ++pass) {
            const int shift = pass == 1 ? 10 : 0, bins = pass == 1 ? 2048 : 1024;
            clear_hist();
            if (tid == 0) nfew = 0;
            for (int i = tid; i < n; i += THREADS) {
                const uint32_t k = kk[i];
                if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & (bins - 1)], 1u);
            }
            __syncthreads();
            const int2 d = find_digit(hist, bins, need, wsum, sh);
            prefix |= static_cast<uint32_t>(d.x) << shift;
            mask |= static_cast<uint32_t>(bins - 1) << shift;
            need -= d.y;
            const int left = static_cast<int>(hist[d.x & (bins - 1)]); // keys matching the prefix now
            __syncthreads();                                               // read before pass 2 clears it
            if (pass == 1 && left <= 32) { // uniform
                for (int i = tid; i < n; i += THREADS) {
                    const uint32_t k = kk[i];
                    if ((k & mask) == prefix) few[atomicAdd(&nfew, 1)] = k;
                }
                __syncthreads();
                if (warp == 0) {
                    const uint32_t k = lane < left ? few[lane] : 0u;
                    int above = 0, at = 0;
                    for (int j = 0; j < left; ++j) {
                        const uint32_t o = few[j];
                        above += o > k ? 1 : 0;
                        at += o >= k ? 1 : 0;
                    }
                    const uint32_t hit = __ballot_sync(FULL, lane < left && above < need && need <= at);
                    const int src = __ffs(hit) - 1;
                    const uint32_t key = __shfl_sync(FULL, k, src);
                    const int ab = __shfl_sync(FULL, above, src);
                    if (lane == 0) {
                        sh[2] = static_cast<int>(key);
                        sh[3] = ab;
                    }
                }
                __syncthreads();
                prefix = static_cast<uint32_t>(sh[2]);
                mask = 0xFFFFFFFFu;
                need -= sh[3];
                __syncthreads();
                break;
            }
        }
    };

    uint32_t prefix = 0u, mask = 0u;
    int need = kb; // rank of the wanted key among the keys that match the prefix
    if constexpr (CL) {
        // ------------------------------------------------ a cluster row
        // Part k: blocks [lo, lo + nown), parts of a multiple of 32 blocks (the host
        // launches clusters only when every part fits P16_CAP prefixes). Every CTA
        // reaches every cluster barrier below, whatever happened before it.
        const int C = csize;
        const int part = (((nb + C - 1) / C) + 31) & ~31;
        const int lo = min(nb, crank * part), nown = min(nb, lo + part) - lo;
        uint16_t* const p16 = reinterpret_cast<uint16_t*>(keys);
        clear_hist();
        if (nown > 0) { // (a part of no blocks streams nothing)
            const bool okc = stream_row(srow + lo, nown, ring, bar0, seq, [&](const float* piece, int base, int n) {
                if (n == PIECE) { // 16-byte loads, 8-byte prefix stores: a thread takes 4 adjacent blocks
                    float4 x[ROUNDS / 4];
#pragma unroll
                    for (int e = 0; e < ROUNDS / 4; ++e)
                        x[e] = reinterpret_cast<const float4*>(piece)[tid + e * THREADS];
#pragma unroll
                    for (int e = 0; e < ROUNDS / 4; ++e) {
                        const uint32_t k0 = order_key(x[e].x), k1 = order_key(x[e].y), k2 = order_key(x[e].z),
                                       k3 = order_key(x[e].w);
                        reinterpret_cast<uint2*>(p16 + base)[tid + e * THREADS] =
                            make_uint2((k0 >> 16) | (k1 & 0xFFFF0000u), (k2 >> 16) | (k3 & 0xFFFF0000u));
                        atomicAdd(&hist[k0 >> 21], 1u);
                        atomicAdd(&hist[k1 >> 21], 1u);
                        atomicAdd(&hist[k2 >> 21], 1u);
                        atomicAdd(&hist[k3 >> 21], 1u);
                    }
                } else {
                    for (int j = tid; j < n; j += THREADS) {
                        const uint32_t k = order_key(piece[j]);
                        p16[base + j] = static_cast<uint16_t>(k >> 16);
                        atomicAdd(&hist[k >> 21], 1u);
                    }
                }
            });
            if (!okc) timed_out(); // (the row's result is then unspecified)
        }
        __syncthreads();
        cluster_sync(); // every part counted
        // The row's histogram, reduced and scattered: CTA k sums bins [k S, (k + 1) S)
        // over every part (S = NBINS / C) into `slice` (over the candidate lists,
        // written only after the next two barriers) and sends its slice's total to
        // every CTA. Then each CTA finds, from the totals, the slice that holds the
        // k-th key and reads only that slice, from its owner. Every remote load of a
        // thread is issued before any is used.
        const int S = NBINS / C;
        uint32_t* const slice = keys + P16_CAP / 2;
        {
            constexpr int PER = NBINS / THREADS; // slice bins per thread, at most
            uint32_t v[PER][MAX_CLUSTER];
#pragma unroll
            for (int q = 0; q < PER; ++q)
#pragma unroll
                for (int k = 0; k < MAX_CLUSTER; ++k) {
                    const int i = tid + q * THREADS;
                    v[q][k] = (i < S && k < C)
                                  ? ld_dsmem(mapa(smem_u32(hist + crank * S + i), static_cast<uint32_t>(k)))
                                  : 0u;
                }
            int mine = 0;
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                uint32_t c = 0u;
#pragma unroll
                for (int k = 0; k < MAX_CLUSTER; ++k) c += v[q][k];
                if (tid + q * THREADS < S) slice[tid + q * THREADS] = c;
                mine += static_cast<int>(c);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(FULL, mine, o);
            const int total = block_prefix(mine, wsum).y;
            if (tid < C) st_dsmem(mapa(smem_u32(&stot[crank]), static_cast<uint32_t>(tid)), static_cast<uint32_t>(total));
        }
        cluster_sync(); // slices summed, totals everywhere
        int js = C - 1, above = 0; // the slice (from the top) that holds the need-th key
        while (js > 0 && above + stot[js] < need) above += stot[js--];
        uint32_t* const htot = reinterpret_cast<uint32_t*>(kept); // that slice in place, zeros elsewhere
        {
            constexpr int PER = NBINS / THREADS;
            uint32_t v[PER];
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                const int i = tid + q * THREADS;
                const bool in = i >= js * S && i < (js + 1) * S;
                v[q] = in ? ld_dsmem(mapa(smem_u32(slice + (i - js * S)), static_cast<uint32_t>(js))) : 0u;
            }
#pragma unroll
            for (int q = 0; q < PER; ++q) htot[tid + q * THREADS] = v[q];
        }
        __syncthreads();
        const int2 dl = find_digit(htot, NBINS, need - above, wsum, sh);
        const int2 d = make_int2(dl.x, dl.y + above);
        const uint32_t d1 = static_cast<uint32_t>(d.x) & (NBINS - 1);
        const int cand = static_cast<int>(htot[d1]);
        int needc = need - d.y;
        uint32_t t16 = d1 << 5, pfx = d1 << 21, msk = 0x7FFu << 21;
        int ng = d.y + cand;
        // (hist is read remotely only before the barrier above: the 5-bit step may reuse it)
        if (ng > CCAP) { // (uniform over the cluster: the same histogram)
            // the 5-bit digit below d1 that holds the k-th key, from every part's prefixes
            if (tid < 32) hist[tid] = 0u;
            __syncthreads();
            for (int j = tid; j < nown; j += THREADS) {
                const uint32_t v = p16[j];
                if ((v >> 5) == d1) atomicAdd(&hist[v & 31u], 1u);
            }
            __syncthreads();
            cluster_sync();
            if (warp == 0) {
                const int bin = 31 - lane;
                const uint32_t a = smem_u32(hist + bin);
                uint32_t v[MAX_CLUSTER];
#pragma unroll
                for (int k = 0; k < MAX_CLUSTER; ++k) v[k] = k < C ? ld_dsmem(mapa(a, static_cast<uint32_t>(k))) : 0u;
                int cnt = 0;
#pragma unroll
                for (int k = 0; k < MAX_CLUSTER; ++k) cnt += static_cast<int>(v[k]);
                int incl = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(FULL, incl, o);
                    if (lane >= o) incl += v;
                }
                if (incl - cnt < needc && needc <= incl) {
                    sh[0] = bin;
                    sh[1] = incl - cnt;
                    sh[2] = cnt;
                }
            }
            __syncthreads();
            t16 = (d1 << 5) | static_cast<uint32_t>(sh[0]);
            pfx = t16 << 16;
            msk = 0xFFFF0000u;
            needc -= sh[1];
            ng = d.y + sh[1] + sh[2];
            cluster_sync(); // every part's 5-bit counts read, sh read
        }
        if (ng <= CCAP) {
            // this part's blocks at or above t16, in index order, to the leader's lists
            // at this part's offset: block index and full key (one score read each)
            uint32_t* const bm = reinterpret_cast<uint32_t*>(kept);
            if (nown > 0) bitmap_ge16(p16, nown, t16, bm);
            const int2 rk = bitmap_ranks(bm, nown, wsum);
            if (tid == 0) st_dsmem(mapa(smem_u32(&ccount[crank]), 0u), static_cast<uint32_t>(rk.y));
            cluster_sync();
            uint32_t cv[MAX_CLUSTER];
#pragma unroll
            for (int k = 0; k < MAX_CLUSTER; ++k) cv[k] = k < crank ? ld_dsmem(mapa(smem_u32(&ccount[k]), 0u)) : 0u;
            int base = 0;
#pragma unroll
            for (int k = 0; k < MAX_CLUSTER; ++k) base += static_cast<int>(cv[k]);
            const uint32_t glr = mapa(smem_u32(keys + P16_CAP / 2), 0u);
            const uint32_t ckr = mapa(smem_u32(keys + P16_CAP / 2 + CCAP), 0u);
            bitmap_emit(bm, nown, base + rk.x, [&](int j, int g) {
                if (g < CCAP) { // exactly ng are emitted; the bound guards the lists
                    const int i = lo + j;
                    st_dsmem(glr + 4u * static_cast<uint32_t>(g), static_cast<uint32_t>(i));
                    st_dsmem(ckr + 4u * static_cast<uint32_t>(g), order_key(__ldg(srow + i)));
                }
            });
            cluster_sync(); // every candidate is in the leader
            if (!leader) return;
            uint32_t* const gl = keys + P16_CAP / 2;
            uint32_t* const ck = gl + CCAP;
            select_in_smem(ck, ng, pfx, msk, needc);
            compact_keys(ck, ng, pfx, needc, [&](int g, int rank) { put_block(static_cast<int>(gl[g]), rank); },
                         wsum);
            write_kept(); // the kept blocks' slots, at their ranks
            for (int t = tid; t < tail; t += THREADS) out[kb * r + t] = slot_of(p, ptrow, nb * r + t, bad);
            if (bad && p.err != nullptr) atomicOr(p.err, QSA_DEVERR_SLOT_RANGE);
            return;
        }
        // too many candidates for the leader: it takes the whole row alone
        if (!leader) return;
    }
    if (nb <= KEYS_CAP) {
        // ------------------------------------------------ the row fits: keys in shared memory
        clear_hist();
        const bool ok = stream_row(srow, nb, ring, bar0, seq, [&](const float* piece, int base, int n) {
            if (n == PIECE) { // 16-byte loads and stores: a thread takes 4 adjacent blocks
                float4 x[ROUNDS / 4];
#pragma unroll
                for (int e = 0; e < ROUNDS / 4; ++e) x[e] = reinterpret_cast<const float4*>(piece)[tid + e * THREADS];
#pragma unroll
                for (int e = 0; e < ROUNDS / 4; ++e) {
                    const uint4 k = make_uint4(order_key(x[e].x), order_key(x[e].y), order_key(x[e].z),
                                               order_key(x[e].w));
                    reinterpret_cast<uint4*>(keys + base)[tid + e * THREADS] = k;
                    atomicAdd(&hist[k.x >> 21], 1u);
                    atomicAdd(&hist[k.y >> 21], 1u);
                    atomicAdd(&hist[k.z >> 21], 1u);
                    atomicAdd(&hist[k.w >> 21], 1u);
                }
            } else {
                for (int j = tid; j < n; j += THREADS) {
                    const uint32_t k = order_key(piece[j]);
                    keys[base + j] = k;
                    atomicAdd(&hist[k >> 21], 1u);
                }
            }
        });
        if (!ok) return timed_out();
        __syncthreads();
        const int2 d = find_digit(hist, NBINS, need, wsum, sh);
        prefix = static_cast<uint32_t>(d.x) << 21;
        mask = 0x7FFu << 21;
        need -= d.y;
        // (16-byte aligned areas: compact_keys reads 4 keys at a time)
        const int nb4 = (nb + 3) & ~3, ng = d.y + static_cast<int>(hist[d.x & (NBINS - 1)]);
        const int ng4 = (ng + 3) & ~3;
        __syncthreads();
        if (nb4 + 2 * ng4 <= KEYS_CAP && 16 * ng <= nb) {
            // the blocks whose top digit is the k-th key's or above, in index order
            // (their indices, then their keys, past the row's keys); the rest of the
            // selection runs on those. Only when they are few: a thread emits a
            // 128-block group's indices one by one.
            uint32_t* const gl = keys + nb4;
            uint32_t* const ck = gl + ng4;
            bitmap_ge32(keys, nb, prefix, reinterpret_cast<uint32_t*>(kept));
            emit_bitmap(reinterpret_cast<uint32_t*>(kept), nb, 0, ng, gl, wsum);
            __syncthreads();
            for (int g = tid; g < ng; g += THREADS) ck[g] = keys[gl[g]];
            __syncthreads();
            select_in_smem(ck, ng, prefix, mask, need);
            compact_keys(ck, ng, prefix, need, [&](int g, int rank) { put_block(static_cast<int>(gl[g]), rank); },
                         wsum);
        } else {
            select_in_smem(keys, nb, prefix, mask, need);
            compact_keys(keys, nb, prefix, need, put_block, wsum);
        }
    } else {
        // ------------------------------------------------ a long row: stream the passes
        // Up to P16_CAP blocks, the first pass also keeps every key's top 16 bits in
        // shared memory; the rest of the selection then reads only the scores of the
        // blocks whose top digit is the k-th key's or above (unless too many are).
        const bool pre16 = nb <= P16_CAP;
        uint16_t* const p16 = reinterpret_cast<uint16_t*>(keys);
        clear_hist();
        bool ok = stream_row(srow, nb, ring, bar0, seq, [&](const float* piece, int base, int n) {
            if (n == PIECE) { // 16-byte loads, 8-byte prefix stores: a thread takes 4 adjacent blocks
                float4 x[ROUNDS / 4];
#pragma unroll
                for (int e = 0; e < ROUNDS / 4; ++e) x[e] = reinterpret_cast<const float4*>(piece)[tid + e * THREADS];
#pragma unroll
                for (int e = 0; e < ROUNDS / 4; ++e) {
                    const uint32_t k0 = order_key(x[e].x), k1 = order_key(x[e].y), k2 = order_key(x[e].z),
                                   k3 = order_key(x[e].w);
                    if (pre16) // the lower index in the lower half of each word
                        reinterpret_cast<uint2*>(p16 + base)[tid + e * THREADS] =
                            make_uint2((k0 >> 16) | (k1 & 0xFFFF0000u), (k2 >> 16) | (k3 & 0xFFFF0000u));
                    atomicAdd(&hist[k0 >> 21], 1u);
                    atomicAdd(&hist[k1 >> 21], 1u);
                    atomicAdd(&hist[k2 >> 21], 1u);
                    atomicAdd(&hist[k3 >> 21], 1u);
                }
            } else {
                for (int j = tid; j < n; j += THREADS) {
                    const uint32_t k = order_key(piece[j]);
                    if (pre16) p16[base + j] = static_cast<uint16_t>(k >> 16);
                    atomicAdd(&hist[k >> 21], 1u);
                }
            }
        });
        if (!ok) return timed_out();
        __syncthreads();
        const int2 d = find_digit(hist, NBINS, need, wsum, sh);
        const uint32_t d1 = static_cast<uint32_t>(d.x) & (NBINS - 1);
        const int cand = static_cast<int>(hist[d1]); // keys in the bin of the k-th key
        need -= d.y;
        __syncthreads();
        bool done = false;
        if (pre16) {
            // Gather, in index order, every block whose key prefix is at or above
            // t16: the kept ones and the rest of the k-th key's bin. The bin is the
            // top 11-bit digit d1, or, when that leaves too many blocks, the 16-bit
            // prefix below it that holds the k-th key.
            uint32_t t16 = d1 << 5, pfx = d1 << 21, msk = 0x7FFu << 21;
            int ng = d.y + cand, needg = need;
            if (ng > CAND_CAP) {
                // key bits 20..16 of the blocks in bin d1, counted from the prefixes
                if (tid < 32) hist[tid] = 0u;
                __syncthreads();
                for (int i = tid; i < nb; i += THREADS) {
                    const uint32_t v = p16[i];
                    if ((v >> 5) == d1) atomicAdd(&hist[v & 31u], 1u);
                }
                __syncthreads();
                if (warp == 0) { // the 5-bit digit (from the top) that holds the need-th key
                    const int bin = 31 - lane;
                    const int cnt = static_cast<int>(hist[bin]);
                    int incl = cnt;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int v = __shfl_up_sync(FULL, incl, o);
                        if (lane >= o) incl += v;
                    }
                    if (incl - cnt < need && need <= incl) {
                        sh[0] = bin;
                        sh[1] = incl - cnt;
                        sh[2] = cnt;
                    }
                }
                __syncthreads();
                t16 = (d1 << 5) | static_cast<uint32_t>(sh[0]);
                pfx = t16 << 16;
                msk = 0xFFFF0000u;
                needg = need - sh[1];
                ng = d.y + sh[1] + sh[2];
                __syncthreads();
            }
            if (ng <= CAND_CAP) {
                uint32_t* const gl = keys + P16_CAP / 2;
                // (the bitmap in the kept-list area, free until the compaction)
                const int n = gather_ge16(p16, nb, t16, reinterpret_cast<uint32_t*>(kept), gl, CAND_CAP, wsum);
                __syncthreads();
                // their full keys, one score read each, over the prefixes (no longer read)
                for (int g = tid; g < n; g += THREADS) keys[g] = order_key(__ldg(srow + gl[g]));
                __syncthreads();
                select_in_smem(keys, n, pfx, msk, needg);
                compact_keys(keys, n, pfx, needg,
                             [&](int g, int rank) { put_block(static_cast<int>(gl[g]), rank); }, wsum);
                done = true;
            }
        }
        if (done) {
            // selected from the prefixes and the gathered keys
        } else if (cand <= KEYS_CAP) {
            // gather that bin's keys, in index order, into shared memory
            int ca = 0, cs = 0;
            ok = stream_row(srow, nb, ring, bar0, seq, [&](const float* piece, int base, int n) {
                scan_piece(n, [&](int j) { return order_key(piece[j]); },
                           [&](uint32_t) { return false; },
                           [&](uint32_t k, bool, int) { return (k >> 21) == d1; },
                           [&](int j, int rank) {
                               if (rank < KEYS_CAP) keys[rank] = order_key(piece[j]);
                           }, ca, cs, wsum);
            });
            if (!ok) return timed_out();
            __syncthreads();
            prefix = d1 << 21;
            mask = 0x7FFu << 21;
            select_in_smem(keys, cand, prefix, mask, need);
            const uint32_t thr = prefix;
            // mark the kept keys of the bin (ties: the first `need` in index order) with
            // 0xFFFFFFFF, a value order_key never returns; a piece's keys are all read
            // before its emits run
            ca = cs = 0;
            for (int base = 0; base < cand; base += PIECE)
                scan_piece(min(PIECE, cand - base), [&](int j) { return keys[base + j]; },
                           [&](uint32_t k) { return k == thr; },
                           [&](uint32_t k, bool eq, int rank) { return k > thr || (eq && rank < need); },
                           [&](int j, int) { keys[base + j] = KEPT; }, ca, cs, wsum);
            __syncthreads();
            // the compaction: bins above d1 are kept, bin d1's keys by their flag
            ca = cs = 0;
            ok = stream_row(srow, nb, ring, bar0, seq, [&](const float* piece, int base, int n) {
                scan_piece(n, [&](int j) { return order_key(piece[j]); },
                           [&](uint32_t k) { return (k >> 21) == d1; },
                           [&](uint32_t k, bool inbin, int rank) {
                               return (k >> 21) > d1 || (inbin && keys[rank] == KEPT);
                           },
                           [&](int j, int rank) { put_block(base + j, rank); }, ca, cs, wsum);
            });
            if (!ok) return timed_out();
        } else {
            // the bin is too large to gather: stream the remaining passes too
            prefix = d1 << 21;
            mask = 0x7FFu << 21;
            for (int pass = 1; pass < 3; ++pass) {
                const int shift = pass == 1 ? 10 : 0, bins = pass == 1 ? 2048 : 1024;
                clear_hist();
                ok = stream_row(srow, nb, ring, bar0, seq, [&](const float* piece, int, int n) {
                    for (int j = tid; j < n; j += THREADS) {
                        const uint32_t k = order_key(piece[j]);
                        if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & (bins - 1)], 1u);
                    }
                });
                if (!ok) return timed_out();
                __syncthreads();
                const int2 dd = find_digit(hist, bins, need, wsum, sh);
                prefix |= static_cast<uint32_t>(dd.x) << shift;
                mask |= static_cast<uint32_t>(bins - 1) << shift;
                need -= dd.y;
            }
            const uint32_t thr = prefix;
            int ca = 0, cs = 0;
            ok = stream_row(srow, nb, ring, bar0, seq, [&](const float* piece, int base, int n) {
                scan_piece(n, [&](int j) { return order_key(piece[j]); },
                           [&](uint32_t k) { return k == thr; },
                           [&](uint32_t k, bool eq, int rank) { return k > thr || (eq && rank < need); },
                           [&](int j, int rank) { put_block(base + j, rank); }, ca, cs, wsum);
            });
            if (!ok) return timed_out();
        }
    }
    write_kept(); // the kept blocks' slots, at their ranks
    // the tail tokens, after the k kept blocks
    for (int t = tid; t < tail; t += THREADS) out[kb * r + t] = slot_of(p, ptrow, nb * r + t, bad);
    if (bad && p.err != nullptr) atomicOr(p.err, QSA_DEVERR_SLOT_RANGE);
    (void)lane;
    (void)warp;
}

__global__ void __launch_bounds__(THREADS, 1) topk_expand_kernel(const Params p) { topk_row<false>(p); }
__global__ void __launch_bounds__(THREADS, 1) topk_cluster_kernel(const Params p) { topk_row<true>(p); }

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
    if ((reinterpret_cast<uintptr_t>(scores->data) & 15u) || scores->stride[0] % 4 != 0)
        return fail(QSA_ERR_MISALIGNED,
                    "scores rows must start on 16-byte boundaries (base 16-byte aligned, row "
                    "stride a multiple of 4)");
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

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(QSA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(QSA_ERR_CUDA, "device ordinal %d out of range", dev);
    static std::mutex mu;
    static bool smem_set[64] = {};
    static int sm_count[64] = {};
    static signed char cluster_ok[64][MAX_CLUSTER + 1] = {}; // 0 unknown, 1 fits, -1 does not
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!smem_set[dev]) {
            for (const void* k : {reinterpret_cast<const void*>(&topk_expand_kernel),
                                  reinterpret_cast<const void*>(&topk_cluster_kernel)}) {
                e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
                if (e != cudaSuccess)
                    return fail(QSA_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            }
            e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess)
                return fail(QSA_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
            smem_set[dev] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    cfg.attrs = attr;
    // Small batches: a cluster of C CTAs per row, the largest C whose clusters fill
    // no more than the SMs, when the longest row spans at least 8 pieces (below
    // that the cluster's barriers cost more than its parts save; 4 CTAs at most
    // below 16 pieces), each part's prefixes fit, and such a cluster can be resident.
    int C = 1;
    const long long nbmax_row = cap / r;
    const int cmax = nbmax_row >= 16LL * PIECE ? MAX_CLUSTER : (nbmax_row >= 8LL * PIECE ? 4 : 1);
    for (int c = cmax; c >= 2; c /= 2) {
        const long long part = (((nbmax_row + c - 1) / c) + 31) & ~31LL;
        if (bs * c > sm_count[dev] || part > P16_CAP) continue;
        std::lock_guard<std::mutex> lk(mu);
        if (cluster_ok[dev][c] == 0) {
            cfg.gridDim = dim3(static_cast<unsigned>(c));
            attr[1].val.clusterDim.x = static_cast<unsigned>(c);
            attr[1].val.clusterDim.y = attr[1].val.clusterDim.z = 1;
            cfg.numAttrs = 2;
            int clusters = 0;
            const cudaError_t q = cudaOccupancyMaxActiveClusters(&clusters, topk_cluster_kernel, &cfg);
            cluster_ok[dev][c] = (q == cudaSuccess && clusters >= 1) ? 1 : -1;
            if (q != cudaSuccess) (void)cudaGetLastError(); // a query that failed: no cluster launch
        }
        if (cluster_ok[dev][c] > 0) {
            C = c;
            break;
        }
    }
    cfg.gridDim = dim3(static_cast<unsigned>(bs * C));
    attr[1].val.clusterDim.x = static_cast<unsigned>(C);
    attr[1].val.clusterDim.y = attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = C > 1 ? 2 : 1;
    e = C > 1 ? cudaLaunchKernelEx(&cfg, topk_cluster_kernel, p) : cudaLaunchKernelEx(&cfg, topk_expand_kernel, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(QSA_ERR_CUDA, "top-k launch: %s", cudaGetErrorString(e));
    qsa_detail_set_error("");
    return QSA_OK;
}
