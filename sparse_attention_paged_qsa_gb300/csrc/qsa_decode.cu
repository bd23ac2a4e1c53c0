// Packed QSA decode for NVIDIA GB300 (sm_103a): one launch per call.
//
// What it computes (sglang PR #36845 "fix(qsa): restore SM121 correctness",
// "Changes" and "Optimized kernel"; sglang PR #37798 "quantized KV pools with
// dequant-on-gather", "Modifications"): for each sequence b and query head h
// (KV head g = h / 12), out = softmax(scale * q . K[I]^T) V[I] over the
// selected slots I = sel[cu[b] : cu[b+1]], duplicates and order kept, with the
// pool rows dequantised on gather. The page's design points kept here: the 12
// query heads of one KV head share one CTA so every K/V row is read once,
// tensor-core QK/PV with FP32 online-softmax state, split-KV across CTAs, and
// a same-launch FP32 log-sum-exp merge whose arrival counter is reset by the
// merging CTA. Lengths are read from cu_seqlens on the device.
//
// GB300 design:
//  * Persistent, balanced grid: the (sequence, KV head, token) space of the
//    live lengths is cut into gridDim.x equal token ranges on the device, so
//    a fixed (graph-captured) grid balances any length mix. Small batches
//    (at most four segments, or up to 64 of nearly equal length) get a whole
//    number of CTAs per segment, each CTA splitting its own segment when every
//    selection is long enough. A CTA whose range covers a whole (sequence, KV
//    head) segment writes the output directly. A segment cut between CTAs is
//    merged in the same launch: the CTA that holds its head at the end of its
//    range merges directly when the other contributors have already arrived
//    (they take their tickets as soon as their piece is done); otherwise the
//    last CTA to arrive merges partials it bulk-copies into shared memory; and
//    when each CTA holds one piece of one segment, all of that segment's CTAs
//    merge a slice each once the last has arrived. Launches are programmatic
//    dependent launches that wait for the previous grid before touching global
//    memory.
//  * Warp-specialised CTA (one per SM): four producer warps, one per SM
//    sub-partition, gather whole K/V rows with 16-byte cp.async into a
//    multi-stage shared-memory ring of 64-token stages, completing each stage
//    on an mbarrier; slot ids are prefetched a ring's depth ahead. Rows are
//    stored with a 16-byte-chunk XOR swizzle (chunk ^ row % 8) so the
//    ldmatrix reads below are bank-conflict free without padding.
//  * Eight consumer warps (two per sub-partition): QK on mma.m16n8k16 with
//    the 12 heads padded to 16 rows, 8 tokens per warp; a per-stage max
//    exchange with lazy rescaling (the reference max only moves when a score
//    exceeds it by 2^8); PV computed transposed, O^T = V^T P^T, with P split
//    into hi + lo columns of the PV operand type (24 columns: 12 heads x {hi,
//    lo}), so P keeps ~16 (bf16) or ~22 (f16) significant bits; each warp owns
//    32 of the 256 output dims.
//  * Quantised pools are converted exactly, in registers, from the raw stage:
//    a K row's ldmatrix word (4 codes of 8 bits, or 8 of 4 bits) becomes the f16
//    pairs of an MMA B fragment (the k-slots follow the word's codes and Q is
//    loaded in that order; Q is rescaled per head by a power of two so it
//    converts to f16 exactly), and ldmatrix.trans of the raw V rows gives each
//    lane one code of two consecutive tokens, the f16 (fp8, int8) or bf16 (int4,
//    grouped) pairs of the PV A fragment (the warp's 32 output dims are spread
//    over its two m-tiles accordingly). Integers use magic-number conversions,
//    e4m3 the hardware conversion; no converted tile and no shared-memory round
//    trip. Per-slot scales scale the scores (K) and the probabilities (V) in
//    FP32 (int8 keeps a per-head power-of-two offset so that P times its V scale
//    fits f16); per-pool fp8 scales fold into constants. The tiered pool, whose
//    rows mix two formats, is converted in shared memory by the consuming warp.
//    Grouped pools (binary16 scale per 64 / 32 channels): QK accumulates each
//    channel group's k-steps apart and adds them with the token's group scale;
//    each consumer warp's 32 PV dims lie in one group, so the warp rebuilds its
//    own P^T with that group's per-token V scales from an FP32 copy of P.
//  * Every wait is bounded; bad slot ids / cu_seqlens set a sticky error
//    word and are clamped, never trapped.

#include <cuda.h> // driver types only (CUcontext, CUresult); nothing links libcuda
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <initializer_list>
#include <mutex>
#include <string>

#include "qsa.h"

namespace qsa {

constexpr int D = 256;
constexpr int GROUP = 12;                   // query heads per KV head
constexpr int T = 64;                       // tokens per pipeline stage
constexpr int NW = 8;                       // consumer warps
constexpr int NP = 4;                       // producer warps
constexpr int NCT = NW * 32;                // consumer threads
constexpr int NTHREADS = (NW + NP) * 32;
constexpr int TPW = T / NW;                 // QK tokens per consumer warp (one n8 tile)
constexpr int DPW = D / NW;                 // PV output dims per consumer warp
constexpr int MT = DPW / 16;                // 16-dim m-tiles per consumer warp
constexpr int KK = T / 16;                  // PV k-steps per stage
constexpr int TPP = T / NP;                 // tokens gathered per producer warp
constexpr int BF_ROW = D * 2;               // bf16 row bytes (swizzled, unpadded)
constexpr int Q_RS = 528;                   // Q tile row stride (512 + 16 pad)
constexpr int PRS = T * 2 + 16;             // P^T row stride (bytes)
constexpr int PFS = T + 8;                  // FP32 P row stride (floats; 72 = 8 mod 32 banks)
constexpr float TAU = 8.0f;                 // lazy-rescale threshold (log2 units)
constexpr int MAX_BS = 128;
constexpr int MAX_CAPACITY = 2055;
constexpr int MIN_TOKENS_PER_CTA = 64;
constexpr unsigned FEW_SEGMENTS = 4;        // up to this many (sequence, KV head) segments ...
constexpr unsigned UNIFORM_SEGMENTS = 64;   // ... or this many of nearly equal length ...
constexpr unsigned MAX_FANIN = 16;          // ... each gets a whole number (<= this) of CTAs
constexpr int PART_BYTES = 12416;           // fp32 O[12][256] + m[12] + l[12], 128-byte multiple
constexpr int MERGE_BATCH = 6;             // partials per bulk-copy batch of the split merge (at most)
constexpr long long WAIT_NS = 2000000000LL; // bounded-wait limit (2 s)
constexpr int BAR_CONSUMERS = 1;            // named barrier id (2..5: consumer warp pairs)
// Register split between the warp roles (setmaxnreg) of the pools whose consumer
// warps set the pace (the dequantising ones): the block is launched with
// LAUNCH_REGS per thread; the producer warpgroup gives registers back and the two
// consumer warpgroups take them, the shares adding up to the launch's total. The
// bf16 pool, bound by its producers' gather, keeps the even split.
constexpr int LAUNCH_REGS = 65536 / NTHREADS / 8 * 8;   // 168
constexpr int PRODUCER_REGS = 56, CONSUMER_REGS = 224;
static_assert(NP * PRODUCER_REGS + NW * CONSUMER_REGS <= (NP + NW) * LAUNCH_REGS, "register split");
static_assert(NP == 4 && NW == 8, "the split works on whole warpgroups");
static_assert(TPW == 8 && MT >= 1 && TPP <= 32, "tile shape");
static_assert(PART_BYTES >= (GROUP * D + 2 * GROUP) * 4, "partial slot size");
static_assert(PART_BYTES % 16 == 0, "bulk copies move 16-byte multiples");

// ROWB: pool row bytes; STAGES: ring depth; RQ: codes are converted in
// registers from the raw stage (K as MMA B fragments, V as PV A fragments), no
// converted tiles; QK_F16: QK runs on f16 operands (exact integer / e4m3 codes,
// Q rescaled per head by a power of two); PV_F16: PV runs on f16
// operands (for int8, with a per-head power-of-two offset that keeps P * s_v in
// range), else bf16; SCALES: per-slot scales (fp32 per (slot, KV head), or
// binary16 per (slot, KV head, channel group) when GROUPS > 0); NIB4: 4-bit
// codes, NIB_OFFSET: stored as code + 8 (else two's complement); TIER: each row
// is an int8_g64 ring row or an int4_g32 pool row, by the owner table; the
// consuming warps widen the int4 rows to int8 codes in shared memory, so the
// stage reads as int8 rows with 32-channel scales (a ring row's 64-channel scales
// serve both of their 32-channel halves).
template <int FMT> struct Traits;
template <> struct Traits<QSA_KV_BF16> {
    static constexpr int ROWB = 512, STAGES = 3, GROUPS = 0;
    static constexpr bool RQ = false, SCALES = false, QK_F16 = false;
    static constexpr bool PV_F16 = false, NIB4 = false, NIB_OFFSET = false, TIER = false;
};
template <> struct Traits<QSA_KV_FP8_E4M3> {
    static constexpr int ROWB = 256, STAGES = 4, GROUPS = 0;
    static constexpr bool RQ = true, SCALES = false, QK_F16 = true;
    static constexpr bool PV_F16 = true, NIB4 = false, NIB_OFFSET = false, TIER = false;
};
template <> struct Traits<QSA_KV_INT8> {
    static constexpr int ROWB = 256, STAGES = 4, GROUPS = 0;
    static constexpr bool RQ = true, SCALES = true, QK_F16 = true;
    static constexpr bool PV_F16 = true, NIB4 = false, NIB_OFFSET = false, TIER = false;
};
template <> struct Traits<QSA_KV_INT4> {
    static constexpr int ROWB = 128, STAGES = 8, GROUPS = 0;
    static constexpr bool RQ = true, SCALES = true, QK_F16 = true;
    static constexpr bool PV_F16 = false, NIB4 = true, NIB_OFFSET = false, TIER = false;
};
template <> struct Traits<QSA_KV_INT8_G64> {
    static constexpr int ROWB = 256, STAGES = 4, GROUPS = 4;
    static constexpr bool RQ = true, SCALES = true, QK_F16 = true;
    static constexpr bool PV_F16 = false, NIB4 = false, NIB_OFFSET = false, TIER = false;
};
template <> struct Traits<QSA_KV_INT4_G32> {
    static constexpr int ROWB = 128, STAGES = 10, GROUPS = 8;
    static constexpr bool RQ = true, SCALES = true, QK_F16 = true;
    static constexpr bool PV_F16 = false, NIB4 = true, NIB_OFFSET = true, TIER = false;
};
template <> struct Traits<QSA_KV_INT8RING_INT4> {
    static constexpr int ROWB = 256, STAGES = 3, GROUPS = 8;
    static constexpr bool RQ = true, SCALES = true, QK_F16 = true;
    static constexpr bool PV_F16 = false, NIB4 = false, NIB_OFFSET = true, TIER = true;
};

template <int FMT> struct Layout {
    using Tr = Traits<FMT>;
    static constexpr int STAGE_KV = T * Tr::ROWB;
    static constexpr int SC_TOK = Tr::GROUPS ? Tr::GROUPS * 2 : 4; // scale bytes per token
    static constexpr int STAGE_SC = Tr::SCALES ? 2 * T * SC_TOK : 0;
    static constexpr int STAGE_FLAGS = Tr::TIER ? T * 4 : 0;    // per token: 1 = ring row
    static constexpr int STAGE_BYTES = 2 * STAGE_KV + STAGE_SC + STAGE_FLAGS;
    static constexpr int PF = Tr::STAGES;       // slot-id prefetch distance (stages)
    static constexpr int R = PF + 1;            // slot-id ring entries
    static constexpr int off_stage = 0;
    // tiered pools: the int4 rows' V codes widened to int8 [T][256] (swizzled);
    // consumer warp w owns 16-byte chunks 2w, 2w + 1 of every row
    static constexpr int off_vexp = off_stage + Tr::STAGES * STAGE_BYTES;
    static constexpr int vexp_bytes = Tr::TIER ? T * 256 : 0;
    static constexpr int off_q = off_vexp + vexp_bytes;
    static constexpr int off_p = off_q + 2 * 16 * Q_RS;
    // P^T hi/lo (two buffers); grouped pools: FP32 P [2][12][PFS], from which each
    // warp builds its PV B fragments in registers (32-channel groups), or each pair
    // of warps sharing a 64-channel group one scaled P^T per stage [4][2][24][PRS]
    static constexpr int off_pw = off_p + 2 * GROUP * PFS * 4;
    static constexpr int p_bytes = Tr::GROUPS == 4 ? 2 * GROUP * PFS * 4 + 8 * 24 * PRS
                                   : Tr::GROUPS    ? 2 * GROUP * PFS * 4
                                                   : 2 * 24 * PRS;
    static constexpr int off_red = off_p + p_bytes;
    static constexpr int off_mref = off_red + 2 * NW * 16 * 4;
    static constexpr int off_lred = off_mref + 2 * 16 * 4;
    // per-slot V scales (f16 PV): per-warp maxima of the scale offsets t, and
    // the per-head offsets E (double-buffered like mref)
    static constexpr bool NUM_REF = Tr::SCALES && Tr::GROUPS == 0 && Tr::PV_F16;
    static constexpr int off_nred = off_lred + NW * 16 * 4;
    static constexpr int off_eref = off_nred + (NUM_REF ? NW * 16 * 4 : 0);
    static constexpr int off_ring = off_eref + (NUM_REF ? 2 * 16 * 4 : 0);
    // tiered pools: per producer warp, its tokens listed by tier (16 hot, 16 cold)
    static constexpr int off_tlist = off_ring + R * T * 4;
    static constexpr int off_segL = off_tlist + (Tr::TIER ? NP * 32 * 4 : 0);
    static constexpr int off_segSrc = off_segL + (MAX_BS + 4) * 4;
    static constexpr int off_segP = off_segSrc + (MAX_BS + 4) * 4;
    static constexpr int off_misc = off_segP + (MAX_BS + 4) * 4;
    static constexpr int off_bar = off_misc + 64 * 4;
    static constexpr int n_bars = 2 * Tr::STAGES + 6; // stages full/empty, Q full/empty, merge
    static constexpr int TOTAL = off_bar + n_bars * 8;
    static_assert(TOTAL <= 227 * 1024, "shared memory budget");
    // the split merge stages two batches of up to MB partials over the (then
    // idle) stage ring, below the Q tiles, then this CTA's own partial of a
    // directly merged segment head
    static constexpr int MB = (off_q / PART_BYTES - 1) / 2 < MERGE_BATCH ? (off_q / PART_BYTES - 1) / 2
                                                                          : MERGE_BATCH;
    static_assert(MB >= 2, "merge buffers");
    static constexpr int off_stash = 2 * MB * PART_BYTES;
    static_assert(off_stash + PART_BYTES <= off_q, "direct-merge stash");
    static_assert(STAGE_BYTES % 128 == 0 && off_vexp % 128 == 0 && off_q % 16 == 0, "alignment");
    static_assert(off_p % 16 == 0 && off_pw % 16 == 0 && off_red % 16 == 0 && off_bar % 8 == 0,
                  "alignment");
};

struct Params {
    const __nv_bfloat16* q;
    long long q_sb, q_sh;
    const uint8_t* kpool;
    const uint8_t* vpool;
    long long num_slots;
    const void* k_scale; // fp32 (fp8: [1]; int8/int4: [slots * Hkv]) or binary16 [slots * Hkv * GROUPS]
    const void* v_scale;
    const int* sel;
    long long n_sel;
    const int* cu;
    __nv_bfloat16* out;
    long long o_sb, o_sh;
    int* err;
    int* cnt;
    uint8_t* part;
    int bs, Hkv, capacity;
    float scale_log2; // softmax_scale * log2(e)
    // tiered pools: int8_g64 ring rows [R, Hkv, 256], binary16 scales [R, Hkv, 4], owner [R]
    const uint8_t* kring;
    const uint8_t* vring;
    const void* kring_scale;
    const void* vring_scale;
    const int* owner;
    int ring_mask; // R - 1
#ifdef QSA_TEST_HOOKS
    int stall_stage; // CTA 0's producers leave this stage incomplete (-1: off)
#endif
};

// Byte offset of 16-byte chunk `chunk` of row `row` in a swizzled row buffer.
template <int ROWB>
__device__ __forceinline__ int swz(int row, int chunk) {
    return row * ROWB + ((chunk ^ (row & 7)) << 4);
}

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    [[maybe_unused]] uint64_t state;
    asm volatile("mbarrier.arrive.shared::cta.b64 %0, [%1];" : "=l"(state) : "r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    [[maybe_unused]] uint64_t state;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 %0, [%1], %2;"
                 : "=l"(state)
                 : "r"(bar), "r"(bytes)
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

// Wait for the phase with `parity` of an mbarrier, for at most WAIT_NS. On
// timeout, record QSA_DEVERR_TIMEOUT, raise the CTA abort flag and return false.
// Inline (a call would make the caller save its live registers around it in the
// hot loop); the error path alone is out of line.
__device__ __noinline__ void wait_timed_out(int* err, volatile int* abort_flag) {
    atomicOr(err, QSA_DEVERR_TIMEOUT);
    *abort_flag = 1;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* err,
                                          volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > (unsigned long long)WAIT_NS) {
                wait_timed_out(err, abort_flag);
                return false;
            }
        }
    }
}

// Wait for bulk copies this CTA issued: bounded like mbar_wait, but blind to the
// abort flag (the copies must land before the CTA may exit).
__device__ __noinline__ bool mbar_wait_copies(uint32_t bar, uint32_t parity, int* err) {
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 63 && globaltimer() - t0 > (unsigned long long)WAIT_NS) {
            atomicOr(err, QSA_DEVERR_TIMEOUT);
            return false;
        }
    }
}

// Wait until a split counter reaches `target` (acquire: the partials stored
// before the increments are visible), for at most WAIT_NS.
__device__ __noinline__ bool wait_count(const int* cnt, int target, int* err) {
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 0;; ++it) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
        if (v >= target) return true;
        if ((it & 63) == 63 && globaltimer() - t0 > (unsigned long long)WAIT_NS) {
            atomicOr(err, QSA_DEVERR_TIMEOUT);
            return false;
        }
        __nanosleep(32);
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

__device__ __forceinline__ void regs_producer() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(PRODUCER_REGS));
}
__device__ __forceinline__ void regs_consumer() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(CONSUMER_REGS));
}

__device__ __forceinline__ int ld_relaxed(const int* ptr) {
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// L2 eviction priorities. The pools with per-slot scales read each K/V row once
// per call but each 32-byte scale sector twice (the sequence's two KV heads sit
// side by side in it, read by different stages or CTAs): rows go first, scales
// last, so the second read of a sector finds it in L2.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void cp_async4_l2(uint32_t dst, const void* src, uint64_t pol) {
    asm volatile("cp.async.ca.shared.global.L2::cache_hint [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void cp_async8_l2(uint32_t dst, const void* src, uint64_t pol) {
    asm volatile("cp.async.ca.shared.global.L2::cache_hint [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void cp_async16_l2(uint32_t dst, const void* src, uint64_t pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_all() {
    asm volatile("fence.proxy.async;" ::: "memory");
}
__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Named barrier over the consumer warps that also ORs a predicate across them.
__device__ __forceinline__ bool consumer_sync_or(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "n"(BAR_CONSUMERS), "n"(NCT)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(BAR_CONSUMERS), "n"(NCT) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                        uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                          uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t& r0, uint32_t& r1, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}

// D += A(16x16, row) * B(16x8, col), bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D += A(16x16, row) * B(16x8, col), f16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <bool F16>
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    if constexpr (F16)
        mma_f16(d, a, b0, b1);
    else
        mma_bf16(d, a, b0, b1);
}

__device__ __forceinline__ void ldsm_x2_t(uint32_t& r0, uint32_t& r1, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float f16_lo(uint32_t v) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(v & 0xFFFFu)));
}
__device__ __forceinline__ float f16_hi(uint32_t v) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(v >> 16)));
}
// Two probabilities as a packed pair of the PV operand type, plus the
// rounding residual pair (the "lo" term of the hi + lo split).
template <bool F16>
__device__ __forceinline__ void split_pair(float a, float b, uint32_t& hi, uint32_t& lo) {
    if constexpr (F16) {
        hi = pack_f16x2(a, b);
        lo = pack_f16x2(a - f16_lo(hi), b - f16_hi(hi));
    } else {
        hi = pack_bf16x2(a, b);
        lo = pack_bf16x2(a - bf16_lo(hi), b - bf16_hi(hi));
    }
}

// ------------------------------------------------------------ exact dequant
//
// Every conversion below is exact: the codes (|int8| <= 128, |int4| <= 8,
// e4m3 with 4 significant bits and |x| <= 448) are representable in f16 and
// bf16. Integers use the magic-number construction: a byte u placed in the
// low mantissa bits of a float whose exponent gives a mantissa step of 1 reads
// as (magic + u); subtracting (magic + offset) leaves the code.

__device__ __forceinline__ uint32_t sub_f16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t sub_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// 4 int8 codes -> 2 f16x2: 0x64uu is 1024 + u; u = code ^ 0x80 = code + 128.
__device__ __forceinline__ void i8x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t x = w ^ 0x80808080u;
    lo = sub_f16x2(__byte_perm(x, 0x64646464u, 0x4140), 0x64806480u); // - 1152
    hi = sub_f16x2(__byte_perm(x, 0x64646464u, 0x4342), 0x64806480u);
}

// 8 int4 codes (channel 2i in the low nibble) -> 4 packed pairs, f16 or bf16:
// nibble u = code + 8 (offset-binary storage as it is; two's complement
// code ^ 8) under the magic 1024 (f16) or 128 (bf16).
template <bool F16, bool OFFSET>
__device__ __forceinline__ void i4x8_to(uint32_t w, uint32_t* o) {
    constexpr uint32_t MAGIC = F16 ? 0x64006400u : 0x43004300u;
    constexpr uint32_t BIAS = F16 ? 0x64086408u : 0x43084308u; // 1032 / 136
    const uint32_t x = OFFSET ? w : w ^ 0x88888888u;
    const uint32_t hs = x >> 4;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t t = __byte_perm(x, hs, k | ((4 + k) << 8));
        const uint32_t v = (t & 0x000F000Fu) | MAGIC;
        o[k] = F16 ? sub_f16x2(v, BIAS) : sub_bf16x2(v, BIAS);
    }
}

// 4 e4m3fn codes -> 2 f16x2 with the hardware conversion (exact).
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// ---------------------------------------------- register-level dequant (RQ pools)
//
// ldmatrix.trans of raw 8-bit rows (8 tokens x 16 codes as 8 x 8 pairs) gives a
// lane the codes [v(2t, 2g), v(2t, 2g+1), v(2t+1, 2g), v(2t+1, 2g+1)] (tokens 2t,
// 2t+1 of the 8, codes 2g, 2g+1 of the 16). Bytes 0, 2 are one code of two
// consecutive tokens: a PV A-fragment pair for code 2g; bytes 1, 3 for code 2g+1.
// `odd` picks which. Exact, as in the shared-memory conversions above.
template <int FMT, bool F16>
__device__ __forceinline__ uint32_t pair8(uint32_t w, bool odd) {
    if constexpr (FMT == QSA_KV_FP8_E4M3) {
        uint32_t lo, hi;
        e4m3x4_to_f16(__byte_perm(w, 0u, 0x3120), lo, hi);
        return odd ? hi : lo;
    } else if constexpr (F16) {
        return sub_f16x2(__byte_perm(w ^ 0x80808080u, 0x64646464u, odd ? 0x4341 : 0x4240), 0x64806480u);
    } else {
        const uint32_t t = __byte_perm(w, 0u, odd ? 0x4341 : 0x4240);
        return sub_bf16x2((t & 0x007F007Fu) | 0x43004300u, (t & 0x00800080u) | 0x43004300u);
    }
}

// ldmatrix.trans of raw 4-bit rows: bytes 0, 2 hold codes 4g, 4g+1 (low, high
// nibble) of tokens 2t, 2t+1 and bytes 1, 3 codes 4g+2, 4g+3. Code 4g + j as a
// pair of the two tokens (f16 or bf16); w already xor-ed with 0x88888888 for
// two's-complement codes, so every nibble reads as code + 8.
template <bool F16>
__device__ __forceinline__ uint32_t pair4(uint32_t w, int j) {
    constexpr uint32_t MAGIC = F16 ? 0x64006400u : 0x43004300u;
    constexpr uint32_t BIAS = F16 ? 0x64086408u : 0x43084308u; // 1032 / 136
    const uint32_t v = ((w >> (4 * j)) & 0x000F000Fu) | MAGIC;
    return F16 ? sub_f16x2(v, BIAS) : sub_bf16x2(v, BIAS);
}

// 16 bytes of an int4 row (32 codes; byte k holds code 2k in its low nibble and
// 2k + 1 in its high one) -> the same 32 codes as int8 values 16 * code (two
// 16-byte chunks): a two's-complement nibble in the high half of a byte reads as
// 16 times its value, so no per-byte carry or sign extension is needed; the
// caller folds the factor 1/16 into the token's scales. Nibbles stored as code +
// 8 (OFFSET) become two's complement by flipping bit 3.
template <bool OFFSET>
__device__ __forceinline__ void widen16_i4x32(const uint4 raw, uint4& o0, uint4& o1) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t r[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t v = OFFSET ? w[k] ^ 0x88888888u : w[k];
        const uint32_t hi = v & 0xF0F0F0F0u, lo = (v << 4) & 0xF0F0F0F0u; // codes 2j+1 / 2j of byte j
        r[2 * k] = __byte_perm(lo, hi, 0x5140);     // codes 8k .. 8k+3
        r[2 * k + 1] = __byte_perm(lo, hi, 0x7362); // codes 8k+4 .. 8k+7
    }
    o0 = make_uint4(r[0], r[1], r[2], r[3]);
    o1 = make_uint4(r[4], r[5], r[6], r[7]);
}

// Q fragments of the register-dequant pools (f16, k16 steps), built from the bf16
// Q tile (rows = heads, 12 real and 4 zero rows, row stride Q_RS). Lane (g, t)
// holds rows g and g + 8. A K B fragment comes from one ldmatrix word of the raw
// rows, so the k-slots follow the codes of that word:
//  * 8-bit codes: a word holds codes 4t .. 4t+3 of a 16-code chunk (the chunk of
//    step c); k-slots {2t, 2t+1, 8+2t, 9+2t} take codes {4t .. 4t+3}: qa[c] = (row g:
//    16c+4t,+1; row g+8: same; row g: 16c+4t+2,+3; row g+8: same).
//  * 4-bit codes: a word holds codes 8t .. 8t+7 of a 32-code chunk c, the pairs
//    (8t, 8t+1), (8t+2, 8t+3) feed step 2c and (8t+4, 8t+5), (8t+6, 8t+7) step 2c+1.
// Each row is scaled by a power of two that brings its largest |q| into
// [2^14, 2^15), so the bf16 values are exact in f16; mul = the inverse factor.
template <int FMT>
__device__ __forceinline__ void build_q_rq(const uint8_t* qt, int lane, uint32_t (&qa)[16][4],
                                           float& mul_a, float& mul_b) {
    using Tr = Traits<FMT>;
    const int g = lane >> 2, t = lane & 3;
    const uint8_t* const ra = qt + g * Q_RS;
    const uint8_t* const rb = qt + (g + 8) * Q_RS;
    if constexpr (!Tr::NIB4) {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const uint2 a = *reinterpret_cast<const uint2*>(ra + (16 * c + 4 * t) * 2);
            const uint2 b = *reinterpret_cast<const uint2*>(rb + (16 * c + 4 * t) * 2);
            qa[c][0] = a.x;
            qa[c][1] = b.x;
            qa[c][2] = a.y;
            qa[c][3] = b.y;
        }
    } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 a = *reinterpret_cast<const uint4*>(ra + (32 * c + 8 * t) * 2);
            const uint4 b = *reinterpret_cast<const uint4*>(rb + (32 * c + 8 * t) * 2);
            qa[2 * c][0] = a.x;
            qa[2 * c][1] = b.x;
            qa[2 * c][2] = a.y;
            qa[2 * c][3] = b.y;
            qa[2 * c + 1][0] = a.z;
            qa[2 * c + 1][1] = b.z;
            qa[2 * c + 1][2] = a.w;
            qa[2 * c + 1][3] = b.w;
        }
    }
    float ma = 0.f, mb = 0.f; // row maxima: rows g (registers 0, 2) and g + 8 (1, 3)
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        ma = fmaxf(ma, fmaxf(fmaxf(fabsf(bf16_lo(qa[c][0])), fabsf(bf16_hi(qa[c][0]))),
                             fmaxf(fabsf(bf16_lo(qa[c][2])), fabsf(bf16_hi(qa[c][2])))));
        mb = fmaxf(mb, fmaxf(fmaxf(fabsf(bf16_lo(qa[c][1])), fabsf(bf16_hi(qa[c][1]))),
                             fmaxf(fabsf(bf16_lo(qa[c][3])), fabsf(bf16_hi(qa[c][3])))));
    }
    ma = fmaxf(ma, __shfl_xor_sync(0xFFFFFFFFu, ma, 1));
    ma = fmaxf(ma, __shfl_xor_sync(0xFFFFFFFFu, ma, 2));
    mb = fmaxf(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 1));
    mb = fmaxf(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 2));
    auto shift_of = [](float m) {
        const int e = static_cast<int>((__float_as_uint(m) >> 23) & 0xFFu) - 127;
        const int sh = m > 0.f ? e - 14 : 0;
        return sh < -100 ? -100 : (sh > 100 ? 100 : sh);
    };
    auto pow2 = [](int e) { return __uint_as_float(static_cast<uint32_t>(127 + e) << 23); };
    const int sa = shift_of(ma), sb = shift_of(mb);
    const float da = pow2(-sa), db = pow2(-sb);
    mul_a = pow2(sa);
    mul_b = pow2(sb);
#pragma unroll
    for (int c = 0; c < 16; ++c)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float d = (j & 1) ? db : da;
            qa[c][j] = pack_f16x2(bf16_lo(qa[c][j]) * d, bf16_hi(qa[c][j]) * d);
        }
}

// ------------------------------------------------------------ work cursor

// Walks the CTA's token range [t, t_end) of the flattened (b, g, j) space in
// stages of at most T tokens that never straddle a (b, g) segment.
struct Cursor {
    long long t;
    int b, g, j, j1, kseg;
    bool segfirst;
};

// The flattened work space is head-major: KV head g's tokens of all sequences,
// [g NT, (g + 1) NT) with NT = segP[bs] the live tokens per head, sequence b's
// at offset segP[b] within it. The CTAs working on head 0 and head 1 of the same
// slots then run at the same time, so the second read of what the heads share
// (slot ids, the 32-byte scale sector of a slot's two heads) hits L2.
__device__ __forceinline__ void cursor_init(Cursor& c, long long t, long long t_end,
                                            const int* segL, const int* segP, int bs, int Hkv) {
    const long long NT = segP[bs];
    c.g = static_cast<int>(t / NT);
    const long long r = t - (long long)c.g * NT;
    int lo = 0, hi = bs - 1; // largest b with segP[b] <= r (a sequence with tokens left)
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (segP[mid] <= r)
            lo = mid;
        else
            hi = mid - 1;
    }
    c.b = lo;
    c.j = static_cast<int>(r - segP[lo]);
    c.t = t;
    c.j1 = static_cast<int>(min((long long)segL[lo], c.j + (t_end - t)));
    c.kseg = 0;
    c.segfirst = true;
}

__device__ __forceinline__ int cursor_n(const Cursor& c) { return min(T, c.j1 - c.j); }

__device__ __forceinline__ void cursor_advance(Cursor& c, long long t_end, const int* segL, int bs) {
    const int n = cursor_n(c);
    c.t += n;
    c.j += n;
    c.segfirst = false;
    if (c.j >= c.j1 && c.t < t_end) {
        do {
            ++c.b;
        } while (c.b < bs && segL[c.b] == 0);
        if (c.b >= bs) { // the next KV head, from its first sequence with tokens
            ++c.g;
            c.b = 0;
            while (segL[c.b] == 0) ++c.b;
        }
        c.j = 0;
        c.j1 = static_cast<int>(min((long long)segL[c.b], t_end - c.t));
        ++c.kseg;
        c.segfirst = true;
    }
}

// CTA index whose range holds flattened token t; first token of CTA c. All
// operands stay below 2^28 (N <= 128 * 2 * 2055 tokens, G <= #SMs), so 32-bit
// unsigned arithmetic is exact.
__device__ __forceinline__ unsigned cta_of(unsigned t, unsigned N, unsigned G) {
    return ((t + 1u) * G - 1u) / N;
}
__device__ __forceinline__ unsigned cta_begin(unsigned c, unsigned N, unsigned G) {
    return c * N / G;
}

// ------------------------------------------------------------------ kernel

template <int FMT>
__global__ void __launch_bounds__(NTHREADS, 1) qsa_decode_kernel(const Params p) {
    using Tr = Traits<FMT>;
    using Ly = Layout<FMT>;
    extern __shared__ __align__(1024) uint8_t smem[];

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    int* segL = reinterpret_cast<int*>(smem + Ly::off_segL);
    int* segSrc = reinterpret_cast<int*>(smem + Ly::off_segSrc);
    int* segP = reinterpret_cast<int*>(smem + Ly::off_segP);
    int* misc = reinterpret_cast<int*>(smem + Ly::off_misc);
    volatile int* abort_flag = misc;
    const uint32_t bar0 = smem_u32(smem + Ly::off_bar);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (Tr::STAGES + s); };
    auto qfull_bar = [&](int i) { return bar0 + 8u * (2 * Tr::STAGES + i); };
    auto qempty_bar = [&](int i) { return bar0 + 8u * (2 * Tr::STAGES + 2 + i); };
    auto merge_bar = [&](int i) { return bar0 + 8u * (2 * Tr::STAGES + 4 + i); };

    // ---------------------------------------------------------------- setup
    if (tid == 0) {
        for (int s = 0; s < Tr::STAGES; ++s) {
            // every producer lane arrives twice: once when its cp.async copies land
            // (noinc), once in program order after its shared-memory stores
            mbar_init(full_bar(s), NP * 64);
            mbar_init(empty_bar(s), NW);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(qfull_bar(i), 1);
            mbar_init(qempty_bar(i), NW);
            mbar_init(merge_bar(i), 1);
        }
        misc[0] = 0;
        // merge bookkeeping of the consumer loop (see mstate below)
        misc[8] = -1;  // pend0
        misc[9] = -1;  // pend1
        misc[10] = -1; // dsid
        misc[11] = 0;  // dn
        misc[12] = -1; // ticket0 (thread 0)
        fence_mbarrier_init();
    }
    // zero the padding rows 12..15 of both Q tiles (rows of the 16-row MMA tile)
    for (int i = tid; i < 2 * 4 * (Q_RS / 16); i += NTHREADS) {
        const int buf = i / (4 * (Q_RS / 16));
        const int rem = i % (4 * (Q_RS / 16));
        uint4* dst = reinterpret_cast<uint4*>(smem + Ly::off_q + buf * 16 * Q_RS +
                                              (12 + rem / (Q_RS / 16)) * Q_RS) +
                     rem % (Q_RS / 16);
        *dst = make_uint4(0, 0, 0, 0);
    }
    // Everything above touched shared memory only; global memory is read and
    // written from here on, after the previous grid in the stream has finished.
    griddep_wait();
    griddep_launch_dependents();
    // sanitised lengths, index offsets and prefix sums (warp 0; bs <= 128)
    if (warp == 0) {
        int bad = 0, Ls[4], run = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int b = lane * 4 + k;
            int L = 0;
            if (b < p.bs) {
                const long long lo = p.cu[b], hi = p.cu[b + 1];
                if (lo < 0 || hi < lo || hi > p.n_sel || hi - lo > p.capacity) bad = 1;
                const long long src = lo < 0 ? 0 : lo;
                long long Ll = hi - lo;
                Ll = Ll < 0 ? 0 : Ll;
                Ll = Ll > p.capacity ? p.capacity : Ll;
                const long long room = p.n_sel - src;
                Ll = Ll > room ? (room < 0 ? 0 : room) : Ll;
                L = static_cast<int>(Ll);
                segL[b] = L;
                segSrc[b] = static_cast<int>(src < p.n_sel ? src : 0);
            }
            Ls[k] = L;
            run += L;
        }
        int incl = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
            if (lane >= off) incl += v;
        }
        int excl = incl - run;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int b = lane * 4 + k;
            if (b < p.bs) segP[b] = excl;
            excl += Ls[k];
        }
        const int total = __shfl_sync(0xFFFFFFFFu, incl, 31);
        int lmax = max(max(Ls[0], Ls[1]), max(Ls[2], Ls[3]));
        int lmin = 0x7fffffff;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (lane * 4 + k < p.bs) lmin = min(lmin, Ls[k]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            lmax = max(lmax, __shfl_xor_sync(0xFFFFFFFFu, lmax, off));
            lmin = min(lmin, __shfl_xor_sync(0xFFFFFFFFu, lmin, off));
        }
        if (lane == 0) {
            segP[p.bs] = total;
            segL[p.bs] = 1; // sentinel for the segment walk
            misc[20] = lmax; // the longest selection
            misc[23] = lmin; // the shortest
        }
        bad = __any_sync(0xFFFFFFFFu, bad);
        if (bad && lane == 0 && blockIdx.x == 0) atomicOr(p.err, QSA_DEVERR_CU_SEQLENS);
    }
    __syncthreads();

    const int Hkv = p.Hkv;
    const unsigned N = static_cast<unsigned>(Hkv) * static_cast<unsigned>(segP[p.bs]);

    // empty selections -> zero rows (spread over all CTAs)
    if (warp < NW) {
        for (int s = blockIdx.x; s < p.bs * Hkv; s += gridDim.x) {
            const int b = s / Hkv, g = s % Hkv;
            if (segL[b] != 0) continue;
            for (int ch = tid; ch < GROUP * (D / 8); ch += NCT) {
                const int h = ch / (D / 8), d0 = (ch % (D / 8)) * 8;
                *reinterpret_cast<uint4*>(p.out + b * p.o_sb + (g * GROUP + h) * p.o_sh + d0) =
                    make_uint4(0, 0, 0, 0);
            }
        }
    }
    if (N == 0) return;
    // Short selections (every one fits a 64-token stage): the CTAs split whole
    // (sequence, KV head) segments, [c S / G, (c + 1) S / G) of the S = bs Hkv in
    // head-major order, so that no segment is cut and nothing is merged.
    const unsigned S_all = static_cast<unsigned>(p.bs * Hkv);
    const bool whole = misc[20] <= T;
    unsigned G = (N + MIN_TOKENS_PER_CTA - 1) / MIN_TOKENS_PER_CTA;
    G = G < gridDim.x ? G : gridDim.x;
    if (whole) G = S_all < gridDim.x ? S_all : gridDim.x;
    // Few segments (bs * Hkv <= FEW_SEGMENTS), or up to UNIFORM_SEGMENTS of nearly
    // equal length (mean at least 7/8 of the longest): a whole number per of CTAs
    // per segment, at most MAX_FANIN. When the shortest selection has at least
    // per tokens, the CTAs split each segment on their own (misc[22] = per): CTA
    // c takes [r L_k / per, (r + 1) L_k / per) of segment k = c / per, r = c mod per
    // (for equal lengths the ranges of the equal-token split), so each CTA holds
    // one piece and every segment's contributors merge it together after the main
    // loop. Otherwise the equal-token split over the per * S CTAs.
    {
        const unsigned S = static_cast<unsigned>(p.bs * Hkv);
        const bool uniform = 8ull * N >= 7ull * S * static_cast<unsigned long long>(misc[20]);
        unsigned local = 0;
        if (!whole && (S <= FEW_SEGMENTS || (S <= UNIFORM_SEGMENTS && uniform)) && 2 * S <= G) {
            const unsigned per = G / S < MAX_FANIN ? G / S : MAX_FANIN;
            G = per * S;
            if (static_cast<unsigned>(misc[23]) >= per) local = per;
        }
        misc[22] = static_cast<int>(local); // every thread writes the same value
    }
    if (blockIdx.x >= G) return;
    long long t_begin, t_end;
    if (whole) { // the first token of segment k = g bs + b is g NT + segP[b]
        const long long NT = segP[p.bs];
        const unsigned k0 = blockIdx.x * S_all / G, k1 = (blockIdx.x + 1) * S_all / G;
        t_begin = (long long)(k0 / p.bs) * NT + segP[k0 % p.bs];
        t_end = k1 >= S_all ? (long long)N : (long long)(k1 / p.bs) * NT + segP[k1 % p.bs];
    } else {
        t_begin = cta_begin(blockIdx.x, N, G);
        t_end = cta_begin(blockIdx.x + 1, N, G);
    }
    if (const unsigned per = static_cast<unsigned>(misc[22]); per != 0) {
        const unsigned k = blockIdx.x / per, r = blockIdx.x - k * per, b = k % static_cast<unsigned>(p.bs),
                       g = k / static_cast<unsigned>(p.bs);
        const unsigned Fs = g * static_cast<unsigned>(segP[p.bs]) + static_cast<unsigned>(segP[b]),
                       L = static_cast<unsigned>(segL[b]);
        t_begin = Fs + r * L / per;
        t_end = Fs + (r + 1) * L / per;
    }

    uint8_t* const stage0 = smem + Ly::off_stage;
    int* const ring = reinterpret_cast<int*>(smem + Ly::off_ring);

    if (warp >= NW) {
        // ============================================================ producers
        // Producer warp pw gathers tokens [pw*TPP, (pw+1)*TPP) of every stage.
        if constexpr (Tr::RQ) regs_producer(); // consumer-bound pools only
        const int pw = warp - NW;
        const int mytok = pw * TPP + lane;
        Cursor pc, ic;
        cursor_init(pc, t_begin, t_end, segL, segP, p.bs, Hkv);
        ic = pc;
        auto prefetch = [&](const Cursor& c, int entry) {
            if (lane < TPP && mytok < cursor_n(c))
                cp_async4(smem_u32(ring + entry * T + mytok), p.sel + segSrc[c.b] + c.j + mytok);
        };
#pragma unroll 1
        for (int i = 0; i < Ly::PF; ++i) {
            if (pc.t < t_end) {
                prefetch(pc, i % Ly::R);
                cursor_advance(pc, t_end, segL, p.bs);
            }
            cp_async_commit();
        }
        constexpr int CPR = Tr::ROWB / 16; // 16-byte chunks per row
        constexpr int RPI = 32 / CPR;      // rows per warp-wide copy instruction
        const uint64_t pol_row = l2_evict_first(), pol_sc = l2_evict_last();
        const int toff = lane / CPR, chunk = lane % CPR;
#pragma unroll 1
        for (int i = 0; ic.t < t_end; ++i) {
            if (pc.t < t_end) {
                prefetch(pc, (i + Ly::PF) % Ly::R);
                cursor_advance(pc, t_end, segL, p.bs);
            }
            cp_async_commit();
            cp_async_wait<Ly::PF>();
            __syncwarp();
            const int n = cursor_n(ic);
            const int b = ic.b, g = ic.g;
            if (ic.segfirst && pw == 0) {
                const int qb = ic.kseg & 1;
                if (!mbar_wait(qempty_bar(qb), ((ic.kseg >> 1) & 1) ^ 1, p.err, abort_flag)) break;
                if (lane == 0) mbar_arrive_expect_tx(qfull_bar(qb), GROUP * D * 2);
                __syncwarp();
                if (lane < GROUP)
                    bulk_g2s(smem_u32(smem + Ly::off_q + qb * 16 * Q_RS + lane * Q_RS),
                             p.q + b * p.q_sb + (g * GROUP + lane) * p.q_sh, D * 2, qfull_bar(qb));
            }
            const int s = i % Tr::STAGES;
            if (!mbar_wait(empty_bar(s), ((i / Tr::STAGES) & 1) ^ 1, p.err, abort_flag)) break;
            uint8_t* const Ks = stage0 + s * Ly::STAGE_BYTES;
            uint8_t* const Vs = Ks + Ly::STAGE_KV;
            long long myrow = 0, myring = 0;
            bool myhot = false;
            const bool valid = lane < TPP && mytok < n;
            if (valid) {
                int slot = ring[(i % Ly::R) * T + mytok];
                if (slot < 0 || (long long)slot >= p.num_slots) {
                    atomicOr(p.err, QSA_DEVERR_SLOT_RANGE);
                    slot = 0;
                }
                myrow = (long long)slot * Hkv + g;
                if constexpr (Tr::TIER) { // hot: the ring position holds this slot's row
                    const int pos = slot & p.ring_mask;
                    myhot = __ldg(p.owner + pos) == slot;
                    myring = (long long)pos * Hkv + g;
                }
            }
            if constexpr (Tr::TIER) {
                // Rows of two sizes: list the warp's tokens by tier (ballot ranks), then
                // copy 256-byte ring rows two per instruction (16 lanes each) and
                // 128-byte pool rows four per instruction (8 lanes each), so no
                // instruction mixes the two and no lane idles inside a pass.
                int* const tlist = reinterpret_cast<int*>(smem + Ly::off_tlist) + pw * 32;
                const unsigned hm = __ballot_sync(0xFFFFFFFFu, valid && myhot);
                const unsigned cm = __ballot_sync(0xFFFFFFFFu, valid && !myhot);
                const unsigned zm = __ballot_sync(0xFFFFFFFFu, lane < TPP && !valid);
                const unsigned below = (1u << lane) - 1u;
                __syncwarp(); // the previous stage's reads of the lists are done
                if (valid) tlist[myhot ? __popc(hm & below) : 16 + __popc(cm & below)] = lane;
                __syncwarp();
                const int nh = __popc(hm), nc = __popc(cm);
#pragma unroll 1
                for (int r0 = 0; r0 < nh; r0 += 2) {
                    const int rr = r0 + (lane >> 4), ch = lane & 15;
                    const int src = tlist[rr < nh ? rr : nh - 1];
                    const long long rrow = __shfl_sync(0xFFFFFFFFu, myring, src);
                    if (rr < nh) {
                        const int t = pw * TPP + src;
                        cp_async16(smem_u32(Ks + swz<Tr::ROWB>(t, ch)), p.kring + rrow * 256 + ch * 16);
                        cp_async16(smem_u32(Vs + swz<Tr::ROWB>(t, ch)), p.vring + rrow * 256 + ch * 16);
                    }
                }
#pragma unroll 1
                for (int r0 = 0; r0 < nc; r0 += 4) {
                    const int rr = r0 + (lane >> 3), ch = lane & 7;
                    const int src = tlist[16 + (rr < nc ? rr : nc - 1)];
                    const long long row = __shfl_sync(0xFFFFFFFFu, myrow, src);
                    if (rr < nc) {
                        const int t = pw * TPP + src;
                        cp_async16_l2(smem_u32(Ks + swz<Tr::ROWB>(t, ch)), p.kpool + row * 128 + ch * 16, pol_row);
                        cp_async16_l2(smem_u32(Vs + swz<Tr::ROWB>(t, ch)), p.vpool + row * 128 + ch * 16, pol_row);
                    }
                }
                if (zm) { // rows past the live length hold zeros (P is 0 there, V must be finite)
#pragma unroll 1
                    for (int t0 = 0; t0 < TPP; t0 += 2) {
                        const int tl = t0 + (lane >> 4);
                        if ((zm >> tl) & 1u)
                            *reinterpret_cast<uint4*>(Vs + swz<Tr::ROWB>(pw * TPP + tl, lane & 15)) =
                                make_uint4(0, 0, 0, 0);
                    }
                }
            } else {
#pragma unroll
                for (int t0 = 0; t0 < TPP; t0 += RPI) {
                    const int tl = t0 + toff;
                    const long long row = __shfl_sync(0xFFFFFFFFu, myrow, tl);
                    const int t = pw * TPP + tl;
                    if (t < n) {
                        if constexpr (Tr::SCALES) {
                            cp_async16_l2(smem_u32(Ks + swz<Tr::ROWB>(t, chunk)),
                                          p.kpool + row * Tr::ROWB + chunk * 16, pol_row);
                            cp_async16_l2(smem_u32(Vs + swz<Tr::ROWB>(t, chunk)),
                                          p.vpool + row * Tr::ROWB + chunk * 16, pol_row);
                        } else {
                            cp_async16(smem_u32(Ks + swz<Tr::ROWB>(t, chunk)),
                                       p.kpool + row * Tr::ROWB + chunk * 16);
                            cp_async16(smem_u32(Vs + swz<Tr::ROWB>(t, chunk)),
                                       p.vpool + row * Tr::ROWB + chunk * 16);
                        }
                    } else {
                        // rows past the live length hold zeros (P is 0 there, V must be finite)
                        *reinterpret_cast<uint4*>(Vs + swz<Tr::ROWB>(t, chunk)) = make_uint4(0, 0, 0, 0);
                    }
                }
            }
            if constexpr (Tr::SCALES) {
                uint8_t* sc = Vs + Ly::STAGE_KV; // K scales [T][SC_TOK], then V scales
                const uint32_t ks = smem_u32(sc + mytok * Ly::SC_TOK);
                const uint32_t vs = ks + T * Ly::SC_TOK;
                const uint8_t* kg = static_cast<const uint8_t*>(p.k_scale) + myrow * Ly::SC_TOK;
                const uint8_t* vg = static_cast<const uint8_t*>(p.v_scale) + myrow * Ly::SC_TOK;
                if constexpr (Tr::TIER) {
                    if (lane < TPP)
                        reinterpret_cast<int*>(Vs + Ly::STAGE_KV + Ly::STAGE_SC)[mytok] = valid && myhot;
                }
                if (Tr::TIER && valid && myhot) { // 4 binary16 scales of the ring row
                    cp_async8(ks, static_cast<const uint8_t*>(p.kring_scale) + myring * 8);
                    cp_async8(vs, static_cast<const uint8_t*>(p.vring_scale) + myring * 8);
                } else if (valid) {
                    if constexpr (Ly::SC_TOK == 4) {
                        cp_async4_l2(ks, kg, pol_sc);
                        cp_async4_l2(vs, vg, pol_sc);
                    } else if constexpr (Ly::SC_TOK == 8) {
                        cp_async8_l2(ks, kg, pol_sc);
                        cp_async8_l2(vs, vg, pol_sc);
                    } else {
                        cp_async16_l2(ks, kg, pol_sc);
                        cp_async16_l2(vs, vg, pol_sc);
                    }
                } else if (Tr::GROUPS && lane < TPP) {
                    // past the live length: zero V scales keep 0 * scale finite in P
                    if constexpr (Ly::SC_TOK == 8)
                        *reinterpret_cast<uint2*>(sc + T * Ly::SC_TOK + mytok * 8) = make_uint2(0, 0);
                    else if constexpr (Ly::SC_TOK == 16)
                        *reinterpret_cast<uint4*>(sc + T * Ly::SC_TOK + mytok * 16) = make_uint4(0, 0, 0, 0);
                }
            }
#ifdef QSA_TEST_HOOKS
            if (blockIdx.x == 0 && i == p.stall_stage) { // test build only: never complete it
                cursor_advance(ic, t_end, segL, p.bs);
                continue;
            }
#endif
            cp_async_arrive_noinc(full_bar(s));
            mbar_arrive(full_bar(s));
            cursor_advance(ic, t_end, segL, p.bs);
        }
        cp_async_wait<0>();
        return;
    }

    // ================================================================ consumers
    if constexpr (Tr::RQ) regs_consumer();
    const int r = lane >> 2, c = lane & 3;
    float kscale_g = 1.0f, out_scale = 1.0f;
    if constexpr (FMT == QSA_KV_FP8_E4M3) {
        kscale_g = __ldg(static_cast<const float*>(p.k_scale));
        out_scale = __ldg(static_cast<const float*>(p.v_scale));
    }
    const float cs_base = p.scale_log2 * kscale_g;
    float* const red = reinterpret_cast<float*>(smem + Ly::off_red);    // [2][NW][16]
    float* const mref = reinterpret_cast<float*>(smem + Ly::off_mref);  // [2][16]
    float* const lred = reinterpret_cast<float*>(smem + Ly::off_lred);  // [NW][16]
    float* const nred = reinterpret_cast<float*>(smem + Ly::off_nred);  // [NW][16]
    float* const eref = reinterpret_cast<float*>(smem + Ly::off_eref);  // [2][16]
    constexpr bool VSH = Ly::NUM_REF;

    uint32_t qa[16][4];
    float qmul_a = 1.f, qmul_b = 1.f; // undo the per-head Q scaling of f16 QK
    // PV n-tiles: f16 P without per-slot V scales (fp8: P <= 2^TAU, 11 significand
    // bits) is used as is, heads 0-7 and 8-11 (+4 zero rows); otherwise P (or
    // P * s_v) is split into hi + lo columns of the PV type, 24 rows in 3 tiles
    constexpr bool P_HI = Tr::PV_F16 && !Tr::SCALES;
    constexpr int NJ = P_HI ? 2 : 3;
    float o[MT][NJ][4];
    float l0 = 0.f, l1 = 0.f;
    // this lane's heads r, r + 8: reference maxima, and (per-slot V scales in f16
    // PV) offsets E and 2^-E, as published in mref / eref; they change only on the
    // slow path, so the fast path keeps them in registers
    float mr_a = 0.f, mr_b = 0.f, er_a = 0.f, er_b = 0.f, fr_a = 1.f, fr_b = 1.f;
    int v = 0, buf = 0, seg_j0 = 0;
    // Merge bookkeeping, kept in shared memory rather than in registers carried
    // through the main loop: [0] pend0 / [1] pend1, the split segments whose
    // partial this CTA wrote (first / last piece of its range); [2] the segment
    // head merged directly after the loop and [3] its other contributors; [4]
    // thread 0's arrival ticket for pend0. Every consumer thread writes the same
    // values, so each reads back what it wrote.
    volatile int* const mstate = misc + 8;
    // contributors of a split segment: CTAs c_first..c_last; c_first's partial
    // sits in its slot 1 when its range began before the segment
    auto seg_range = [&](int sid, unsigned& Fs, unsigned& c_first, unsigned& c_last) {
        const int b = sid / Hkv, g = sid - (sid / Hkv) * Hkv, L = segL[b];
        Fs = static_cast<unsigned>(g * segP[p.bs] + segP[b]);
        c_first = cta_of(Fs, N, G);
        c_last = cta_of(Fs + static_cast<unsigned>(L) - 1u, N, G);
    };
    const int tok_base = warp * TPW;
    const int tk0 = tok_base + 2 * c;
    const int xs = lane & 7;                 // row % 8 of every row this lane addresses
    // QK B-fragment chunk pattern: matrix (lane >> 3) covers chunk 2*ks + cb
    const int kx = ((((lane >> 3) & 1) + (lane >> 4) * 2) ^ xs) << 4;
    // PV A-fragment chunk pattern: chunk 4*warp + 2*mt + ((lane >> 3) & 1)
    const int vx = ((((lane >> 3) & 1)) ^ xs) << 4;

    if constexpr (P_HI) { // the padding rows 12-15 of both P^T buffers, read as zeros
        for (int k = tid; k < 2 * 4 * PRS / 4; k += NCT) {
            const int bsel = k / (4 * PRS / 4), w = k - bsel * (4 * PRS / 4);
            reinterpret_cast<int*>(smem + Ly::off_p + bsel * 24 * PRS + 12 * PRS)[w] = 0;
        }
    }
    Cursor cc;
    cursor_init(cc, t_begin, t_end, segL, segP, p.bs, Hkv);
#pragma unroll 1
    for (int i = 0; cc.t < t_end; ++i) {
        const int n = cursor_n(cc);
        const bool first = cc.segfirst;
        const bool last = cc.j + n >= cc.j1;
        const int b = cc.b, g = cc.g;
        if (first) {
            seg_j0 = cc.j;
            const int qb = cc.kseg & 1;
            if (!mbar_wait(qfull_bar(qb), (cc.kseg >> 1) & 1, p.err, abort_flag)) break;
            const uint32_t qbase = smem_u32(smem + Ly::off_q + qb * 16 * Q_RS);
            if constexpr (Tr::RQ) {
                build_q_rq<FMT>(smem + Ly::off_q + qb * 16 * Q_RS, lane, qa, qmul_a, qmul_b);
            } else {
#pragma unroll
                for (int ks = 0; ks < 16; ++ks) {
                    const int mi = lane >> 3;
                    const uint32_t addr =
                        qbase + ((mi & 1) * 8 + (lane & 7)) * Q_RS + (ks * 16 + (mi >> 1) * 8) * 2;
                    ldsm_x4(qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], addr);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(qempty_bar(qb));
            if constexpr (Tr::QK_F16 && !Tr::RQ) {
                // Q to f16, exactly: scale each head (row) by a power of two that
                // brings its largest |q| into [2^14, 2^15); undo it on the scores.
                float mr = 0.f, mr8 = 0.f;
#pragma unroll
                for (int ks = 0; ks < 16; ++ks) {
                    mr = fmaxf(mr, fmaxf(fmaxf(fabsf(bf16_lo(qa[ks][0])), fabsf(bf16_hi(qa[ks][0]))),
                                         fmaxf(fabsf(bf16_lo(qa[ks][2])), fabsf(bf16_hi(qa[ks][2])))));
                    mr8 = fmaxf(mr8, fmaxf(fmaxf(fabsf(bf16_lo(qa[ks][1])), fabsf(bf16_hi(qa[ks][1]))),
                                           fmaxf(fabsf(bf16_lo(qa[ks][3])), fabsf(bf16_hi(qa[ks][3])))));
                }
                mr = fmaxf(mr, __shfl_xor_sync(0xFFFFFFFFu, mr, 1));
                mr = fmaxf(mr, __shfl_xor_sync(0xFFFFFFFFu, mr, 2));
                mr8 = fmaxf(mr8, __shfl_xor_sync(0xFFFFFFFFu, mr8, 1));
                mr8 = fmaxf(mr8, __shfl_xor_sync(0xFFFFFFFFu, mr8, 2));
                auto shift_of = [](float m) {
                    const int e = static_cast<int>((__float_as_uint(m) >> 23) & 0xFFu) - 127;
                    const int sh = m > 0.f ? e - 14 : 0;
                    return sh < -100 ? -100 : (sh > 100 ? 100 : sh);
                };
                const int sa = shift_of(mr), sb = shift_of(mr8);
                const float da = __uint_as_float(static_cast<uint32_t>(127 - sa) << 23);
                const float db = __uint_as_float(static_cast<uint32_t>(127 - sb) << 23);
                qmul_a = __uint_as_float(static_cast<uint32_t>(127 + sa) << 23);
                qmul_b = __uint_as_float(static_cast<uint32_t>(127 + sb) << 23);
#pragma unroll
                for (int ks = 0; ks < 16; ++ks) {
                    qa[ks][0] = pack_f16x2(bf16_lo(qa[ks][0]) * da, bf16_hi(qa[ks][0]) * da);
                    qa[ks][2] = pack_f16x2(bf16_lo(qa[ks][2]) * da, bf16_hi(qa[ks][2]) * da);
                    qa[ks][1] = pack_f16x2(bf16_lo(qa[ks][1]) * db, bf16_hi(qa[ks][1]) * db);
                    qa[ks][3] = pack_f16x2(bf16_lo(qa[ks][3]) * db, bf16_hi(qa[ks][3]) * db);
                }
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int j = 0; j < NJ; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[mt][j][e] = 0.f;
            l0 = l1 = 0.f;
        }
        const int s = i % Tr::STAGES;
        if (!mbar_wait(full_bar(s), (i / Tr::STAGES) & 1, p.err, abort_flag)) break;
        uint8_t* const Ks = stage0 + s * Ly::STAGE_BYTES;
        uint8_t* const Vs = Ks + Ly::STAGE_KV;
        float skr[2] = {1.f, 1.f}, svr[2] = {1.f, 1.f};
        // grouped pools: K scales (binary16 pairs) of tokens tk0, tk0 + 1, and V
        // scales of tokens 2 lane, 2 lane + 1 in this warp's channel group
        constexpr int GP = Tr::GROUPS ? Tr::GROUPS / 2 : 1;
        uint32_t ksw[2][GP];
        float svw[2] = {0.f, 0.f};

        // per-slot scales, into registers while the stage is held
        if constexpr (Tr::SCALES && !Tr::GROUPS) {
            const float* sc = reinterpret_cast<const float*>(Vs + Ly::STAGE_KV);
            skr[0] = sc[tk0];
            skr[1] = sc[tk0 + 1];
            svr[0] = sc[T + tk0];
            svr[1] = sc[T + tk0 + 1];
        }
        if constexpr (Tr::GROUPS) { // read before the stage is released
            constexpr int G = Tr::GROUPS;
            const uint32_t* sk = reinterpret_cast<const uint32_t*>(Vs + Ly::STAGE_KV);
#pragma unroll
            for (int k = 0; k < GP; ++k) {
                ksw[0][k] = sk[tk0 * GP + k];
                ksw[1][k] = sk[(tk0 + 1) * GP + k];
            }
            const __half* sv = reinterpret_cast<const __half*>(Vs + Ly::STAGE_KV + T * Ly::SC_TOK);
            const int gv = warp * G / NW;
            if constexpr (Tr::TIER) {
                // a ring row holds 4 scales of 64 channels: 32-channel group k reads k / 2
                const int* flag = reinterpret_cast<const int*>(Vs + Ly::STAGE_KV + Ly::STAGE_SC);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    if (flag[tk0 + u]) {
                        const uint32_t e0 = ksw[u][0], e1 = ksw[u][1];
                        ksw[u][0] = __byte_perm(e0, 0, 0x1010);
                        ksw[u][1] = __byte_perm(e0, 0, 0x3232);
                        ksw[u][2] = __byte_perm(e1, 0, 0x1010);
                        ksw[u][3] = __byte_perm(e1, 0, 0x3232);
                    } else {
                        skr[u] = 0.0625f; // the int4 row's codes are widened as 16 * code
                    }
                }
                const bool h0 = flag[2 * lane] != 0, h1 = flag[2 * lane + 1] != 0;
                svw[0] = __half2float(sv[(2 * lane) * G + (h0 ? gv >> 1 : gv)]) * (h0 ? 1.f : 0.0625f);
                svw[1] = __half2float(sv[(2 * lane + 1) * G + (h1 ? gv >> 1 : gv)]) * (h1 ? 1.f : 0.0625f);
            } else {
                svw[0] = __half2float(sv[(2 * lane) * G + gv]);
                svw[1] = __half2float(sv[(2 * lane + 1) * G + gv]);
            }
        }

        uint32_t hot_lo = 0, hot_hi = 0; // tiered pools: ring-row tokens of the stage (bit t)
        if constexpr (Tr::TIER) {
            // Widen the stage's int4 rows to int8 (16 * code): K in place, for this warp's
            // own 8 tokens (only this warp reads them); V into this warp's chunks
            // 2w, 2w + 1 of the side buffer, for every token (only this warp reads
            // them). Everything read comes before everything written (__syncwarp).
            const int* flag = reinterpret_cast<const int*>(Vs + Ly::STAGE_KV + Ly::STAGE_SC);
            hot_lo = __ballot_sync(0xFFFFFFFFu, flag[lane] != 0);
            hot_hi = __ballot_sync(0xFFFFFFFFu, flag[lane + 32] != 0);
            const int tt = tok_base + (lane & 7), kc = lane >> 3; // K: token, chunks kc, kc + 4
            const bool kcold = !(((tt < 32 ? hot_lo : hot_hi) >> (tt & 31)) & 1u);
            uint4 kr[2], vr[2];
            if (kcold) {
                kr[0] = *reinterpret_cast<const uint4*>(Ks + swz<Tr::ROWB>(tt, kc));
                kr[1] = *reinterpret_cast<const uint4*>(Ks + swz<Tr::ROWB>(tt, kc + 4));
            }
            const bool vcold0 = !((hot_lo >> lane) & 1u), vcold1 = !((hot_hi >> lane) & 1u);
            if (vcold0) vr[0] = *reinterpret_cast<const uint4*>(Vs + swz<Tr::ROWB>(lane, warp));
            if (vcold1) vr[1] = *reinterpret_cast<const uint4*>(Vs + swz<Tr::ROWB>(lane + 32, warp));
            __syncwarp();
            if (kcold) {
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    uint4 o0, o1;
                    widen16_i4x32<Tr::NIB_OFFSET>(kr[u], o0, o1);
                    *reinterpret_cast<uint4*>(Ks + swz<Tr::ROWB>(tt, 2 * (kc + 4 * u))) = o0;
                    *reinterpret_cast<uint4*>(Ks + swz<Tr::ROWB>(tt, 2 * (kc + 4 * u) + 1)) = o1;
                }
            }
            uint8_t* const vexp = smem + Ly::off_vexp;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                if (u == 0 ? vcold0 : vcold1) {
                    const int tv = lane + 32 * u;
                    uint4 o0, o1;
                    widen16_i4x32<Tr::NIB_OFFSET>(vr[u], o0, o1);
                    *reinterpret_cast<uint4*>(vexp + swz<Tr::ROWB>(tv, 2 * warp)) = o0;
                    *reinterpret_cast<uint4*>(vexp + swz<Tr::ROWB>(tv, 2 * warp + 1)) = o1;
                }
            }
            __syncwarp();
        }

        // ---------------------------------------------------------------- QK
        float sacc[4][4] = {};
        // a stage past the live length (a piece's last, partial stage): warps whose
        // 8 tokens are all masked skip their MMAs and (bf16) PV runs the live k16
        // steps only; kept to the pools where it measured faster (elsewhere the
        // extra branches cost more than the skipped work)
        constexpr bool SKIP_QK = !Tr::SCALES, SKIP_PV = !Tr::RQ;
        if (SKIP_QK && tok_base >= n) {
            // nothing: every score of this warp is masked below
        } else if constexpr (Tr::RQ) {
            // this warp's 8 tokens from the raw stage: ldmatrix matrix (lane >> 3) of
            // word set j reads 16-byte chunk 4j + (lane >> 3) of its token's row; each
            // word becomes f16 B fragments in registers (k16 step ks: chunk ks for
            // 8-bit codes, half of chunk ks / 2 for 4-bit codes)
            const uint32_t krow = smem_u32(Ks) + (tok_base + (lane & 7)) * Tr::ROWB;
            constexpr int G = Tr::GROUPS ? Tr::GROUPS : 1, KPG = 16 / G; // k16 steps per group
            float acc[4][4] = {};
            uint32_t w[4], nb[4];
#pragma unroll
            for (int ks = 0; ks < 16; ++ks) {
                uint32_t b0, b1;
                if constexpr (Tr::NIB4) {
                    if ((ks & 7) == 0)
                        ldsm_x4(w[0], w[1], w[2], w[3], krow + ((((ks >> 1) + (lane >> 3)) ^ xs) << 4));
                    if ((ks & 1) == 0) i4x8_to<true, Tr::NIB_OFFSET>(w[(ks >> 1) & 3], nb);
                    b0 = nb[2 * (ks & 1)];
                    b1 = nb[2 * (ks & 1) + 1];
                } else {
                    if ((ks & 3) == 0) ldsm_x4(w[0], w[1], w[2], w[3], krow + (((ks + (lane >> 3)) ^ xs) << 4));
                    if constexpr (FMT == QSA_KV_FP8_E4M3)
                        e4m3x4_to_f16(w[ks & 3], b0, b1);
                    else
                        i8x4_to_f16(w[ks & 3], b0, b1);
                }
                mma_f16(acc[ks & 3], qa[ks], b0, b1);
                if constexpr (Tr::GROUPS) {
                    if ((ks + 1) % KPG == 0) { // a group's end: fold with the token's group scale
                        const int gi = ks / KPG;
                        float t4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            t4[e] = (acc[0][e] + acc[1][e]) + (acc[2][e] + acc[3][e]);
                            acc[0][e] = acc[1][e] = acc[2][e] = acc[3][e] = 0.f;
                        }
                        const uint32_t w0 = ksw[0][gi >> 1], w1 = ksw[1][gi >> 1];
                        const float s0 = __half2float(__ushort_as_half(static_cast<unsigned short>(gi & 1 ? w0 >> 16 : w0)));
                        const float s1 = __half2float(__ushort_as_half(static_cast<unsigned short>(gi & 1 ? w1 >> 16 : w1)));
                        sacc[0][0] += t4[0] * s0;
                        sacc[0][1] += t4[1] * s1;
                        sacc[0][2] += t4[2] * s0;
                        sacc[0][3] += t4[3] * s1;
                    }
                }
            }
            if constexpr (!Tr::GROUPS) {
#pragma unroll
                for (int e = 0; e < 4; ++e) sacc[0][e] = (acc[0][e] + acc[1][e]) + (acc[2][e] + acc[3][e]);
            }
        } else { // bf16 rows
            const uint32_t krow = smem_u32(Ks) + (tok_base + (lane & 7)) * BF_ROW;
#pragma unroll
            for (int ks = 0; ks < 16; ks += 2) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(b0, b1, b2, b3, krow + ((ks * 32) ^ kx));
                float* acc = sacc[(ks >> 1) & 1];
                mma16816<Tr::QK_F16>(acc, qa[ks], b0, b1);
                mma16816<Tr::QK_F16>(sacc[2 + ((ks >> 1) & 1)], qa[ks + 1], b2, b3);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) sacc[0][e] += sacc[1][e] + sacc[2][e] + sacc[3][e];
        }
        const bool v0 = tk0 < n, v1 = tk0 + 1 < n;
        const bool row8 = r < 4; // head r + 8 is a real head (8..11)
        const float ninf = -INFINITY;
        float x[4];
        const float csa = cs_base * qmul_a, csb = cs_base * qmul_b;
        x[0] = v0 ? sacc[0][0] * csa * skr[0] : ninf;
        x[1] = v1 ? sacc[0][1] * csa * skr[1] : ninf;
        x[2] = (v0 && row8) ? sacc[0][2] * csb * skr[0] : ninf;
        x[3] = (v1 && row8) ? sacc[0][3] * csb * skr[1] : ninf;
        float ma = fmaxf(x[0], x[1]), mb = fmaxf(x[2], x[3]);
        ma = fmaxf(ma, __shfl_xor_sync(0xFFFFFFFFu, ma, 1));
        ma = fmaxf(ma, __shfl_xor_sync(0xFFFFFFFFu, ma, 2));
        mb = fmaxf(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 1));
        mb = fmaxf(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 2));
        float* const redb = red + buf * NW * 16;
        if (c == 0) {
            redb[warp * 16 + r] = ma;
            redb[warp * 16 + r + 8] = mb;
        }
        const float* const mrefv = mref + v * 16;
        const float mo_a = first ? ninf : mr_a;
        const float mo_b = first ? ninf : mr_b;
        // Per-slot V scales in f16 PV (int8): PV runs on pn = p * s_v * 2^-E_h,
        // p = 2^(x - m_h). The per-head offset E_h is kept at or above every
        // t = (x - m_h) + floor(log2 |s_v|) - 14 of the piece, so pn < 2^15 (when
        // a t exceeds it, it rises to that t + TAU, so it seldom rises again); it
        // is held relative to the reference m_h, so that a huge score cannot
        // absorb the scale's exponent. O is accumulated against m_h + E_h,
        // rescaled when that rises and multiplied by 2^E_h in the epilogue.
        // E_h >= -119 keeps 2^-E_h and p * 2^-E_h finite.
        float fa = 1.f, fb = 1.f, eo_a = 0.f, eo_b = 0.f, g0 = 0.f, g1 = 0.f;
        const float* const erefv = eref + v * 16;
        bool vraise = false;
        if constexpr (VSH) {
            auto lgs = [](float sv) {
                return static_cast<float>(static_cast<int>((__float_as_uint(sv) >> 23) & 0xFFu) - 141);
            };
            g0 = lgs(svr[0]);
            g1 = lgs(svr[1]);
            if (!first) {
                eo_a = er_a;
                eo_b = er_b;
                fa = fr_a;
                fb = row8 ? fr_b : 0.f;
                const float ta = fmaxf((x[0] - mo_a) + g0, (x[1] - mo_a) + g1);
                const float tb = fmaxf((x[2] - mo_b) + g0, (x[3] - mo_b) + g1);
                vraise = ta > eo_a || (row8 && tb > eo_b);
            }
        }

        uint8_t* const Pb = smem + Ly::off_p + buf * 24 * PRS;
        float pr[4];
        auto compute_p = [&](float ra, float rb) {
            pr[0] = x[0] == ninf ? 0.f : ex2(x[0] - ra);
            pr[1] = x[1] == ninf ? 0.f : ex2(x[1] - ra);
            pr[2] = x[2] == ninf ? 0.f : ex2(x[2] - rb);
            pr[3] = x[3] == ninf ? 0.f : ex2(x[3] - rb);
        };
        float* const Pf = reinterpret_cast<float*>(smem + Ly::off_p) + buf * GROUP * PFS;
        auto write_p = [&]() {
            // p * s_v * f in an order whose partial product stays finite: with f <= 1,
            // s_v * f <= s_v; with f > 1, p * f <= 2^TAU * 2^119 (masked tokens have p = 0)
            auto pnum = [](float pp, float sv, float f) { return f <= 1.f ? pp * (sv * f) : (pp * f) * sv; };
            float pv[4] = {pnum(pr[0], svr[0], fa), pnum(pr[1], svr[1], fa), pnum(pr[2], svr[0], fb),
                           pnum(pr[3], svr[1], fb)};
            pv[0] = v0 ? pv[0] : 0.f;
            pv[1] = v1 ? pv[1] : 0.f;
            pv[2] = v0 ? pv[2] : 0.f;
            pv[3] = v1 ? pv[3] : 0.f;
            if constexpr (Tr::GROUPS) { // FP32 P; each warp scales and splits its own fragments
                *reinterpret_cast<float2*>(Pf + r * PFS + tk0) = make_float2(pv[0], pv[1]);
                if (row8) *reinterpret_cast<float2*>(Pf + (8 + r) * PFS + tk0) = make_float2(pv[2], pv[3]);
                return;
            }
            if constexpr (P_HI) { // P^T rows: heads 0-11; rows 12-15 stay zero
                *reinterpret_cast<uint32_t*>(Pb + r * PRS + tk0 * 2) = pack_f16x2(pv[0], pv[1]);
                if (row8) *reinterpret_cast<uint32_t*>(Pb + (8 + r) * PRS + tk0 * 2) = pack_f16x2(pv[2], pv[3]);
                return;
            }
            uint32_t hi_a, lo_a;
            split_pair<Tr::PV_F16>(pv[0], pv[1], hi_a, lo_a);
            *reinterpret_cast<uint32_t*>(Pb + r * PRS + tk0 * 2) = hi_a;
            *reinterpret_cast<uint32_t*>(Pb + (8 + r) * PRS + tk0 * 2) = lo_a;
            if (row8) {
                uint32_t hi_b, lo_b;
                split_pair<Tr::PV_F16>(pv[2], pv[3], hi_b, lo_b);
                *reinterpret_cast<uint32_t*>(Pb + (16 + r) * PRS + tk0 * 2) = hi_b;
                *reinterpret_cast<uint32_t*>(Pb + (20 + r) * PRS + tk0 * 2) = lo_b;
            }
        };
        compute_p(mo_a, mo_b);
        write_p();
        // One barrier publishes P and the per-warp maxima and ORs "some score of
        // this stage exceeds its head's reference by more than TAU" over all warps.
        const bool nd_local = first || ma > mo_a + TAU || (row8 && mb > mo_b + TAU) || vraise;
        if (consumer_sync_or(nd_local)) {
            // stage maximum per head vs the running reference
            auto stage_max = [&](int h) {
                float m = redb[h];
#pragma unroll
                for (int w = 1; w < NW; ++w) m = fmaxf(m, redb[w * 16 + h]);
                return m;
            };
            auto old_ref = [&](int h) { return first ? ninf : mrefv[h]; };
            // slow path (uniform over the consumer warps): raise the reference max
            auto new_ref = [&](int h) { return fmaxf(old_ref(h), stage_max(h)); };
            auto alpha = [&](int h) {
                const float mo = old_ref(h);
                return mo == ninf ? 0.f : ex2(mo - new_ref(h));
            };
            const float na = new_ref(r), nb = row8 ? new_ref(r + 8) : 0.f;
            mr_a = na;
            mr_b = nb;
            l0 *= alpha(r);
            l1 *= row8 ? alpha(r + 8) : 0.f;
            // per-slot V scales: the stage's largest offset t per head against the
            // new references (one more exchange), then the new E_h
            if constexpr (VSH) {
                float ta = fmaxf((x[0] - na) + g0, (x[1] - na) + g1);
                float tb = fmaxf((x[2] - nb) + g0, (x[3] - nb) + g1);
                ta = fmaxf(ta, __shfl_xor_sync(0xFFFFFFFFu, ta, 1));
                ta = fmaxf(ta, __shfl_xor_sync(0xFFFFFFFFu, ta, 2));
                tb = fmaxf(tb, __shfl_xor_sync(0xFFFFFFFFu, tb, 1));
                tb = fmaxf(tb, __shfl_xor_sync(0xFFFFFFFFu, tb, 2));
                if (c == 0) {
                    nred[warp * 16 + r] = ta;
                    nred[warp * 16 + r + 8] = row8 ? tb : ninf;
                }
                consumer_sync();
            }
            // E_h after this stage: the old offset carried to the new reference or,
            // when the stage's largest t exceeds it, that t plus TAU of slack (as the
            // lazy maximum has), so that E_h rarely needs to rise again; at least
            // -119 (fmaxf drops the NaN of -inf - -inf)
            auto new_e = [&](int h) {
                float t = nred[h];
#pragma unroll
                for (int w = 1; w < NW; ++w) t = fmaxf(t, nred[w * 16 + h]);
                const float carried = first ? ninf : erefv[h] + (old_ref(h) - new_ref(h));
                return fmaxf(t > carried ? t + TAU : carried, -119.f);
            };
            auto o_scale = [&](int h) {
                if constexpr (!VSH) return alpha(h);
                if (first || old_ref(h) == ninf) return 0.f; // O is still zero then
                return ex2((old_ref(h) - new_ref(h)) + (erefv[h] - new_e(h)));
            };
            if constexpr (VSH) {
                er_a = new_e(r);
                er_b = row8 ? new_e(r + 8) : 0.f;
                fr_a = ex2(-er_a);
                fr_b = row8 ? ex2(-er_b) : 0.f;
                fa = fr_a;
                fb = fr_b;
            }
            compute_p(na, nb);
            write_p();
            const float a0 = o_scale(2 * c), a1 = o_scale(2 * c + 1);
            const float a2 = o_scale(8 + ((2 * c) & 3)), a3 = o_scale(8 + ((2 * c + 1) & 3));
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                for (int j = 0; j < NJ - 1; ++j) {
                    o[mt][j][0] *= a0;
                    o[mt][j][1] *= a1;
                    o[mt][j][2] *= a0;
                    o[mt][j][3] *= a1;
                }
                o[mt][NJ - 1][0] *= a2;
                o[mt][NJ - 1][1] *= a3;
                o[mt][NJ - 1][2] *= a2;
                o[mt][NJ - 1][3] *= a3;
            }
            if (warp == 0 && lane < GROUP) mref[(v ^ 1) * 16 + lane] = new_ref(lane);
            if (VSH && warp == 1 && lane < GROUP) eref[(v ^ 1) * 16 + lane] = new_e(lane);
            v ^= 1;
            consumer_sync();
        }
        l0 += pr[0] + pr[1];
        l1 += pr[2] + pr[3];

        // ---------------------------------------------------------------- PV
        const uint8_t* Pt = Pb;
        if constexpr (Tr::GROUPS == 4) {
            // 64-channel groups: warps 2k and 2k + 1 share group k and need the same
            // scaled P^T, so the pair builds one copy (six heads each, double-buffered
            // by stage) and meets at a named barrier; each P times its token's V
            // scale, split into bf16 hi + lo
            const int pair = warp >> 1, h0 = 6 * (warp & 1);
            uint8_t* const Pw = smem + Ly::off_pw + (pair * 2 + buf) * 24 * PRS;
            const int t = 2 * lane;
            const float sv0 = svw[0], sv1 = svw[1];
#pragma unroll
            for (int hh = 0; hh < 6; ++hh) {
                const int h = h0 + hh;
                const float2 pp = *reinterpret_cast<const float2*>(Pf + h * PFS + t);
                uint32_t hi, lo;
                split_pair<false>(pp.x * sv0, pp.y * sv1, hi, lo);
                const int rh = h < 8 ? h : 8 + h, rl = h < 8 ? 8 + h : 12 + h;
                *reinterpret_cast<uint32_t*>(Pw + rh * PRS + t * 2) = hi;
                *reinterpret_cast<uint32_t*>(Pw + rl * PRS + t * 2) = lo;
            }
            asm volatile("bar.sync %0, 64;" ::"r"(BAR_CONSUMERS + 1 + pair) : "memory");
            Pt = Pw;
        }
        {
            const uint32_t pbase = smem_u32(Pt);
            const uint32_t vrow = smem_u32(Vs) + ((lane >> 4) * 8 + (lane & 7)) * BF_ROW;
#pragma unroll
            for (int kk = 0; kk < KK; ++kk) {
                if (!SKIP_PV || kk * 16 < n) { // P is 0 past n (V rows past n are zero-filled)
                    uint32_t pb[NJ][2];
                    if constexpr (Tr::GROUPS == 8) {
                        // 32-channel groups: the B fragments of P^T scaled per token by this
                        // warp's group V scale, built in registers. Lane (r, c) takes
                        // heads r (hi, lo: tiles 0, 1) and 8 + (r & 3) (tile 2: hi for
                        // r < 4, lo above), tokens 2c, 2c + 1 and 8 + 2c, 9 + 2c of the
                        // k-step; token 2l + u's scale is lane l's svw[u]
                        const int ta = kk * 16 + 2 * c, tb = ta + 8;
                        const float s0 = __shfl_sync(0xFFFFFFFFu, svw[0], ta >> 1);
                        const float s1 = __shfl_sync(0xFFFFFFFFu, svw[1], ta >> 1);
                        const float s8 = __shfl_sync(0xFFFFFFFFu, svw[0], tb >> 1);
                        const float s9 = __shfl_sync(0xFFFFFFFFu, svw[1], tb >> 1);
                        const float* const Pr = Pf + r * PFS;
                        const float* const P2 = Pf + (8 + (r & 3)) * PFS;
                        const float2 p0 = *reinterpret_cast<const float2*>(Pr + ta);
                        const float2 p1 = *reinterpret_cast<const float2*>(Pr + tb);
                        const float2 p2 = *reinterpret_cast<const float2*>(P2 + ta);
                        const float2 p3 = *reinterpret_cast<const float2*>(P2 + tb);
                        split_pair<false>(p0.x * s0, p0.y * s1, pb[0][0], pb[1][0]);
                        split_pair<false>(p1.x * s8, p1.y * s9, pb[0][1], pb[1][1]);
                        uint32_t h2a, l2a, h2b, l2b;
                        split_pair<false>(p2.x * s0, p2.y * s1, h2a, l2a);
                        split_pair<false>(p3.x * s8, p3.y * s9, h2b, l2b);
                        pb[NJ - 1][0] = r < 4 ? h2a : l2a;
                        pb[NJ - 1][1] = r < 4 ? h2b : l2b;
                    } else {
                        ldsm_x4(pb[0][0], pb[0][1], pb[1][0], pb[1][1],
                                pbase + ((lane >> 4) * 8 + (lane & 7)) * PRS +
                                    (kk * 16 + ((lane >> 3) & 1) * 8) * 2);
                        if constexpr (NJ == 3)
                            ldsm_x2(pb[NJ - 1][0], pb[NJ - 1][1],
                                    pbase + (16 + (lane & 7)) * PRS + (kk * 16 + ((lane >> 3) & 1) * 8) * 2);
                    }
                    if constexpr (Tr::RQ) {
                        // V^T fragments straight from the raw stage (ldmatrix.trans of the
                        // codes, converted in registers); the warp's 32 dims are spread
                        // over its two m-tiles as the epilogue's dim map says
                        uint32_t a[MT][4];
                        const uint32_t vst = smem_u32(Vs);
                        if constexpr (Tr::NIB4) { // chunk `warp` (32 codes) of tokens 0-7 / 8-15
                            const int tv = kk * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
                            uint32_t r0, r1;
                            ldsm_x2_t(r0, r1, vst + tv * Tr::ROWB + ((warp ^ xs) << 4));
                            if constexpr (!Tr::NIB_OFFSET) {
                                r0 ^= 0x88888888u;
                                r1 ^= 0x88888888u;
                            }
    #pragma unroll
                            for (int mt = 0; mt < MT; ++mt) {
                                a[mt][0] = pair4<Tr::PV_F16>(r0, 2 * mt);
                                a[mt][1] = pair4<Tr::PV_F16>(r0, 2 * mt + 1);
                                a[mt][2] = pair4<Tr::PV_F16>(r1, 2 * mt);
                                a[mt][3] = pair4<Tr::PV_F16>(r1, 2 * mt + 1);
                            }
                        } else { // chunks 2 warp, 2 warp + 1 (16 codes each) of tokens 0-7 / 8-15
                            const int mi = lane >> 3;
                            const int tv = kk * 16 + (mi >> 1) * 8 + (lane & 7);
                            uint32_t vrow_base = vst;
                            if constexpr (Tr::TIER) // int4 rows: their widened codes in the side buffer
                                if (!((((tv < 32) ? hot_lo : hot_hi) >> (tv & 31)) & 1u))
                                    vrow_base = smem_u32(smem + Ly::off_vexp);
                            uint32_t r[4];
                            ldsm_x4_t(r[0], r[1], r[2], r[3],
                                      vrow_base + tv * Tr::ROWB + (((2 * warp + (mi & 1)) ^ xs) << 4));
    #pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                a[0][q] = pair8<FMT, Tr::PV_F16>(r[q], false);
                                a[1][q] = pair8<FMT, Tr::PV_F16>(r[q], true);
                            }
                        }
    #pragma unroll
                        for (int mt = 0; mt < MT; ++mt)
    #pragma unroll
                            for (int j = 0; j < NJ; ++j) mma16816<Tr::PV_F16>(o[mt][j], a[mt], pb[j][0], pb[j][1]);
                    } else {
    #pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            uint32_t a[4];
                            ldsm_x4_t(a[0], a[1], a[2], a[3],
                                      vrow + kk * 16 * BF_ROW + (((4 * warp + 2 * mt) << 4) ^ vx));
    #pragma unroll
                            for (int j = 0; j < NJ; ++j) mma16816<Tr::PV_F16>(o[mt][j], a, pb[j][0], pb[j][1]);
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(s));

        // ------------------------------------------------------------ epilogue
        if (last) {
            const int L = segL[b];
            const bool complete = (seg_j0 == 0) && (cc.j1 == L);
            const int sid = b * Hkv + g;
            // The head of a segment that this CTA's range ends in. Every other
            // contributor starts its range inside the segment, so it has usually
            // finished its piece and taken its ticket long before: then (at most
            // two of them) this CTA merges their partials with its own right after
            // the loop, and neither writes its own partial nor takes a ticket.
            const bool head_split = !complete && cc.kseg != 0;
            int n_other = 0;
            if (head_split) {
                unsigned Fs, c_first, c_last;
                seg_range(sid, Fs, c_first, c_last);
                n_other = static_cast<int>(c_last - c_first); // c_first is this CTA
                if (tid == 0) {
                    const bool all_in = n_other <= 2 && ld_relaxed(p.cnt + sid) == n_other;
                    if (all_in) fence_acq_rel_gpu(); // acquire: their partials precede
                    misc[4] = all_in ? 1 : 0;
                }
            }
            float la = l0, lb = l1;
            la += __shfl_xor_sync(0xFFFFFFFFu, la, 1);
            la += __shfl_xor_sync(0xFFFFFFFFu, la, 2);
            lb += __shfl_xor_sync(0xFFFFFFFFu, lb, 1);
            lb += __shfl_xor_sync(0xFFFFFFFFu, lb, 2);
            if (c == 0) {
                lred[warp * 16 + r] = la;
                lred[warp * 16 + r + 8] = lb;
            }
            consumer_sync();
            auto ltot = [&](int h) {
                float t = 0.f;
#pragma unroll
                for (int w = 0; w < NW; ++w) t += lred[w * 16 + h];
                return t;
            };
            const int hA = 2 * c, hB = 2 * c + 1, hC = 8 + 2 * c, hD = 9 + 2 * c;
            // output dims of accumulator rows r and r + 8 of m-tile mt: 16-dim blocks,
            // or (register-dequant pools) the warp's 32 dims spread over its two
            // m-tiles -- 8-bit codes: tile mt holds dims 2i + mt of both 16-dim chunks;
            // 4-bit codes: tile mt holds dims 4i + 2 mt and 4i + 2 mt + 1
            auto dim_a = [&](int mt) {
                return Tr::RQ ? (Tr::NIB4 ? warp * DPW + 4 * r + 2 * mt : warp * DPW + 2 * r + mt)
                              : warp * DPW + mt * 16 + r;
            };
            auto dim_b = [&](int mt) { return dim_a(mt) + (Tr::RQ ? (Tr::NIB4 ? 1 : 16) : 8); };
            // per-slot V scales: O was accumulated against m_h + E_h; back to m_h
            auto esc = [&](int h) { return VSH ? ex2(eref[v * 16 + h]) : 1.f; };
            const float eA = esc(hA), eB = esc(hB);
            const float eC = c < 2 ? esc(hC) : 1.f, eD = c < 2 ? esc(hD) : 1.f;
            const float fA = complete ? __fdividef(out_scale, ltot(hA)) * eA : eA;
            const float fB = complete ? __fdividef(out_scale, ltot(hB)) * eB : eB;
            const float fC = (complete && c < 2) ? __fdividef(out_scale, ltot(hC)) * eC : eC;
            const float fD = (complete && c < 2) ? __fdividef(out_scale, ltot(hD)) * eD : eD;
            __nv_bfloat16* const outb = p.out + b * p.o_sb + (long long)(g * GROUP) * p.o_sh;
            float* const part = reinterpret_cast<float*>(
                p.part + ((long long)blockIdx.x * 2 + (cc.kseg == 0 ? 0 : 1)) * PART_BYTES);
            auto put = [&](int h, int d, float val) {
                if (complete)
                    outb[h * p.o_sh + d] = __float2bfloat16_rn(val);
                else
                    part[h * D + d] = val;
            };
            // this thread's values: [mt][A dA, B dA, A dB, B dB, C dA, D dA, C dB, D dB]
            float val[MT][8];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if constexpr (NJ == 3) { // hi + lo columns
                        val[mt][e] = o[mt][0][e] + o[mt][1][e];
                        val[mt][4 + e] = o[mt][2][e] + __shfl_xor_sync(0xFFFFFFFFu, o[mt][2][e], 2);
                    } else {
                        val[mt][e] = o[mt][0][e];
                        val[mt][4 + e] = o[mt][1][e];
                    }
                }
            }
            if (head_split && misc[4] != 0) {
                // keep the unnormalised own partial in shared memory; it is merged
                // with the other contributors' after the loop (this is the range's
                // last piece)
                float* const st = reinterpret_cast<float*>(smem + Ly::off_stash);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const int dA = dim_a(mt), dB = dim_b(mt);
                    st[hA * D + dA] = val[mt][0] * eA;
                    st[hB * D + dA] = val[mt][1] * eB;
                    st[hA * D + dB] = val[mt][2] * eA;
                    st[hB * D + dB] = val[mt][3] * eB;
                    if (c < 2) {
                        st[hC * D + dA] = val[mt][4] * eC;
                        st[hD * D + dA] = val[mt][5] * eD;
                        st[hC * D + dB] = val[mt][6] * eC;
                        st[hD * D + dB] = val[mt][7] * eD;
                    }
                }
                if (tid < GROUP) {
                    st[GROUP * D + tid] = mref[v * 16 + tid];
                    st[GROUP * D + GROUP + tid] = ltot(tid);
                }
                mstate[2] = sid;
                mstate[3] = n_other;
            } else {
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const int dA = dim_a(mt), dB = dim_b(mt);
                    put(hA, dA, val[mt][0] * fA);
                    put(hB, dA, val[mt][1] * fB);
                    put(hA, dB, val[mt][2] * fA);
                    put(hB, dB, val[mt][3] * fB);
                    if (c < 2) {
                        put(hC, dA, val[mt][4] * fC);
                        put(hD, dA, val[mt][5] * fD);
                        put(hC, dB, val[mt][6] * fC);
                        put(hD, dB, val[mt][7] * fD);
                    }
                }
                if (!complete) {
                    // split segment: leave the partial (m, l next to O) for the merge
                    if (tid < GROUP) {
                        part[GROUP * D + tid] = mref[v * 16 + tid];
                        part[GROUP * D + GROUP + tid] = ltot(tid);
                    }
                    if (cc.kseg == 0) {
                        // the range's first piece: take its arrival ticket now, so the
                        // CTA holding the segment's head can merge it directly
                        mstate[0] = sid;
                        consumer_sync();
                        if (tid == 0) {
                            __threadfence(); // release: the partial precedes the ticket
                            mstate[4] = atomicAdd(p.cnt + sid, 1);
                        }
                    } else {
                        mstate[1] = sid; // ticket taken after the whole range is streamed
                    }
                }
            }
            // no trailing barrier: lred is next written in a later epilogue, and
            // every stage in between passes the per-stage consumer barrier
        }
        cursor_advance(cc, t_end, segL, p.bs);
        buf ^= 1;
    }

    // ------------------------------------------------ direct merge of the last head
    const int pend0 = mstate[0], pend1 = mstate[1], dsid = mstate[2], dn = mstate[3];
    // Other contributors (CTAs blockIdx+1 .. blockIdx+dn, slot 0: the segment is the
    // first piece of their ranges) had all arrived when the epilogue checked.
    if (dsid >= 0) {
        consumer_sync(); // the stash is complete
        constexpr int CH = GROUP * (D / 4) / NCT;
        const float* const st = reinterpret_cast<const float*>(smem + Ly::off_stash);
        const int b = dsid / Hkv, g = dsid - b * Hkv;
        __nv_bfloat16* const outb = p.out + b * p.o_sb + (long long)(g * GROUP) * p.o_sh;
        const float ninf = -INFINITY;
#pragma unroll
        for (int e = 0; e < CH; ++e) {
            const int ch = tid + e * NCT, h = ch / (D / 4), d0 = (ch % (D / 4)) * 4;
            float mk[2], lk[2];
            float4 ok[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                if (k >= dn) continue;
                const float* const pk = reinterpret_cast<const float*>(
                    p.part + static_cast<size_t>((blockIdx.x + 1u + k) * 2u) * PART_BYTES);
                mk[k] = __ldcg(pk + GROUP * D + h);
                lk[k] = __ldcg(pk + GROUP * D + GROUP + h);
                ok[k] = __ldcg(reinterpret_cast<const float4*>(pk + h * D + d0));
            }
            const float mo = st[GROUP * D + h];
            float M = mo;
#pragma unroll
            for (int k = 0; k < 2; ++k)
                if (k < dn) M = fmaxf(M, mk[k]);
            const float wo = ex2(mo - M);
            float den = wo * st[GROUP * D + GROUP + h];
            float4 acc = *reinterpret_cast<const float4*>(st + h * D + d0);
            acc.x *= wo;
            acc.y *= wo;
            acc.z *= wo;
            acc.w *= wo;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                if (k >= dn) continue;
                const float w = mk[k] == ninf ? 0.f : ex2(mk[k] - M);
                den = fmaf(w, lk[k], den);
                acc.x = fmaf(w, ok[k].x, acc.x);
                acc.y = fmaf(w, ok[k].y, acc.y);
                acc.z = fmaf(w, ok[k].z, acc.z);
                acc.w = fmaf(w, ok[k].w, acc.w);
            }
            const float f = __fdividef(out_scale, den);
            *reinterpret_cast<uint2*>(outb + h * p.o_sh + d0) =
                make_uint2(pack_bf16x2(acc.x * f, acc.y * f), pack_bf16x2(acc.z * f, acc.w * f));
        }
        if (tid == 0) atomicExch(p.cnt + dsid, 0);
    }

    // ------------------------------------------------ deferred split merges
    // Each split segment's partials are merged by the CTA that arrives last on
    // its counter; the merger resets the counter to zero. The partial stores of
    // all consumer threads precede thread 0's acq_rel ticket through the
    // barrier (release), and the merger's reads follow its ticket (acquire).
    // Segments split on their own (misc[22] = n): this CTA's one piece is
    // contributor r of the n CTAs of segment pend0, all of which stored their
    // partial and took a ticket.
    // Once the n tickets are in, each contributor merges float4 columns r, r + n,
    // ... of the segment's 12 x 256 outputs from the n partials in CTA order; a
    // second round of arrivals on the counter ends at 2n, and the contributor
    // that brings it there resets it.
    if (pend0 >= 0 && misc[22] != 0) {
        const unsigned n = static_cast<unsigned>(misc[22]), r = blockIdx.x % n, cf = blockIdx.x - r;
        if (tid == 0) {
            bool ok = true;
            if (mstate[4] == static_cast<int>(n) - 1)
                fence_acq_rel_gpu(); // the last ticket: every other partial precedes it
            else
                ok = wait_count(p.cnt + pend0, static_cast<int>(n), p.err);
            misc[2] = ok ? 1 : 0;
        }
        if (consumer_sync_or(*abort_flag != 0) || misc[2] == 0) return;
        const int b = pend0 / Hkv, g = pend0 - b * Hkv;
        __nv_bfloat16* const outb = p.out + b * p.o_sb + (long long)(g * GROUP) * p.o_sh;
        const float ninf = -INFINITY;
        for (unsigned f = r + n * static_cast<unsigned>(tid); f < GROUP * D / 4; f += n * NCT) {
            const int h = static_cast<int>(f) / (D / 4), d0 = (static_cast<int>(f) % (D / 4)) * 4;
            const float* const p0 = reinterpret_cast<const float*>(p.part + static_cast<size_t>(cf * 2u) * PART_BYTES);
            constexpr size_t PSTEP = 2 * PART_BYTES / 4; // floats from one CTA's slot 0 to the next's
            float M = ninf;
#pragma unroll 4
            for (unsigned i = 0; i < n; ++i) M = fmaxf(M, __ldcg(p0 + i * PSTEP + GROUP * D + h));
            float den = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
            for (unsigned i = 0; i < n; ++i) {
                const float* const pk = p0 + i * PSTEP;
                const float m = __ldcg(pk + GROUP * D + h);
                const float w = m == ninf ? 0.f : ex2(m - M);
                const float l = __ldcg(pk + GROUP * D + GROUP + h);
                const float4 o = __ldcg(reinterpret_cast<const float4*>(pk + h * D + d0));
                den = fmaf(w, l, den);
                acc.x = fmaf(w, o.x, acc.x);
                acc.y = fmaf(w, o.y, acc.y);
                acc.z = fmaf(w, o.z, acc.z);
                acc.w = fmaf(w, o.w, acc.w);
            }
            const float fo = __fdividef(out_scale, den);
            *reinterpret_cast<uint2*>(outb + h * p.o_sh + d0) =
                make_uint2(pack_bf16x2(acc.x * fo, acc.y * fo), pack_bf16x2(acc.z * fo, acc.w * fo));
        }
        consumer_sync(); // every consumer thread's reads precede the release
        if (tid == 0) {
            __threadfence();
            if (atomicAdd(p.cnt + pend0, 1) == static_cast<int>(2 * n) - 1) atomicExch(p.cnt + pend0, 0);
        }
        return;
    }

    if (pend0 >= 0 || pend1 >= 0) {
        consumer_sync(); // every consumer thread's partial stores precede the release below
        if (tid == 0) {
            int last[2] = {0, 0};
            // pend0's ticket was taken when its partial was stored; pend1's is now
            if (pend1 >= 0) __threadfence(); // release: the partial stores precede it
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int sid = q == 0 ? pend0 : pend1;
                if (sid < 0) continue;
                unsigned Fs, cf, cl;
                seg_range(sid, Fs, cf, cl);
                const int ticket = q == 0 ? mstate[4] : atomicAdd(p.cnt + sid, 1);
                last[q] = ticket == static_cast<int>(cl - cf) ? 1 : 0;
            }
            if (last[0] || last[1]) __threadfence(); // acquire: the merge reads follow
            misc[2] = last[0];
            misc[3] = last[1];
        }
        // The merges this CTA owns (at most two segments) are cut into batches of
        // up to MERGE_BATCH contributors. Whole partials come by bulk copy (TMA
        // engine) into two alternating shared-memory buffers over the idle stage
        // ring, so one batch lands while the previous one is combined; a
        // segment's running (M, den, acc) is rescaled once per batch.
        if (consumer_sync_or(*abort_flag != 0)) return; // a wait ran out: partials untrustworthy
        int nq0 = 0, nq1 = 0;
        unsigned cf0 = 0, cf1 = 0, fs0 = 0, fs1 = 0;
        {
            unsigned Fs, c_first, c_last;
            if (pend0 >= 0 && misc[2]) {
                seg_range(pend0, Fs, c_first, c_last);
                nq0 = static_cast<int>(c_last - c_first) + 1;
                cf0 = c_first;
                fs0 = cta_begin(c_first, N, G) < Fs ? 1u : 0u;
            }
            if (pend1 >= 0 && misc[3]) {
                seg_range(pend1, Fs, c_first, c_last);
                nq1 = static_cast<int>(c_last - c_first) + 1;
                cf1 = c_first;
                fs1 = cta_begin(c_first, N, G) < Fs ? 1u : 0u;
            }
        }
        constexpr int MB = Ly::MB;
        const int nb0 = (nq0 + MB - 1) / MB;
        const int nbatch = nb0 + (nq1 + MB - 1) / MB;
        if (nbatch == 0) return;
        uint8_t* const mbuf = smem + Ly::off_stage;
        // batch k -> (segment q, first contributor, count)
        auto batch = [&](int k, int& q, int& k0, int& n) {
            q = k < nb0 ? 0 : 1;
            k0 = (q == 0 ? k : k - nb0) * MB;
            n = min(MB, (q == 0 ? nq0 : nq1) - k0);
        };
        auto issue = [&](int k) { // thread 0 only
            int q, k0, n;
            batch(k, q, k0, n);
            const uint32_t bar = merge_bar(k & 1);
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n * PART_BYTES));
            for (int j = 0; j < n; ++j) {
                const unsigned cta = (q == 0 ? cf0 : cf1) + static_cast<unsigned>(k0 + j);
                const unsigned slot = j + k0 == 0 ? (q == 0 ? fs0 : fs1) : 0u;
                bulk_g2s(smem_u32(mbuf + ((k & 1) * MB + j) * PART_BYTES),
                         p.part + static_cast<size_t>(cta * 2u + slot) * PART_BYTES, PART_BYTES,
                         bar);
            }
        };
        // earlier generic accesses of the stage ring (this CTA) and the other
        // CTAs' partial stores (acquired through the tickets) before the async proxy
        fence_proxy_async_all();
        consumer_sync();
        if (tid == 0) {
            issue(0);
            if (nbatch > 1) issue(1);
        }
        constexpr int CH = GROUP * (D / 4) / NCT; // float4 chunks per thread (3)
        static_assert(GROUP * (D / 4) % NCT == 0, "merge chunking");
        const float ninf = -INFINITY;
        int hh[CH], dd[CH];
        float M[CH], den[CH];
        float4 acc[CH];
#pragma unroll
        for (int e = 0; e < CH; ++e) {
            const int ch = tid + e * NCT;
            hh[e] = ch / (D / 4);
            dd[e] = (ch % (D / 4)) * 4;
            M[e] = ninf;
            den[e] = 0.f;
            acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll 1
        for (int k = 0; k < nbatch; ++k) {
            int q, k0, n;
            batch(k, q, k0, n);
            const bool landed = mbar_wait_copies(merge_bar(k & 1), (k >> 1) & 1, p.err);
            const float* const pb =
                reinterpret_cast<const float*>(mbuf + (k & 1) * MB * PART_BYTES);
            constexpr int PF = PART_BYTES / 4;
            float Mb[CH];
#pragma unroll
            for (int e = 0; e < CH; ++e) Mb[e] = M[e];
            for (int j = 0; j < n; ++j) {
#pragma unroll
                for (int e = 0; e < CH; ++e) Mb[e] = fmaxf(Mb[e], pb[j * PF + GROUP * D + hh[e]]);
            }
#pragma unroll
            for (int e = 0; e < CH; ++e) {
                // a contributor's m never exceeds Mb; an empty one (m = -inf) weighs 0
                const float r = M[e] == ninf ? 0.f : ex2(M[e] - Mb[e]);
                den[e] *= r;
                acc[e].x *= r;
                acc[e].y *= r;
                acc[e].z *= r;
                acc[e].w *= r;
                M[e] = Mb[e];
            }
            for (int j = 0; j < n; ++j) {
                const float* const pk = pb + j * PF;
#pragma unroll
                for (int e = 0; e < CH; ++e) {
                    const float mv = pk[GROUP * D + hh[e]];
                    const float w = mv == ninf ? 0.f : ex2(mv - M[e]);
                    const float4 ov = *reinterpret_cast<const float4*>(pk + hh[e] * D + dd[e]);
                    den[e] = fmaf(w, pk[GROUP * D + GROUP + hh[e]], den[e]);
                    acc[e].x = fmaf(w, ov.x, acc[e].x);
                    acc[e].y = fmaf(w, ov.y, acc[e].y);
                    acc[e].z = fmaf(w, ov.z, acc[e].z);
                    acc[e].w = fmaf(w, ov.w, acc[e].w);
                }
            }
            // this buffer's reads precede the bulk copy that refills it; a batch
            // that did not land in time ends the merge for every consumer thread
            // (after one more bounded wait for copies still in flight)
            fence_proxy_async();
            if (consumer_sync_or(!landed)) {
                mbar_wait_copies(merge_bar(k & 1), (k >> 1) & 1, p.err);
                if (nbatch > k + 1) mbar_wait_copies(merge_bar((k + 1) & 1), ((k + 1) >> 1) & 1, p.err);
                return;
            }
            if (tid == 0 && k + 2 < nbatch) issue(k + 2);
            if (k0 + n == (q == 0 ? nq0 : nq1)) { // the segment's last batch: normalise and store
                const int sid = q == 0 ? pend0 : pend1;
                const int b = sid / Hkv, g = sid - b * Hkv;
                __nv_bfloat16* const outb = p.out + b * p.o_sb + (long long)(g * GROUP) * p.o_sh;
#pragma unroll
                for (int e = 0; e < CH; ++e) {
                    const float f = __fdividef(out_scale, den[e]);
                    *reinterpret_cast<uint2*>(outb + hh[e] * p.o_sh + dd[e]) =
                        make_uint2(pack_bf16x2(acc[e].x * f, acc[e].y * f),
                                   pack_bf16x2(acc[e].z * f, acc[e].w * f));
                    M[e] = ninf;
                    den[e] = 0.f;
                    acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
                if (tid == 0) atomicExch(p.cnt + sid, 0);
            }
        }
    }
}

} // namespace qsa

// ====================================================================== host

// Shared with the other translation units of libqsa (not exported): record the
// message qsa_last_error_message() returns on this thread.
__attribute__((visibility("hidden"))) void qsa_detail_set_error(const char* msg);

namespace {

using namespace qsa;

thread_local std::string g_last_error;

} // namespace

__attribute__((visibility("hidden"))) void qsa_detail_set_error(const char* msg) {
    g_last_error = msg ? msg : "";
}

namespace {

int fail(int code, const char* fmt, ...) {
    char msg[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(msg, sizeof msg, fmt, ap);
    va_end(ap);
    g_last_error = msg;
    return code;
}

struct DeviceState {
    int sms = 0;
    bool smem_set[QSA_KV_INT8RING_INT4 + 1] = {};
};

std::mutex g_mu;
DeviceState g_dev[64];

int current_device(int* dev, int* sms) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return fail(QSA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (*dev < 0 || *dev >= 64) return fail(QSA_ERR_CUDA, "device ordinal %d out of range", *dev);
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& st = g_dev[*dev];
    if (st.sms == 0) {
        e = cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, *dev);
        if (e != cudaSuccess)
            return fail(QSA_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    }
    *sms = st.sms;
    return QSA_OK;
}

int check_sizes(int32_t bs, int32_t num_q_heads, int32_t capacity) {
    if (bs < 1 || bs > MAX_BS)
        return fail(QSA_ERR_UNSUPPORTED, "batch size %d outside the supported 1..%d", bs, MAX_BS);
    if (num_q_heads != 12 && num_q_heads != 24)
        return fail(QSA_ERR_UNSUPPORTED,
                    "%d query heads: the decode contract is 24 (TP1, 2 KV heads) or 12 (TP2, 1 KV head)",
                    num_q_heads);
    if (capacity < 1 || capacity > MAX_CAPACITY)
        return fail(QSA_ERR_UNSUPPORTED, "selected-KV capacity %d outside the supported 1..%d",
                    capacity, MAX_CAPACITY);
    return QSA_OK;
}

long long grid_for(int32_t bs, int32_t num_q_heads, int32_t capacity, int32_t max_ctas, int sms) {
    const long long hkv = num_q_heads / GROUP;
    const long long work = (long long)bs * hkv * capacity;
    long long g = (work + MIN_TOKENS_PER_CTA - 1) / MIN_TOKENS_PER_CTA;
    if (g > sms) g = sms;
    if (max_ctas > 0 && g > max_ctas) g = max_ctas;
    return g < 1 ? 1 : g;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

void layout_for(int32_t bs, int32_t num_q_heads, long long grid, qsa_scratch_layout* ly) {
    const size_t hkv = num_q_heads / GROUP;
    ly->error_word_offset = 0;
    ly->counters_offset = 256;
    ly->counters_count = (size_t)bs * hkv;
    ly->partials_offset = 256 + align_up(ly->counters_count * 4, 256);
    ly->partial_slot_bytes = PART_BYTES;
    ly->total_bytes = ly->partials_offset + (size_t)grid * 2 * PART_BYTES;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

#ifdef QSA_TEST_HOOKS
// Test build only (libqsa_testhooks.so, compiled with -DQSA_TEST_HOOKS; the shipped
// libqsa.so has none of this): qsa_test_set_stall_stage(k) makes CTA 0's producers
// of the following launches never complete their k-th stage. Its consumers' wait
// then runs out (WAIT_NS), the launch records QSA_DEVERR_TIMEOUT and ends; nothing
// faults and nothing spins without a limit. k < 0 turns it off.
int g_test_stall_stage = -1;
#endif

int check_row_tensor(const qsa_tensor* t, const char* name, int bs, int hq) {
    if (t->dtype != QSA_DTYPE_BF16)
        return fail(QSA_ERR_UNSUPPORTED, "%s must be bf16 (dtype %d given)", name, t->dtype);
    if (t->ndim != 3 || t->shape[0] != bs || t->shape[1] != hq || t->shape[2] != D)
        return fail(QSA_ERR_INVALID_ARGUMENT, "%s must be [bs=%d, Hq=%d, 256]", name, bs, hq);
    if (t->stride[2] != 1)
        return fail(QSA_ERR_INVALID_ARGUMENT, "%s must be contiguous along the head dimension", name);
    if (t->stride[0] % 8 != 0 || t->stride[1] % 8 != 0 || t->stride[0] < 0 || t->stride[1] < 0)
        return fail(QSA_ERR_MISALIGNED, "%s strides must be non-negative multiples of 8 elements",
                    name);
    if (t->data == nullptr) return fail(QSA_ERR_INVALID_ARGUMENT, "%s data is NULL", name);
    if (!aligned16(t->data)) return fail(QSA_ERR_MISALIGNED, "%s must be 16-byte aligned", name);
    return QSA_OK;
}

template <int FMT> const void* kernel_ptr() { return reinterpret_cast<const void*>(&qsa_decode_kernel<FMT>); }

template <int FMT>
int launch(const Params& prm, int grid, int dev, cudaStream_t stream) {
    constexpr int smem = Layout<FMT>::TOTAL;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_dev[dev].smem_set[FMT]) {
            cudaError_t e = cudaFuncSetAttribute(qsa_decode_kernel<FMT>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess)
                return fail(QSA_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            g_dev[dev].smem_set[FMT] = true;
        }
    }
    // programmatic dependent launch: the kernel waits for the previous grid
    // itself (griddepcontrol.wait) before it touches global memory. Small
    // batches (at most 64 segments, whose CTAs may wait for each other in the
    // merge) launch cooperatively, so all their CTAs are resident together
    // whatever else runs on the device (the grid is at most one CTA per SM).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = prm.bs * prm.Hkv <= static_cast<int>(UNIFORM_SEGMENTS) ? 2 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, qsa_decode_kernel<FMT>, prm);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(QSA_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
    return QSA_OK;
}

} // namespace

extern "C" {

int qsa_version(void) { return 100; }

const char* qsa_strerror(int code) {
    switch (code) {
    case QSA_OK: return "success";
    case QSA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case QSA_ERR_UNSUPPORTED: return "outside the packed QSA decode contract";
    case QSA_ERR_SCRATCH_TOO_SMALL: return "scratch buffer too small";
    case QSA_ERR_MISALIGNED: return "misaligned pointer or stride";
    case QSA_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown error";
    }
}

const char* qsa_last_error_message(void) { return g_last_error.c_str(); }

int32_t qsa_decode_grid(int32_t bs, int32_t num_q_heads, int32_t capacity, int32_t max_ctas) {
    int rc = check_sizes(bs, num_q_heads, capacity);
    if (rc != QSA_OK) return rc;
    int dev, sms;
    rc = current_device(&dev, &sms);
    if (rc != QSA_OK) return rc;
    return static_cast<int32_t>(grid_for(bs, num_q_heads, capacity, max_ctas, sms));
}

int qsa_decode_scratch_layout(int32_t bs, int32_t num_q_heads, int32_t capacity,
                              qsa_scratch_layout* layout) {
    if (layout == nullptr) return fail(QSA_ERR_INVALID_ARGUMENT, "layout is NULL");
    int rc = check_sizes(bs, num_q_heads, capacity);
    if (rc != QSA_OK) return rc;
    int dev, sms;
    rc = current_device(&dev, &sms);
    if (rc != QSA_OK) return rc;
    layout_for(bs, num_q_heads, grid_for(bs, num_q_heads, capacity, 0, sms), layout);
    return QSA_OK;
}

size_t qsa_decode_scratch_bytes(int32_t bs, int32_t num_q_heads, int32_t capacity) {
    qsa_scratch_layout ly;
    if (qsa_decode_scratch_layout(bs, num_q_heads, capacity, &ly) != QSA_OK) return 0;
    return ly.total_bytes;
}

int qsa_scratch_init(void* scratch, size_t scratch_bytes, void* stream) {
    if (scratch == nullptr) return fail(QSA_ERR_INVALID_ARGUMENT, "scratch is NULL");
    cudaError_t e = cudaMemsetAsync(scratch, 0, scratch_bytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(QSA_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
    return QSA_OK;
}

int qsa_scratch_error(const void* scratch, int32_t* flags, int32_t clear, void* stream) {
    if (scratch == nullptr || flags == nullptr)
        return fail(QSA_ERR_INVALID_ARGUMENT, "scratch and flags must be non-NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t host = 0;
    cudaError_t e = cudaMemcpyAsync(&host, scratch, sizeof host, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && clear)
        e = cudaMemsetAsync(const_cast<void*>(scratch), 0, sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return fail(QSA_ERR_CUDA, "error-word readback: %s", cudaGetErrorString(e));
    *flags = host;
    return QSA_OK;
}

int qsa_decode(const qsa_tensor* q, const qsa_tensor* k_pool, const qsa_tensor* v_pool,
               const qsa_kv_quant_meta* meta, const qsa_tensor* sel, const qsa_tensor* cu,
               const qsa_tensor* out, void* scratch, size_t scratch_bytes, void* stream) {
    if (!q || !k_pool || !v_pool || !meta || !sel || !cu || !out)
        return fail(QSA_ERR_INVALID_ARGUMENT, "a descriptor pointer is NULL");
    const int fmt = meta->format;
    if (fmt < QSA_KV_BF16 || fmt > QSA_KV_INT8RING_INT4)
        return fail(QSA_ERR_UNSUPPORTED, "unknown K/V pool format %d", fmt);
    if (q->ndim != 3) return fail(QSA_ERR_INVALID_ARGUMENT, "q must be [bs, Hq, 256]");
    const int64_t bs64 = q->shape[0], hq64 = q->shape[1];
    if (q->shape[2] != D)
        return fail(QSA_ERR_UNSUPPORTED, "head dim %lld: the decode contract is D = 256",
                    (long long)q->shape[2]);
    if (bs64 < 1 || bs64 > MAX_BS)
        return fail(QSA_ERR_UNSUPPORTED, "batch size %lld outside the supported 1..%d",
                    (long long)bs64, MAX_BS);
    if (hq64 != 12 && hq64 != 24)
        return fail(QSA_ERR_UNSUPPORTED,
                    "%lld query heads: the decode contract is 24 (TP1, 2 KV heads) or 12 (TP2, 1 KV head)",
                    (long long)hq64);
    const int bs = (int)bs64, hq = (int)hq64, hkv = hq / GROUP;
    int rc = check_sizes(bs, hq, meta->capacity);
    if (rc != QSA_OK) return rc;
    if ((rc = check_row_tensor(q, "q", bs, hq)) != QSA_OK) return rc;
    if ((rc = check_row_tensor(out, "out", bs, hq)) != QSA_OK) return rc;

    const int want_dtype = fmt == QSA_KV_BF16                              ? QSA_DTYPE_BF16
                           : (fmt == QSA_KV_INT8 || fmt == QSA_KV_INT8_G64) ? QSA_DTYPE_INT8
                                                                            : QSA_DTYPE_UINT8;
    const int64_t row_elems =
        (fmt == QSA_KV_INT4 || fmt == QSA_KV_INT4_G32 || fmt == QSA_KV_INT8RING_INT4) ? D / 2 : D;
    for (const qsa_tensor* pool : {k_pool, v_pool}) {
        const char* nm = pool == k_pool ? "k_pool" : "v_pool";
        if (pool->dtype != want_dtype)
            return fail(QSA_ERR_INVALID_ARGUMENT, "%s dtype %d does not match pool format %d", nm,
                        pool->dtype, fmt);
        if (pool->ndim != 3 || pool->shape[1] != hkv || pool->shape[2] != row_elems ||
            pool->shape[0] < 1)
            return fail(QSA_ERR_INVALID_ARGUMENT, "%s must be [num_slots, Hkv=%d, %lld]", nm, hkv,
                        (long long)row_elems);
        if (pool->stride[2] != 1 || pool->stride[1] != row_elems ||
            pool->stride[0] != hkv * row_elems)
            return fail(QSA_ERR_INVALID_ARGUMENT, "%s must be contiguous", nm);
        if (pool->data == nullptr) return fail(QSA_ERR_INVALID_ARGUMENT, "%s data is NULL", nm);
        if (!aligned16(pool->data)) return fail(QSA_ERR_MISALIGNED, "%s must be 16-byte aligned", nm);
    }
    if (k_pool->shape[0] != v_pool->shape[0])
        return fail(QSA_ERR_INVALID_ARGUMENT, "k_pool and v_pool hold different slot counts");
    if (sel->dtype != QSA_DTYPE_INT32 || sel->ndim != 1 || (sel->shape[0] > 1 && sel->stride[0] != 1) ||
        sel->shape[0] < 0)
        return fail(QSA_ERR_INVALID_ARGUMENT, "sel_indices must be a contiguous int32 vector");
    if (sel->shape[0] > 0 && sel->data == nullptr)
        return fail(QSA_ERR_INVALID_ARGUMENT, "sel_indices data is NULL");
    if (sel->shape[0] > INT32_MAX)
        return fail(QSA_ERR_UNSUPPORTED, "sel_indices longer than 2^31 - 1");
    if (cu->dtype != QSA_DTYPE_INT32 || cu->ndim != 1 || cu->shape[0] != bs + 1 ||
        cu->stride[0] != 1 || cu->data == nullptr)
        return fail(QSA_ERR_INVALID_ARGUMENT, "cu_seqlens must be a contiguous int32 [bs + 1]");
    if (!std::isfinite(meta->softmax_scale))
        return fail(QSA_ERR_INVALID_ARGUMENT, "softmax_scale must be finite");
    if (fmt != QSA_KV_BF16) {
        if (meta->k_scale == nullptr || meta->v_scale == nullptr)
            return fail(QSA_ERR_INVALID_ARGUMENT, "quantised pools need k_scale and v_scale");
        // grouped pools read a token's binary16 scales with one 8- or 16-byte copy
        const uintptr_t al = fmt == QSA_KV_INT8_G64                                  ? 8
                             : (fmt == QSA_KV_INT4_G32 || fmt == QSA_KV_INT8RING_INT4) ? 16
                                                                                       : 4;
        if ((reinterpret_cast<uintptr_t>(meta->k_scale) & (al - 1)) ||
            (reinterpret_cast<uintptr_t>(meta->v_scale) & (al - 1)))
            return fail(QSA_ERR_MISALIGNED, "scales must be %d-byte aligned for this format", (int)al);
    }
    const qsa_kv_tier* tier = meta->tier;
    if (fmt == QSA_KV_INT8RING_INT4) {
        if (tier == nullptr) return fail(QSA_ERR_INVALID_ARGUMENT, "the tiered format needs kv_quant_meta->tier");
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
    }
    if (scratch == nullptr) return fail(QSA_ERR_INVALID_ARGUMENT, "scratch is NULL");
    if (reinterpret_cast<uintptr_t>(scratch) & 255u)
        return fail(QSA_ERR_MISALIGNED, "scratch must be 256-byte aligned");

    int dev, sms;
    if ((rc = current_device(&dev, &sms)) != QSA_OK) return rc;
    const long long grid = grid_for(bs, hq, meta->capacity, meta->max_ctas, sms);
    qsa_scratch_layout ly;
    layout_for(bs, hq, grid, &ly);
    if (scratch_bytes < ly.total_bytes)
        return fail(QSA_ERR_SCRATCH_TOO_SMALL, "scratch holds %zu bytes, this call needs %zu",
                    scratch_bytes, ly.total_bytes);

    Params prm;
    prm.q = static_cast<const __nv_bfloat16*>(q->data);
    prm.q_sb = q->stride[0];
    prm.q_sh = q->stride[1];
    prm.kpool = static_cast<const uint8_t*>(k_pool->data);
    prm.vpool = static_cast<const uint8_t*>(v_pool->data);
    prm.num_slots = k_pool->shape[0];
    prm.k_scale = meta->k_scale;
    prm.v_scale = meta->v_scale;
    prm.sel = static_cast<const int*>(sel->data);
    prm.n_sel = sel->shape[0];
    prm.cu = static_cast<const int*>(cu->data);
    prm.out = static_cast<__nv_bfloat16*>(out->data);
    prm.o_sb = out->stride[0];
    prm.o_sh = out->stride[1];
    uint8_t* base = static_cast<uint8_t*>(scratch);
    prm.err = reinterpret_cast<int*>(base + ly.error_word_offset);
    prm.cnt = reinterpret_cast<int*>(base + ly.counters_offset);
    prm.part = base + ly.partials_offset;
    prm.bs = bs;
    prm.Hkv = hkv;
    prm.capacity = meta->capacity;
    prm.scale_log2 = meta->softmax_scale * 1.4426950408889634f;
    prm.kring = prm.vring = nullptr;
    prm.kring_scale = prm.vring_scale = nullptr;
    prm.owner = nullptr;
    prm.ring_mask = 0;
#ifdef QSA_TEST_HOOKS
    prm.stall_stage = g_test_stall_stage;
#endif
    if (fmt == QSA_KV_INT8RING_INT4) {
        prm.kring = static_cast<const uint8_t*>(tier->k_ring);
        prm.vring = static_cast<const uint8_t*>(tier->v_ring);
        prm.kring_scale = tier->k_ring_scale;
        prm.vring_scale = tier->v_ring_scale;
        prm.owner = tier->owner;
        prm.ring_mask = tier->ring_slots - 1;
    }

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (fmt) {
    case QSA_KV_BF16: rc = launch<QSA_KV_BF16>(prm, (int)grid, dev, st); break;
    case QSA_KV_FP8_E4M3: rc = launch<QSA_KV_FP8_E4M3>(prm, (int)grid, dev, st); break;
    case QSA_KV_INT8: rc = launch<QSA_KV_INT8>(prm, (int)grid, dev, st); break;
    case QSA_KV_INT4: rc = launch<QSA_KV_INT4>(prm, (int)grid, dev, st); break;
    case QSA_KV_INT8_G64: rc = launch<QSA_KV_INT8_G64>(prm, (int)grid, dev, st); break;
    case QSA_KV_INT4_G32: rc = launch<QSA_KV_INT4_G32>(prm, (int)grid, dev, st); break;
    default: rc = launch<QSA_KV_INT8RING_INT4>(prm, (int)grid, dev, st); break;
    }
    if (rc == QSA_OK) g_last_error.clear();
    return rc;
}

#ifdef QSA_TEST_HOOKS
void qsa_test_set_stall_stage(int stage) { g_test_stall_stage = stage; }
#endif

} // extern "C"

// ============================================ decode without caller-provided scratch
//
// qsa_decode_static_scratch is qsa_decode for callers that cannot allocate
// device memory at call time. Its scratch is one file-scope device array of
// fixed size, created when the library is loaded and held by every GPU that
// loads it until the process exits.

namespace {

constexpr int STATIC_MAX_CTAS = 160;                 // grid cap of this entry point
constexpr size_t STATIC_HEADER_BYTES = 256 + 1024;   // error word + 256 counters
constexpr size_t STATIC_SCRATCH_BYTES =
    STATIC_HEADER_BYTES + (size_t)STATIC_MAX_CTAS * 2 * PART_BYTES; // 3,974,400 bytes

// Per device: the array's device address and the id of the context it was looked
// up in (under g_mu). A device reset (cudaDeviceReset) ends the primary context and
// unloads the module; the next context gets a new id and the address is looked up
// again instead of reusing the stale one.
struct StaticScratch {
    void* ptr = nullptr;
    unsigned long long ctx_id = 0;
};
StaticScratch g_static[64];

// Id of the calling thread's current CUDA context, unique for the life of the
// process (the CUDA driver API's cuCtxGetId, reached through the runtime's entry-point
// query); 0 when there is no current context or the query is unavailable.
unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(fn);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS ||
        ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

} // namespace

static __device__ __align__(256) unsigned char g_static_scratch[STATIC_SCRATCH_BYTES];

extern "C" int qsa_decode_static_scratch(const qsa_tensor* q, const qsa_tensor* k_pool,
                                         const qsa_tensor* v_pool,
                                         const qsa_kv_quant_meta* kv_quant_meta,
                                         const qsa_tensor* sel_indices,
                                         const qsa_tensor* cu_seqlens, const qsa_tensor* out,
                                         void* stream) {
    if (kv_quant_meta == nullptr) return fail(QSA_ERR_INVALID_ARGUMENT, "kv_quant_meta is NULL");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(QSA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(QSA_ERR_CUDA, "device ordinal %d out of range", dev);
    void* ptr = nullptr;
    {
        // Set-up, once per device (and again after a reset of its context), with that
        // device current: the array's name is only a host-side stand-in, so look up
        // its device address.
        std::lock_guard<std::mutex> lk(g_mu);
        StaticScratch& st = g_static[dev];
        const unsigned long long id = st.ptr ? current_context_id() : 0;
        if (st.ptr == nullptr || id == 0 || id != st.ctx_id) {
            void* addr = nullptr;
            e = cudaGetSymbolAddress(&addr, g_static_scratch);
            if (e != cudaSuccess)
                return fail(QSA_ERR_CUDA, "cudaGetSymbolAddress(static scratch): %s",
                            cudaGetErrorString(e));
            st.ptr = addr;
            st.ctx_id = current_context_id(); // the lookup made the primary context current
        }
        ptr = st.ptr;
    }
    // Cap the grid so the partial results fit the fixed array; any size the
    // decode contract admits then fits, and qsa_decode rejects the rest.
    qsa_kv_quant_meta meta = *kv_quant_meta;
    if (meta.max_ctas <= 0 || meta.max_ctas > STATIC_MAX_CTAS) meta.max_ctas = STATIC_MAX_CTAS;
    // The array keeps the previous call's contents: the error word and the
    // arrival counters must start at zero.
    e = cudaMemsetAsync(ptr, 0, STATIC_HEADER_BYTES, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(QSA_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
    return qsa_decode(q, k_pool, v_pool, &meta, sel_indices, cu_seqlens, out, ptr,
                      STATIC_SCRATCH_BYTES, stream);
}
