/*
 * qsa.h -- C ABI of libqsa: packed Qwen-sparse-attention (QSA) decode over a
 * paged, optionally quantised K/V pool, on one NVIDIA GB300 (sm_103a).
 *
 * The operation (sglang PR #36845 "fix(qsa): restore SM121 correctness",
 * sections "Changes" and "Optimized kernel"; sglang PR #37798 "quantized KV
 * pools with dequant-on-gather", section "Modifications"):
 *
 *   For every sequence b (one BF16 query token, Hq heads, head dim 256) with
 *   L_b = cu_seqlens[b+1] - cu_seqlens[b] selected token slots
 *   I_j = sel_indices[cu_seqlens[b] + j] (order and duplicates kept), and
 *   every query head h, whose KV head is g = h / 12 (12:1 GQA):
 *
 *     out[b,h,:] = sum_j softmax_j(softmax_scale * q[b,h,:] . K[I_j,g,:]) V[I_j,g,:]
 *
 *   with K/V dequantised from the pool format on gather. L_b == 0 gives a
 *   zero row. Supported geometry (the pages' contract): BF16 query/output,
 *   D = 256, Hq = 24 with Hkv = 2 (TP1) or Hq = 12 with Hkv = 1 (TP2),
 *   1 <= bs <= 128, 1 <= capacity <= 2055 selected slots per sequence.
 *   Calls outside it fail with QSA_ERR_UNSUPPORTED and a descriptive message.
 *
 * Ownership and ordering. The caller owns every buffer. The library never
 * allocates, frees or synchronises inside qsa_decode: it validates the
 * descriptors on the host (reading no device memory) and enqueues exactly one
 * kernel on `stream`. Live lengths are read from cu_seqlens on the device,
 * so a captured CUDA graph stays valid when cu_seqlens and sel_indices
 * change between replays. Kernels are launched with programmatic stream
 * serialization: a launch may become resident while the previous grid in the
 * stream drains, but it waits for that grid (griddepcontrol.wait) before it
 * reads or writes any global memory, so stream order holds as usual.
 *
 * Scratch. A caller-owned device buffer of qsa_decode_scratch_bytes() bytes,
 * zeroed once with qsa_scratch_init(). It holds a sticky device error word,
 * one arrival counter per (sequence, KV head) -- zero before and after every
 * launch, the kernel resets them in the same launch -- and the split-KV
 * partial results. Launches that share a scratch buffer must be ordered
 * (same stream or explicit dependencies).
 *
 * Residency. A small batch (at most 64 (sequence, KV head) segments) is
 * launched cooperatively: all its CTAs (never more than one per SM) become
 * resident together, waiting for SMs that kernels on other streams hold, so
 * the merge in which the CTAs of one segment wait, for at most 2 s, for each
 * other's partials always has all of them running.
 */
#ifndef QSA_H_
#define QSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types of qsa_tensor.dtype. */
enum {
    QSA_DTYPE_BF16 = 1,
    QSA_DTYPE_UINT8 = 2, /* fp8 e4m3fn codes and packed int4 nibbles */
    QSA_DTYPE_INT8 = 3,
    QSA_DTYPE_INT32 = 4,
    QSA_DTYPE_FLOAT32 = 5
};

/* K/V pool formats (qsa_kv_quant_meta.format), sglang PR #37798, "Modifications". */
enum {
    QSA_KV_BF16 = 0,     /* [slots, Hkv, 256] bf16 */
    QSA_KV_FP8_E4M3 = 1, /* [slots, Hkv, 256] uint8 e4m3fn codes, one fp32 scale per pool */
    QSA_KV_INT8 = 2,     /* [slots, Hkv, 256] int8, fp32 scale per (slot, KV head) */
    QSA_KV_INT4 = 3,     /* [slots, Hkv, 128] uint8: two's-complement nibbles, channel 2i
                            in the low nibble, fp32 scale per (slot, KV head) */
    QSA_KV_INT8_G64 = 4, /* [slots, Hkv, 256] int8, binary16 scale per (slot, KV head,
                            64-channel group): [slots, Hkv, 4]; group 0 = the rotary dims */
    QSA_KV_INT4_G32 = 5, /* [slots, Hkv, 128] uint8: offset-binary nibbles (code + 8,
                            code in [-7, 7]), channel 2i in the low nibble, binary16 scale
                            per (slot, KV head, 32-channel group): [slots, Hkv, 8] */
    QSA_KV_INT8RING_INT4 = 6 /* tiered: the pools and scales are the int4_g32 rows of every
                                slot; qsa_kv_quant_meta.tier holds the int8_g64 ring */
};

/* Return codes. Nothing is enqueued when a call returns an error. */
enum {
    QSA_OK = 0,
    QSA_ERR_INVALID_ARGUMENT = -1, /* NULL pointer, dtype/ndim/shape/stride mismatch */
    QSA_ERR_UNSUPPORTED = -2,      /* well-formed but outside the decode contract */
    QSA_ERR_SCRATCH_TOO_SMALL = -3,
    QSA_ERR_MISALIGNED = -4,       /* a base address or stride breaks 16-byte alignment */
    QSA_ERR_CUDA = -5              /* a CUDA runtime call or the launch failed */
};

/* Bits of the sticky device error word (see qsa_scratch_error). Bad data
 * never traps or hangs the GPU: the kernel records it and carries on with a
 * safe substitute, and the affected sequences' outputs are unspecified. */
enum {
    QSA_DEVERR_SLOT_RANGE = 1, /* a selected slot id outside [0, num_slots); slot 0 read instead */
    QSA_DEVERR_CU_SEQLENS = 2, /* cu_seqlens decreasing, negative, past the index buffer,
                                  or a length above capacity; the length is clamped */
    QSA_DEVERR_TIMEOUT = 4,    /* an internal wait exceeded its limit (2 s) and the launch
                                  gave up early (a library fault, not a data fault) */
    QSA_DEVERR_CTX_LEN = 8     /* qsa_topk_expand: a context length outside [0, capacity];
                                  it is clamped into that range */
};

/* A strided view of caller memory. `data` is a device pointer for
 * qsa_decode; strides are in elements. */
typedef struct {
    void* data;
    int32_t dtype;
    int32_t ndim;
    int64_t shape[4];
    int64_t stride[4];
} qsa_tensor;

/* The hot tier of a QSA_KV_INT8RING_INT4 pool (sglang PR #37798, "Modifications",
 * the tiered KV pool module): a ring of R int8_g64 rows with an owner table. Row
 * (slot, g) is read from ring row (slot & (R - 1), g) when owner[slot & (R - 1)]
 * == slot (hot), else from the int4_g32 pool (cold). Every token is written to
 * both (qsa_kv_write_tiered). The caller owns all of it; sizes are not checked. */
typedef struct {
    void* k_ring;       /* int8 [R, Hkv, 256] contiguous, 16-byte aligned */
    void* v_ring;
    void* k_ring_scale; /* binary16 [R, Hkv, 4] (per 64-channel group), 8-byte aligned */
    void* v_ring_scale;
    int32_t* owner;     /* int32 [R]: the slot whose row a ring position holds; -1: none */
    int32_t ring_slots; /* R: a power of two, 1 .. 2^30 */
} qsa_kv_tier;

/* Pool format and softmax parameters of one call. */
typedef struct {
    int32_t format;       /* QSA_KV_* */
    int32_t capacity;     /* max selected slots per sequence, 1..2055; bounds the split plan */
    const void* k_scale;  /* device; fp8: float [1]; int8/int4: float [slots * Hkv];
                             int8_g64 / int4_g32: binary16 [slots * Hkv * 4 / 8], 8- / 16-byte
                             aligned; bf16: NULL */
    const void* v_scale;  /* same layout as k_scale */
    float softmax_scale;  /* finite; 1/16 = 1/sqrt(256) for the pages' model */
    int32_t max_ctas;     /* 0: library chooses the grid; > 0: cap on CTAs (e.g. 1 forces
                             one CTA to do all the work, which tests the no-split path) */
    const qsa_kv_tier* tier; /* QSA_KV_INT8RING_INT4: the hot ring (host struct, read at
                                the call); other formats: ignored, may be NULL */
} qsa_kv_quant_meta;

/*
 * qsa_decode -- enqueue one packed QSA decode.
 *
 *  q           bf16 [bs, Hq, 256]; stride[2] == 1; stride[0], stride[1] multiples of 8;
 *              base 16-byte aligned.
 *  k_pool,     [num_slots, Hkv, row] contiguous; row = 256 elements (bf16, fp8 as
 *  v_pool      uint8, int8 and int8_g64 as int8) or 128 bytes (int4 / int4_g32 as uint8);
 *              identical shapes; base 16-byte aligned. Row (slot, g) is read whole, once
 *              per selecting (sequence, g), with its scales.
 *  kv_quant_meta  format, scales, softmax scale, capacity, optional CTA cap.
 *  sel_indices int32 [n_sel], contiguous: the packed selected slot ids.
 *  cu_seqlens  int32 [bs + 1], device, read on the device only.
 *  out         bf16 [bs, Hq, 256]; stride[2] == 1; stride[0], stride[1] multiples of 8;
 *              base 16-byte aligned. Fully written (zeros for empty selections).
 *  scratch     device buffer of at least qsa_decode_scratch_bytes(bs, Hq, capacity)
 *              bytes, 256-byte aligned, initialised once by qsa_scratch_init.
 *  stream      cudaStream_t (NULL: the legacy default stream).
 *
 * Returns QSA_OK or a negative QSA_ERR_*; see qsa_last_error_message().
 */
int qsa_decode(const qsa_tensor* q, const qsa_tensor* k_pool, const qsa_tensor* v_pool,
               const qsa_kv_quant_meta* kv_quant_meta, const qsa_tensor* sel_indices,
               const qsa_tensor* cu_seqlens, const qsa_tensor* out, void* scratch,
               size_t scratch_bytes, void* stream);

/*
 * qsa_kv_write -- quantise new K/V rows and scatter them into the pools: the
 * write that fills what qsa_decode gathers (sglang PR #37798, "Modifications":
 * one fused quantise + scatter launch per write; part 1, mem_cache/memory_pool.py:
 * the fp8 write saturates to +-448 before the e4m3 cast).
 *
 *  format      QSA_KV_* of the pools.
 *  k_new,      bf16 [n, Hkv, 256] (Hkv 1 or 2); stride[2] == 1, other strides
 *  v_new       non-negative multiples of 8; base 16-byte aligned. n may be 0.
 *  slots       int32 [n], contiguous: destination slot of token i. Slots must be
 *              distinct within a call: each (token, head, K or V) row is written by
 *              its own warp, so a repeated slot leaves that row's codes and scale
 *              unspecified (they may mix the repeated tokens' writes).
 *  k_pool,     pools as for qsa_decode; row slot[i] * Hkv + g receives token i, head g.
 *  v_pool
 *  k_scale,    fp8: the pool's fp32 scale [1] (read; must be finite and > 0);
 *  v_scale     int8/int4: fp32 [num_slots * Hkv], entry of each written row set to
 *              absmax(row) / 127 (int8) or / 7 (int4); int8_g64 / int4_g32: binary16
 *              [num_slots * Hkv * 4 / 8] (8- / 16-byte aligned), the written row's
 *              group entries set to binary16(min(absmax(group) / 127 or / 7, 65504));
 *              bf16: unused (may be NULL).
 *  device_error  optional int32 device word: QSA_DEVERR_SLOT_RANGE is OR-ed in when a
 *              slot is outside [0, num_slots); that row is skipped. May be NULL.
 *  stream      cudaStream_t.
 *
 * Codes, in binary32 with IEEE division and round-to-nearest-even: bf16 rows are
 * copied; fp8 = e4m3fn(x / s) saturating at +-448; int8 = clamp(rint(x / s), -127, 127);
 * int4 = clamp(rint(x / s), -8, 7), two's-complement nibbles, channel 2i in the low
 * nibble; int8_g64 / int4_g32 = clamp(rint(x / s16), -127, 127) / (-7, 7) with the
 * group's binary16 scale s16, int4_g32 as offset-binary nibbles code + 8; an all-zero
 * row (group) gets scale 0 and zero codes. Inputs must be finite.
 * Validates on the host, enqueues one kernel, allocates nothing.
 */
int qsa_kv_write(int32_t format, const qsa_tensor* k_new, const qsa_tensor* v_new,
                 const qsa_tensor* slots, const qsa_tensor* k_pool, const qsa_tensor* v_pool,
                 void* k_scale, void* v_scale, int32_t* device_error, void* stream);

/*
 * qsa_kv_write_tiered -- the write of a QSA_KV_INT8RING_INT4 pool: every token i is
 * written twice, as the int4_g32 row of slot[i] (k_pool / v_pool, binary16 scales
 * k_scale / v_scale [num_slots * Hkv * 8], 16-byte aligned) and as the int8_g64 row
 * of ring position p = slot[i] & (R - 1), whose owner entry becomes slot[i]. When
 * several tokens of one call (with distinct slots) share a ring position, the last
 * of them (largest i) owns it, as if the tokens were written in order; owner and
 * ring row then agree. Slots must be distinct within a call, as for qsa_kv_write: a
 * repeated slot leaves its rows, its ring row and the owner entry unspecified.
 * Arguments otherwise as for qsa_kv_write. Enqueues two kernels on `stream` (claim
 * the ring positions, then write); allocates nothing. Between the two, the owner
 * entries of the positions being written hold claim marks (negative values); a
 * decode ordered after the call sees the final owners.
 */
int qsa_kv_write_tiered(const qsa_tensor* k_new, const qsa_tensor* v_new, const qsa_tensor* slots,
                        const qsa_tensor* k_pool, const qsa_tensor* v_pool, void* k_scale,
                        void* v_scale, const qsa_kv_tier* tier, int32_t* device_error,
                        void* stream);

/* Scratch bytes a qsa_decode call with these sizes needs on the current
 * device (0 when the sizes are outside the contract). Split-KV partials take
 * two 12 KiB slots per CTA of the grid the library would choose.
 * Source: sglang PR #36845, "Optimized kernel" (long KV rows split across CTAs,
 * whose partial results the final split merges; its device counter lives here)
 * and "Changes" (the contract that bounds the size: 1 <= bs <= 128, TP1 24Q or TP2
 * 12Q, selected capacity <= 2055; the pages give 32.3 MiB as their worst case at
 * TP1 bs=128, this layout needs under 4 MB). */
size_t qsa_decode_scratch_bytes(int32_t bs, int32_t num_q_heads, int32_t capacity);

/* Number of CTAs qsa_decode launches for these sizes on the current device
 * (after applying max_ctas when > 0); negative QSA_ERR_* on bad sizes.
 * Source: sglang PR #36845, "Optimized kernel" (the split of long KV rows across
 * CTAs); the grid is fixed by the sizes, so a captured graph keeps it. */
int32_t qsa_decode_grid(int32_t bs, int32_t num_q_heads, int32_t capacity, int32_t max_ctas);

/* Offsets of the scratch regions, for callers that inspect them (tests):
 * the error word (int32), the counters (int32 [bs * Hkv]) and the partials.
 * Source: sglang PR #36845, "Optimized kernel" (the per-split device counters that
 * the final split resets in the same launch; the pages check them zero after
 * 150,000 consecutive launches). */
typedef struct {
    size_t error_word_offset;
    size_t counters_offset;
    size_t counters_count;
    size_t partials_offset;
    size_t partial_slot_bytes;
    size_t total_bytes;
} qsa_scratch_layout;

int qsa_decode_scratch_layout(int32_t bs, int32_t num_q_heads, int32_t capacity,
                              qsa_scratch_layout* layout);

/* Zero a scratch buffer (cudaMemsetAsync on `stream`). Call once after
 * allocating it; counters then stay zero across launches by themselves.
 * Source: sglang PR #36845, "Optimized kernel": the final split resets its device
 * counter in the same launch, and every counter is back at zero after 150,000
 * consecutive launches, so one zeroing at allocation is all the state needs. */
int qsa_scratch_init(void* scratch, size_t scratch_bytes, void* stream);

/* Read the sticky device error word into *flags (QSA_DEVERR_* bits). This
 * is the library's only device readback: it copies 4 bytes on `stream` and
 * synchronises that stream. With clear != 0 the word is reset to zero.
 * Source: sglang PR #36845, "Changes" (lengths are read on the device, so the
 * decode itself never reads back to the host) and "Motivation" (the failure the
 * pages fight is silent: wrong outputs while the server stays healthy; bad device
 * data is therefore recorded here instead of being passed over). */
int qsa_scratch_error(const void* scratch, int32_t* flags, int32_t clear, void* stream);

/* Static description of a return code.
 * Source: sglang PR #36845, "Changes": unsupported calls fail with a descriptive
 * contract error. */
const char* qsa_strerror(int code);

/* Descriptive message of the last failing call on this host thread ("" if none):
 * which argument broke which rule of the contract.
 * Source: sglang PR #36845, "Changes": unsupported calls fail with a descriptive
 * contract error. */
const char* qsa_last_error_message(void);

/*
 * qsa_decode_static_scratch -- qsa_decode without a caller-provided scratch
 * buffer. The pages have no counterpart to this entry point.
 *
 * For callers that cannot allocate device memory when they call: code whose
 * memory is fixed up front and that may not call cudaMalloc (or a framework
 * allocator) on the call path, e.g. an inference-engine plugin with a preset
 * memory budget or a host loop where an allocation would synchronise the
 * device, and bindings that hold pointers to tensors but own no allocator.
 * It allocates nothing: its scratch is one file-scope device array of
 * 3,974,400 bytes (256-byte aligned) that every GPU which loads libqsa holds
 * until the process exits.
 *
 * Arguments as for qsa_decode, minus scratch. The grid is capped at 160 CTAs
 * so the split-KV partials fit the array; kv_quant_meta->max_ctas may lower
 * that cap. Every size the decode contract admits fits; anything else is
 * rejected like qsa_decode does (QSA_ERR_UNSUPPORTED, QSA_ERR_SCRATCH_TOO_SMALL,
 * ... with qsa_last_error_message()).
 *
 * The first call on each device (with that device current) looks up the
 * array's device address; make that first call before any stream capture.
 * Each call enqueues a 1,280-byte memset that clears the array's error word
 * and counters, then the decode kernel, both on `stream`. All calls on a
 * device share the one array, which keeps the last call's contents: calls
 * that overlap on the GPU (unordered streams, concurrent host threads) race
 * on it and must be serialised by the caller. The device error word is not
 * readable through this entry point.
 */
int qsa_decode_static_scratch(const qsa_tensor* q, const qsa_tensor* k_pool,
                              const qsa_tensor* v_pool, const qsa_kv_quant_meta* kv_quant_meta,
                              const qsa_tensor* sel_indices, const qsa_tensor* cu_seqlens,
                              const qsa_tensor* out, void* stream);

/* Sizes of one qsa_topk_expand call. */
typedef struct {
    int32_t token_topk;     /* tokens kept from whole blocks per sequence: a positive multiple
                               of compress_ratio; token_topk + compress_ratio - 1 <= 2055 */
    int32_t compress_ratio; /* tokens per compressed block, 1..64 (the pages use 4, 8, 16) */
    int32_t capacity;       /* largest context length, 1..262144 (the pages' 256K) */
    int32_t page_size;      /* page_table's page size, a power of two (the pages use 64);
                               0: no page table, the ids are logical token positions */
} qsa_topk_params;

/*
 * qsa_topk_expand -- the step that produces qsa_decode's sel_indices and
 * cu_seqlens: exact top-k over compressed-block scores, then index expansion
 * (1Cat-vLLM PR #523, "Follow-up: device-planned MQA and QSA quality
 * attribution": exact top-k + index expansion at a fixed 256K capacity; sglang
 * PR #37798, "Decode routing": index-row width token_topk + compress_ratio - 1 =
 * 2048 + 4 - 1 = 2051, 64-token pages). The scores themselves come from the
 * caller; the pages give no formula for them.
 *
 * For sequence b with context length T = ctx_lens[b] and r = compress_ratio,
 * block i covers tokens [i r, (i + 1) r); the floor(T / r) complete blocks carry
 * scores[b][i]; the last T mod r tokens are in no block yet. k = token_topk / r
 * blocks are kept: all of them when there are at most k, else the k ranked first
 * -- higher score first, equal scores by lower block index, NaN below every
 * number, -0.0 equal to +0.0. Row b lists the kept blocks' tokens in ascending
 * position, then the tail tokens: r * min(floor(T / r), k) + T mod r <=
 * token_topk + r - 1 ids. With a page table, position p becomes slot
 * page_table[b][p / page_size] * page_size + p % page_size. Rows are packed in
 * sequence order from sel_indices[0]; cu_seqlens[0] = 0 and cu_seqlens[b + 1] is
 * the end of row b, as qsa_decode reads them.
 *
 *  scores       float32 [bs, >= capacity / compress_ratio], unit stride along the
 *               blocks; row stride >= the row length. Entries past a row's
 *               floor(T / r) blocks are not read.
 *  ctx_lens     int32 [bs], contiguous, 1 <= bs <= 128, read on the device only.
 *               A length outside [0, capacity] is clamped into it and sets
 *               QSA_DEVERR_CTX_LEN.
 *  page_table   int32 [bs, >= ceil(capacity / page_size)], unit stride along the
 *               pages, when page_size > 0 (else ignored, may be NULL). A page id
 *               that puts a slot outside [0, 2^31) writes -1 there and sets
 *               QSA_DEVERR_SLOT_RANGE.
 *  params       the sizes above (host struct, read at the call).
 *  sel_indices  int32, contiguous, at least bs * (token_topk + compress_ratio - 1)
 *               entries; entries past cu_seqlens[bs] are left as they were.
 *  cu_seqlens   int32 [bs + 1], contiguous.
 *  device_error optional int32 device word the QSA_DEVERR_* bits are OR-ed into.
 *  stream       cudaStream_t.
 *
 * Validates on the host, enqueues one kernel (one CTA per sequence, or for small
 * batches of rows of at least 32,768 blocks a cluster of up to 8 CTAs per
 * sequence, the cluster size chosen from bs, capacity / compress_ratio and the
 * device's SM count, the same on every call with those), allocates nothing and
 * needs no scratch; a captured graph stays valid when ctx_lens and scores change
 * between replays. Returns QSA_OK or a negative QSA_ERR_*.
 */
int qsa_topk_expand(const qsa_tensor* scores, const qsa_tensor* ctx_lens,
                    const qsa_tensor* page_table, const qsa_topk_params* params,
                    const qsa_tensor* sel_indices, const qsa_tensor* cu_seqlens,
                    int32_t* device_error, void* stream);

/* Library version, major * 10000 + minor * 100 + patch. The pages have no
 * counterpart; a caller checks it against the header it was built with. */
int qsa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H_ */
