/*
 * A plain C client of libqsa (no Python, no PyTorch): it uses only qsa.h and the
 * CUDA runtime. Test infrastructure for tests/test_c_client.py.
 *
 *   qsa_c_client host          host-side checks: version, error strings, rejection
 *                              of bad descriptors before any CUDA call
 *   qsa_c_client gpu DIR       one TP2 bf16 decode (12 query heads, 1 KV head,
 *                              bs = 3, lengths 1 / 77 / 300, a 4096-slot pool) on
 *                              cudaMalloc'd buffers; inputs and output are written
 *                              to DIR as raw little-endian files for the oracle
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "qsa.h"

#define CHECK(x)                                                                        \
    do {                                                                                \
        cudaError_t e_ = (x);                                                           \
        if (e_ != cudaSuccess) {                                                        \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));                    \
            return 2;                                                                   \
        }                                                                               \
    } while (0)

/* splitmix64: a small deterministic generator for the synthetic inputs */
static uint64_t mix(uint64_t* s) {
    uint64_t z = (*s += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* uniform in [-1, 1) rounded to bf16 (truncation of a value with <= 8 bits) */
static uint16_t rand_bf16(uint64_t* s) {
    const int v = (int)(mix(s) % 256) - 128; /* exact in bf16 once scaled */
    float f = (float)v / 128.0f;
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

static qsa_tensor tensor(void* data, int dtype, int ndim, const int64_t* shape) {
    qsa_tensor t;
    memset(&t, 0, sizeof t);
    t.data = data;
    t.dtype = dtype;
    t.ndim = ndim;
    int64_t st = 1;
    for (int i = ndim - 1; i >= 0; --i) {
        t.shape[i] = shape[i];
        t.stride[i] = st;
        st *= shape[i];
    }
    return t;
}

static int write_file(const char* dir, const char* name, const void* p, size_t n) {
    char path[1024];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE* f = fopen(path, "wb");
    if (!f) return 1;
    const size_t w = fwrite(p, 1, n, f);
    fclose(f);
    return w != n;
}

static int host_checks(void) {
    if (qsa_version() < 100) return 1;
    if (strcmp(qsa_strerror(QSA_OK), "success") != 0) return 1;
    if (qsa_decode(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL) != QSA_ERR_INVALID_ARGUMENT)
        return 1;
    if (strstr(qsa_last_error_message(), "NULL") == NULL) return 1;
    /* a 16-head query is outside the contract: rejected on the host */
    static uint16_t qbuf[2 * 16 * 256], pool[8 * 256];
    static int32_t sel[4], cu[3];
    int64_t qs[3] = {2, 16, 256}, ps[3] = {8, 1, 256}, ss[1] = {4}, cs[1] = {3};
    qsa_tensor q = tensor(qbuf, QSA_DTYPE_BF16, 3, qs), k = tensor(pool, QSA_DTYPE_BF16, 3, ps);
    qsa_tensor s = tensor(sel, QSA_DTYPE_INT32, 1, ss), c = tensor(cu, QSA_DTYPE_INT32, 1, cs);
    qsa_kv_quant_meta meta;
    memset(&meta, 0, sizeof meta);
    meta.format = QSA_KV_BF16;
    meta.capacity = 4;
    meta.softmax_scale = 1.0f / 16.0f;
    if (qsa_decode(&q, &k, &k, &meta, &s, &c, &q, NULL, 0, NULL) != QSA_ERR_UNSUPPORTED) return 1;
    if (strstr(qsa_last_error_message(), "query heads") == NULL) return 1;
    printf("host ok: version %d\n", qsa_version());
    return 0;
}

static int gpu_decode(const char* dir) {
    enum { BS = 3, HQ = 12, HKV = 1, D = 256, SLOTS = 4096 };
    const int lengths[BS] = {1, 77, 300};
    int32_t cu[BS + 1] = {0};
    for (int b = 0; b < BS; ++b) cu[b + 1] = cu[b] + lengths[b];
    const int n_sel = cu[BS];
    uint64_t seed = 12345;
    uint16_t* q = malloc(sizeof(uint16_t) * BS * HQ * D);
    uint16_t* kp = malloc(sizeof(uint16_t) * SLOTS * HKV * D);
    uint16_t* vp = malloc(sizeof(uint16_t) * SLOTS * HKV * D);
    int32_t* sel = malloc(sizeof(int32_t) * n_sel);
    uint16_t* out = malloc(sizeof(uint16_t) * BS * HQ * D);
    for (int i = 0; i < BS * HQ * D; ++i) q[i] = rand_bf16(&seed);
    for (int i = 0; i < SLOTS * HKV * D; ++i) kp[i] = rand_bf16(&seed);
    for (int i = 0; i < SLOTS * HKV * D; ++i) vp[i] = rand_bf16(&seed);
    for (int i = 0; i < n_sel; ++i) sel[i] = (int32_t)(mix(&seed) % SLOTS);

    void *dq, *dk, *dv, *ds, *dc, *dout, *scratch;
    const size_t sbytes = qsa_decode_scratch_bytes(BS, HQ, 300);
    if (sbytes == 0) return 3;
    CHECK(cudaMalloc(&dq, sizeof(uint16_t) * BS * HQ * D));
    CHECK(cudaMalloc(&dk, sizeof(uint16_t) * SLOTS * HKV * D));
    CHECK(cudaMalloc(&dv, sizeof(uint16_t) * SLOTS * HKV * D));
    CHECK(cudaMalloc(&ds, sizeof(int32_t) * n_sel));
    CHECK(cudaMalloc(&dc, sizeof(int32_t) * (BS + 1)));
    CHECK(cudaMalloc(&dout, sizeof(uint16_t) * BS * HQ * D));
    CHECK(cudaMalloc(&scratch, sbytes));
    CHECK(cudaMemcpy(dq, q, sizeof(uint16_t) * BS * HQ * D, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(dk, kp, sizeof(uint16_t) * SLOTS * HKV * D, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(dv, vp, sizeof(uint16_t) * SLOTS * HKV * D, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(ds, sel, sizeof(int32_t) * n_sel, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(dc, cu, sizeof(int32_t) * (BS + 1), cudaMemcpyHostToDevice));
    cudaStream_t st;
    CHECK(cudaStreamCreate(&st));
    if (qsa_scratch_init(scratch, sbytes, st) != QSA_OK) return 4;

    int64_t qs[3] = {BS, HQ, D}, ps[3] = {SLOTS, HKV, D}, ss[1] = {n_sel}, cs[1] = {BS + 1};
    qsa_tensor tq = tensor(dq, QSA_DTYPE_BF16, 3, qs), tk = tensor(dk, QSA_DTYPE_BF16, 3, ps);
    qsa_tensor tv = tensor(dv, QSA_DTYPE_BF16, 3, ps), ts = tensor(ds, QSA_DTYPE_INT32, 1, ss);
    qsa_tensor tc = tensor(dc, QSA_DTYPE_INT32, 1, cs), to = tensor(dout, QSA_DTYPE_BF16, 3, qs);
    qsa_kv_quant_meta meta;
    memset(&meta, 0, sizeof meta);
    meta.format = QSA_KV_BF16;
    meta.capacity = 300;
    meta.softmax_scale = 1.0f / 16.0f;
    const int rc = qsa_decode(&tq, &tk, &tv, &meta, &ts, &tc, &to, scratch, sbytes, st);
    if (rc != QSA_OK) {
        fprintf(stderr, "qsa_decode: %s\n", qsa_last_error_message());
        return 5;
    }
    int32_t flags = -1;
    if (qsa_scratch_error(scratch, &flags, 0, st) != QSA_OK || flags != 0) return 6;
    CHECK(cudaMemcpy(out, dout, sizeof(uint16_t) * BS * HQ * D, cudaMemcpyDeviceToHost));
    if (write_file(dir, "q.bin", q, sizeof(uint16_t) * BS * HQ * D) ||
        write_file(dir, "k.bin", kp, sizeof(uint16_t) * SLOTS * HKV * D) ||
        write_file(dir, "v.bin", vp, sizeof(uint16_t) * SLOTS * HKV * D) ||
        write_file(dir, "sel.bin", sel, sizeof(int32_t) * n_sel) ||
        write_file(dir, "cu.bin", cu, sizeof(int32_t) * (BS + 1)) ||
        write_file(dir, "out.bin", out, sizeof(uint16_t) * BS * HQ * D))
        return 7;
    cudaFree(dq); cudaFree(dk); cudaFree(dv); cudaFree(ds); cudaFree(dc); cudaFree(dout);
    cudaFree(scratch);
    cudaStreamDestroy(st);
    free(q); free(kp); free(vp); free(sel); free(out);
    printf("gpu ok\n");
    return 0;
}

int main(int argc, char** argv) {
    if (argc >= 2 && strcmp(argv[1], "host") == 0) return host_checks();
    if (argc >= 3 && strcmp(argv[1], "gpu") == 0) return gpu_decode(argv[2]);
    fprintf(stderr, "usage: %s host | gpu DIR\n", argv[0]);
    return 64;
}
