/* A plain C (C11) caller of libattn.so on the GPU: device buffers from
 * cudaMalloc, one causal GQA prefill, one KV-cache append and one paged
 * decode through include/attn.h, results copied back and written to files.
 * tests/test_c_abi.py writes the inputs (raw little-endian arrays) into the
 * directory given as argv[1], runs this program and gates the outputs
 * against the fp64 oracle.
 *
 * Sizes (mirrored by the Python test):
 *   prefill  B = 1, Hq = 4, Hkv = 2, n = 300, d = 128, causal, bf16 -> fp32 + lse
 *   decode   3 sequences, Hq = 8, Hkv = 2, d = 128, 16-token blocks, one new
 *            token appended per sequence at position seq_lens[s] - 1, then one
 *            query token per sequence over the whole cache, bf16 -> fp32 + lse */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "attn.h"

enum { PB = 1, PHQ = 4, PHKV = 2, PN = 300, D = 128 };
enum { S = 3, DHQ = 8, DHKV = 2, BS = 16, MAXB = 32, MAXLEN = 512 };

static const char *dir;

static void *read_file(const char *name, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "rb");
    if (!f) {
        fprintf(stderr, "cannot open %s\n", path);
        exit(2);
    }
    void *buf = malloc(bytes);
    if (!buf || fread(buf, 1, bytes, f) != bytes) {
        fprintf(stderr, "short read %s\n", path);
        exit(2);
    }
    fclose(f);
    return buf;
}

static void write_file(const char *name, const void *buf, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "wb");
    if (!f || fwrite(buf, 1, bytes, f) != bytes) {
        fprintf(stderr, "cannot write %s\n", path);
        exit(2);
    }
    fclose(f);
}

/* host file -> new device buffer */
static void *upload(const char *name, size_t bytes) {
    void *h = read_file(name, bytes);
    void *d = NULL;
    if (cudaMalloc(&d, bytes) != cudaSuccess ||
        cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
        fprintf(stderr, "upload %s failed\n", name);
        exit(3);
    }
    free(h);
    return d;
}

static void *dalloc(size_t bytes) {
    void *d = NULL;
    if (cudaMalloc(&d, bytes) != cudaSuccess) {
        fprintf(stderr, "cudaMalloc failed\n");
        exit(3);
    }
    return d;
}

/* device buffer -> host file */
static void download(const char *name, const void *d, size_t bytes) {
    void *h = malloc(bytes);
    if (!h || cudaMemcpy(h, d, bytes, cudaMemcpyDeviceToHost) != cudaSuccess) {
        fprintf(stderr, "download %s failed\n", name);
        exit(3);
    }
    write_file(name, h, bytes);
    free(h);
}

#define CALL(x)                                                                    \
    do {                                                                           \
        attn_status st_ = (x);                                                     \
        if (st_ != ATTN_OK) {                                                      \
            fprintf(stderr, "%s:%d: %s -> %s\n", __FILE__, __LINE__, #x,           \
                    attn_status_str(st_));                                         \
            return 1;                                                              \
        }                                                                          \
    } while (0)

int main(int argc, char **argv) {
    if (argc != 2) {
        fprintf(stderr, "usage: abi_gpu <dir>\n");
        return 2;
    }
    dir = argv[1];
    int *nblk = (int *)read_file("num_blocks.i32", sizeof(int));
    const int num_blocks = *nblk;
    free(nblk);

    /* ---- prefill */
    const size_t q_el = (size_t)PB * PHQ * PN * D, kv_el = (size_t)PB * PHKV * PN * D;
    void *Q = upload("Q.bf16", q_el * 2);
    void *K = upload("K.bf16", kv_el * 2);
    void *V = upload("V.bf16", kv_el * 2);
    float *O = (float *)dalloc(q_el * 4);
    float *lse = (float *)dalloc((size_t)PB * PHQ * PN * 4);
    CALL(attn_prefill(Q, K, V, O, lse, PB, PHQ, PHKV, PN, PN, D, 1, 0.08838834764831845f,
                      ATTN_BF16, ATTN_F32, NULL, NULL, NULL, NULL));
    if (attn_last_launch_count() != 1)
        return 4;

    /* ---- append one token per sequence, then decode */
    const size_t cache_el = (size_t)num_blocks * DHKV * BS * D;
    void *Kc = upload("Kc.bf16", cache_el * 2);
    void *Vc = upload("Vc.bf16", cache_el * 2);
    void *q = upload("q.bf16", (size_t)S * DHQ * D * 2);
    int32_t *table = (int32_t *)upload("block_table.i32", (size_t)S * MAXB * 4);
    int32_t *lens = (int32_t *)upload("seq_lens.i32", (size_t)S * 4);
    void *kn = upload("k_new.bf16", (size_t)S * DHKV * D * 2);
    void *vn = upload("v_new.bf16", (size_t)S * DHKV * D * 2);
    int32_t *sid = (int32_t *)upload("seq_ids.i32", (size_t)S * 4);
    int32_t *pos = (int32_t *)upload("positions.i32", (size_t)S * 4);
    CALL(attn_kv_append(kn, vn, Kc, Vc, table, sid, pos, S, S, DHKV, D, BS, MAXB, num_blocks,
                        ATTN_BF16, ATTN_BF16, NULL, NULL, NULL));
    const size_t ws_bytes = attn_decode_workspace_bytes(S, DHQ, D, MAXLEN);
    if (ws_bytes == 0)
        return 4;
    void *ws = dalloc(ws_bytes);
    float *Od = (float *)dalloc((size_t)S * DHQ * D * 4);
    float *lsed = (float *)dalloc((size_t)S * DHQ * 4);
    CALL(attn_decode(q, Kc, Vc, table, lens, Od, lsed, S, DHQ, DHKV, D, BS, MAXB, num_blocks,
                     MAXLEN, 0.08838834764831845f, ATTN_BF16, ATTN_BF16, ATTN_F32, NULL, NULL,
                     ws, ws_bytes, NULL));
    if (attn_last_launch_count() != 2)
        return 4;
    CALL(attn_last_error(NULL)); /* synchronises; no device-side error recorded */

    download("O.f32", O, q_el * 4);
    download("lse.f32", lse, (size_t)PB * PHQ * PN * 4);
    download("Kc_out.bf16", Kc, cache_el * 2);
    download("Vc_out.bf16", Vc, cache_el * 2);
    download("Od.f32", Od, (size_t)S * DHQ * D * 4);
    download("lsed.f32", lsed, (size_t)S * DHQ * 4);
    printf("c abi gpu ok\n");
    return 0;
}
