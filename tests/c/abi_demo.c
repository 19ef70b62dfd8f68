/*
 * A plain C caller of libdsv4kv: no Python, no torch.  Reads the inputs of one
 * fused step from raw files, runs dsv4_qnorm_rope_kv_quant_insert on the
 * legacy default stream with buffers from cudaMalloc, and writes q and the
 * FP8 cache back out.  The GPU test that builds it compares the outputs with
 * the oracle.
 *
 * usage: abi_demo DIR T H NUM_BLOCKS BLOCK_SIZE MAX_POSITION
 *   DIR holds q.bin (bf16 [T,H,512]), kv.bin (bf16 [T,512]), w.bin (bf16 [512]),
 *   pos.bin, slot.bin (int64 [T]), cs.bin (fp32 [MAX_POSITION,64]), cache.bin
 *   (uint8, the cache pre-image); writes q_out.bin, cache_out.bin, err.txt.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "dsv4kv.h"

static void *load(const char *dir, const char *name, size_t bytes)
{
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "rb");
    if (!f) {
        fprintf(stderr, "cannot open %s\n", path);
        exit(2);
    }
    void *host = malloc(bytes ? bytes : 1);
    if (fread(host, 1, bytes, f) != bytes) {
        fprintf(stderr, "short read on %s\n", path);
        exit(2);
    }
    fclose(f);
    void *dev = NULL;
    if (cudaMalloc(&dev, bytes ? bytes : 1) != cudaSuccess ||
        cudaMemcpy(dev, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
        fprintf(stderr, "device copy of %s failed\n", name);
        exit(3);
    }
    free(host);
    return dev;
}

static void store(const char *dir, const char *name, const void *dev, size_t bytes)
{
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    void *host = malloc(bytes ? bytes : 1);
    if (cudaMemcpy(host, dev, bytes, cudaMemcpyDeviceToHost) != cudaSuccess) {
        fprintf(stderr, "copy back of %s failed\n", name);
        exit(3);
    }
    FILE *f = fopen(path, "wb");
    if (!f || fwrite(host, 1, bytes, f) != bytes) {
        fprintf(stderr, "cannot write %s\n", path);
        exit(2);
    }
    fclose(f);
    free(host);
}

int main(int argc, char **argv)
{
    if (argc != 7) {
        fprintf(stderr, "usage: %s DIR T H NUM_BLOCKS BLOCK_SIZE MAX_POSITION\n", argv[0]);
        return 1;
    }
    const char *dir = argv[1];
    const int64_t T = atoll(argv[2]);
    const int32_t H = atoi(argv[3]);
    const int64_t nb = atoll(argv[4]);
    const int32_t bs = atoi(argv[5]);
    const int64_t max_pos = atoll(argv[6]);
    const size_t q_bytes = (size_t)T * H * DSV4_HEAD_DIM * 2;
    const size_t cache_bytes = dsv4_fp8_cache_bytes(nb, bs);

    void *q = load(dir, "q.bin", q_bytes);
    void *kv = load(dir, "kv.bin", (size_t)T * DSV4_HEAD_DIM * 2);
    void *w = load(dir, "w.bin", DSV4_HEAD_DIM * 2);
    int64_t *pos = load(dir, "pos.bin", (size_t)T * 8);
    int64_t *slot = load(dir, "slot.bin", (size_t)T * 8);
    float *cs = load(dir, "cs.bin", (size_t)max_pos * DSV4_ROPE_DIM * 4);
    uint8_t *cache = load(dir, "cache.bin", cache_bytes);
    int32_t *err = NULL;
    if (cudaMalloc((void **)&err, sizeof(int32_t)) != cudaSuccess ||
        cudaMemset(err, 0, sizeof(int32_t)) != cudaSuccess)
        return 3;

    const int st = dsv4_qnorm_rope_kv_quant_insert(q, kv, w, pos, cs, max_pos, slot, cache, nb, bs,
                                                   T, H, 1e-6f, err, NULL);
    if (st != DSV4_OK) {
        fprintf(stderr, "dsv4_qnorm_rope_kv_quant_insert: %s\n", dsv4_status_string(st));
        return 4;
    }
    if (cudaDeviceSynchronize() != cudaSuccess)
        return 5;
    store(dir, "q_out.bin", q, q_bytes);
    store(dir, "cache_out.bin", cache, cache_bytes);
    int32_t herr = -1;
    cudaMemcpy(&herr, err, sizeof herr, cudaMemcpyDeviceToHost);
    char path[4096];
    snprintf(path, sizeof path, "%s/err.txt", dir);
    FILE *f = fopen(path, "w");
    fprintf(f, "%d\n", (int)herr);
    fclose(f);
    /* a bad argument comes back as a status, with nothing launched */
    if (dsv4_qnorm_rope_kv_quant_insert(q, kv, w, pos, cs, max_pos, slot, cache, nb, bs, T, H,
                                        -1.0f, err, NULL) != DSV4_ERR_VALUE)
        return 6;
    printf("ok\n");
    return 0;
}
