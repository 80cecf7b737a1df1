/*
 * A C client of libpkv with no Python and no torch: it loads a decode-step
 * case from raw files, allocates and fills device buffers with the CUDA
 * runtime, runs pkv_decode_step (the cache write, then the paged decode)
 * and writes o back to a file.
 *
 *   decode_step <dir>
 *
 * <dir>/meta.txt holds, whitespace separated: n_layers size n_kv_heads
 * head_dim num_reqs max_ctx_len batch n_heads layer_id max_len; the other
 * files are the raw arrays: k_buffer.bin v_buffer.bin (bf16 bits),
 * req_to_token.bin req_pool_indices.bin seq_lens.bin kv_indptr.bin
 * out_cache_loc.bin (int32), q.bin k_new.bin v_new.bin (bf16 bits).  Writes
 * <dir>/o.bin.  Exit status 0 on success.
 */
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "pkv.h"

static void *load(const char *dir, const char *name, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "rb");
    if (!f) return NULL;
    void *h = malloc(bytes ? bytes : 1);
    size_t got = fread(h, 1, bytes, f);
    fclose(f);
    if (got != bytes) {
        free(h);
        return NULL;
    }
    void *d = NULL;
    if (cudaMalloc(&d, bytes ? bytes : 16) != cudaSuccess ||
        cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
        free(h);
        return NULL;
    }
    free(h);
    return d;
}

int main(int argc, char **argv) {
    if (argc != 2) return 2;
    const char *dir = argv[1];
    char path[4096];
    snprintf(path, sizeof path, "%s/meta.txt", dir);
    FILE *mf = fopen(path, "r");
    if (!mf) return 3;
    long long n_layers, size, hk, d, num_reqs, max_ctx, batch, n_heads, layer, max_len;
    if (fscanf(mf, "%lld %lld %lld %lld %lld %lld %lld %lld %lld %lld", &n_layers, &size, &hk, &d,
               &num_reqs, &max_ctx, &batch, &n_heads, &layer, &max_len) != 10)
        return 4;
    fclose(mf);

    const size_t pool = (size_t)(n_layers * size * hk * d) * 2;
    pkv_kvcache c;
    memset(&c, 0, sizeof c);
    c.k_buffer = load(dir, "k_buffer.bin", pool);
    c.v_buffer = load(dir, "v_buffer.bin", pool);
    c.dtype = PKV_BF16;
    c.n_layers = (int32_t)n_layers;
    c.n_kv_heads = (int32_t)hk;
    c.head_dim = (int32_t)d;
    c.size = size;
    c.req_to_token = load(dir, "req_to_token.bin", (size_t)(num_reqs * max_ctx) * 4);
    c.num_reqs = (int32_t)num_reqs;
    c.max_ctx_len = (int32_t)max_ctx;
    c.req_pool_indices = load(dir, "req_pool_indices.bin", (size_t)batch * 4);
    c.seq_lens = load(dir, "seq_lens.bin", (size_t)batch * 4);
    c.kv_indptr = load(dir, "kv_indptr.bin", (size_t)(batch + 1) * 4);
    c.out_cache_loc = load(dir, "out_cache_loc.bin", (size_t)batch * 4);
    c.batch = (int32_t)batch;
    c.max_len = (int32_t)max_len;
    const size_t qbytes = (size_t)(batch * n_heads * d) * 2, rowbytes = (size_t)(batch * hk * d) * 2;
    void *q = load(dir, "q.bin", qbytes), *kn = load(dir, "k_new.bin", rowbytes),
         *vn = load(dir, "v_new.bin", rowbytes);
    if (!c.k_buffer || !c.v_buffer || !c.req_to_token || !c.req_pool_indices || !c.seq_lens ||
        !c.kv_indptr || !c.out_cache_loc || !q || !kn || !vn)
        return 5;
    void *o = NULL;
    if (cudaMalloc(&o, qbytes) != cudaSuccess) return 6;

    /* the workspace: allocated once, described once */
    const int32_t splits = 256;
    const size_t wbytes = pkv_workspace_bytes((int32_t)batch, (int32_t)n_heads, (int32_t)d, splits);
    void *wbase = NULL;
    if (wbytes == 0 || cudaMalloc(&wbase, wbytes) != cudaSuccess) return 7;
    pkv_workspace ws;
    int rc = pkv_workspace_init(wbase, wbytes, (int32_t)batch, (int32_t)n_heads, (int32_t)d, splits, &ws);
    if (rc != PKV_OK) return 8;

    cudaStream_t s;
    if (cudaStreamCreate(&s) != cudaSuccess) return 9;
    rc = pkv_decode_step(&c, (int32_t)layer, kn, vn, (int32_t)batch, q, o, (int32_t)n_heads,
                         (float)(1.0 / sqrt((double)d)), &ws, s);
    if (rc != PKV_OK) {
        fprintf(stderr, "pkv_decode_step: %s\n", pkv_status_string(rc));
        return 10;
    }
    int64_t detail = 0;
    rc = pkv_last_device_error(s, &detail);
    if (rc != PKV_OK) {
        fprintf(stderr, "device error %lld\n", (long long)detail);
        return 11;
    }
    void *oh = malloc(qbytes);
    if (cudaMemcpy(oh, o, qbytes, cudaMemcpyDeviceToHost) != cudaSuccess) return 12;
    snprintf(path, sizeof path, "%s/o.bin", dir);
    FILE *of = fopen(path, "wb");
    if (!of || fwrite(oh, 1, qbytes, of) != qbytes) return 13;
    fclose(of);
    free(oh);
    printf("ok\n");
    return 0;
}
