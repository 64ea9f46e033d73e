/*
 * A plain C caller of the boundary library (include/lb.h): reads a boundary's inputs
 * from raw little-endian files, runs lb_fold_norm_fp8 on device buffers it allocates
 * with the CUDA runtime, and writes residual', the E4M3 codes and the scales back to
 * files.  Used by tests/test_c_abi_gpu.py, which compares the files with the CPU
 * oracle.
 *
 *   abi_fold_fp8 DIR K T H EPS
 *   inputs  DIR/p0.bin .. DIR/p{K-1}.bin (bf16 [T,H]), DIR/res.bin (bf16 [T,H]),
 *           DIR/gamma.bin (float32 [H])
 *   outputs DIR/res_out.bin (bf16 [T,H]), DIR/q.bin (uint8 [T,H]), DIR/scale.bin
 *           (float32 [T])
 * Exit status 0 on success; the library status or CUDA error is printed otherwise.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "lb.h"

static void *read_file(const char *dir, const char *name, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "rb");
    if (!f) return NULL;
    void *buf = malloc(bytes);
    size_t got = buf ? fread(buf, 1, bytes, f) : 0;
    fclose(f);
    if (got != bytes) { free(buf); return NULL; }
    return buf;
}

static int write_file(const char *dir, const char *name, const void *buf, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "wb");
    if (!f) return 1;
    size_t put = fwrite(buf, 1, bytes, f);
    fclose(f);
    return put != bytes;
}

static void *to_device(const void *host, size_t bytes) {
    void *d = NULL;
    if (cudaMalloc(&d, bytes) != cudaSuccess) return NULL;
    if (cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
    return d;
}

int main(int argc, char **argv) {
    if (argc != 6) {
        fprintf(stderr, "usage: %s DIR K T H EPS\n", argv[0]);
        return 2;
    }
    const char *dir = argv[1];
    const int K = atoi(argv[2]);
    const int64_t T = atoll(argv[3]), H = atoll(argv[4]);
    const float eps = (float)atof(argv[5]);
    if (K < 1 || K > LB_MAX_K || T < 1 || H < 8) return 2;
    const size_t row_bytes = (size_t)T * (size_t)H * 2;

    const void *partials[LB_MAX_K];
    for (int k = 0; k < K; ++k) {
        char name[32];
        snprintf(name, sizeof name, "p%d.bin", k);
        void *h = read_file(dir, name, row_bytes);
        if (!h) { fprintf(stderr, "cannot read %s\n", name); return 1; }
        partials[k] = to_device(h, row_bytes);
        free(h);
        if (!partials[k]) { fprintf(stderr, "device copy failed\n"); return 1; }
    }
    void *hres = read_file(dir, "res.bin", row_bytes);
    void *hgamma = read_file(dir, "gamma.bin", (size_t)H * 4);
    if (!hres || !hgamma) { fprintf(stderr, "cannot read inputs\n"); return 1; }
    void *res = to_device(hres, row_bytes);
    float *gamma = (float *)to_device(hgamma, (size_t)H * 4);
    void *res_out = NULL, *q = NULL, *scale = NULL;
    if (!res || !gamma || cudaMalloc(&res_out, row_bytes) != cudaSuccess ||
        cudaMalloc(&q, (size_t)T * (size_t)H) != cudaSuccess ||
        cudaMalloc(&scale, (size_t)T * 4) != cudaSuccess) {
        fprintf(stderr, "device allocation failed\n");
        return 1;
    }
    cudaStream_t stream;
    if (cudaStreamCreate(&stream) != cudaSuccess) return 1;

    lb_status st = lb_fold_norm_fp8(partials, K, res, res_out, gamma, (uint8_t *)q,
                                    (float *)scale, NULL, T, H, eps, NULL,
                                    (lb_stream_t)stream);
    if (st != LB_OK) {
        fprintf(stderr, "lb_fold_norm_fp8: %s (cuda %d)\n", lb_status_string(st),
                lb_last_cuda_error());
        return 1;
    }
    if (cudaStreamSynchronize(stream) != cudaSuccess) { fprintf(stderr, "sync failed\n"); return 1; }
    unsigned int flags = 0;
    if (lb_device_error(&flags, 1) != LB_OK || flags != 0) {
        fprintf(stderr, "device error flags %u\n", flags);
        return 1;
    }

    void *hout = malloc(row_bytes), *hq = malloc((size_t)T * (size_t)H),
         *hs = malloc((size_t)T * 4);
    if (!hout || !hq || !hs) return 1;
    if (cudaMemcpy(hout, res_out, row_bytes, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(hq, q, (size_t)T * (size_t)H, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(hs, scale, (size_t)T * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
        return 1;
    if (write_file(dir, "res_out.bin", hout, row_bytes) ||
        write_file(dir, "q.bin", hq, (size_t)T * (size_t)H) ||
        write_file(dir, "scale.bin", hs, (size_t)T * 4))
        return 1;
    printf("lb_fold_norm_fp8 K=%d T=%lld H=%lld: ok\n", K, (long long)T, (long long)H);
    return 0;
}
