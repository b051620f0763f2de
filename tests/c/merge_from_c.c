/*
 * A C caller of the merge's C ABI (include/dcp_lse_reduce.h), with no Python
 * in the call path: device buffers from cudaMalloc, the legacy default
 * stream, plain pointer arrays. It reads one merge's inputs from a file,
 * calls dcp_lse_reduce, and writes the merged outputs and LSEs to another
 * file, which the test compares with the oracle. It also makes one call that
 * the library must reject on the host (cp = 0) and prints its status code
 * and message.
 *
 * Input file (little endian): int32 cp, H, D, lse_base_e; int64 B, lse_stride;
 * then cp sources of B*H*D bf16 bits, then cp LSE arrays of B*lse_stride fp32.
 * Output file: cp destinations of B*(H/cp)*D bf16 bits, then cp merged LSE
 * arrays of B*(H/cp) fp32.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "dcp_lse_reduce.h"

#define CHECK_CUDA(call)                                                              \
    do {                                                                              \
        cudaError_t e_ = (call);                                                      \
        if (e_ != cudaSuccess) {                                                      \
            fprintf(stderr, "%s failed: %s\n", #call, cudaGetErrorString(e_));        \
            return 4;                                                                 \
        }                                                                             \
    } while (0)

static int read_exact(FILE* f, void* dst, size_t n) { return fread(dst, 1, n, f) == n; }

int main(int argc, char** argv) {
    if (argc != 3) {
        fprintf(stderr, "usage: %s INPUT OUTPUT\n", argv[0]);
        return 2;
    }
    FILE* in = fopen(argv[1], "rb");
    if (in == NULL) {
        fprintf(stderr, "cannot open %s\n", argv[1]);
        return 2;
    }
    int32_t hdr[4];
    int64_t dims[2];
    if (!read_exact(in, hdr, sizeof hdr) || !read_exact(in, dims, sizeof dims)) {
        fprintf(stderr, "short header\n");
        return 2;
    }
    const int cp = hdr[0], H = hdr[1], D = hdr[2], base_e = hdr[3];
    const int64_t B = dims[0], lse_stride = dims[1];
    if (cp < 1 || cp > DCP_LSE_REDUCE_CP_MAX || H < cp || H % cp != 0 || D < 8 || B < 1 || lse_stride < H) {
        fprintf(stderr, "bad header\n");
        return 2;
    }
    const int Hl = H / cp;
    const size_t src_bytes = (size_t)B * H * D * 2, lse_bytes = (size_t)B * lse_stride * 4;
    const size_t dst_bytes = (size_t)B * Hl * D * 2, lout_bytes = (size_t)B * Hl * 4;

    const void* srcs[DCP_LSE_REDUCE_CP_MAX];
    const float* lses[DCP_LSE_REDUCE_CP_MAX];
    void* dsts[DCP_LSE_REDUCE_CP_MAX];
    float* louts[DCP_LSE_REDUCE_CP_MAX];
    void* host = malloc(src_bytes > lse_bytes ? src_bytes : lse_bytes);
    if (host == NULL) return 2;
    for (int j = 0; j < cp; ++j) {
        void* d = NULL;
        if (!read_exact(in, host, src_bytes)) {
            fprintf(stderr, "short source %d\n", j);
            return 2;
        }
        CHECK_CUDA(cudaMalloc(&d, src_bytes));
        CHECK_CUDA(cudaMemcpy(d, host, src_bytes, cudaMemcpyHostToDevice));
        srcs[j] = d;
    }
    for (int j = 0; j < cp; ++j) {
        void* d = NULL;
        if (!read_exact(in, host, lse_bytes)) {
            fprintf(stderr, "short LSE %d\n", j);
            return 2;
        }
        CHECK_CUDA(cudaMalloc(&d, lse_bytes));
        CHECK_CUDA(cudaMemcpy(d, host, lse_bytes, cudaMemcpyHostToDevice));
        lses[j] = (const float*)d;
    }
    fclose(in);
    for (int r = 0; r < cp; ++r) {
        void* d = NULL;
        CHECK_CUDA(cudaMalloc(&d, dst_bytes));
        dsts[r] = d;
        CHECK_CUDA(cudaMalloc(&d, lout_bytes));
        louts[r] = (float*)d;
    }

    int rc = dcp_lse_reduce(srcs, lses, lse_stride, cp, B, H, D, base_e, dsts, louts, NULL);
    if (rc != 0) {
        fprintf(stderr, "dcp_lse_reduce returned %d: %s\n", rc, dcp_lse_reduce_strerror(rc));
        return 3;
    }
    CHECK_CUDA(cudaDeviceSynchronize());

    FILE* out = fopen(argv[2], "wb");
    if (out == NULL) return 2;
    void* back = malloc(dst_bytes);
    if (back == NULL) return 2;
    for (int r = 0; r < cp; ++r) {
        CHECK_CUDA(cudaMemcpy(back, dsts[r], dst_bytes, cudaMemcpyDeviceToHost));
        fwrite(back, 1, dst_bytes, out);
    }
    for (int r = 0; r < cp; ++r) {
        CHECK_CUDA(cudaMemcpy(back, louts[r], lout_bytes, cudaMemcpyDeviceToHost));
        fwrite(back, 1, lout_bytes, out);
    }
    fclose(out);

    const int bad = dcp_lse_reduce(srcs, lses, lse_stride, 0, B, H, D, base_e, dsts, louts, NULL);
    printf("version %d\n", dcp_lse_reduce_version());
    printf("cp=0 -> %d: %s\n", bad, dcp_lse_reduce_strerror(bad));

    for (int j = 0; j < cp; ++j) {
        cudaFree((void*)srcs[j]);
        cudaFree((void*)lses[j]);
        cudaFree(dsts[j]);
        cudaFree(louts[j]);
    }
    free(host);
    free(back);
    return 0;
}
