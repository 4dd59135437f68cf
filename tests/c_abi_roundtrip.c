/*
 * Round trip through the C ABI alone, with no Python and no PyTorch: prepare
 * a small seeded NVFP4 stack on the GPU with csf_prepare, decode it with
 * csf_decode (whole, then routed into a poisoned workspace), and compare the
 * bytes on the host.  Built and run by tests/test_gpu_c_abi.py.  Prints "ok"
 * and exits 0 on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "csf.h"

#define CHECK_CUDA(x)                                                              \
    do {                                                                           \
        cudaError_t e_ = (x);                                                      \
        if (e_ != cudaSuccess) {                                                   \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));               \
            return 2;                                                              \
        }                                                                          \
    } while (0)
#define CHECK_CSF(x)                                                               \
    do {                                                                           \
        csf_status s_ = (x);                                                       \
        if (s_ != CSF_OK) {                                                        \
            fprintf(stderr, "%s: %s\n", #x, csf_status_string(s_));                \
            return 3;                                                              \
        }                                                                          \
    } while (0)

static uint32_t lcg(uint32_t *s) {
    *s = *s * 1664525u + 1013904223u;
    return *s >> 8;
}

int main(void) {
    const int E = 3, R = 200, C = 100;
    const size_t n = (size_t)E * R * C, rows = (size_t)E * R;
    uint8_t *h = (uint8_t *)malloc(n), *back = (uint8_t *)malloc(n);
    uint32_t seed = 12345u;
    for (size_t r = 0; r < rows; ++r) {                 /* base 40..80, offsets 0..14, 3% random bytes */
        const uint32_t base = 40 + lcg(&seed) % 41;
        for (int c = 0; c < C; ++c) {
            const uint32_t v = (lcg(&seed) % 100 < 3) ? lcg(&seed) % 256 : base + lcg(&seed) % 15;
            h[r * C + c] = (uint8_t)v;
        }
    }
    if (csf_abi_version() != CSF_ABI_VERSION) {
        fprintf(stderr, "ABI version %d, header %d\n", csf_abi_version(), CSF_ABI_VERSION);
        return 4;
    }
    const csf_geometry g = {CSF_NVFP4, E, R, C};
    csf_sizes_t sz;
    CHECK_CSF(csf_sizes(&g, &sz));

    uint8_t *dense, *base, *offsets, *exc_bytes, *ws, *scratch;
    uint32_t *exc_index, *err;
    CHECK_CUDA(cudaMalloc((void **)&dense, n));
    CHECK_CUDA(cudaMalloc((void **)&base, sz.base));
    CHECK_CUDA(cudaMalloc((void **)&offsets, sz.offsets));
    CHECK_CUDA(cudaMalloc((void **)&exc_index, sz.exc_index));
    CHECK_CUDA(cudaMalloc((void **)&exc_bytes, (n + 15) & ~(size_t)15));
    CHECK_CUDA(cudaMalloc((void **)&ws, n));
    CHECK_CUDA(cudaMalloc((void **)&scratch, sz.prepare_scratch));
    CHECK_CUDA(cudaMalloc((void **)&err, sizeof(uint32_t)));
    CHECK_CUDA(cudaMemset(err, 0, sizeof(uint32_t)));
    CHECK_CUDA(cudaMemset(offsets, 0, sz.offsets));
    CHECK_CUDA(cudaMemcpy(dense, h, n, cudaMemcpyHostToDevice));

    csf_stack st;
    memset(&st, 0, sizeof st);
    st.g = g;
    st.base = base;
    st.offsets = offsets;
    st.escapes = NULL;
    st.exc_index = exc_index;
    st.exc_bytes = exc_bytes;
    st.error_word = err;
    CHECK_CSF(csf_prepare(dense, &st, n, scratch, sz.prepare_scratch, NULL));
    uint32_t total = 0;
    CHECK_CUDA(cudaMemcpy(&total, exc_index + rows, sizeof total, cudaMemcpyDeviceToHost));
    st.num_exc = total;

    /* whole stack */
    CHECK_CSF(csf_decode(&st, ws, n, NULL, 0, NULL));
    CHECK_CUDA(cudaMemcpy(back, ws, n, cudaMemcpyDeviceToHost));
    if (memcmp(back, h, n) != 0) {
        fprintf(stderr, "decode differs from the dense input\n");
        return 5;
    }
    /* routed: experts 0 and 2 active (int32 prefix), expert 1's plane untouched */
    const int32_t start_h[4] = {0, 1, 1, 3};
    int32_t *start;
    CHECK_CUDA(cudaMalloc((void **)&start, sizeof start_h));
    CHECK_CUDA(cudaMemcpy(start, start_h, sizeof start_h, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemset(ws, 0xFF, n));
    CHECK_CSF(csf_decode(&st, ws, n, start, 0, NULL));
    CHECK_CUDA(cudaMemcpy(back, ws, n, cudaMemcpyDeviceToHost));
    const size_t plane = (size_t)R * C;
    for (size_t i = 0; i < n; ++i) {
        const int e = (int)(i / plane);
        const uint8_t want = (e == 1) ? 0xFF : h[i];
        if (back[i] != want) {
            fprintf(stderr, "routed decode differs at byte %zu (expert %d)\n", i, e);
            return 6;
        }
    }
    uint32_t word = 0;
    CHECK_CUDA(cudaMemcpy(&word, err, sizeof word, cudaMemcpyDeviceToHost));
    if (word != 0) {
        fprintf(stderr, "device error word %#x\n", word);
        return 7;
    }
    printf("ok %u exceptions\n", total);
    cudaFree(dense); cudaFree(base); cudaFree(offsets); cudaFree(exc_index); cudaFree(exc_bytes);
    cudaFree(ws); cudaFree(scratch); cudaFree(err); cudaFree(start);
    free(h); free(back);
    return 0;
}
