/*
 * A C caller of the library through include/gbmoe.h alone: the whole
 * Standard layer (moe_forward, bf16, softmax top-2) on seeded inputs, its
 * workspace sized by moe_workspace_size, device memory from the CUDA
 * runtime.  Exits 0 and prints the output's checksum when every call returns
 * GBMOE_OK, the device error word stays 0, every output is finite and a
 * second run gives the same bits; exits 1 otherwise.  With a file name as
 * its argument it also writes there, raw and in this order, x (M, K) bf16,
 * the logits (M, E) fp32, w1 (E, 2N, K) bf16, w2 (E, K, N) bf16 and the
 * output (M, K) bf16, for a check against an independent implementation.
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "gbmoe.h"

enum { M = 64, K = 256, N = 128, E = 8, TOPK = 2 };

static uint32_t lcg_state = 12345u;

/* uniform in [-1, 1) */
static float next_uniform(void) {
    lcg_state = lcg_state * 1664525u + 1013904223u;
    return (float)(lcg_state >> 8) / 8388608.0f - 1.0f;
}

/* bf16 bits of a float, rounded to nearest even (inputs are finite) */
static uint16_t bf16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float bf16_value(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

#define CUDA_OK(call)                                                          \
    do {                                                                       \
        cudaError_t e_ = (call);                                               \
        if (e_ != cudaSuccess) {                                               \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));        \
            return 1;                                                          \
        }                                                                      \
    } while (0)

static void fill_bf16(uint16_t *h, size_t n, float scale) {
    size_t i;
    for (i = 0; i < n; ++i)
        h[i] = bf16_bits(next_uniform() * scale);
}

int main(int argc, char **argv) {
    const size_t nx = (size_t)M * K, nl = (size_t)M * E;
    const size_t nw1 = (size_t)E * 2 * N * K, nw2 = (size_t)E * K * N;
    uint16_t *hx = malloc(nx * 2), *hw1 = malloc(nw1 * 2), *hw2 = malloc(nw2 * 2);
    uint16_t *hout = malloc(nx * 2), *hout2 = malloc(nx * 2);
    float *hl = malloc(nl * 4);
    uint16_t *dx, *dw1, *dw2, *dout;
    float *dl;
    int32_t *derr, herr = -1;
    void *ws;
    size_t wsb, i;
    double checksum = 0.0;
    int run;
    gbmoe_status_t st;

    if (!hx || !hw1 || !hw2 || !hout || !hout2 || !hl) return 1;
    fill_bf16(hx, nx, 1.0f);
    for (i = 0; i < nl; ++i) hl[i] = next_uniform() * 2.0f;
    fill_bf16(hw1, nw1, 1.0f / 16.0f); /* about N(0, 1/K) in scale */
    fill_bf16(hw2, nw2, 1.0f / 11.0f);

    wsb = moe_workspace_size(GBMOE_WS_FORWARD, M, E, N, K, TOPK, GBMOE_BF16);
    if (wsb == 0) {
        fprintf(stderr, "moe_workspace_size refused the shapes\n");
        return 1;
    }
    CUDA_OK(cudaMalloc((void **)&dx, nx * 2));
    CUDA_OK(cudaMalloc((void **)&dl, nl * 4));
    CUDA_OK(cudaMalloc((void **)&dw1, nw1 * 2));
    CUDA_OK(cudaMalloc((void **)&dw2, nw2 * 2));
    CUDA_OK(cudaMalloc((void **)&dout, nx * 2));
    CUDA_OK(cudaMalloc((void **)&derr, 4));
    CUDA_OK(cudaMalloc(&ws, wsb));
    CUDA_OK(cudaMemcpy(dx, hx, nx * 2, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dl, hl, nl * 4, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dw1, hw1, nw1 * 2, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dw2, hw2, nw2 * 2, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemset(derr, 0, 4));

    /* a bad argument is refused on the host, before anything is enqueued */
    st = moe_forward(dx, dl, NULL, M, K, N, E, NULL, E, E + 1, GBMOE_SOFTMAX, 1, 1, 1, 0,
                     GBMOE_ACT_SILU, GBMOE_BF16, dw1, NULL, dw2, NULL, NULL, NULL, dout, NULL,
                     NULL, ws, wsb, derr, NULL);
    if (st != GBMOE_INVALID_ARG) {
        fprintf(stderr, "topk > E was not refused: %s\n", gbmoe_status_string(st));
        return 1;
    }

    for (run = 0; run < 2; ++run) {
        st = moe_forward(dx, dl, NULL, M, K, N, E, NULL, E, TOPK, GBMOE_SOFTMAX, 1, 1, 1, 0,
                         GBMOE_ACT_SILU, GBMOE_BF16, dw1, NULL, dw2, NULL, NULL, NULL, dout,
                         NULL, NULL, ws, wsb, derr, NULL);
        if (st != GBMOE_OK) {
            fprintf(stderr, "moe_forward: %s (cuda error %d)\n", gbmoe_status_string(st),
                    gbmoe_last_cuda_error());
            return 1;
        }
        CUDA_OK(cudaDeviceSynchronize());
        CUDA_OK(cudaMemcpy(run == 0 ? hout : hout2, dout, nx * 2, cudaMemcpyDeviceToHost));
    }
    CUDA_OK(cudaMemcpy(&herr, derr, 4, cudaMemcpyDeviceToHost));
    if (herr != 0) {
        fprintf(stderr, "device error word %d\n", herr);
        return 1;
    }
    for (i = 0; i < nx; ++i) {
        const float v = bf16_value(hout[i]);
        if (!isfinite(v)) {
            fprintf(stderr, "output %zu is not finite\n", i);
            return 1;
        }
        checksum += fabs((double)v);
    }
    if (memcmp(hout, hout2, nx * 2) != 0) {
        fprintf(stderr, "two runs differ\n");
        return 1;
    }
    if (argc > 1) {
        FILE *f = fopen(argv[1], "wb");
        if (!f || fwrite(hx, 2, nx, f) != nx || fwrite(hl, 4, nl, f) != nl ||
            fwrite(hw1, 2, nw1, f) != nw1 || fwrite(hw2, 2, nw2, f) != nw2 ||
            fwrite(hout, 2, nx, f) != nx || fclose(f) != 0) {
            fprintf(stderr, "could not write %s\n", argv[1]);
            return 1;
        }
    }
    printf("c_abi_forward ok: M=%d K=%d N=%d E=%d top-%d, sum|out| = %.6f\n", M, K, N, E, TOPK,
           checksum);
    cudaFree(dx); cudaFree(dl); cudaFree(dw1); cudaFree(dw2); cudaFree(dout);
    cudaFree(derr); cudaFree(ws);
    free(hx); free(hw1); free(hw2); free(hout); free(hout2); free(hl);
    return 0;
}
