/* A plain C11 program that runs the forward and backward through the C ABI
 * with its own device buffers (CUDA runtime only, no Python): SReLU, MXFP8,
 * rowwise and columnwise copies, on a deterministic ragged problem.  Writes,
 * as raw little-endian bytes to stdout: the split (E int64), X and dY (BF16),
 * p (FP32), then Y's rowwise data and scales, columnwise data and scales,
 * dX (BF16), dprobs (FP32), dX's rowwise data and scales, columnwise data and
 * scales.  The test compares them with the oracle. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "gsa.h"

#define E 3
#define W 256

static uint32_t lcg = 12345u;
static uint32_t next_u32(void) {
    lcg = lcg * 1664525u + 1013904223u;
    return lcg;
}
/* a BF16 value with a random sign, exponent in [-4, 3] and mantissa */
static uint16_t rand_bf16(void) {
    const uint32_t r = next_u32();
    const uint32_t sign = (r >> 31) << 15, ex = 123u + ((r >> 8) & 7u), man = r & 0x7Fu;
    return (uint16_t)(sign | (ex << 7) | man);
}

static int check(cudaError_t e, const char *what) {
    if (e != cudaSuccess) {
        fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
        return 1;
    }
    return 0;
}

static void *dev(size_t bytes) {
    void *p = NULL;
    if (bytes == 0) bytes = 16;
    if (cudaMalloc(&p, bytes) != cudaSuccess) return NULL;
    cudaMemset(p, 0, bytes);
    return p;
}

static int dump(const void *d, size_t bytes) {
    void *h = malloc(bytes ? bytes : 1);
    if (!h || cudaMemcpy(h, d, bytes, cudaMemcpyDeviceToHost) != cudaSuccess) return 1;
    fwrite(h, 1, bytes, stdout);
    free(h);
    return 0;
}

int main(void) {
    const int64_t split[E] = {45, 0, 70};
    const int64_t M = 115;
    gsa_layout_info li;
    gsa_recipe r = {GSA_MXFP8, 0, 0, GSA_SCALES_COMPACT};
    gsa_act_params ap = {4.0f, 7.0f, 1.702f, 1.0f};
    uint16_t *hx = malloc(sizeof(uint16_t) * M * W), *hdy = malloc(sizeof(uint16_t) * M * W);
    float *hp = malloc(sizeof(float) * M);
    int64_t i;
    gsa_status st;
    if (!hx || !hdy || !hp) return 2;
    for (i = 0; i < M * W; ++i) hx[i] = rand_bf16();
    for (i = 0; i < M * W; ++i) hdy[i] = rand_bf16();
    for (i = 0; i < M; ++i) hp[i] = (float)(next_u32() >> 8) / 16777216.0f;
    if (gsa_layout(E, split, W, GSA_MXFP8, &li, NULL, NULL) != GSA_OK) return 3;
    {
        const size_t ws_bytes = gsa_workspace_size(E, split, W, GSA_ACT_SRELU, GSA_MXFP8);
        void *x = dev(sizeof(uint16_t) * M * W), *dy = dev(sizeof(uint16_t) * M * W), *p = dev(sizeof(float) * M);
        void *ws = dev(ws_bytes);
        gsa_qout yq = {dev(li.row_data_bytes), dev(li.row_scale_bytes), dev(li.col_data_bytes), dev(li.col_scale_bytes),
                       NULL, NULL};
        gsa_qout dq = {dev(li.row_data_bytes), dev(li.row_scale_bytes), dev(li.col_data_bytes), dev(li.col_scale_bytes),
                       NULL, NULL};
        void *dx = dev(sizeof(uint16_t) * M * W);
        float *dpr = (float *)dev(sizeof(float) * M);
        if (!x || !dy || !p || !ws || !dx || !dpr) return 4;
        if (check(cudaMemcpy(x, hx, sizeof(uint16_t) * M * W, cudaMemcpyHostToDevice), "copy x") ||
            check(cudaMemcpy(dy, hdy, sizeof(uint16_t) * M * W, cudaMemcpyHostToDevice), "copy dy") ||
            check(cudaMemcpy(p, hp, sizeof(float) * M, cudaMemcpyHostToDevice), "copy p"))
            return 5;
        st = grouped_scaled_act_fwd(x, (const float *)p, split, E, W, GSA_ACT_SRELU, &ap, &r, &yq, NULL, ws, ws_bytes,
                                    NULL);
        if (st != GSA_OK) {
            fprintf(stderr, "fwd: %s\n", gsa_status_string(st));
            return 6;
        }
        st = grouped_scaled_act_bwd(dy, x, (const float *)p, split, E, W, GSA_ACT_SRELU, &ap, &r, dx, &dq, dpr, NULL, ws,
                                    ws_bytes, NULL);
        if (st != GSA_OK) {
            fprintf(stderr, "bwd: %s\n", gsa_status_string(st));
            return 7;
        }
        if (check(cudaDeviceSynchronize(), "sync") || gsa_workspace_status(ws, NULL) != GSA_OK) return 8;
        fwrite(split, sizeof(int64_t), E, stdout);
        fwrite(hx, sizeof(uint16_t), M * W, stdout);
        fwrite(hdy, sizeof(uint16_t), M * W, stdout);
        fwrite(hp, sizeof(float), M, stdout);
        if (dump(yq.row_data, li.row_data_bytes) || dump(yq.row_scale, li.row_scale_bytes) ||
            dump(yq.col_data, li.col_data_bytes) || dump(yq.col_scale, li.col_scale_bytes) ||
            dump(dx, sizeof(uint16_t) * M * W) || dump(dpr, sizeof(float) * M) || dump(dq.row_data, li.row_data_bytes) ||
            dump(dq.row_scale, li.row_scale_bytes) || dump(dq.col_data, li.col_data_bytes) ||
            dump(dq.col_scale, li.col_scale_bytes))
            return 9;
    }
    free(hx);
    free(hdy);
    free(hp);
    return 0;
}
