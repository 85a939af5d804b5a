/* A plain C caller of the C ABI (no Python, no torch): the loss 1 - SSIM of a
 * small image pair, forward with saved fields, stored backward, and the
 * recompute backward, on the CUDA runtime's own device buffers.
 *
 * The pair is generated here from a closed formula that the test restates in
 * numpy:  img1[c][i][j] = 0.5 + 0.4 sin(0.37 i + 0.11 j + c),
 *         img2[c][i][j] = img1 + 0.05 cos(0.23 i - 0.19 j + 2 c).
 * Prints the mean, then every gradient value of img1 (stored, then recompute).
 * Exit status: 0 on success, 1 on any non-zero status from the library or the
 * runtime. */
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <cuda_runtime.h>

#include "gbssim.h"

#define CHECK_CUDA(x)                                                     \
    do {                                                                  \
        cudaError_t e_ = (x);                                             \
        if (e_ != cudaSuccess) {                                          \
            fprintf(stderr, "cuda: %s\n", cudaGetErrorString(e_));        \
            return 1;                                                     \
        }                                                                 \
    } while (0)
#define CHECK_GB(x)                                                       \
    do {                                                                  \
        int s_ = (x);                                                     \
        if (s_ != 0) {                                                    \
            fprintf(stderr, "gbssim: %s\n", gbssim_strerror(s_));         \
            return 1;                                                     \
        }                                                                 \
    } while (0)

int main(void)
{
    const int N = 1, C = 2, H = 24, W = 30, padding = 0; /* valid */
    const size_t n = (size_t)N * C * H * W;
    float *h1 = (float *)malloc(n * sizeof(float));
    float *h2 = (float *)malloc(n * sizeof(float));
    float *hg = (float *)malloc(n * sizeof(float));
    if (!h1 || !h2 || !hg) return 1;
    for (int c = 0; c < C; ++c)
        for (int i = 0; i < H; ++i)
            for (int j = 0; j < W; ++j) {
                const size_t k = ((size_t)c * H + i) * W + j;
                h1[k] = (float)(0.5 + 0.4 * sin(0.37 * i + 0.11 * j + c));
                h2[k] = (float)(h1[k] + 0.05 * cos(0.23 * i - 0.19 * j + 2.0 * c));
            }
    const size_t ws_bytes = gbssim_workspace_bytes(N, C, H, W, padding);
    const size_t saved_bytes = gbssim_saved_bytes(N, C, H, W, 0);
    float *d1, *d2, *dmean, *dsaved, *dg, *ddl;
    void *dws;
    CHECK_CUDA(cudaMalloc((void **)&d1, n * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void **)&d2, n * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void **)&dmean, N * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void **)&dsaved, saved_bytes));
    CHECK_CUDA(cudaMalloc((void **)&dg, n * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void **)&ddl, N * sizeof(float)));
    CHECK_CUDA(cudaMalloc(&dws, ws_bytes));
    CHECK_CUDA(cudaMemset(dws, 0, ws_bytes));
    CHECK_CUDA(cudaMemcpy(d1, h1, n * sizeof(float), cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d2, h2, n * sizeof(float), cudaMemcpyHostToDevice));
    const float dl = -1.0f; /* loss = 1 - mean */
    CHECK_CUDA(cudaMemcpy(ddl, &dl, sizeof(float), cudaMemcpyHostToDevice));

    CHECK_GB(ssim_fwd(d1, d2, N, C, H, W, padding, dmean, NULL, dsaved, saved_bytes, 0, dws,
                      ws_bytes, NULL));
    CHECK_GB(ssim_bwd(ddl, d1, d2, N, C, H, W, padding, dsaved, saved_bytes, dg, NULL, NULL));
    float mean = 0.0f;
    CHECK_CUDA(cudaMemcpy(&mean, dmean, sizeof(float), cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(hg, dg, n * sizeof(float), cudaMemcpyDeviceToHost));
    printf("%.9g\n", mean);
    for (size_t k = 0; k < n; ++k) printf("%.9g\n", hg[k]);
    CHECK_GB(ssim_bwd(ddl, d1, d2, N, C, H, W, padding, NULL, 0, dg, NULL, NULL));
    CHECK_CUDA(cudaMemcpy(hg, dg, n * sizeof(float), cudaMemcpyDeviceToHost));
    for (size_t k = 0; k < n; ++k) printf("%.9g\n", hg[k]);
    CHECK_CUDA(cudaDeviceSynchronize());
    return 0;
}
