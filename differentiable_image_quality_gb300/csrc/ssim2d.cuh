// Launch interface of the 2D SSIM kernels (host side of ssim2d.cu).
#pragma once

#include <cstddef>
#include <cuda_runtime.h>

namespace gbssim {

constexpr int kThreads2d = 128;

// Arguments of the 2D streaming kernel.  The grid is one block per
// (plane, row segment, column strip), flattened with the strip fastest.
struct Ssim2dArgs {
    const float *x;  // img1 [planes, H, W]
    const float *y;  // img2
    int H, W;        // input extent
    int Ho, Wo;      // output-domain extent (valid: H-10, W-10; same: H, W)
    int off;         // window offset: 0 valid, 5 same
    int C;           // channels (plane / C = image index)
    int strips, segs, seg_rows;
    int vec16;       // 1: W % 4 == 0 and x, y 16-byte aligned (16-byte staging)
    // gradient mode: fields written here (grad of mean[n] * dL[n]); out2 may be null
    float *out1, *out2;
    const float *dL;  // [N] or null (then dL = 1)
    float inv_count;  // 1 / (C * Ho * Wo)
    float *map;       // [planes, Ho, Wo] or null
    // mean reduction (null partials: no mean)
    double *partials;
    unsigned *counter;
    float *mean;
    int images, blocks_per_image;
    double count;
};

size_t ssim2d_smem_bytes(bool grad, bool g2);
// Column strips of a plane in gradient mode (over W) or forward-only mode (over Wo).
int ssim2d_strips(bool grad, int W, int Wo, int off);
const void *ssim2d_kernel_ptr(bool grad, bool g2);
cudaError_t ssim2d_launch(const Ssim2dArgs &a, bool grad, bool g2, int blocks, cudaStream_t s);

// g = f * dL[i / per_image] * inv_count for one or two fields (f2/g2 may be null).
cudaError_t scale_fields_launch(const float *f1, const float *f2, float *g1, float *g2,
                                const float *dL, float inv_count, size_t per_image, size_t total,
                                int sm_count, cudaStream_t s);

}  // namespace gbssim
