// Launch interface of the 3D SSIM kernels (host side of ssim3d.cu).
#pragma once

#include <cstddef>
#include <cuda_runtime.h>

namespace gbssim {

constexpr int kThreads3d = 256;
constexpr int kTile3dY = 16;  // tile rows (one thread per column of the tile)
constexpr int kTile3dX = 16;

// Arguments of both 3D kernels.  Grid: one block per (plane, z segment, tile
// row, tile column), flattened with the tile column fastest.  The statistics
// kernel tiles the output domain (Do x Ho x Wo); the adjoint kernel tiles the
// volume (D x H x W).
struct Ssim3dArgs {
    const float *x, *y;        // img1, img2 [planes, D, H, W]
    int D, H, W;
    int Do, Ho, Wo;
    int off;                   // 0 valid, 5 same
    int vec16;                 // statistics staging in 16-byte chunks (see fill3d)
    int C;
    int tiles_x, tiles_y, zsegs, zseg_len;
    float *gfield;             // [planes, Do, Ho, Wo] float4 derivatives (workspace)
    float *out1, *out2;        // adjoint: gradients or saved fields
    const float *dL;           // [N] or null (dL = 1)
    float inv_count;           // 1 / (C * Do * Ho * Wo)
    float *map;                // statistics: [planes, Do, Ho, Wo] or null
    double *partials;          // statistics: null = no mean
    unsigned *counter;
    float *mean;
    int images, blocks_per_image;
    double count;
};

size_t ssim3d_stats_smem();
size_t ssim3d_adjoint_smem();
// Per-device set-up (shared-memory limits); occ[0] / occ[1] = resident CTAs per
// SM of the statistics / adjoint kernels.
cudaError_t ssim3d_prepare(int occ[2]);
cudaError_t ssim3d_stats_launch(const Ssim3dArgs &a, bool grad, int blocks, cudaStream_t s);
cudaError_t ssim3d_adjoint_launch(const Ssim3dArgs &a, bool g2, int blocks, cudaStream_t s);

}  // namespace gbssim
