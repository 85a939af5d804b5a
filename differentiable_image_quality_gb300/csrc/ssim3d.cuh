// Launch interface of the 3D SSIM kernels (host side of ssim3d.cu).
#pragma once

#include <cstddef>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gbssim {

constexpr int kTile3dY = 16;   // tile rows (one thread per column of the tile)
constexpr int kStats3dX = 8;   // statistics kernel tiles: 16 x 8 columns (output domain)
constexpr int kAdj3dX = 16;    // adjoint kernel tiles: 16 x 16 columns (volume)

// Arguments of both 3D kernels.  Grid: one block per (plane, z segment, tile
// row, tile column), flattened with the tile column fastest.  The statistics
// kernel tiles the output domain (Do x Ho x Wo); the adjoint kernel tiles the
// volume (D x H x W).
struct Ssim3dArgs {
    // tensor staging (tma = 1): x, y as [planes][D][H][W] with the box of a
    // staged slice tile (statistics) and of a chain-rule pixel tile (adjoint);
    // the derivative field as [planes][Do][Ho][4 Wo] floats with the box of a
    // staged derivative tile.  Passed as a grid constant: read in place.
    CUtensorMap tm_x, tm_y, tm_g, tm_cx, tm_cy;
    int tma;
    unsigned tx_extra;         // test hook: bytes announced beyond the copies (0)
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
// Tensor maps of a's staging (a.x, a.y, a.gfield and the extents set); sets
// a.tma = 1 when every map was encoded and the tiles start on 16-byte columns
// (valid padding, W % 4 == 0, 16-byte aligned volumes), else 0 (cp.async).
void ssim3d_prepare_staging(Ssim3dArgs &a, long long planes);
// Reads (and with clear, resets) the 3D kernels' record of staging waits that
// ran out of time (bit 0).  Synchronous.
cudaError_t ssim3d_staging_status(unsigned *flags, bool clear);
size_t ssim3d_adjoint_smem();
// Per-device set-up (shared-memory limits); occ[0] / occ[1] = resident CTAs per
// SM of the statistics / adjoint kernels.
cudaError_t ssim3d_prepare(int occ[2]);
cudaError_t ssim3d_stats_launch(const Ssim3dArgs &a, bool grad, int blocks, cudaStream_t s);
cudaError_t ssim3d_adjoint_launch(const Ssim3dArgs &a, bool g2, int blocks, cudaStream_t s);

}  // namespace gbssim
