// Launch interface of the 3D SSIM kernels (host side of ssim3d.cu).
#pragma once

#include <cstddef>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gbssim {

constexpr int kTile3dY = 16;   // XY tile rows of the two slice kernels
constexpr int kXy3dX = 8;      // XY statistics kernel: 16 x 8 tiles of the output domain (Ho x Wo)
constexpr int kAdj3dX = 16;    // XY adjoint kernel: 16 x 16 tiles of the volume (H x W)
constexpr int kZThreads = 128; // Z kernel: columns per block

// Arguments of the three 3D kernels.
//   xy   grid: one block per (plane, z segment, tile row, tile column), tile
//        column fastest; writes the XY-blurred shifted statistics of every
//        slice into tfield.
//   z    grid: one block per (plane, z segment, column block), column block
//        fastest; reads tfield, writes SSIM (mean, map) and, for gradients,
//        the Z-adjoint of the SSIM derivatives into ufield.
//   adj  grid as xy over the volume's tiles; reads ufield and the images,
//        writes the gradients (or the saved fields).
struct Ssim3dArgs {
    // tensor staging: x, y as [planes][D][H][W] with the box of a staged slice
    // tile (xy kernel, tma) and of a chain-rule pixel tile (adjoint kernel,
    // tma_adj); ufield as [planes][D][Ho][4 Wo] floats with the box of a staged
    // derivative tile.  Passed as a grid constant: read in place.
    CUtensorMap tm_x, tm_y, tm_g, tm_cx, tm_cy;
    int tma, tma_adj;
    unsigned tx_extra;         // test hook: bytes announced beyond the copies (0)
    const float *x, *y;        // img1, img2 [planes, D, H, W]
    int D, H, W;
    int Do, Ho, Wo;
    int off;                   // 0 valid, 5 same
    int vec16;                 // xy staging in 16-byte chunks (see fill3d)
    int C;
    int tiles_x, tiles_y, zsegs, zseg_len;
    int col_blocks;            // z kernel: blocks of kZThreads columns per plane
    float4 *tfield;            // [planes, D, Ho, Wo] XY-blurred (m1, m2, es, ed)
    float4 *ufield;            // [planes, D, Ho, Wo] Z-adjoint of (g_f1, g_es, g_ed, g_f2)
    float *out1, *out2;        // adjoint: gradients or saved fields
    const float *dL;           // [N] or null (dL = 1)
    float inv_count;           // 1 / (C * Do * Ho * Wo)
    float *map;                // z kernel: [planes, Do, Ho, Wo] or null
    double *partials;          // z kernel: null = no mean
    unsigned *counter;
    float *mean;
    int images, blocks_per_image;
    double count;
};

// Tensor maps of a's staging (a.x, a.y, a.ufield and the extents set); sets
// a.tma = 1 when the xy kernel's maps were encoded and its tiles start on
// 16-byte columns (valid padding, W % 4 == 0, 16-byte aligned volumes), and
// a.tma_adj = 1 when the adjoint kernel's were (W % 4 == 0, aligned volumes);
// else 0 (cp.async).
void ssim3d_prepare_staging(Ssim3dArgs &a, long long planes);
// Reads (and with clear, resets) the 3D kernels' record of staging waits that
// ran out of time (bit 0).  Synchronous.
cudaError_t ssim3d_staging_status(unsigned *flags, bool clear);
// Per-device set-up (shared-memory limits); occ[0..4] = resident CTAs per SM of
// the xy kernel, the z kernel (forward, gradient, gradient + grad2) and the
// adjoint kernel.
cudaError_t ssim3d_prepare(int occ[5]);
cudaError_t ssim3d_xy_launch(const Ssim3dArgs &a, int blocks, cudaStream_t s);
// The z and adjoint kernels launch early (programmatic dependent launch) and
// wait for the kernel ahead of them before reading its output.
cudaError_t ssim3d_z_launch(const Ssim3dArgs &a, bool grad, bool g2, int blocks, cudaStream_t s);
cudaError_t ssim3d_adjoint_launch(const Ssim3dArgs &a, bool g2, int blocks, cudaStream_t s);

}  // namespace gbssim
