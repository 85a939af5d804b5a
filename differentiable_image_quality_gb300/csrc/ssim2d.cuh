// Launch interface of the 2D SSIM kernels (host side of ssim2d.cu).
#pragma once

#include <cstddef>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gbssim {

constexpr int kThreads2d = 128;

// Arguments of the 2D streaming kernel.  The grid is one block per (plane,
// column strip, row segment); strips may have different numbers of segments.
// Passed as a grid constant: the tensor maps are read in place.
struct Ssim2dArgs {
    // tensor staging (tma = 1): maps of img1 / img2 as [planes][H][W] with the
    // boxes of a staged row block and of a block of chain-rule pixel rows
    CUtensorMap tm_x, tm_y, tm_cx, tm_cy;
    int tma;
    unsigned tx_extra;  // test hook: bytes announced beyond the copies (0)
    const float *x;  // img1 [planes, H, W]
    const float *y;  // img2
    int H, W;        // input extent
    int Ho, Wo;      // output-domain extent (valid: H-10, W-10; same: H, W)
    int off;         // window offset: 0 valid, 5 same
    int C;           // channels (plane / C = image index)
    // segmentation (see segment_of): rows = H (gradient mode) or Ho; per_plane
    // blocks per plane; long_blocks = planes * (strips - seg_extra) * seg_base
    int strips, rows, per_plane, seg_base, seg_extra, long_blocks;
    int vec16;       // 1: W % 4 == 0 and x, y 16-byte aligned (16-byte staging)
    int pair_out;    // 1: vec16 and out1 (out2) 8-byte aligned: gradients stored in pairs
    int no_wait;     // 1: x, y are inputs that the kernel ahead did not write (no wait for it)
    // gradient mode: fields written here (grad of mean[n] * dL[n]); out2 may be null
    float *out1, *out2;
    const float *dL;  // [N] or null (then dL = 1)
    float inv_count;  // 1 / (C * Ho * Wo)
    float *map;       // [planes, Ho, Wo] or null
    size_t map_stride;  // components mode: floats from the l map to the cs map (cs to S)
    int segments;       // blocks of the launch (components mode: partials are [3][segments])
    // test build only: per output pixel, float4 statistics (mu1, mu2, sigma11 +
    // sigma22, sigma12) and float4 derivatives of S (see ssim2d_dump_launch)
    float *dump_stats, *dump_grads;
    // mean reduction (null partials: no mean)
    double *partials;
    unsigned *counter;
    float *mean;
    int images, blocks_per_image;
    double count;
};

size_t ssim2d_smem_bytes(bool grad, bool g2);
// Tensor maps of the staging copies for a.x / a.y ([planes][H][W]); sets a.tma to
// 1 when every map was encoded (a.vec16 required), else 0 (cp.async staging).
void ssim2d_prepare_staging(Ssim2dArgs &a, long long planes, bool grad);
// Reads (and with clear, resets) the device's record of staging waits that ran
// out of time (bit 0).  Synchronous.
cudaError_t ssim2d_staging_status(unsigned *flags, bool clear);
// Staging mode: 0 tensor copies where possible, 1 cp.async only, 2 tensor copies
// that announce 16 bytes more than they deliver, so that every wait runs out
// (test of the failure path).
void ssim2d_set_staging_mode(int mode);
int staging_mode();  // the mode set last (also applied to the 3D kernels)
// A tiled float32 tensor map: rank dims (innermost first), rank - 1 byte strides,
// box extents; out-of-range elements read as zeros.  False if encoding fails.
bool encode_tiled_f32(CUtensorMap &m, const void *ptr, int rank, const unsigned long long *dims,
                      const unsigned long long *strides, const unsigned *box);
// Column strips of a plane in gradient mode (over W) or forward-only mode (over Wo).
int ssim2d_strips(bool grad, int W, int Wo, int off);
const void *ssim2d_kernel_ptr(bool grad, bool g2);
cudaError_t ssim2d_launch(const Ssim2dArgs &a, bool grad, bool g2, int blocks, cudaStream_t s);
// Forward-only kernel in components mode: l, cs and S maps (a.map, a.map_stride
// apart) and their per-image means a.mean[j * images + n], j = 0 (l), 1 (cs),
// 2 (S); a.partials holds 3 x a.segments doubles.  Same plan as the forward.
// early: launch with programmatic stream serialisation (the kernel waits for
// the kernel ahead on the stream before reading anything).
cudaError_t ssim2d_components_launch(const Ssim2dArgs &a, int blocks, cudaStream_t s,
                                     bool early);
const void *ssim2d_components_kernel_ptr();
// Several octaves of the per-octave stage in one components-mode launch
// (launched early; every block waits for the kernel ahead first).  Octave o
// owns blocks first[o] .. first[o + 1] - 1 of the grid, each with its own
// partial-sum area (oct[o].partials, 3 x oct[o].segments); the launch's last
// block reduces all their means and resets *counter.
constexpr int kMaxMulti = 8;
struct Ssim2dMulti {
    Ssim2dArgs oct[kMaxMulti];
    int first[kMaxMulti + 1];
    int count;
    unsigned *counter;
};
cudaError_t ssim2d_components_multi_launch(const Ssim2dMulti &m, cudaStream_t s);
const void *ssim2d_components_multi_kernel_ptr();

// The forward-only walk split between two warpgroups of a 256-thread CTA (the
// column pass of step t beside the row pass of step t+1); needs a.tma.  kind:
// 0 forward (mean, map), 1 components mode, 2 several octaves in components
// mode.  Same plans and results as the stream kernel's forward modes.
constexpr int kThreads2dFsplit = 256;
size_t ssim2d_fsplit_smem_bytes();
const void *ssim2d_fsplit_kernel_ptr(int kind);
cudaError_t ssim2d_fsplit_launch(const Ssim2dArgs &a, bool comp, int blocks, cudaStream_t s,
                                 bool early);
cudaError_t ssim2d_fsplit_multi_launch(const Ssim2dMulti &m, cudaStream_t s);

// Octaves lo + 1 .. lo + levels (levels <= kChainLevels) of both images from
// octave lo in one launch: 2x2 box means, ragged edges over in-range pixels.
// Launched early; with wait_first the kernel ahead wrote octave lo, otherwise
// the launch runs beside the kernel ahead and waits for it only at its end.
constexpr int kChainLevels = 5;
constexpr int kChainTile = 1 << kChainLevels;  // octave-lo tile of a block: kChainTile rows,
constexpr int kChainG = 4;                      // kChainTile * kChainG columns
struct OctaveChainArgs {
    const float *x, *y;                                // octave lo, [planes][H[0]][W[0]]
    float *ox[kChainLevels], *oy[kChainLevels];        // octaves lo + 1 .. lo + levels
    int H[kChainLevels + 1], W[kChainLevels + 1];      // extents of octaves lo .. lo + levels
    int levels, tiles_x, tiles_y, wait_first;          // tiles over octave lo
    long long planes;
};
cudaError_t octave_chain_launch(const OctaveChainArgs &m, cudaStream_t s);

#ifdef GBSSIM_TEST_HOOKS
// Test build: the gradient-mode kernel with grad2 that also writes, for every
// output pixel it owns, the window statistics and the derivatives of S with
// respect to the unshifted moments (mu1, mu2, E[x^2] = E[y^2], E[xy]) into
// a.dump_stats / a.dump_grads ([planes][Ho][Wo] float4 each).
cudaError_t ssim2d_dump_launch(const Ssim2dArgs &a, int blocks, cudaStream_t s);
#endif

// g = f * dL[i / per_image] * inv_count for one or two fields (f2/g2 may be null).
cudaError_t scale_fields_launch(const float *f1, const float *f2, float *g1, float *g2,
                                const float *dL, float inv_count, size_t per_image, size_t total,
                                int sm_count, cudaStream_t s);

}  // namespace gbssim
