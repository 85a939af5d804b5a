/*
 * gbssim.h -- C ABI of a fused, differentiable SSIM loss for NVIDIA GB300 (sm_103a).
 *
 * What is computed (per image n, channel c, output pixel p of the domain Omega):
 *   mu1, mu2, E[x^2], E[y^2], E[xy] under an 11x11 Gaussian window (sigma 1.5,
 *   weights normalised to sum to one) -- the five blurred quantities of the
 *   TriSSIM README, "How it works", with the fixed 11x11 window of the fused-ssim
 *   README introduction;
 *   S(p) = (2 mu1 mu2 + C1)(2 sigma12 + C2) / ((mu1^2 + mu2^2 + C1)(sigma11 + sigma22 + C2)),
 *   C1 = 0.01^2, C2 = 0.03^2 (images in [0, 1]: fused-ssim README, "Constraints");
 *   mean[n] = average of S over the channels and Omega of image n (fused-ssim
 *   README, "Usage", returns this mean).
 * The backward applies the adjoint of the blur (a "full" correlation) to the
 * upstream gradients of the statistics and combines them by the chain rule of
 * the TriSSIM README, "How it works":
 *   grad_img1 = B^T(g_mu1) + 2 img1 B^T(g_s11) + img2 B^T(g_s12), grad_img2 likewise.
 *
 * Padding (fused-ssim README, "Usage"):
 *   GBSSIM_VALID      Omega = (H-10) x (W-10): windows that lie inside the image.
 *                     Needs H, W >= 11 (and D >= 11 in 3D).
 *   GBSSIM_SAME_ZERO  Omega = H x W: the image is extended by zeros; border
 *                     windows are not renormalised.  Needs H, W >= 1.
 *
 * Conventions shared by every call below:
 *   - Images are contiguous float32, NCHW (2D) or NCDHW (3D), in DEVICE memory,
 *     4-byte aligned.  Values are expected in [0, 1] but are not checked; NaN
 *     propagates.
 *   - All pointers are caller-owned.  The library allocates no memory and keeps
 *     no state between calls except small per-device launch caches.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call
 *     is asynchronous on that stream.  Argument errors are returned before any
 *     launch; a failed launch returns GBSSIM_ECUDA.
 *   - Return value: GBSSIM_OK (0) or a negative status; nothing aborts.
 *   - Calls are deterministic: the same inputs give bit-identical outputs.
 *
 * Accuracy.  The arithmetic is float32 (the means are summed in double).  The
 * kernels evaluate an exactly equivalent form of the definition: values are
 * shifted by one pixel of their neighbourhood before they are squared (2D; a
 * constant 1/2 in 3D), the fourth blurred quantity is E[(x - y)^2] instead of
 * E[xy], and the chain rule is taken through x - y.  Against a double-precision
 * evaluation of the definition, for images in [0, 1], the test suite holds
 * per-image means to 1e-5, gradients to 1e-4 of their largest element, 2D SSIM
 * maps to 5e-6 and 3D maps to 3e-5, flat (constant) regions included.
 */
#ifndef GBSSIM_H
#define GBSSIM_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GBSSIM_ABI_VERSION 1

typedef enum { GBSSIM_VALID = 0, GBSSIM_SAME_ZERO = 1 } gbssim_padding;

enum {
    GBSSIM_OK = 0,
    GBSSIM_EINVAL = -1,     /* null pointer where one is required, bad enum, aliasing */
    GBSSIM_ESHAPE = -2,     /* N, C < 1, a spatial extent too small, or sizes too large */
    GBSSIM_EALIGN = -3,     /* a pointer not 4-byte aligned */
    GBSSIM_EWORKSPACE = -4, /* workspace or saved buffer missing or too small */
    GBSSIM_ECUDA = -5,      /* a CUDA runtime call or launch failed */
    GBSSIM_ETOOLARGE = -6   /* too large for the fixed scratch of ssim_fwd_noalloc */
};

/* ABI version of the loaded library (GBSSIM_ABI_VERSION at its build). */
int gbssim_abi_version(void);

/* A static, human-readable description of a status code. */
const char *gbssim_strerror(int status);

/* The eleven float32 taps the kernels use (host copy), w[0..10].  They are the
 * float32 roundings of exp(-(k-5)^2 / 4.5), k = 0..10, divided by their sum. */
void gbssim_window(float w[11]);

/* Kernel-side failures recorded on the current device since the previous call,
 * as bit flags in *flags_out, which this call then clears.
 *   bit 0 (GBSSIM_DEV_STAGING_TIMEOUT): a 2D kernel waited about a second for
 *   its staged input rows without them arriving; its blocks stopped early, so
 *   that call's gradients and map are not valid, and the mean of each image
 *   with a stopped block is NaN.
 * Synchronises the device: a diagnostic, not part of the hot path.  Returns
 * GBSSIM_OK, GBSSIM_EINVAL (null flags_out) or GBSSIM_ECUDA. */
#define GBSSIM_DEV_STAGING_TIMEOUT 1u
int gbssim_device_status(unsigned *flags_out);

/* ------------------------------------------------------------------ 2D ----- */

/* Bytes of scratch that ssim_fwd needs for the given shape (per-block partial
 * sums and a completion counter).  Returns 0 if the shape is invalid.  The
 * buffer must be zero-filled once before its first use; every completed call
 * leaves it zero-filled again.  Two calls that run at the same time must not
 * share one workspace. */
size_t gbssim_workspace_bytes(int N, int C, int H, int W, int padding);

/* Bytes of the optional `saved` buffer of ssim_fwd: one float32 field the size
 * of the input for grad_img1, plus one more when want_grad2 != 0. */
size_t gbssim_saved_bytes(int N, int C, int H, int W, int want_grad2);

/* Forward.
 *   img1, img2       [N, C, H, W] float32, device.
 *   out_mean         [N] float32, device: mean SSIM of each image.
 *   out_map_or_null  [N, C, Ho, Wo] float32, device, or NULL: the SSIM map.
 *   saved_or_null    device buffer of saved_bytes >= gbssim_saved_bytes(..., want_grad2),
 *                    or NULL.  When given, the forward also computes, for each
 *                    image, the gradient of mean[n] itself (i.e. with dL = 1)
 *                    with respect to img1 (and img2 when want_grad2 != 0), so
 *                    that ssim_bwd is a single scaling pass.  NULL is the
 *                    inference mode ("train=False" of the fused-ssim README,
 *                    "Usage"): only the mean (and map) are computed.
 *   workspace        device buffer of workspace_bytes >= gbssim_workspace_bytes(...).
 */
int ssim_fwd(const float *img1, const float *img2, int N, int C, int H, int W, int padding,
             float *out_mean, float *out_map_or_null, float *saved_or_null, size_t saved_bytes,
             int want_grad2, void *workspace, size_t workspace_bytes, void *stream);

/* Backward of loss = sum_n dL[n] * mean[n] (dL = dLoss/dmean, [N] float32, device).
 *   saved_or_null    the buffer written by a matching ssim_fwd (same images, shape
 *                    and padding; want_grad2 set there if grad_img2 is wanted
 *                    here), or NULL to recompute everything from img1 and img2.
 *   grad_img1        [N, C, H, W] float32, device; overwritten (not accumulated).
 *   grad_img2_or_null  likewise, or NULL to skip it (fused-ssim README,
 *                    "Constraints": by default only img1 is differentiable).
 * Gradient buffers must not overlap img1, img2 or each other. */
int ssim_bwd(const float *dL, const float *img1, const float *img2, int N, int C, int H, int W,
             int padding, const float *saved_or_null, size_t saved_bytes, float *grad_img1,
             float *grad_img2_or_null, void *stream);

/* Forward and backward in one call, for a loss whose derivative with respect to
 * each image's mean SSIM is known before the forward -- the usual training loss
 * 1 - mean over the batch has dL[n] = -1/N.  One kernel pass computes the
 * means (and the map), the upstream gradients of the statistics, the adjoint
 * and the chain rule (TriSSIM README, "How it works"), so the statistics are
 * formed once and no intermediate field is written.  Arguments as in ssim_fwd
 * and ssim_bwd; dL is [N] float32 on the device, read by the kernel.  The
 * workspace is sized by gbssim_workspace_bytes. */
int ssim_fwd_bwd(const float *img1, const float *img2, int N, int C, int H, int W, int padding,
                 const float *dL, float *out_mean, float *out_map_or_null, float *grad_img1,
                 float *grad_img2_or_null, void *workspace, size_t workspace_bytes, void *stream);

/* Size of the device array behind ssim_fwd_noalloc (per GPU, for the process's life). */
#define GBSSIM_NOALLOC_SCRATCH_BYTES (1u << 20)

/* ssim_fwd for callers that cannot allocate device memory.  The pages describe
 * no such call; it exists for users of this library.  A plug-in running inside
 * an application that owns the device memory, or code on a latency-critical
 * path that must not call cudaMalloc (which can also synchronise the device),
 * cannot provide ssim_fwd's workspace.  This call takes the same arguments minus
 * the workspace and uses a fixed array that the library defines in device
 * memory instead: GBSSIM_NOALLOC_SCRATCH_BYTES on every GPU that loads the
 * library, held until the process exits.  It allocates nothing.
 *   - Shapes whose workspace (gbssim_workspace_bytes) would exceed that array
 *     return GBSSIM_ETOOLARGE; use ssim_fwd for them.  A 1 x 3 x 1080 x 1920
 *     pair needs about 35 KB of it.  This size check comes first: such a shape
 *     returns GBSSIM_ETOOLARGE whatever the other arguments are.  Any other
 *     argument error is reported as ssim_fwd reports it.
 *   - All calls on a device share the one array and it keeps the previous
 *     call's contents; the call clears the part that must start at zero, on
 *     `stream`, before its kernel.  Calls whose work overlaps on the GPU (other
 *     streams, other threads) race on it: order them on one stream.
 *   - Every call looks up the array's address on the current device (nothing
 *     is cached, so a device reset cannot leave a stale address).  The first
 *     call on each device also does the per-device set-up ssim_fwd does; make
 *     that first call before any stream capture.
 * Results are identical to ssim_fwd's. */
int ssim_fwd_noalloc(const float *img1, const float *img2, int N, int C, int H, int W,
                     int padding, float *out_mean, float *out_map_or_null, float *saved_or_null,
                     size_t saved_bytes, int want_grad2, void *stream);

/* ------------------------------------------------------- per-octave maps --- */
/* The per-octave stage of the ssimulacra2 hand-off page ("blur -> pointwise
 * sigma11 / sigma22 / sigma12 -> error maps", once per octave of a 2x pyramid),
 * with this library's 11x11 Gaussian window in place of that metric's
 * recursive blur and with SSIM's own three per-pixel maps as the error maps:
 *   l  = (2 mu1 mu2 + C1) / (mu1^2 + mu2^2 + C1)       luminance
 *   cs = (2 sigma12 + C2) / (sigma11 + sigma22 + C2)   contrast-structure
 *   S  = l * cs                                         SSIM (as ssim_fwd)
 * Octave 0 is the input pair; octave o + 1 is octave o downscaled 2x: each pixel
 * is the mean of the pixels of its 2x2 block that lie inside the image (so
 * ceil(H/2) x ceil(W/2); a ragged last row or column averages one or two
 * pixels).  The page gives no formula for the downscale or the error maps;
 * these are the plain readings.  Forward only; no gradients. */

/* Extents (H_o, W_o) of octave o: H_0 = H, H_{o+1} = ceil(H_o / 2). */

/* Workspace bytes of ssim_pyramid (0 if a shape or octave count is invalid:
 * octaves >= 1 and every octave extent must suit the padding, i.e. >= 11 for
 * valid).  Same zero-fill rule as gbssim_workspace_bytes.  It holds the
 * downscaled images of octaves 1 .. octaves-1 and the block partial sums. */
size_t gbssim_pyramid_workspace_bytes(int N, int C, int H, int W, int padding, int octaves);

/* Floats of the optional maps buffer: per octave o, three maps of
 * N*C*Ho_o*Wo_o floats (l, then cs, then S), octaves one after another.  0 if
 * invalid. */
size_t gbssim_pyramid_map_floats(int N, int C, int H, int W, int padding, int octaves);

/* Per-octave means and maps.
 *   img1, img2    [N, C, H, W] float32, device.
 *   octaves       number of octaves (>= 1).
 *   out_means     [octaves][3][N] float32, device: per octave the mean of l, of
 *                 cs and of S over the channels and output pixels of image n.
 *   maps_or_null  device buffer of gbssim_pyramid_map_floats(...) floats, or NULL.
 *   workspace     device buffer of gbssim_pyramid_workspace_bytes(...) bytes.
 * Octave 0's S mean equals ssim_fwd's mean. */
int ssim_pyramid(const float *img1, const float *img2, int N, int C, int H, int W, int padding,
                 int octaves, float *out_means, float *maps_or_null, void *workspace,
                 size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------ 3D ----- */
/* fused-ssim README, "3D data": the same statistics with an 11x11x11 window on
 * NCDHW volumes.  Arguments mean what they mean in 2D, with D added; both
 * paddings apply to all three axes (valid needs D, H, W >= 11).
 * The 3D calls keep two fields between their three kernels in the workspace:
 * the XY-blurred statistics of every slice and the Z-blurred derivatives of
 * SSIM, one float4 per (slice, output column) each; so ssim3d_bwd takes a
 * workspace too (it is only used when saved_or_null is NULL). */

/* Workspace bytes of ssim3d_fwd / ssim3d_bwd (0 for an invalid shape).  Same
 * zero-fill rule as gbssim_workspace_bytes. */
size_t gbssim3d_workspace_bytes(int N, int C, int D, int H, int W, int padding);

/* Bytes of the optional saved buffer (one field the size of the input per
 * wanted gradient). */
size_t gbssim3d_saved_bytes(int N, int C, int D, int H, int W, int want_grad2);

int ssim3d_fwd(const float *img1, const float *img2, int N, int C, int D, int H, int W,
               int padding, float *out_mean, float *out_map_or_null, float *saved_or_null,
               size_t saved_bytes, int want_grad2, void *workspace, size_t workspace_bytes,
               void *stream);

int ssim3d_bwd(const float *dL, const float *img1, const float *img2, int N, int C, int D,
               int H, int W, int padding, const float *saved_or_null, size_t saved_bytes,
               float *grad_img1, float *grad_img2_or_null, void *workspace,
               size_t workspace_bytes, void *stream);

/* The single-call forward + backward of ssim_fwd_bwd for volumes. */
int ssim3d_fwd_bwd(const float *img1, const float *img2, int N, int C, int D, int H, int W,
                   int padding, const float *dL, float *out_mean, float *out_map_or_null,
                   float *grad_img1, float *grad_img2_or_null, void *workspace,
                   size_t workspace_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GBSSIM_H */
