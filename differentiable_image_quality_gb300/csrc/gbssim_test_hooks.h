/*
 * gbssim_test_hooks.h -- entry points of the test build libgbssim_test.so only
 * (sources compiled with -DGBSSIM_TEST_HOOKS).  The product library libgbssim.so
 * does not export them: they change process-wide behaviour or exist only to
 * check the kernels stage by stage.
 */
#ifndef GBSSIM_TEST_HOOKS_H
#define GBSSIM_TEST_HOOKS_H

#ifdef __cplusplus
extern "C" {
#endif

/* Make the 2D planner cut every strip into ceil(rows / `rows`) equal row
 * segments (0 restores the planner).  Affects every later call in the process. */
void gbssim_tune_seg_rows(int rows);

/* Staging of every later 2D / 3D call in the process: 0 tensor copies where the
 * images allow them (the product behaviour), 1 cp.async copies only, 2 tensor
 * copies that announce 16 bytes more than they deliver, so that every bounded
 * staging wait runs out (the failure path: NaN means, the device status bit). */
void gbssim_tune_staging(int mode);

/* Force the stream kernel for every later forward-only and per-octave launch
 * in the process (on = 0), or let the forward split kernel run where the
 * inputs allow tensor copies (on = 1, the default). */
void gbssim_tune_fwd_split(int on);

/* Stage-by-stage parity of the 2D gradient kernel: one run of the kernel of
 * ssim_fwd's stored variant with grad2 on img1 / img2 ([N, C, H, W] float32,
 * device) that also writes, for every output pixel of [N, C, Ho, Wo]:
 *   out_stats  float4 (mu1, mu2, sigma11 + sigma22, sigma12) of the window;
 *   out_grads  float4 (dS/dmu1, dS/dmu2, dS/dE[x^2] = dS/dE[y^2], dS/dE[xy]),
 *              the derivatives of S with respect to the unshifted moments;
 * both 16-byte aligned, and the two gradient fields of the per-image means
 * (dL = 1) into field1 / field2 ([N, C, H, W] each).  No mean is reduced.
 * Returns a gbssim status. */
int gbssim_test_stage_dump2d(const float *img1, const float *img2, int N, int C, int H, int W,
                             int padding, float *out_stats, float *out_grads, float *field1,
                             float *field2, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GBSSIM_TEST_HOOKS_H */
