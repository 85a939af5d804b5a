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

#ifdef __cplusplus
}
#endif

#endif /* GBSSIM_TEST_HOOKS_H */
