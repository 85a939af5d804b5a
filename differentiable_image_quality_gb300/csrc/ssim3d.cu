// 3D SSIM (fused-ssim README, "3D data").
#include "../../include/gbssim.h"
#include "common.cuh"
#include "ssim3d.cuh"

namespace gbssim {
int ssim3d_prepare_device() { return GBSSIM_OK; }
}  // namespace gbssim

extern "C" {

size_t gbssim3d_workspace_bytes(int, int, int, int, int, int) { return 0; }
size_t gbssim3d_saved_bytes(int, int, int, int, int, int) { return 0; }

int ssim3d_fwd(const float *, const float *, int, int, int, int, int, int, float *, float *,
               float *, size_t, int, void *, size_t, void *)
{
    return GBSSIM_EINVAL;
}

int ssim3d_bwd(const float *, const float *, const float *, int, int, int, int, int, int,
               const float *, size_t, float *, float *, void *)
{
    return GBSSIM_EINVAL;
}

}  // extern "C"
