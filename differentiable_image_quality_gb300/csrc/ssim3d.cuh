// Launch interface of the 3D SSIM kernels (host side of ssim3d.cu).
#pragma once

#include <cstddef>
#include <cuda_runtime.h>

namespace gbssim {

// Per-device set-up of the 3D kernels (shared-memory limits); GBSSIM_OK or a status.
int ssim3d_prepare_device();

}  // namespace gbssim
