// ssim_fwd_noalloc: the 2D forward for callers that cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc: a plug-in or custom operator
// living inside a host application whose allocator owns all device memory, or
// code on a latency-critical path where an allocation (and the device-wide
// synchronisation cudaMalloc / cudaFree can imply) is not acceptable.  Such a
// caller still owns its inputs and outputs, but cannot hand ssim_fwd the small
// scratch buffer it needs (per-block partial sums and a completion counter).
// This entry point takes that scratch from a fixed array in device memory that
// the library itself defines; every GPU that loads the library holds the array
// (GBSSIM_NOALLOC_SCRATCH_BYTES) until the process exits.
#include <cstddef>

#include <cuda_runtime.h>

#include "gbssim.h"

namespace {

constexpr size_t kScratchBytes = GBSSIM_NOALLOC_SCRATCH_BYTES;
constexpr size_t kCounterBytes = 256;  // ssim_fwd keeps its completion counter here

// The scratch.  In host code this name is only a stand-in for the device
// array: its device address comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the scratch on the current device.  Looked up on every
// call and never cached: a cached address would go stale if the application
// reset the device or its primary context was destroyed and created again.
int scratch_on_current_device(void **out)
{
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
        (void)cudaGetLastError();
        return GBSSIM_ECUDA;
    }
    *out = p;
    return GBSSIM_OK;
}

}  // namespace

extern "C" int ssim_fwd_noalloc(const float *img1, const float *img2, int N, int C, int H, int W,
                                int padding, float *out_mean, float *out_map_or_null,
                                float *saved_or_null, size_t saved_bytes, int want_grad2,
                                void *stream)
{
    // the size check comes first: a problem beyond the array is refused whatever
    // the other arguments are, before anything touches the device
    const size_t need = gbssim_workspace_bytes(N, C, H, W, padding);
    if (need == 0)  // invalid shape or padding: let ssim_fwd report which argument
        return ssim_fwd(img1, img2, N, C, H, W, padding, out_mean, out_map_or_null,
                        saved_or_null, saved_bytes, want_grad2, nullptr, 0, stream);
    if (need > kScratchBytes) return GBSSIM_ETOOLARGE;
    void *scratch = nullptr;
    const int rc = scratch_on_current_device(&scratch);
    if (rc != GBSSIM_OK) return rc;
    // The array keeps whatever the previous call left; the counter must start at zero.
    if (cudaMemsetAsync(scratch, 0, kCounterBytes, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return GBSSIM_ECUDA;
    }
    return ssim_fwd(img1, img2, N, C, H, W, padding, out_mean, out_map_or_null, saved_or_null,
                    saved_bytes, want_grad2, scratch, kScratchBytes, stream);
}
