// Shared device helpers of the SSIM kernels (sm_103a).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace gbssim {

// The eleven taps of the window: float32 roundings of exp(-(k-5)^2 / (2 * 1.5^2)),
// k = 0..10, divided by their sum (fused-ssim README introduction: a fixed 11x11
// Gaussian window "as per the original SSIM paper"; sigma 1.5).  Symmetric:
// w(k) = w(10 - k), six distinct values.
__host__ __device__ constexpr float tap(int k)
{
    return (k == 0 || k == 10)  ? 1.028380124e-03f
           : (k == 1 || k == 9) ? 7.598758209e-03f
           : (k == 2 || k == 8) ? 3.600077331e-02f
           : (k == 3 || k == 7) ? 1.093606874e-01f
           : (k == 4 || k == 6) ? 2.130055428e-01f
                                : 2.660117149e-01f;
}

constexpr int kTaps = 11;
constexpr int kRadius = 5;

// Stabilising constants for data range 1 (fused-ssim README, "Constraints").
constexpr float kC1 = 1.0e-4f;  // (0.01 * 1)^2
constexpr float kC2 = 9.0e-4f;  // (0.03 * 1)^2

// Values enter the products shifted: x' = x - s, y' = y - t, the image being
// extended by zeros, i.e. the shifted image by -s (-t).  The variances and
// covariance are invariant under a common shift of a window's values when the
// window's weights sum to one, which they do once the zero extension is
// counted; the shift only reduces float32 cancellation in E[x'^2] - E[x']^2,
// which is smallest when s is close to the window's own values.  The 2D kernels
// take s and t from one in-image pixel near each 11-row band of an 8-column
// group of windows (the shift is exact for any value, as long as all pixels of
// one window share it); the 3D kernels use the constant kShift.
constexpr float kShift = 0.5f;

// ------------------------------------------------------------ cp.async helpers

__device__ __forceinline__ void cp_async4(void *smem, const void *gmem, bool in_bounds)
{
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    const int src_bytes = in_bounds ? 4 : 0;  // 0: write zeros, read nothing
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(s), "l"(gmem),
                 "r"(src_bytes)
                 : "memory");
}

// 16-byte copy (global and shared addresses 16-byte aligned), L2 only.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool in_bounds)
{
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    const int src_bytes = in_bounds ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem),
                 "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int Pending>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;\n" ::"n"(Pending) : "memory");
}

// ------------------------------------------------- TMA and mbarrier helpers

// Shared-memory address of a generic pointer into shared memory.
__device__ __forceinline__ unsigned smem_u32(const void *p)
{
    return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Makes initialised barriers visible to the tensor-copy unit.
__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// One arrival that also announces `bytes` of incoming copies.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, unsigned bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity)
{
    unsigned done;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for the phase of `bar` with the given parity to complete, for at most
// `max_cycles` SM clocks; false if it did not.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, unsigned parity,
                                                  long long max_cycles)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > max_cycles) return false;
    return true;
}

// Tiled tensor copy global -> shared of the box at (x, y, z); completion is
// signalled on `bar` as transferred bytes.  `map` is a tensor map in parameter,
// constant or global memory; `dst` is 128-byte aligned.
__device__ __forceinline__ void tma_load_3d(void *dst, const void *map, int x, int y, int z,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// The same for a 4D box at (x, y, z, w).
__device__ __forceinline__ void tma_load_4d(void *dst, const void *map, int x, int y, int z, int w,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];\n" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
        : "memory");
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start before the kernel ahead of it on the stream has
// finished, once every block of that kernel has called pdl_trigger (or
// exited); it must call pdl_wait before touching that kernel's results.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Approximate reciprocal (the hardware instruction, relative error ~1 ulp).
// Its argument here is a product of two sums each >= C1 or C2, never zero,
// infinite or subnormal.
__device__ __forceinline__ float rcp_approx(float x)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// ------------------------------------------------------------ SSIM at a pixel

// Statistics of one window in shifted form: m1 = E[x'], m2 = E[y'],
// es = E[x'^2] + E[y'^2], ed = E[(x' - y')^2], with x' = x - s, y' = y - t for
// the window's shift sh = (s, t).  The fourth statistic is the blurred squared
// difference rather than E[x'y'] (which is (es - ed) / 2): SSIM's
// contrast-structure term is
//   cs = (2 sigma12 + C2) / (sigma_sum + C2) = 1 - D / (sigma_sum + C2),
//   D = sigma_sum - 2 sigma12 = ed - (m1 - m2)^2,
// and D, taken from ed, carries no rounding of the images' common level: where
// the two images agree it is near zero whatever the shift, while es - 2 E[x'y']
// would cancel two terms of the size of the shifted values squared.
struct Moments {
    float m1, m2, es, ed;
};

// Upstream gradients of S for the backward.  g_es and g_ed are the derivatives
// with respect to the shifted moments es and ed (because sigma11 and sigma22
// enter S only as their sum, dS/dE[x'^2] and dS/dE[y'^2] are one value, g_es).
// g_f1 and g_f2 are the first-moment maps of the chain rule with the window's
// shift (s, t) folded in, so that every pixel takes the same form
//   grad1 = B^T g_f1 + 2 (x - 1/2) B^T g_es + 2 (x - y) B^T g_ed:
//   g_f1 = dS/dm1 + 2 (1/2 - s) g_es - 2 (s - t) g_ed
//        = 2 cs (mu2 - mu1 l) / B1 + (1 - 2 mu1) g_es - 2 (mu1 - mu2) g_ed
// (the shift cancels; g_f2 likewise with the images swapped).  In a flat
// window g_ed is of order 1 / C2 and g_es small; g_ed meets only differences
// of the two images.
struct MomentGrads {
    float g_f1, g_f2, g_es, g_ed;
};

// S = l * cs with
//   mu = m + sh, sigma_sum = es - m1^2 - m2^2, D = ed - (m1 - m2)^2,
//   l = A1 / B1, A1 = 2 mu1 mu2 + C1, B1 = mu1^2 + mu2^2 + C1,
//   cs = 1 - D / B2, B2 = sigma_sum + C2,
// each product fused into the sum that uses it (one rounding per term).
struct SsimTerms {
    float mu1, mu2, A1, B1, B2, D;
};

__device__ __forceinline__ SsimTerms ssim_terms(const Moments &m, float2 sh)
{
    SsimTerms t;
    t.mu1 = m.m1 + sh.x;
    t.mu2 = m.m2 + sh.y;
    t.B1 = fmaf(t.mu1, t.mu1, fmaf(t.mu2, t.mu2, kC1));
    t.B2 = fmaf(-m.m1, m.m1, fmaf(-m.m2, m.m2, m.es + kC2));
    t.A1 = fmaf(t.mu1 + t.mu1, t.mu2, kC1);
    const float dm = m.m1 - m.m2;
    t.D = fmaf(-dm, dm, m.ed);
    return t;
}

// The two factors of S: (l, cs).
__device__ __forceinline__ float2 ssim_factors(const Moments &m, float2 sh)
{
    const SsimTerms t = ssim_terms(m, sh);
    return make_float2(t.A1 * rcp_approx(t.B1), fmaf(-t.D, rcp_approx(t.B2), 1.0f));
}

// S = A1 (B2 - D) / (B1 B2): one reciprocal.  B2 - D is the numerator of cs,
// so B2's rounding still reaches S only through D / B2.
__device__ __forceinline__ float ssim_value(const Moments &m, float2 sh)
{
    const SsimTerms t = ssim_terms(m, sh);
    return (t.A1 * (t.B2 - t.D)) * rcp_approx(t.B1 * t.B2);
}

// S and its derivatives:
//   dS/des = l D / B2^2,   dS/ded = -l / B2,
//   dS/dmu1 (sigma_sum and D fixed) = 2 cs (mu2 - mu1 l) / B1,
// and through sigma_sum = es - m1^2 - m2^2, D = ed - (m1 - m2)^2:
//   dS/dm1 = 2 cs (mu2 - mu1 l) / B1 - 2 m1 dS/des - 2 (m1 - m2) dS/ded,
// which with the fold of MomentGrads gives g_f1 (g_f2 likewise).
// When `valid` is false every derivative (and S) comes out as exactly zero:
// l is zeroed before it is used.
template <bool WANT_G2>
__device__ __forceinline__ float ssim_and_grads(const Moments &m, float2 sh, bool valid,
                                                MomentGrads &g)
{
    const SsimTerms t = ssim_terms(m, sh);
    const float r1 = rcp_approx(t.B1), r2 = rcp_approx(t.B2);
    const float l = valid ? t.A1 * r1 : 0.0f;
    const float Dr2 = t.D * r2;
    const float cs = 1.0f - Dr2;
    const float S = l * cs;
    const float lr2 = l * r2;
    g.g_ed = -lr2;
    g.g_es = lr2 * Dr2;
    const float cr1x2 = valid ? cs * (r1 + r1) : 0.0f;
    const float du2 = 2.0f * (t.mu1 - t.mu2);
    g.g_f1 = fmaf(cr1x2, fmaf(-t.mu1, l, t.mu2), fmaf(fmaf(-2.0f, t.mu1, 1.0f), g.g_es, -du2 * g.g_ed));
    if (WANT_G2)
        g.g_f2 = fmaf(cr1x2, fmaf(-t.mu2, l, t.mu1), fmaf(fmaf(-2.0f, t.mu2, 1.0f), g.g_es, du2 * g.g_ed));
    return S;
}

// ------------------------------------------------------------ block reduction

// Sum of one float per thread over a block of NT threads (NT a multiple of 32),
// in double; returns the total in thread 0.  Fixed order: deterministic.
template <int NT>
__device__ __forceinline__ double block_sum(float v, double *scratch /* NT/32 doubles */)
{
    double d = static_cast<double>(v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d += __shfl_down_sync(0xffffffffu, d, o);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) scratch[warp] = d;
    __syncthreads();
    double t = 0.0;
    if (threadIdx.x == 0) {
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) t += scratch[w];
    }
    return t;
}

// Last-block ticket of a grid-wide finish: every block calls this once, after
// its partial sums are written; true (in every thread) in the block that
// arrives last, whose view of all partials is then complete.
template <int NT>
__device__ __forceinline__ bool finish_ticket(unsigned *counter)
{
    __shared__ bool last;
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned ticket = atomicAdd(counter, 1u);
        last = (ticket == gridDim.x - 1);
    }
    __syncthreads();
    if (last) __threadfence();
    return last;
}

// Per-image means from block partial sums: for every quantity k < K and image
// n, the blocks_per_image consecutive partials at partials[k * stride +
// n * blocks_per_image ...] -- one warp per (k, n), its lanes striding the
// partials, then a fixed shuffle tree: a fixed order, so the result is
// deterministic -- give mean[k * images + n] = sum / count.  The (k, n)
// reductions run in parallel: each costs one round of L2 loads.
template <int NT, int K>
__device__ __forceinline__ void reduce_means_k(const double *partials, int stride, float *mean,
                                               int images, int blocks_per_image, double count)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int q = warp; q < K * images; q += NT / 32) {
        const int k = q / images, n = q - k * images;
        const double *p = partials + size_t(k) * stride + size_t(n) * blocks_per_image;
        double s = 0.0;
        for (int b = lane; b < blocks_per_image; b += 32) s += __ldcg(p + b);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xffffffffu, s, o);
        if (lane == 0) mean[k * images + n] = static_cast<float>(s / count);
    }
}

// Grid-wide finish of per-image means: the last block to arrive reduces them
// (reduce_means_k) and resets the counter to zero for the next call.
template <int NT, int K>
__device__ __forceinline__ void finish_means_k(double *partials, int stride, unsigned *counter,
                                               float *mean, int images, int blocks_per_image,
                                               double count)
{
    if (!finish_ticket<NT>(counter)) return;
    reduce_means_k<NT, K>(partials, stride, mean, images, blocks_per_image, count);
    if (threadIdx.x == 0) *counter = 0u;
}

// One quantity: partials[slot], mean[n].
template <int NT>
__device__ __forceinline__ void finish_means(double *partials, unsigned *counter, float *mean,
                                             int images, int blocks_per_image, double count)
{
    finish_means_k<NT, 1>(partials, 0, counter, mean, images, blocks_per_image, count);
}

}  // namespace gbssim
