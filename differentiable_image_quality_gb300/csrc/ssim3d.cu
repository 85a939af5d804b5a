// 3D SSIM (fused-ssim README, "3D data"): the same statistics and adjoint as in
// 2D with an 11x11x11 separable window on NCDHW volumes.
//
// Following that page's plan -- keep the 2D convolution on XY slices, and do
// the Z convolution and SSIM through a ring buffer, one depth row per thread --
// a CTA owns an XY tile of 16 x 32 columns and walks along Z one slice per step:
//   XY  the slice's row pass and column pass in shared memory (cp.async staging
//       of the slice tile plus its 10-pixel halo, three buffers);
//   Z   each thread keeps an 11-slice register ring of its column's XY-blurred
//       values; the ring's weighted sum is the full 3D window.
// Two kernels:
//   stats    statistics -> SSIM (mean, map) and, for gradients, the derivatives
//            of SSIM with respect to the four shifted moments, one float4 per
//            output voxel, into the workspace;
//   adjoint  the same walk over those derivative fields (the blur's adjoint is
//            the blur with the window mirrored, which for a symmetric window is
//            the same correlation with the "full" extent), then the chain rule
//            grad1 = B^T g_mu1 + 2 x B^T g_e + y B^T g_e12 (grad2 likewise).
#include "common.cuh"
#include "ssim3d.cuh"

namespace gbssim {
namespace {

constexpr int NT = kThreads3d;  // 512
constexpr int TY = kTile3dY;    // 16 rows of columns per tile
constexpr int TX = kTile3dX;    // 32 columns per row
constexpr int IY = TY + 10, IX = TX + 10;
constexpr int IXP = IX + 2;     // float pitch of the staged input rows (float4 aligned)
constexpr int KX = 4, NXG = TX / KX, NXI = IY * NXG;  // row-pass items per slice
constexpr int KY = 4, NYG = TY / KY, NYI = NYG * TX;  // column-pass items per slice
constexpr int NBUF = 3;

static_assert(NT == TY * TX, "one thread per column of the tile");

constexpr size_t kStatsInBytes = size_t(2) * NBUF * IY * IXP * sizeof(float);
constexpr size_t kAdjInBytes = size_t(NBUF) * IY * IX * sizeof(float4);
constexpr size_t kXBytes = size_t(2) * IY * TX * sizeof(float4);
constexpr size_t kYBytes = size_t(TY) * TX * sizeof(float4);

__device__ __forceinline__ int swz(int c) { return (c & ~7) | ((c + (c >> 3)) & 7); }

__device__ __forceinline__ float4 wsum_ring(const float4 (&ring)[kTaps], int newest)
{
    // sum_a w_a ring[(newest + 1 + a) % 11]: the oldest slice gets w_0
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int a = 0; a < kTaps; ++a) {
        const float4 h = ring[(newest + 1 + a) % kTaps];
        const float w = tap(a);
        s.x = fmaf(w, h.x, s.x);
        s.y = fmaf(w, h.y, s.y);
        s.z = fmaf(w, h.z, s.z);
        s.w = fmaf(w, h.w, s.w);
    }
    return s;
}

// ------------------------------------------------------------------ kernel A

template <bool GRAD>
__global__ void __launch_bounds__(NT, 1) ssim3d_stats_kernel(const Ssim3dArgs a)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float *xs = reinterpret_cast<float *>(smem_raw);
    float *ys = xs + NBUF * IY * IXP;
    float4 *hx = reinterpret_cast<float4 *>(smem_raw + kStatsInBytes);
    float4 *hy = hx + 2 * IY * TX;
    __shared__ double red[NT / 32];

    const int tid = threadIdx.x;
    int b = blockIdx.x;
    const int tile_x = b % a.tiles_x; b /= a.tiles_x;
    const int tile_y = b % a.tiles_y; b /= a.tiles_y;
    const int zseg = b % a.zsegs;
    const int plane = b / a.zsegs;
    const size_t vol = size_t(a.D) * a.H * a.W;
    const float *__restrict__ xp = a.x + size_t(plane) * vol;
    const float *__restrict__ yp = a.y + size_t(plane) * vol;

    const int y0 = tile_y * TY, x0 = tile_x * TX;       // statistic coordinates
    const int z0 = zseg * a.zseg_len;
    const int z1 = min(z0 + a.zseg_len, a.Do);
    const int iy0 = y0 - a.off, ix0 = x0 - a.off, iz0 = z0 - a.off;
    const int nz = z1 - z0 + 10;                        // input slices walked

    auto load_slice = [&](int s) {
        const int buf = s % NBUF;
        const int Z = iz0 + s;
        const bool zin = (Z >= 0) && (Z < a.D);
        for (int e = tid; e < IY * IX; e += NT) {
            const int r = e / IX, c = e - r * IX;
            const int Y = iy0 + r, X = ix0 + c;
            const bool inb = zin && (Y >= 0) && (Y < a.H) && (X >= 0) && (X < a.W);
            const size_t gi = inb ? (size_t(Z) * a.H + Y) * a.W + X : 0;
            const int si = (buf * IY + r) * IXP + c;
            cp_async4(xs + si, xp + gi, inb);
            cp_async4(ys + si, yp + gi, inb);
        }
    };

    // row pass of slice s: row r of the staged tile, columns [KX g, KX g + KX)
    auto x_item = [&](int s, int item) {
        const int r = item / NXG, g = item - r * NXG;
        const int base = ((s % NBUF) * IY + r) * IXP + g * KX;
        float xv[KX + 10], yv[KX + 10];
#pragma unroll
        for (int m = 0; m < KX + 8; m += 4) {
            const float4 u = *reinterpret_cast<const float4 *>(xs + base + m);
            const float4 v = *reinterpret_cast<const float4 *>(ys + base + m);
            xv[m] = u.x; xv[m + 1] = u.y; xv[m + 2] = u.z; xv[m + 3] = u.w;
            yv[m] = v.x; yv[m + 1] = v.y; yv[m + 2] = v.z; yv[m + 3] = v.w;
        }
        {
            const float2 u = *reinterpret_cast<const float2 *>(xs + base + KX + 8);
            const float2 v = *reinterpret_cast<const float2 *>(ys + base + KX + 8);
            xv[KX + 8] = u.x; xv[KX + 9] = u.y;
            yv[KX + 8] = v.x; yv[KX + 9] = v.y;
        }
        float acc[KX][4];
#pragma unroll
        for (int m = 0; m < KX + 10; ++m) {
            const float xx = xv[m] - kShift, yy = yv[m] - kShift;
            const float pe = fmaf(xx, xx, yy * yy);
            const float pc = xx * yy;
#pragma unroll
            for (int o = 0; o < KX; ++o) {
                const int t = m - o;
                if (t < 0 || t > 10) continue;
                const float w = tap(t);
                if (t == 0) {
                    acc[o][0] = w * xx; acc[o][1] = w * yy; acc[o][2] = w * pe; acc[o][3] = w * pc;
                } else {
                    acc[o][0] = fmaf(w, xx, acc[o][0]);
                    acc[o][1] = fmaf(w, yy, acc[o][1]);
                    acc[o][2] = fmaf(w, pe, acc[o][2]);
                    acc[o][3] = fmaf(w, pc, acc[o][3]);
                }
            }
        }
        float4 *dst = hx + (s & 1) * IY * TX + r * TX;
#pragma unroll
        for (int o = 0; o < KX; ++o)
            dst[swz(g * KX + o)] = make_float4(acc[o][0], acc[o][1], acc[o][2], acc[o][3]);
    };

    // column pass of slice s: column tx, rows [KY g, KY g + KY)
    auto y_item = [&](int s, int item) {
        const int g = item / TX, tx = item - g * TX;
        const float4 *src = hx + (s & 1) * IY * TX;
        float4 acc[KY];
#pragma unroll
        for (int m = 0; m < KY + 10; ++m) {
            const float4 v = src[(g * KY + m) * TX + swz(tx)];
#pragma unroll
            for (int o = 0; o < KY; ++o) {
                const int t = m - o;
                if (t < 0 || t > 10) continue;
                const float w = tap(t);
                if (t == 0) {
                    acc[o] = make_float4(w * v.x, w * v.y, w * v.z, w * v.w);
                } else {
                    acc[o].x = fmaf(w, v.x, acc[o].x);
                    acc[o].y = fmaf(w, v.y, acc[o].y);
                    acc[o].z = fmaf(w, v.z, acc[o].z);
                    acc[o].w = fmaf(w, v.w, acc[o].w);
                }
            }
        }
#pragma unroll
        for (int o = 0; o < KY; ++o) hy[(g * KY + o) * TX + tx] = acc[o];
    };

    const int ty = tid / TX, tx = tid - ty * TX;
    const int py = y0 + ty, px = x0 + tx;
    const bool col_ok = (py < a.Ho) && (px < a.Wo);
    float4 ring[kTaps];
#pragma unroll
    for (int k = 0; k < kTaps; ++k) ring[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    float ssum = 0.0f;

    // Z step: push this column's XY-blurred value of slice s, finish slice s - 10.
    auto z_step = [&](auto K_, int s) {
        constexpr int K = decltype(K_)::value;
        ring[K] = hy[ty * TX + tx];
        const int p = z0 + s - 10;
        if (s >= 10 && p < z1 && col_ok) {
            const float4 h = wsum_ring(ring, K);
            const Moments mo{h.x, h.y, h.z, h.w};
            float S;
            if (GRAD) {
                MomentGrads gg;
                S = ssim_and_grads<true>(mo, true, gg);
                const size_t oi = ((size_t(plane) * a.Do + p) * a.Ho + py) * a.Wo + px;
                reinterpret_cast<float4 *>(a.gfield)[oi] = make_float4(gg.g_m1, gg.g_e, gg.g_e12, gg.g_m2);
            } else {
                S = ssim_value(mo);
            }
            ssum += S;
            if (a.map) a.map[((size_t(plane) * a.Do + p) * a.Ho + py) * a.Wo + px] = S;
        }
    };

    load_slice(0);
    cp_async_commit();
    if (nz > 1) load_slice(1);
    cp_async_commit();
    if (nz > 2) load_slice(2);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    for (int i = tid; i < NXI; i += NT) x_item(0, i);
    __syncthreads();

    for (int s = 0; s < nz; ++s) {
        const int nx = (s + 1 < nz) ? NXI : 0;
        for (int i = tid; i < NYI + nx; i += NT) {
            if (i < NYI)
                y_item(s, i);
            else
                x_item(s + 1, i - NYI);
        }
        __syncthreads();
        if (s + 3 < nz) load_slice(s + 3);  // into the buffer x_item(s) released
        cp_async_commit();
        switch (s % kTaps) {
        case 0: z_step(std::integral_constant<int, 0>{}, s); break;
        case 1: z_step(std::integral_constant<int, 1>{}, s); break;
        case 2: z_step(std::integral_constant<int, 2>{}, s); break;
        case 3: z_step(std::integral_constant<int, 3>{}, s); break;
        case 4: z_step(std::integral_constant<int, 4>{}, s); break;
        case 5: z_step(std::integral_constant<int, 5>{}, s); break;
        case 6: z_step(std::integral_constant<int, 6>{}, s); break;
        case 7: z_step(std::integral_constant<int, 7>{}, s); break;
        case 8: z_step(std::integral_constant<int, 8>{}, s); break;
        case 9: z_step(std::integral_constant<int, 9>{}, s); break;
        default: z_step(std::integral_constant<int, 10>{}, s); break;
        }
        cp_async_wait<1>();  // slice s + 2 has landed
        __syncthreads();
    }
    cp_async_wait<0>();

    if (a.partials) {
        const double tot = block_sum<NT>(ssum, red);
        if (tid == 0) a.partials[blockIdx.x] = tot;
        finish_means<NT>(a.partials, a.counter, a.mean, a.images, a.blocks_per_image, a.count);
    }
}

// ------------------------------------------------------------------ kernel B

template <bool G2>
__global__ void __launch_bounds__(NT, 1) ssim3d_adjoint_kernel(const Ssim3dArgs a)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float4 *gs = reinterpret_cast<float4 *>(smem_raw);                   // [NBUF][IY][IX]
    float4 *ux = reinterpret_cast<float4 *>(smem_raw + kAdjInBytes);     // [2][IY][TX]
    float4 *uy = ux + 2 * IY * TX;                                        // [TY][TX]

    const int tid = threadIdx.x;
    int b = blockIdx.x;
    const int tile_x = b % a.tiles_x; b /= a.tiles_x;
    const int tile_y = b % a.tiles_y; b /= a.tiles_y;
    const int zseg = b % a.zsegs;
    const int plane = b / a.zsegs;
    const int n = plane / a.C;
    const size_t vol = size_t(a.D) * a.H * a.W;
    const size_t plane_off = size_t(plane) * vol;
    const float4 *__restrict__ gf = reinterpret_cast<const float4 *>(a.gfield) +
                                    size_t(plane) * a.Do * a.Ho * a.Wo;

    const int y0 = tile_y * TY, x0 = tile_x * TX;  // gradient (image) coordinates
    const int q0 = zseg * a.zseg_len;
    const int q1 = min(q0 + a.zseg_len, a.D);
    // derivative positions feeding gradient q: q + off - 10 .. q + off per axis
    const int gy0 = y0 + a.off - 10, gx0 = x0 + a.off - 10, gz0 = q0 + a.off - 10;
    const int nz = q1 - q0 + 10;
    const float scale = a.dL ? a.dL[n] * a.inv_count : a.inv_count;

    auto load_slice = [&](int s) {
        const int buf = s % NBUF;
        const int P = gz0 + s;
        const bool zin = (P >= 0) && (P < a.Do);
        for (int e = tid; e < IY * IX; e += NT) {
            const int r = e / IX, c = e - r * IX;
            const int Y = gy0 + r, X = gx0 + c;
            const bool inb = zin && (Y >= 0) && (Y < a.Ho) && (X >= 0) && (X < a.Wo);
            const size_t gi = inb ? (size_t(P) * a.Ho + Y) * a.Wo + X : 0;
            cp_async16(gs + (buf * IY + r) * IX + c, gf + gi, inb);
        }
    };

    // adjoint row pass: gradient columns [KX g, KX g + KX) of staged row r
    auto x_item = [&](int s, int item) {
        const int r = item / NXG, g = item - r * NXG;
        const float4 *src = gs + ((s % NBUF) * IY + r) * IX + g * KX;
        float4 acc[KX];
#pragma unroll
        for (int m = 0; m < KX + 10; ++m) {
            const float4 v = src[m];
#pragma unroll
            for (int o = 0; o < KX; ++o) {
                const int t = m - o;
                if (t < 0 || t > 10) continue;
                const float w = tap(t);
                if (t == 0) {
                    acc[o] = make_float4(w * v.x, w * v.y, w * v.z, G2 ? w * v.w : 0.f);
                } else {
                    acc[o].x = fmaf(w, v.x, acc[o].x);
                    acc[o].y = fmaf(w, v.y, acc[o].y);
                    acc[o].z = fmaf(w, v.z, acc[o].z);
                    if (G2) acc[o].w = fmaf(w, v.w, acc[o].w);
                }
            }
        }
        float4 *dst = ux + (s & 1) * IY * TX + r * TX;
#pragma unroll
        for (int o = 0; o < KX; ++o) dst[swz(g * KX + o)] = acc[o];
    };

    auto y_item = [&](int s, int item) {
        const int g = item / TX, tx = item - g * TX;
        const float4 *src = ux + (s & 1) * IY * TX;
        float4 acc[KY];
#pragma unroll
        for (int m = 0; m < KY + 10; ++m) {
            const float4 v = src[(g * KY + m) * TX + swz(tx)];
#pragma unroll
            for (int o = 0; o < KY; ++o) {
                const int t = m - o;
                if (t < 0 || t > 10) continue;
                const float w = tap(t);
                if (t == 0) {
                    acc[o] = make_float4(w * v.x, w * v.y, w * v.z, G2 ? w * v.w : 0.f);
                } else {
                    acc[o].x = fmaf(w, v.x, acc[o].x);
                    acc[o].y = fmaf(w, v.y, acc[o].y);
                    acc[o].z = fmaf(w, v.z, acc[o].z);
                    if (G2) acc[o].w = fmaf(w, v.w, acc[o].w);
                }
            }
        }
#pragma unroll
        for (int o = 0; o < KY; ++o) uy[(g * KY + o) * TX + tx] = acc[o];
    };

    const int ty = tid / TX, tx = tid - ty * TX;
    const int qy = y0 + ty, qx = x0 + tx;
    const bool col_ok = (qy < a.H) && (qx < a.W);
    float4 ring[kTaps];
#pragma unroll
    for (int k = 0; k < kTaps; ++k) ring[k] = make_float4(0.f, 0.f, 0.f, 0.f);

    auto z_step = [&](auto K_, int s) {
        constexpr int K = decltype(K_)::value;
        ring[K] = uy[ty * TX + tx];
        const int q = q0 + s - 10;
        if (s >= 10 && q < q1 && col_ok) {
            const size_t gi = plane_off + (size_t(q) * a.H + qy) * a.W + qx;
            const float x = __ldg(a.x + gi) - kShift, y = __ldg(a.y + gi) - kShift;
            const float4 v = wsum_ring(ring, K);  // (B^T g_m1, B^T g_e, B^T g_e12, B^T g_m2)
            a.out1[gi] = scale * fmaf(2.0f * x, v.y, fmaf(y, v.z, v.x));
            if (G2) a.out2[gi] = scale * fmaf(2.0f * y, v.y, fmaf(x, v.z, v.w));
        }
    };

    load_slice(0);
    cp_async_commit();
    if (nz > 1) load_slice(1);
    cp_async_commit();
    if (nz > 2) load_slice(2);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    for (int i = tid; i < NXI; i += NT) x_item(0, i);
    __syncthreads();

    for (int s = 0; s < nz; ++s) {
        const int nx = (s + 1 < nz) ? NXI : 0;
        for (int i = tid; i < NYI + nx; i += NT) {
            if (i < NYI)
                y_item(s, i);
            else
                x_item(s + 1, i - NYI);
        }
        __syncthreads();
        if (s + 3 < nz) load_slice(s + 3);
        cp_async_commit();
        switch (s % kTaps) {
        case 0: z_step(std::integral_constant<int, 0>{}, s); break;
        case 1: z_step(std::integral_constant<int, 1>{}, s); break;
        case 2: z_step(std::integral_constant<int, 2>{}, s); break;
        case 3: z_step(std::integral_constant<int, 3>{}, s); break;
        case 4: z_step(std::integral_constant<int, 4>{}, s); break;
        case 5: z_step(std::integral_constant<int, 5>{}, s); break;
        case 6: z_step(std::integral_constant<int, 6>{}, s); break;
        case 7: z_step(std::integral_constant<int, 7>{}, s); break;
        case 8: z_step(std::integral_constant<int, 8>{}, s); break;
        case 9: z_step(std::integral_constant<int, 9>{}, s); break;
        default: z_step(std::integral_constant<int, 10>{}, s); break;
        }
        cp_async_wait<1>();
        __syncthreads();
    }
    cp_async_wait<0>();
}

template <typename K>
cudaError_t prepare(K kernel, size_t smem, int *occ)
{
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, kernel, NT, smem);
}

}  // namespace

size_t ssim3d_stats_smem() { return kStatsInBytes + kXBytes + kYBytes; }
size_t ssim3d_adjoint_smem() { return kAdjInBytes + kXBytes + kYBytes; }

cudaError_t ssim3d_prepare(int occ[2])
{
    int o[4] = {0, 0, 0, 0};
    cudaError_t e;
    if ((e = prepare(ssim3d_stats_kernel<false>, ssim3d_stats_smem(), &o[0])) != cudaSuccess) return e;
    if ((e = prepare(ssim3d_stats_kernel<true>, ssim3d_stats_smem(), &o[1])) != cudaSuccess) return e;
    if ((e = prepare(ssim3d_adjoint_kernel<false>, ssim3d_adjoint_smem(), &o[2])) != cudaSuccess) return e;
    if ((e = prepare(ssim3d_adjoint_kernel<true>, ssim3d_adjoint_smem(), &o[3])) != cudaSuccess) return e;
    occ[0] = o[0] < o[1] ? o[0] : o[1];
    occ[1] = o[2] < o[3] ? o[2] : o[3];
    return (occ[0] < 1 || occ[1] < 1) ? cudaErrorInvalidConfiguration : cudaSuccess;
}

cudaError_t ssim3d_stats_launch(const Ssim3dArgs &a, bool grad, int blocks, cudaStream_t s)
{
    if (grad)
        ssim3d_stats_kernel<true><<<blocks, NT, ssim3d_stats_smem(), s>>>(a);
    else
        ssim3d_stats_kernel<false><<<blocks, NT, ssim3d_stats_smem(), s>>>(a);
    return cudaGetLastError();
}

cudaError_t ssim3d_adjoint_launch(const Ssim3dArgs &a, bool g2, int blocks, cudaStream_t s)
{
    if (g2)
        ssim3d_adjoint_kernel<true><<<blocks, NT, ssim3d_adjoint_smem(), s>>>(a);
    else
        ssim3d_adjoint_kernel<false><<<blocks, NT, ssim3d_adjoint_smem(), s>>>(a);
    return cudaGetLastError();
}

}  // namespace gbssim
