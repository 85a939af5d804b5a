// 3D SSIM (fused-ssim README, "3D data"): the same statistics and adjoint as in
// 2D with an 11x11x11 separable window on NCDHW volumes.
//
// Three passes whose intermediates stay in L2 (at 128^3 the two volumes, the
// statistics field and the derivative field together take well under its
// 129 MB), so that each axis's halo is computed once:
//   xy   per slice, the row pass and column pass of the four shifted statistics
//        on an XY tile plus its 10-pixel halo in shared memory -> tfield, one
//        float4 per (slice, output column); the slice tiles are staged by
//        tensor copies (one thread issues them, a transaction barrier per
//        buffer tracks them, every wait bounded) or by cp.async where the tile
//        does not start on a 16-byte column, into three buffers, each refilled
//        two steps before its row pass;
//   z    one thread per output column walks along Z: the Z window sums as a
//        shift register of pending sums, SSIM (mean, map) and, for gradients,
//        the derivatives of SSIM with respect to the four shifted moments,
//        whose Z adjoint (the same correlation with the "full" extent, the
//        window being symmetric) runs as a second shift register -> ufield;
//   adj  per slice, the XY adjoint of those four fields on a tile plus halo
//        in shared memory, then the chain rule
//        grad1 = B^T g_mu1 + 2 x' B^T g_e + y' B^T g_e12 (grad2 likewise), taken
//        with the derivatives with respect to es = E[x'^2] + E[y'^2] and
//        ed = E[(x - y)^2]: B^T g_mu1 + 2 x' B^T g_es + 2 (x - y) B^T g_ed.
// The page's own plan keeps the 2D convolution per slice and runs Z per depth
// row in one kernel; walking Z inside the slice kernels re-runs the XY work of
// each Z segment's 10-slice warm-up, which these passes avoid.
// All window sums run on float pairs (fma.rn.f32x2): (mu1, mu2), (es, ed) for
// the statistics, (g_mu1, g_es), (g_ed, g_mu2) for the adjoint.  Work items of
// the row passes are numbered row-fastest over odd shared-memory pitches, so
// the threads of a quarter warp hit distinct bank groups.
#include "common.cuh"
#include "ssim2d.cuh"
#include "ssim3d.cuh"

namespace gbssim {
namespace {

// Tile geometry of a slice kernel: TY x TX columns, one thread per column; a
// row-pass item covers KX columns of one row, a column-pass item KY rows of
// one column (wider items load fewer shared values per output).  The xy kernel
// runs 16 x 8 tiles (128 threads) with 4 x 4 items, the adjoint kernel 16 x 16
// tiles (256 threads) with row items of 8 columns and column items of 4 rows.
template <int TX_, int KY_, int KX_>
struct Geo {
    static constexpr int TY = kTile3dY, TX = TX_, NT = TY * TX;
    static constexpr int IY = TY + 10, IX = TX + 10;  // staged slice tile
    // float pitch of a staged input row: a multiple of 16 bytes, an odd number of
    // 16-byte units (28 for 16 columns, 20 for 8)
    static constexpr int IXU = (IX + 3) / 4, IXP = 4 * (IXU % 2 ? IXU : IXU + 1);
    static constexpr int GXP = IX + 1;  // float4 pitch of a staged derivative row (odd)
    static constexpr int HXP = TX + 1;  // float4 pitch of a row-pass output row
    static constexpr int KX = KX_, NXG = TX / KX, NXI = IY * NXG;  // row-pass items per slice
    static constexpr int KY = KY_, NYG = TY / KY, NYI = NYG * TX;  // column-pass items per slice
    // staging buffers, each a multiple of 128 bytes (tensor-copy destinations)
    static constexpr int XSTAGE = (IY * IXP + 31) / 32 * 32;  // floats of a staged input tile
    static constexpr int GSTAGE = (IY * GXP + 7) / 8 * 8;     // float4 of a staged derivative tile
    static constexpr int CSTAGE = TY * TX;                     // floats of a chain-rule pixel tile
    static_assert(TX % KX == 0 && TY % KY == 0, "items tile the columns");
    static_assert(NYI % 32 == 0, "column-pass items fill whole warps");
    static_assert(IXP % 4 == 0 && IXP >= IX, "input pitch");
    static_assert((CSTAGE * 4) % 128 == 0, "chain tiles stay 128-byte aligned");
};
using GS = Geo<kXy3dX, 4, 4>;   // xy kernel
using GA = Geo<kAdj3dX, 4, 8>;  // adjoint kernel

constexpr int NBUF = 3;            // xy kernel: staged slices
constexpr int NBUF_A = 3;          // adjoint kernel: staged derivative slices
constexpr int CBUF_A = NBUF_A + 2; // adjoint kernel: chain-rule pixel tiles in flight
constexpr unsigned kStatsTx = 2u * GS::IY * GS::IXP * sizeof(float);
constexpr unsigned kAdjTx =
    unsigned(GA::IY * GA::GXP * sizeof(float4) + 2 * GA::CSTAGE * sizeof(float));
constexpr long long kWaitCycles = 1LL << 31;   // staging wait limit (about a second)
constexpr long long kDrainCycles = 1LL << 27;  // after a failed wait: copies still in flight
constexpr int kZPrefetch = 8;                  // z kernel: slices loaded ahead

__device__ unsigned g_staging3d_status;  // bit 0: a staging wait ran out of time

constexpr size_t kStatsInBytes = size_t(2) * NBUF * GS::XSTAGE * sizeof(float);
constexpr size_t kStatsXBytes = size_t(2) * GS::IY * GS::HXP * sizeof(float4);
constexpr size_t kStatsYBytes = size_t(2) * GS::TY * GS::TX * sizeof(float4);  // two slices
constexpr size_t kAdjInBytes = size_t(NBUF_A) * GA::GSTAGE * sizeof(float4);
constexpr size_t kChainBytes = size_t(2) * CBUF_A * GA::CSTAGE * sizeof(float);
constexpr size_t kAdjXBytes = size_t(2) * GA::IY * GA::HXP * sizeof(float4);
constexpr size_t kAdjYBytes = size_t(2) * GA::TY * GA::TX * sizeof(float4);

size_t xy_smem() { return 128 + kStatsInBytes + kStatsXBytes + kStatsYBytes; }
size_t adjoint_smem() { return 128 + kAdjInBytes + kChainBytes + kAdjXBytes + kAdjYBytes; }

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }
__device__ __forceinline__ float2 splat(float w) { return make_float2(w, w); }
__device__ __forceinline__ float2 lo(const float4 &v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi(const float4 &v) { return make_float2(v.z, v.w); }

// 11-tap pass over float4 values loaded from smem at src[stride * m],
// m = 0 .. K + 9, giving K outputs (two float pairs each).
template <int K>
__device__ __forceinline__ void taps4(const float4 *src, int stride, float2 (&oa)[K], float2 (&ob)[K])
{
#pragma unroll
    for (int m = 0; m < K + 10; ++m) {
        const float4 v = src[m * stride];
#pragma unroll
        for (int o = 0; o < K; ++o) {
            const int t = m - o;
            if (t < 0 || t > 10) continue;
            const float2 w = splat(tap(t));
            oa[o] = (t == 0) ? __fmul2_rn(w, lo(v)) : __ffma2_rn(w, lo(v), oa[o]);
            ob[o] = (t == 0) ? __fmul2_rn(w, hi(v)) : __ffma2_rn(w, hi(v), ob[o]);
        }
    }
}

// The same pass over the first three components only (x, y as a pair, z
// alone): the adjoint for grad_img1 needs B^T of g_mu1, g_es and g_ed, not g_mu2.
template <int K>
__device__ __forceinline__ void taps3(const float4 *src, int stride, float2 (&oa)[K], float (&oc)[K])
{
#pragma unroll
    for (int m = 0; m < K + 10; ++m) {
        const float4 v = src[m * stride];
#pragma unroll
        for (int o = 0; o < K; ++o) {
            const int t = m - o;
            if (t < 0 || t > 10) continue;
            oa[o] = (t == 0) ? __fmul2_rn(splat(tap(t)), lo(v)) : __ffma2_rn(splat(tap(t)), lo(v), oa[o]);
            oc[o] = (t == 0) ? tap(t) * v.z : fmaf(tap(t), v.z, oc[o]);
        }
    }
}

// A Z pass as a shift register of pending window sums.  P[j] holds, after
// slice s, the part of the window that completes at slice s + j + 1 contributed
// by slices <= s.  Slice s with value h completes the window of P[0] (h is its
// newest slice, weight w_10) and shifts the rest:
//   out = P[0] + w_10 h,  P[j] = P[j + 1] + w_{9-j} h (j < 9),  P[9] = w_0 h.
// Every register index is fixed, so no step dispatches on s % 11, and the 11
// updates are independent.
__device__ __forceinline__ float2 zshift2(float2 (&P)[kTaps - 1], float2 h)
{
    const float2 out = __ffma2_rn(splat(tap(10)), h, P[0]);
#pragma unroll
    for (int j = 0; j < kTaps - 2; ++j) P[j] = __ffma2_rn(splat(tap(9 - j)), h, P[j + 1]);
    P[kTaps - 2] = __fmul2_rn(splat(tap(0)), h);
    return out;
}

__device__ __forceinline__ float zshift1(float (&P)[kTaps - 1], float h)
{
    const float out = fmaf(tap(10), h, P[0]);
#pragma unroll
    for (int j = 0; j < kTaps - 2; ++j) P[j] = fmaf(tap(9 - j), h, P[j + 1]);
    P[kTaps - 2] = tap(0) * h;
    return out;
}

// The same register fed a zero (a slice past the end of the domain).
__device__ __forceinline__ float2 zshift2_zero(float2 (&P)[kTaps - 1])
{
    const float2 out = P[0];
#pragma unroll
    for (int j = 0; j < kTaps - 2; ++j) P[j] = P[j + 1];
    P[kTaps - 2] = f2(0.f, 0.f);
    return out;
}

__device__ __forceinline__ float zshift1_zero(float (&P)[kTaps - 1])
{
    const float out = P[0];
#pragma unroll
    for (int j = 0; j < kTaps - 2; ++j) P[j] = P[j + 1];
    P[kTaps - 2] = 0.f;
    return out;
}

// Slices j < waited have been waited for, j < issued copied (slice j on barrier
// j % NB): after a failed wait, let the copies still in flight land (bounded),
// then record the failure.
template <int NB>
__device__ __forceinline__ void drain_failed(uint64_t *bars, int waited, int issued)
{
    const long long t0 = clock64();
    for (int j = waited; j < issued; ++j) {
        const long long left = kDrainCycles - (clock64() - t0);
        if (left > 0) mbar_wait_bounded(&bars[j % NB], (j / NB) & 1, left);
    }
    atomicOr(&g_staging3d_status, 1u);
}

__device__ __forceinline__ float4 nan4()
{
    const float q = __int_as_float(0x7fc00000);
    return make_float4(q, q, q, q);
}

// ------------------------------------------------------------------ xy kernel

__global__ void __launch_bounds__(GS::NT, 4) ssim3d_xy_kernel(const __grid_constant__ Ssim3dArgs a)
{
    constexpr int NT = GS::NT, TY = GS::TY, TX = GS::TX, IY = GS::IY, IX = GS::IX,
                  IXP = GS::IXP, HXP = GS::HXP, KX = GS::KX, NXI = GS::NXI, KY = GS::KY,
                  NYI = GS::NYI, XSTAGE = GS::XSTAGE;
    extern __shared__ __align__(128) unsigned char smem_dyn[];
    unsigned char *smem_raw = smem_dyn + ((128 - (smem_u32(smem_dyn) & 127)) & 127);
    float *xs = reinterpret_cast<float *>(smem_raw);
    float *ys = xs + NBUF * XSTAGE;
    float4 *hx = reinterpret_cast<float4 *>(smem_raw + kStatsInBytes);
    float4 *hy = hx + 2 * IY * HXP;  // kStatsXBytes after hx
    __shared__ uint64_t bars[NBUF];
    pdl_trigger();

    const int tid = threadIdx.x;
    int b = blockIdx.x;
    const int tile_x = b % a.tiles_x; b /= a.tiles_x;
    const int tile_y = b % a.tiles_y; b /= a.tiles_y;
    const int zseg = b % a.zsegs;
    const int plane = b / a.zsegs;
    const size_t vol = size_t(a.D) * a.H * a.W;
    const float *__restrict__ xp = a.x + size_t(plane) * vol;
    const float *__restrict__ yp = a.y + size_t(plane) * vol;

    const int y0 = tile_y * TY, x0 = tile_x * TX;  // output-domain coordinates
    const int z0 = zseg * a.zseg_len;
    const int z1 = min(z0 + a.zseg_len, a.D);
    const int iy0 = y0 - a.off, ix0 = x0 - a.off;
    const int nz = z1 - z0;  // slices walked

    auto load_slice = [&](int s) {
        const int buf = s % NBUF;
        const int Z = z0 + s;
        if (a.tma) {
            if (tid == 0) {
                mbar_arrive_expect_tx(&bars[buf], kStatsTx + a.tx_extra);
                tma_load_4d(xs + buf * XSTAGE, &a.tm_x, ix0, iy0, Z, plane, &bars[buf]);
                tma_load_4d(ys + buf * XSTAGE, &a.tm_y, ix0, iy0, Z, plane, &bars[buf]);
            }
            return;
        }
        if (a.vec16) {
            // the tile origin ix0 is a multiple of 4 and W % 4 == 0: 16-byte chunks,
            // each entirely inside or outside the volume
            constexpr int NCH = IXP / 4;
            for (int e = tid; e < IY * NCH; e += NT) {
                const int r = e / NCH, ch = e - r * NCH;
                const int Y = iy0 + r, X = ix0 + 4 * ch;
                const bool inb = (Y >= 0) && (Y < a.H) && (X >= 0) && (X < a.W);
                const size_t gi = inb ? (size_t(Z) * a.H + Y) * a.W + X : 0;
                const int si = buf * XSTAGE + r * IXP + 4 * ch;
                cp_async16(xs + si, xp + gi, inb);
                cp_async16(ys + si, yp + gi, inb);
            }
            return;
        }
        for (int e = tid; e < IY * IX; e += NT) {
            const int r = e / IX, c = e - r * IX;
            const int Y = iy0 + r, X = ix0 + c;
            const bool inb = (Y >= 0) && (Y < a.H) && (X >= 0) && (X < a.W);
            const size_t gi = inb ? (size_t(Z) * a.H + Y) * a.W + X : 0;
            const int si = buf * XSTAGE + r * IXP + c;
            cp_async4(xs + si, xp + gi, inb);
            cp_async4(ys + si, yp + gi, inb);
        }
    };

    // row pass of slice s: staged row r, columns [KX g, KX g + KX)
    auto x_item = [&](int s, int item) {
        const int g = item / IY, r = item - g * IY;
        const int base = (s % NBUF) * XSTAGE + r * IXP + g * KX;
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
        float2 accA[KX], accB[KX];
#pragma unroll
        for (int m = 0; m < KX + 10; ++m) {
            const float2 p = f2(xv[m] - kShift, yv[m] - kShift);
            const float2 sq = __fmul2_rn(p, p);
            const float dd = p.x - p.y;
            const float2 q = f2(sq.x + sq.y, dd * dd);
#pragma unroll
            for (int o = 0; o < KX; ++o) {
                const int t = m - o;
                if (t < 0 || t > 10) continue;
                const float2 w = splat(tap(t));
                accA[o] = (t == 0) ? __fmul2_rn(w, p) : __ffma2_rn(w, p, accA[o]);
                accB[o] = (t == 0) ? __fmul2_rn(w, q) : __ffma2_rn(w, q, accB[o]);
            }
        }
        float4 *dst = hx + ((s & 1) * IY + r) * HXP + g * KX;
#pragma unroll
        for (int o = 0; o < KX; ++o)
            dst[o] = make_float4(accA[o].x, accA[o].y, accB[o].x, accB[o].y);
    };

    // column pass of slice s: column tx, rows [KY g, KY g + KY)
    auto y_item = [&](int s, int item) {
        const int g = item / TX, tx = item - g * TX;
        float2 oa[KY], ob[KY];
        taps4<KY>(hx + ((s & 1) * IY + g * KY) * HXP + tx, HXP, oa, ob);
#pragma unroll
        for (int o = 0; o < KY; ++o)
            hy[((s & 1) * TY + g * KY + o) * TX + tx] = make_float4(oa[o].x, oa[o].y, ob[o].x, ob[o].y);
    };

    const int ty = tid / TX, tx = tid - ty * TX;
    const int py = y0 + ty, px = x0 + tx;
    const bool col_ok = (py < a.Ho) && (px < a.Wo);
    float4 *__restrict__ tcol =
        a.tfield + (size_t(plane) * a.D + z0) * a.Ho * a.Wo + size_t(col_ok ? py : 0) * a.Wo + px;
    const size_t tstride = size_t(a.Ho) * a.Wo;

    // Pipeline: step s stores slice s, runs the column pass of slice s + 1 and
    // the row pass of slice s + 2, then one barrier.  The row and column results
    // are double-buffered by slice parity, so each buffer a step writes was last
    // read in the step before.  Slices 0 .. NBUF-1 are in flight from the start
    // (one commit group each) and slice NBUF follows the row pass of slice 0;
    // as step s starts, the buffer whose row pass ran in the step before (slice
    // s + 1) takes slice s + 1 + NBUF, NBUF - 1 steps ahead of its row pass.
    // With cp.async staging every wait leaves the one newest group pending.
    // Tensor staging waits on slice j's barrier (use j / NBUF of buffer
    // j % NBUF); a wait that runs out stops the walk and the block's slices
    // come out NaN.
    auto landed = [&](int j) {
        return j >= nz || mbar_wait_bounded(&bars[j % NBUF], (j / NBUF) & 1, kWaitCycles);
    };
    if (a.tma) {
        if (tid == 0) {
#pragma unroll
            for (int b2 = 0; b2 < NBUF; ++b2) mbar_init(&bars[b2], 1);
            mbar_init_fence();
        }
        __syncthreads();
    }
    int issued = 0, waited = 0;  // slices copied / waited for (uniform)
#pragma unroll
    for (int k = 0; k < NBUF; ++k) {
        if (k < nz) {
            load_slice(k);
            ++issued;
        }
        cp_async_commit();
    }
    bool ok = true;
    if (a.tma) ok = landed(0) && landed(1);
    else cp_async_wait<NBUF - 2>();  // slices 0 and 1
    bool failed = __syncthreads_or(!ok);
    if (!failed) {
        waited = min(nz, 2);
        for (int i = tid; i < NXI; i += NT) x_item(0, i);
        __syncthreads();
        if (NBUF < nz) {  // slice 0's buffer is free
            load_slice(NBUF);
            ++issued;
        }
        cp_async_commit();
        const int nx = (1 < nz) ? NXI : 0;
        for (int i = tid; i < NYI + nx; i += NT) {
            if (i < NYI) y_item(0, i);
            else x_item(1, i - NYI);
        }
        if (a.tma) ok = landed(2);
        else cp_async_wait<NBUF - 2>();  // slice 2
        failed = __syncthreads_or(!ok);
        if (!failed) waited = min(nz, 3);
    }

    for (int s = 0; s < nz && !failed; ++s) {
        if (s + 1 + NBUF < nz) {
            load_slice(s + 1 + NBUF);
            ++issued;
        }
        cp_async_commit();
        if (col_ok) tcol[s * tstride] = hy[((s & 1) * TY + ty) * TX + tx];
        const int ny = (s + 1 < nz) ? NYI : 0;
        const int nx = (s + 2 < nz) ? NXI : 0;
        for (int i = tid; i < ny + nx; i += NT) {
            if (i < ny) y_item(s + 1, i);
            else x_item(s + 2, i - ny);
        }
        if (a.tma) ok = landed(s + 3);
        else cp_async_wait<NBUF - 2>();  // slice s + 3 has landed
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        waited = min(nz, s + 4);
    }
    cp_async_wait<0>();
    if (failed) {
        if (a.tma && tid == 0) drain_failed<NBUF>(bars, waited, issued);
        if (col_ok)
            for (int s = 0; s < nz; ++s) tcol[s * tstride] = nan4();
    }
}

// ------------------------------------------------------------------- z kernel

// Shifted statistics of a slice of padding (same padding, outside the volume):
// every pixel is 0, i.e. -kShift after the shift, blurred by the XY window (the
// two images' difference is 0 there).
__device__ __forceinline__ float4 pad_stats()
{
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < kTaps; ++k) t += tap(k);
    const float s2 = t * t;
    return make_float4(-kShift * s2, -kShift * s2, 2.0f * kShift * kShift * s2, 0.0f);
}

// One thread per output column (Ho x Wo, flattened) and z segment.  With
// gradients the segments cut the volume's slices [0, D): segment [z0, z1) of
// ufield needs the derivatives of output slices z0 + off - 10 .. z1 + off - 1,
// hence the statistics of slices z0 - 10 .. z1 + 9 (20 slices of warm-up).
// Without, they cut the output slices [0, Do) (10 slices of warm-up).  SSIM
// of output slice p counts (mean, map) in the segment that holds p.  SAME:
// same padding (slices outside the volume enter as padding statistics); in
// valid padding every slice read lies inside the volume.
template <bool GRAD, bool G2, bool SAME>
__global__ void __launch_bounds__(kZThreads) ssim3d_z_kernel(const __grid_constant__ Ssim3dArgs a)
{
    __shared__ double red[kZThreads / 32];
    pdl_trigger();
    int b = blockIdx.x;
    const int cb = b % a.col_blocks; b /= a.col_blocks;
    const int zseg = b % a.zsegs;
    const int plane = b / a.zsegs;
    const int cols = a.Ho * a.Wo;
    const int c = cb * kZThreads + threadIdx.x;
    const bool col_ok = c < cols;
    const size_t base = size_t(plane) * a.D * cols + (col_ok ? c : 0);
    const float4 *__restrict__ tcol = a.tfield + base;
    float4 *__restrict__ ucol = a.ufield + base;
    constexpr int off = SAME ? kRadius : 0;
    const int z0 = zseg * a.zseg_len;
    const int z1 = min(z0 + a.zseg_len, GRAD ? a.D : a.Do);
    const int plo = GRAD ? max(z0 + off - 10, 0) : z0;       // output slices computed
    const int phi = GRAD ? min(z1 + off, a.Do) : z1;
    const int t0 = plo - off;                                  // first statistics slice
    const int nfeed = phi - plo + 10;
    const float4 kpad = pad_stats();
    const size_t ostride = size_t(cols);
    float *mapc = a.map ? a.map + (size_t(plane) * a.Do) * cols + (col_ok ? c : 0) : nullptr;

    float2 PA[kTaps - 1], PB[kTaps - 1];  // pending Z sums of (m1, m2), (es, ed)
    float2 QA[kTaps - 1], QB[kTaps - 1];  // adjoint: of (g_f1, g_es), (g_ed, g_f2)
    float QC[kTaps - 1];                  // adjoint: of g_ed alone without grad_img2
#pragma unroll
    for (int k = 0; k < kTaps - 1; ++k) {
        PA[k] = PB[k] = QA[k] = QB[k] = f2(0.f, 0.f);
        QC[k] = 0.f;
    }
    float ssum = 0.f;

    auto emit = [&](int p, const float2 &vA, const float2 &vB, float v12) {
        const int z = p - off;  // ufield slice completed by output slice p
        if (z >= z0 && col_ok)
            ucol[size_t(z) * ostride] = G2 ? make_float4(vA.x, vA.y, vB.x, vB.y)
                                           : make_float4(vA.x, vA.y, v12, 0.f);
    };

    // feed i: statistics slice t0 + i; from i = 10 on it completes output slice
    // plo + i - 10
    auto step = [&](int i, const float4 &h) {
        const float2 M = zshift2(PA, lo(h)), E = zshift2(PB, hi(h));
        if (i < 10) return;
        const int p = plo + i - 10;
        const Moments mo{M.x, M.y, E.x, E.y};
        const bool own = GRAD ? (p >= z0 && p < z1) : true;
        float S;
        if (GRAD) {
            MomentGrads g;
            S = ssim_and_grads<G2>(mo, make_float2(kShift, kShift), true, g);
            const float2 vA = zshift2(QA, f2(g.g_f1, g.g_es));
            float2 vB = f2(0.f, 0.f);
            float v12 = 0.f;
            if (G2) vB = zshift2(QB, f2(g.g_ed, g.g_f2));
            else v12 = zshift1(QC, g.g_ed);
            emit(p, vA, vB, v12);
        } else {
            S = ssim_value(mo, make_float2(kShift, kShift));
        }
        if (own && col_ok) {
            ssum += S;
            if (mapc) mapc[size_t(p) * ostride] = S;
        }
    };

    // valid padding reads only slices inside the volume
    const float4 *tnext = tcol + size_t(SAME ? 0 : t0) * ostride;
    auto fetch = [&](int i) -> float4 {
        if (i >= nfeed || !col_ok) return make_float4(0.f, 0.f, 0.f, 0.f);
        if (SAME) {
            const int t = t0 + i;
            if (t < 0 || t >= a.D) return kpad;
            return __ldcg(tcol + size_t(t) * ostride);
        }
        return __ldcg(tnext + size_t(i) * ostride);
    };

    pdl_wait();  // tfield of the xy kernel ahead on the stream
    // rolling prefetch: slot j holds feed i0 + j; it is refilled with feed
    // i0 + j + kZPrefetch as soon as it is taken
    float4 q[kZPrefetch];
#pragma unroll
    for (int j = 0; j < kZPrefetch; ++j) q[j] = fetch(j);
    for (int i0 = 0; i0 < nfeed; i0 += kZPrefetch) {
#pragma unroll
        for (int j = 0; j < kZPrefetch; ++j) {
            const float4 h = q[j];
            q[j] = fetch(i0 + j + kZPrefetch);
            if (i0 + j < nfeed) step(i0 + j, h);
        }
    }
    if (GRAD) {
        // derivative slices past the output domain are zero: flush the rest
        for (int p = phi; p < z1 + off; ++p) {
            const float2 vA = zshift2_zero(QA);
            float2 vB = f2(0.f, 0.f);
            float v12 = 0.f;
            if (G2) vB = zshift2_zero(QB);
            else v12 = zshift1_zero(QC);
            emit(p, vA, vB, v12);
        }
    }

    if (a.partials) {
        const double tot = block_sum<kZThreads>(ssum, red);
        if (threadIdx.x == 0) a.partials[blockIdx.x] = tot;
        finish_means<kZThreads>(a.partials, a.counter, a.mean, a.images, a.blocks_per_image, a.count);
    }
}

// ------------------------------------------------------------- adjoint kernel

template <bool G2>
__global__ void __launch_bounds__(GA::NT, 3) ssim3d_adjoint_kernel(const __grid_constant__ Ssim3dArgs a)
{
    constexpr int NT = GA::NT, TY = GA::TY, TX = GA::TX, IY = GA::IY, IX = GA::IX,
                  GXP = GA::GXP, HXP = GA::HXP, KX = GA::KX, NXI = GA::NXI, KY = GA::KY,
                  NYI = GA::NYI, GSTAGE = GA::GSTAGE, CSTAGE = GA::CSTAGE;
    extern __shared__ __align__(128) unsigned char smem_dyn[];
    unsigned char *smem_raw = smem_dyn + ((128 - (smem_u32(smem_dyn) & 127)) & 127);
    float4 *gs = reinterpret_cast<float4 *>(smem_raw);                   // [NBUF_A][GSTAGE]
    float *cbx = reinterpret_cast<float *>(smem_raw + kAdjInBytes);      // [CBUF_A][TY][TX]
    float *cby = cbx + CBUF_A * CSTAGE;
    float4 *ux = reinterpret_cast<float4 *>(smem_raw + kAdjInBytes + kChainBytes);  // [2][IY][HXP]
    float4 *uy = ux + 2 * IY * HXP;                                       // [2][TY][TX]
    __shared__ uint64_t bars[NBUF_A];
    pdl_trigger();
    pdl_wait();  // ufield of the z kernel ahead on the stream

    const int tid = threadIdx.x;
    int b = blockIdx.x;
    const int tile_x = b % a.tiles_x; b /= a.tiles_x;
    const int tile_y = b % a.tiles_y; b /= a.tiles_y;
    const int zseg = b % a.zsegs;
    const int plane = b / a.zsegs;
    const int n = plane / a.C;
    const size_t vol = size_t(a.D) * a.H * a.W;
    const size_t plane_off = size_t(plane) * vol;
    const float4 *__restrict__ gf = a.ufield + size_t(plane) * a.D * a.Ho * a.Wo;

    const int y0 = tile_y * TY, x0 = tile_x * TX;  // gradient (image) coordinates
    const int q0 = zseg * a.zseg_len;
    const int q1 = min(q0 + a.zseg_len, a.D);
    // derivative positions feeding gradient q: q + off - 10 .. q + off per axis
    const int gy0 = y0 + a.off - 10, gx0 = x0 + a.off - 10;
    const int nz = q1 - q0;
    const float scale = a.dL ? a.dL[n] * a.inv_count : a.inv_count;

    // derivative slice q0 + s and the input pixels of the same slice into
    // chain buffer s % CBUF_A
    auto load_slice = [&](int s) {
        const int buf = s % NBUF_A;
        const int q = q0 + s;
        if (a.tma_adj) {
            // zeros outside the derivative domain
            if (tid == 0) {
                mbar_arrive_expect_tx(&bars[buf], kAdjTx + a.tx_extra);
                tma_load_4d(gs + buf * GSTAGE, &a.tm_g, 4 * gx0, gy0, q, plane, &bars[buf]);
                tma_load_4d(cbx + (s % CBUF_A) * CSTAGE, &a.tm_cx, x0, y0, q, plane, &bars[buf]);
                tma_load_4d(cby + (s % CBUF_A) * CSTAGE, &a.tm_cy, x0, y0, q, plane, &bars[buf]);
            }
            return;
        }
        for (int e = tid; e < IY * IX; e += NT) {
            const int r = e / IX, c = e - r * IX;
            const int Y = gy0 + r, X = gx0 + c;
            const bool inb = (Y >= 0) && (Y < a.Ho) && (X >= 0) && (X < a.Wo);
            const size_t gi = inb ? (size_t(q) * a.Ho + Y) * a.Wo + X : 0;
            cp_async16(gs + buf * GSTAGE + r * GXP + c, gf + gi, inb);
        }
        const int ty = tid / TX, tx = tid - ty * TX;  // one pixel per thread (NT == TY * TX)
        const int qy = y0 + ty, qx = x0 + tx;
        const bool inb = (qy < a.H) && (qx < a.W);
        const size_t gi = inb ? plane_off + (size_t(q) * a.H + qy) * a.W + qx : 0;
        cp_async4(cbx + (s % CBUF_A) * CSTAGE + tid, a.x + gi, inb);
        cp_async4(cby + (s % CBUF_A) * CSTAGE + tid, a.y + gi, inb);
    };

    // adjoint row pass: gradient columns [KX g, KX g + KX) of staged row r
    // (grad_img1 only: the fourth component, g_mu2, is not blurred; its slot
    // carries zero)
    auto x_item = [&](int s, int item) {
        const int g = item / IY, r = item - g * IY;
        float2 oa[KX], ob[KX];
        const float4 *src = gs + (s % NBUF_A) * GSTAGE + r * GXP + g * KX;
        if (G2) {
            taps4<KX>(src, 1, oa, ob);
        } else {
            float oc[KX];
            taps3<KX>(src, 1, oa, oc);
#pragma unroll
            for (int o = 0; o < KX; ++o) ob[o] = f2(oc[o], 0.f);
        }
        float4 *dst = ux + ((s & 1) * IY + r) * HXP + g * KX;
#pragma unroll
        for (int o = 0; o < KX; ++o) dst[o] = make_float4(oa[o].x, oa[o].y, ob[o].x, ob[o].y);
    };

    auto y_item = [&](int s, int item) {
        const int g = item / TX, tx = item - g * TX;
        float2 oa[KY], ob[KY];
        const float4 *src = ux + ((s & 1) * IY + g * KY) * HXP + tx;
        if (G2) {
            taps4<KY>(src, HXP, oa, ob);
        } else {
            float oc[KY];
            taps3<KY>(src, HXP, oa, oc);
#pragma unroll
            for (int o = 0; o < KY; ++o) ob[o] = f2(oc[o], 0.f);
        }
#pragma unroll
        for (int o = 0; o < KY; ++o)
            uy[((s & 1) * TY + g * KY + o) * TX + tx] = make_float4(oa[o].x, oa[o].y, ob[o].x, ob[o].y);
    };

    const int ty = tid / TX, tx = tid - ty * TX;
    const int qy = y0 + ty, qx = x0 + tx;
    const bool col_ok = (qy < a.H) && (qx < a.W);
    const size_t gbase = plane_off + size_t(col_ok ? qy : 0) * a.W + qx;
    const size_t gstride = size_t(a.H) * a.W;

    // chain rule of slice s from (B^T g_f1, B^T g_es, B^T g_ed, B^T g_f2) at this
    // pixel: per window (shift 1/2 for both images),
    //   g_m1 + 2 x' g_es + 2 (x' - y') g_ed = g_f1 + 2 (x - 1/2) g_es + 2 (x - y) g_ed;
    // in a flat window g_ed is of order 1 / C2 and meets x - y
    auto chain_step = [&](int s) {
        if (!col_ok) return;
        const float4 h = uy[((s & 1) * TY + ty) * TX + tx];
        const size_t gi = gbase + size_t(q0 + s) * gstride;
        const float x = cbx[(s % CBUF_A) * CSTAGE + tid];
        const float y = cby[(s % CBUF_A) * CSTAGE + tid];
        const float dxy2 = 2.0f * (x - y);
        a.out1[gi] = scale * fmaf(dxy2, h.z, fmaf(2.0f * (x - kShift), h.y, h.x));
        if (G2) a.out2[gi] = scale * fmaf(-dxy2, h.z, fmaf(2.0f * (y - kShift), h.y, h.w));
    };

    // The pipeline of the xy kernel, with the chain rule in place of the store,
    // on NBUF_A staging buffers: at step s the chain rule of slice s, the column
    // pass of slice s + 1 and the row pass of slice s + 2 run; the buffer whose
    // row pass ran in the step before (slice s + 1) takes slice s + 1 + NBUF_A as
    // the step starts, two steps before its row pass.  Chain tiles live from the
    // slice's copy to its chain rule: NBUF_A + 2 of them.  With cp.async staging
    // every wait leaves the one newest group pending.
    auto landed = [&](int j) {
        return j >= nz || mbar_wait_bounded(&bars[j % NBUF_A], (j / NBUF_A) & 1, kWaitCycles);
    };
    if (a.tma_adj) {
        if (tid == 0) {
#pragma unroll
            for (int b2 = 0; b2 < NBUF_A; ++b2) mbar_init(&bars[b2], 1);
            mbar_init_fence();
        }
        __syncthreads();
    }
    int issued = 0, waited = 0;
#pragma unroll
    for (int k = 0; k < NBUF_A; ++k) {
        if (k < nz) {
            load_slice(k);
            ++issued;
        }
        cp_async_commit();
    }
    bool ok = true;
    if (a.tma_adj) ok = landed(0) && landed(1);
    else cp_async_wait<1>();  // slices 0 and 1
    bool failed = __syncthreads_or(!ok);
    if (!failed) {
        waited = min(nz, 2);
        for (int i = tid; i < NXI; i += NT) x_item(0, i);
        __syncthreads();
        // slice 0's buffer is free: slice NBUF_A
        if (NBUF_A < nz) {
            load_slice(NBUF_A);
            ++issued;
        }
        cp_async_commit();
        const int nx = (1 < nz) ? NXI : 0;
        for (int i = tid; i < NYI + nx; i += NT) {
            if (i < NYI) y_item(0, i);
            else x_item(1, i - NYI);
        }
        if (a.tma_adj) ok = landed(2);
        else cp_async_wait<1>();  // slice 2
        failed = __syncthreads_or(!ok);
        if (!failed) waited = min(nz, 3);
    }

    for (int s = 0; s < nz && !failed; ++s) {
        if (s + 1 + NBUF_A < nz) {
            load_slice(s + 1 + NBUF_A);
            ++issued;
        }
        cp_async_commit();
        chain_step(s);
        const int ny = (s + 1 < nz) ? NYI : 0;
        const int nx = (s + 2 < nz) ? NXI : 0;
        for (int i = tid; i < ny + nx; i += NT) {
            if (i < ny) y_item(s + 1, i);
            else x_item(s + 2, i - ny);
        }
        if (a.tma_adj) ok = landed(s + 3);
        else cp_async_wait<1>();  // slice s + 3 (and its chain tile) landed
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        waited = min(nz, s + 4);
    }
    cp_async_wait<0>();
    if (failed) {
        if (a.tma_adj && tid == 0) drain_failed<NBUF_A>(bars, waited, issued);
        if (col_ok)
            for (int s = 0; s < nz; ++s) {
                const size_t gi = gbase + size_t(q0 + s) * gstride;
                a.out1[gi] = nan4().x;
                if (G2) a.out2[gi] = nan4().x;
            }
    }
}

template <typename K>
cudaError_t prepare(K kernel, int threads, size_t smem, int *occ)
{
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, kernel, threads, smem);
}

template <typename K>
cudaError_t launch_early(K kernel, const Ssim3dArgs &a, int blocks, int threads, size_t smem,
                         cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(unsigned(threads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace

void ssim3d_prepare_staging(Ssim3dArgs &a, long long planes)
{
    const int mode = staging_mode();
    // the volumes as [planes][D][H][W]: W % 4 == 0, 16-byte aligned
    const bool aligned = mode != 1 && a.W % 4 == 0 && reinterpret_cast<uintptr_t>(a.x) % 16 == 0 &&
                         reinterpret_cast<uintptr_t>(a.y) % 16 == 0 && planes < (1LL << 31);
    const unsigned long long W = a.W, H = a.H, D = a.D, P = planes;
    const unsigned long long dims[4] = {W, H, D, P};
    const unsigned long long st[3] = {W * 4, H * W * 4, D * H * W * 4};
    // xy kernel: tiles start at x0 - off, on 16-byte columns in valid padding
    bool xy = aligned && a.off == 0;
    if (xy) {
        const unsigned bx[4] = {GS::IXP, GS::IY, 1, 1};
        xy = encode_tiled_f32(a.tm_x, a.x, 4, dims, st, bx) &&
             encode_tiled_f32(a.tm_y, a.y, 4, dims, st, bx);
    }
    // adjoint kernel: chain tiles at multiples of 16 columns, derivative tiles
    // at 4 (x0 + off - 10) floats of float4 rows (16-byte columns in both paddings)
    bool adj = aligned && a.ufield;
    if (adj) {
        const unsigned bc[4] = {GA::TX, GA::TY, 1, 1};
        adj = encode_tiled_f32(a.tm_cx, a.x, 4, dims, st, bc) &&
              encode_tiled_f32(a.tm_cy, a.y, 4, dims, st, bc);
    }
    if (adj) {
        const unsigned long long Wo = a.Wo, Ho = a.Ho;
        const unsigned long long gdims[4] = {4 * Wo, Ho, D, P};
        const unsigned long long gst[3] = {Wo * 16, Ho * Wo * 16, D * Ho * Wo * 16};
        const unsigned bg[4] = {4 * GA::GXP, GA::IY, 1, 1};
        adj = encode_tiled_f32(a.tm_g, a.ufield, 4, gdims, gst, bg);
    }
    a.tma = xy ? 1 : 0;
    a.tma_adj = adj ? 1 : 0;
    a.tx_extra = ((xy || adj) && mode == 2) ? 16u : 0u;
}

cudaError_t ssim3d_staging_status(unsigned *flags, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_staging3d_status, sizeof(unsigned));
    if (e == cudaSuccess && clear) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_staging3d_status, &zero, sizeof(unsigned));
    }
    return e;
}

cudaError_t ssim3d_prepare(int occ[5])
{
    int o[6] = {0, 0, 0, 0, 0, 0};
    cudaError_t e;
    if ((e = prepare(ssim3d_xy_kernel, GS::NT, xy_smem(), &o[0])) != cudaSuccess) return e;
    if ((e = prepare(ssim3d_z_kernel<false, false, true>, kZThreads, 0, &o[1])) != cudaSuccess) return e;
    if ((e = prepare(ssim3d_z_kernel<true, false, true>, kZThreads, 0, &o[2])) != cudaSuccess) return e;
    if ((e = prepare(ssim3d_z_kernel<true, true, true>, kZThreads, 0, &o[3])) != cudaSuccess) return e;
    if ((e = prepare(ssim3d_adjoint_kernel<false>, GA::NT, adjoint_smem(), &o[4])) != cudaSuccess)
        return e;
    if ((e = prepare(ssim3d_adjoint_kernel<true>, GA::NT, adjoint_smem(), &o[5])) != cudaSuccess)
        return e;
    for (int i = 0; i < 4; ++i) occ[i] = o[i];
    occ[4] = o[4] < o[5] ? o[4] : o[5];
    for (int i = 0; i < 5; ++i)
        if (occ[i] < 1) return cudaErrorInvalidConfiguration;
    return cudaSuccess;
}

cudaError_t ssim3d_xy_launch(const Ssim3dArgs &a, int blocks, cudaStream_t s)
{
    ssim3d_xy_kernel<<<blocks, GS::NT, xy_smem(), s>>>(a);
    return cudaGetLastError();
}

cudaError_t ssim3d_z_launch(const Ssim3dArgs &a, bool grad, bool g2, int blocks, cudaStream_t s)
{
    if (a.off) {
        if (!grad) return launch_early(ssim3d_z_kernel<false, false, true>, a, blocks, kZThreads, 0, s);
        if (g2) return launch_early(ssim3d_z_kernel<true, true, true>, a, blocks, kZThreads, 0, s);
        return launch_early(ssim3d_z_kernel<true, false, true>, a, blocks, kZThreads, 0, s);
    }
    if (!grad) return launch_early(ssim3d_z_kernel<false, false, false>, a, blocks, kZThreads, 0, s);
    if (g2) return launch_early(ssim3d_z_kernel<true, true, false>, a, blocks, kZThreads, 0, s);
    return launch_early(ssim3d_z_kernel<true, false, false>, a, blocks, kZThreads, 0, s);
}

cudaError_t ssim3d_adjoint_launch(const Ssim3dArgs &a, bool g2, int blocks, cudaStream_t s)
{
    if (g2) return launch_early(ssim3d_adjoint_kernel<true>, a, blocks, GA::NT, adjoint_smem(), s);
    return launch_early(ssim3d_adjoint_kernel<false>, a, blocks, GA::NT, adjoint_smem(), s);
}

}  // namespace gbssim
