// 2D SSIM: one streaming kernel for the forward, the training forward and the
// recompute backward, plus the scaling pass of the stored backward.
//
// Method (TriSSIM README, "How it works"; fused-ssim README introduction):
//   forward   five Gaussian-blurred quantities -- here four, because sigma11 and
//             sigma22 enter SSIM only as their sum -- from one row pass and one
//             column pass, SSIM in registers, and the mean;
//   backward  the blur's adjoint (a "full" correlation) applied to the upstream
//             gradients of the statistics, then the chain rule
//             grad1 = B^T g_mu1 + 2 x B^T g_e + y B^T g_e12 (grad2 likewise).
//
// Design.  A CTA owns a vertical strip of columns of one (n, c) plane and walks
// down a segment of its rows, 11 rows per step.  Per step:
//   H  row pass: 11 input rows (staged in shared memory by cp.async, three
//      buffers) -> the four row-blurred statistics of 128 columns (hb);
//   V  column pass, one thread per column: an 11-row register ring of hb gives
//      the window statistics, then SSIM and its derivatives in registers; in
//      gradient mode a second 11-row register ring of those derivatives gives
//      the column pass of the adjoint (vb);
//   A  row pass of the adjoint over vb, the chain rule with the input pixel, and
//      the store of the gradient row.
// H of step t+1 and A of step t share one barrier interval.  Streaming down the
// rows computes every statistic of the strip once (no vertical halo recompute
// except the 20-row warm-up of a segment).
//
// Gradient mode has two uses:
//   training forward: the gradient fields of mean[n] itself (dL = 1) go to the
//                     caller's `saved` buffer, and the mean is reduced too;
//   recompute backward: the fields times dL[n] go to grad_img1 / grad_img2.
#include "common.cuh"
#include "ssim2d.cuh"

namespace gbssim {
namespace {

constexpr int NT = kThreads2d;         // threads per CTA = statistic columns per strip
constexpr int SW = NT;                 // statistic columns held by a strip
constexpr int GW = SW - 10;            // gradient columns produced by a strip
constexpr int IW = SW + 10;            // input columns staged per row
constexpr int IWP = IW + 2;            // padded pitch (multiple of 4 floats)
constexpr int STEP = kTaps;            // rows per step = ring length
constexpr int KH = 8;                  // columns per row-pass work item
constexpr int NGH = SW / KH;           // row-pass items per row
constexpr int KA = 8;                  // columns per adjoint row-pass work item
constexpr int NGA = (GW + KA - 1) / KA;
constexpr int NBUF = 3;                // input row blocks in flight

static_assert(SW % KH == 0, "strip width must be a multiple of the row-pass block");
static_assert(IWP % 4 == 0, "input pitch must keep float4 alignment");

// Shared-memory layout: xs, ys [NBUF][STEP][IWP] floats, hb [STEP][SW] float4,
// vb [STEP][SW] float4 (gradient mode only).
constexpr size_t kInBytes = size_t(2) * NBUF * STEP * IWP * sizeof(float);
constexpr size_t kRowBytes = size_t(STEP) * SW * sizeof(float4);

// Column swizzle of hb / vb: writers with a stride of 8 columns and readers with
// a stride of 1 both hit eight distinct 16-byte bank groups per quarter warp.
__device__ __forceinline__ int swz(int c) { return (c & ~7) | ((c + (c >> 3)) & 7); }

__device__ __forceinline__ float4 f4(float a, float b, float c, float d)
{
    return make_float4(a, b, c, d);
}

template <bool GRAD, bool G2>
__global__ void __launch_bounds__(NT, 2) ssim2d_stream_kernel(const Ssim2dArgs a)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float *xs = reinterpret_cast<float *>(smem_raw);
    float *ys = xs + NBUF * STEP * IWP;
    float4 *hb = reinterpret_cast<float4 *>(smem_raw + kInBytes);
    float4 *vb = hb + STEP * SW;
    __shared__ double red[NT / 32];

    const int tid = threadIdx.x;
    int bidx = blockIdx.x;
    const int strip = bidx % a.strips;
    bidx /= a.strips;
    const int seg = bidx % a.segs;
    const int plane = bidx / a.segs;
    const int n = plane / a.C;
    const size_t plane_off = size_t(plane) * size_t(a.H) * size_t(a.W);
    const float *__restrict__ xp = a.x + plane_off;
    const float *__restrict__ yp = a.y + plane_off;

    // Geometry of the walk.  Input row r completes statistic row p = r + off - 10;
    // in gradient mode statistic row p completes gradient row q = p - off = r - 10.
    int j0 = 0, sc0, ic0, R0, nrows, q0 = 0, q1 = 0;
    if (GRAD) {
        j0 = strip * GW;
        q0 = seg * a.seg_rows;
        q1 = min(q0 + a.seg_rows, a.H);
        sc0 = j0 + a.off - 10;
        ic0 = j0 - 10;
        R0 = q0 - 10;
        nrows = q1 - q0 + 20;
    } else {
        sc0 = strip * SW;
        const int r0 = seg * a.seg_rows;
        const int r1 = min(r0 + a.seg_rows, a.Ho);
        ic0 = sc0 - a.off;
        R0 = r0 - a.off;
        nrows = r1 - r0 + 10;
    }
    const int steps = (nrows + STEP - 1) / STEP;
    const int Rend = R0 + nrows;

    // ---- stage one block of STEP input rows into buffer t % NBUF (zeros outside)
    auto load_block = [&](int t) {
        const int buf = t % NBUF;
        const int rbase = R0 + t * STEP;
        for (int e = tid; e < STEP * IW; e += NT) {
            const int ri = e / IW, ci = e - ri * IW;
            const int R = rbase + ri, Cc = ic0 + ci;
            const bool inb = (R >= 0) && (R < a.H) && (Cc >= 0) && (Cc < a.W);
            const size_t gi = inb ? size_t(R) * a.W + Cc : 0;
            const int si = (buf * STEP + ri) * IWP + ci;
            cp_async4(xs + si, xp + gi, inb);
            cp_async4(ys + si, yp + gi, inb);
        }
    };

    // ---- row pass of the statistics: row k of block t, columns [KH g, KH g + KH)
    auto h_item = [&](int t, int item) {
        const int k = item / NGH, g = item - k * NGH;
        const int base = ((t % NBUF) * STEP + k) * IWP + g * KH;
        float xv[KH + 10], yv[KH + 10];
#pragma unroll
        for (int m = 0; m < KH + 8; m += 4) {
            const float4 u = *reinterpret_cast<const float4 *>(xs + base + m);
            const float4 v = *reinterpret_cast<const float4 *>(ys + base + m);
            xv[m] = u.x; xv[m + 1] = u.y; xv[m + 2] = u.z; xv[m + 3] = u.w;
            yv[m] = v.x; yv[m + 1] = v.y; yv[m + 2] = v.z; yv[m + 3] = v.w;
        }
        {
            const float2 u = *reinterpret_cast<const float2 *>(xs + base + KH + 8);
            const float2 v = *reinterpret_cast<const float2 *>(ys + base + KH + 8);
            xv[KH + 8] = u.x; xv[KH + 9] = u.y;
            yv[KH + 8] = v.x; yv[KH + 9] = v.y;
        }
        float acc[KH][4];
#pragma unroll
        for (int m = 0; m < KH + 10; ++m) {
            const float x = xv[m] - kShift, y = yv[m] - kShift;
            const float pe = fmaf(x, x, y * y);
            const float pc = x * y;
#pragma unroll
            for (int o = 0; o < KH; ++o) {
                const int b = m - o;
                if (b < 0 || b > 10) continue;
                const float w = tap(b);
                if (b == 0) {
                    acc[o][0] = w * x; acc[o][1] = w * y; acc[o][2] = w * pe; acc[o][3] = w * pc;
                } else {
                    acc[o][0] = fmaf(w, x, acc[o][0]);
                    acc[o][1] = fmaf(w, y, acc[o][1]);
                    acc[o][2] = fmaf(w, pe, acc[o][2]);
                    acc[o][3] = fmaf(w, pc, acc[o][3]);
                }
            }
        }
#pragma unroll
        for (int o = 0; o < KH; ++o)
            hb[k * SW + swz(g * KH + o)] = f4(acc[o][0], acc[o][1], acc[o][2], acc[o][3]);
    };

    const float scale = (GRAD && a.dL) ? a.dL[n] * a.inv_count : a.inv_count;

    // ---- row pass of the adjoint for gradient row of (block t, row k), chain rule, store
    auto a_item = [&](int t, int item) {
        const int k = item / NGA, g = item - k * NGA;
        const int q = R0 + t * STEP + k - 10;
        if (q < q0 || q >= q1) return;
        // input row q: block t row 0 when k == 10, else block t-1 row k+1
        const int tq = (k == STEP - 1) ? t : t - 1;
        const int kq = (k == STEP - 1) ? 0 : k + 1;
        const int xbase = ((tq % NBUF) * STEP + kq) * IWP + 10;
        float acc[KA][4];
#pragma unroll
        for (int m = 0; m < KA + 10; ++m) {
            const int c = min(g * KA + m, SW - 1);  // past the strip only for unused outputs
            const float4 v = vb[k * SW + swz(c)];
#pragma unroll
            for (int o = 0; o < KA; ++o) {
                const int b = m - o;
                if (b < 0 || b > 10) continue;
                const float w = tap(b);
                if (b == 0) {
                    acc[o][0] = w * v.x; acc[o][1] = w * v.y; acc[o][2] = w * v.z;
                    if (G2) acc[o][3] = w * v.w;
                } else {
                    acc[o][0] = fmaf(w, v.x, acc[o][0]);
                    acc[o][1] = fmaf(w, v.y, acc[o][1]);
                    acc[o][2] = fmaf(w, v.z, acc[o][2]);
                    if (G2) acc[o][3] = fmaf(w, v.w, acc[o][3]);
                }
            }
        }
        float *o1 = a.out1 + plane_off + size_t(q) * a.W;
        float *o2 = G2 ? a.out2 + plane_off + size_t(q) * a.W : nullptr;
#pragma unroll
        for (int o = 0; o < KA; ++o) {
            const int jj = g * KA + o;
            const int j = j0 + jj;
            if (jj < GW && j < a.W) {
                const float x = xs[xbase + jj] - kShift;
                const float y = ys[xbase + jj] - kShift;
                // acc = (B^T g_m1, B^T g_e, B^T g_e12, B^T g_m2)
                o1[j] = scale * fmaf(2.0f * x, acc[o][1], fmaf(y, acc[o][2], acc[o][0]));
                if (G2) o2[j] = scale * fmaf(2.0f * y, acc[o][1], fmaf(x, acc[o][2], acc[o][3]));
            }
        }
    };

    // ---- column pass state: registers of thread tid (statistic column sc0 + tid)
    float4 hr[STEP];
    float4 gr[STEP];
#pragma unroll
    for (int k = 0; k < STEP; ++k) {
        hr[k] = f4(0.f, 0.f, 0.f, 0.f);
        gr[k] = f4(0.f, 0.f, 0.f, 0.f);
    }
    const int pc = sc0 + tid;
    const bool col_ok = (pc >= 0) && (pc < a.Wo);
    const bool col_own = GRAD ? (tid >= 10 || strip == 0) : true;
    const bool want_mean = (a.partials != nullptr);
    float ssum = 0.0f;

    // ---- prologue
    load_block(0);
    cp_async_commit();
    if (steps > 1) load_block(1);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    for (int i = tid; i < STEP * NGH; i += NT) h_item(0, i);
    __syncthreads();

    for (int t = 0; t < steps; ++t) {
        // ---- V: column passes of step t
#pragma unroll
        for (int k = 0; k < STEP; ++k) {
            hr[k] = hb[k * SW + swz(tid)];
            Moments mo{0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int aa = 0; aa < STEP; ++aa) {
                const float4 h = hr[(k + 1 + aa) % STEP];
                const float w = tap(aa);
                mo.m1 = fmaf(w, h.x, mo.m1);
                mo.m2 = fmaf(w, h.y, mo.m2);
                mo.es = fmaf(w, h.z, mo.es);
                mo.e12 = fmaf(w, h.w, mo.e12);
            }
            const int r = R0 + t * STEP + k;
            const int p = r + a.off - 10;
            const bool ok = col_ok && (r >= R0 + 10) && (r < Rend) && (p >= 0) && (p < a.Ho);
            if (GRAD) {
                MomentGrads gg;
                const float S = ssim_and_grads(mo, gg);
                gr[k] = ok ? f4(gg.g_m1, gg.g_e, gg.g_e12, gg.g_m2) : f4(0.f, 0.f, 0.f, 0.f);
                const bool own = ok && col_own && (r - 10 >= q0 || seg == 0);
                if (own) {
                    ssum += S;
                    if (a.map) a.map[(size_t(plane) * a.Ho + p) * a.Wo + pc] = S;
                }
                float4 v = f4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int aa = 0; aa < STEP; ++aa) {
                    const float4 gv = gr[(k + 1 + aa) % STEP];
                    const float w = tap(aa);
                    v.x = fmaf(w, gv.x, v.x);
                    v.y = fmaf(w, gv.y, v.y);
                    v.z = fmaf(w, gv.z, v.z);
                    if (G2) v.w = fmaf(w, gv.w, v.w);
                }
                vb[k * SW + swz(tid)] = v;
            } else {
                const float S = ssim_value(mo);
                if (ok) {
                    ssum += S;
                    if (a.map) a.map[(size_t(plane) * a.Ho + p) * a.Wo + pc] = S;
                }
            }
        }
        cp_async_wait<0>();  // block t+1 has landed
        __syncthreads();
        // ---- H of step t+1 and A of step t
        const int nh = (t + 1 < steps) ? STEP * NGH : 0;
        const int na = GRAD ? STEP * NGA : 0;
        for (int i = tid; i < nh + na; i += NT) {
            if (i < nh)
                h_item(t + 1, i);
            else
                a_item(t, i - nh);
        }
        __syncthreads();
        if (t + 2 < steps) load_block(t + 2);  // into the buffer A(t) just released
        cp_async_commit();
    }
    cp_async_wait<0>();

    if (want_mean) {
        const double tot = block_sum<NT>(ssum, red);
        if (tid == 0) a.partials[blockIdx.x] = tot;
        finish_means<NT>(a.partials, a.counter, a.mean, a.images, a.blocks_per_image, a.count);
    }
}

// grad = field * dL[n] / count, elementwise; n = index / per_image.
// A field may be scaled in place (g == f).
__global__ void __launch_bounds__(256) scale_fields_vec4(const float4 *f1, const float4 *f2,
                                                         float4 *g1, float4 *g2,
                                                         const float *__restrict__ dL,
                                                         float inv_count, size_t per_image4,
                                                         size_t total4)
{
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total4;
         i += size_t(gridDim.x) * blockDim.x) {
        const float s = dL[i / per_image4] * inv_count;
        float4 v = __ldcs(f1 + i);
        v.x *= s; v.y *= s; v.z *= s; v.w *= s;
        __stcs(g1 + i, v);
        if (g2) {
            float4 u = __ldcs(f2 + i);
            u.x *= s; u.y *= s; u.z *= s; u.w *= s;
            __stcs(g2 + i, u);
        }
    }
}

__global__ void __launch_bounds__(256) scale_fields_scalar(const float *f1, const float *f2,
                                                           float *g1, float *g2,
                                                           const float *__restrict__ dL,
                                                           float inv_count, size_t per_image,
                                                           size_t total)
{
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += size_t(gridDim.x) * blockDim.x) {
        const float s = dL[i / per_image] * inv_count;
        g1[i] = f1[i] * s;
        if (g2) g2[i] = f2[i] * s;
    }
}

template <bool GRAD, bool G2>
cudaError_t launch_stream(const Ssim2dArgs &a, int blocks, cudaStream_t s)
{
    const size_t smem = kInBytes + (GRAD ? 2 : 1) * kRowBytes;
    ssim2d_stream_kernel<GRAD, G2><<<blocks, NT, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

size_t ssim2d_smem_bytes(bool grad) { return kInBytes + (grad ? 2 : 1) * kRowBytes; }

int ssim2d_grad_cols() { return GW; }
int ssim2d_stat_cols() { return SW; }

const void *ssim2d_kernel_ptr(bool grad, bool g2)
{
    if (!grad) return reinterpret_cast<const void *>(ssim2d_stream_kernel<false, false>);
    return g2 ? reinterpret_cast<const void *>(ssim2d_stream_kernel<true, true>)
              : reinterpret_cast<const void *>(ssim2d_stream_kernel<true, false>);
}

cudaError_t ssim2d_launch(const Ssim2dArgs &a, bool grad, bool g2, int blocks, cudaStream_t s)
{
    if (!grad) return launch_stream<false, false>(a, blocks, s);
    return g2 ? launch_stream<true, true>(a, blocks, s) : launch_stream<true, false>(a, blocks, s);
}

cudaError_t scale_fields_launch(const float *f1, const float *f2, float *g1, float *g2,
                                const float *dL, float inv_count, size_t per_image, size_t total,
                                int sm_count, cudaStream_t s)
{
    const bool vec = (per_image % 4 == 0) &&
                     ((reinterpret_cast<uintptr_t>(f1) | reinterpret_cast<uintptr_t>(g1) |
                       reinterpret_cast<uintptr_t>(f2) | reinterpret_cast<uintptr_t>(g2)) % 16 == 0);
    const size_t work = vec ? total / 4 : total;
    size_t blocks = (work + 255) / 256;
    const size_t cap = size_t(sm_count) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (vec)
        scale_fields_vec4<<<unsigned(blocks), 256, 0, s>>>(
            reinterpret_cast<const float4 *>(f1), reinterpret_cast<const float4 *>(f2),
            reinterpret_cast<float4 *>(g1), reinterpret_cast<float4 *>(g2), dL, inv_count,
            per_image / 4, total / 4);
    else
        scale_fields_scalar<<<unsigned(blocks), 256, 0, s>>>(f1, f2, g1, g2, dL, inv_count,
                                                             per_image, total);
    return cudaGetLastError();
}

}  // namespace gbssim
