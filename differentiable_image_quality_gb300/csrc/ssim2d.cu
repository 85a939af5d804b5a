// 2D SSIM: one streaming kernel for the forward, the training forward and the
// recompute backward, plus the scaling pass of the stored backward.
//
// Method (TriSSIM README, "How it works"; fused-ssim README introduction):
//   forward   five Gaussian-blurred quantities -- here four, because sigma11 and
//             sigma22 enter SSIM only as their sum -- from one row pass and one
//             column pass, SSIM in registers, and the mean;
//   backward  the blur's adjoint (a "full" correlation) applied to the upstream
//             gradients of the statistics, then the chain rule
//             grad1 = B^T g_mu1 + 2 x B^T g_e + y B^T g_e12 (grad2 likewise),
//             evaluated here with the derivatives of S with respect to
//             es = E[x^2] + E[y^2] and ed = E[(x - y)^2] (E[xy] = (es - ed) / 2):
//             grad1 = B^T g_f1 + 2 (x - 1/2) B^T g_es + 2 (x - y) B^T g_ed.
//
// Design.  A CTA owns a vertical strip of columns of one (n, c) plane and walks
// down a segment of its rows, 11 rows per step.  Per step:
//   H  row pass: 11 input rows (staged in shared memory by cp.async, two
//      buffers) -> the four row-blurred statistics of 128 columns (hb);
//   V  column pass, one thread per column: an 11-row register ring of hb gives
//      the window statistics, then SSIM and its derivatives in registers; in
//      gradient mode a second 11-row register ring of those derivatives gives
//      the column pass of the adjoint (va, vc);
//   A  row pass of the adjoint over va / vc, the chain rule with the input
//      pixels of the gradient rows (prefetched into cb by cp.async while V
//      runs), and the store of the gradient.
// H of step t+1 and A of step t share one barrier interval.  Streaming down the
// rows computes every statistic of the strip once (no vertical halo recompute
// except the 20-row warm-up of a segment).
//
// The window sums run on pairs of float32 values with packed instructions
// (fma.rn.f32x2 and friends): the statistics as (mu1, mu2) and (E[x^2]+E[y^2],
// E[(x-y)^2]), the adjoint maps as (g_mu1, g_es) and (g_ed, g_mu2).  The column
// passes use the window's symmetry (w_k = w_{10-k}): five paired sums, then six
// multiply-adds, which also halves the length of each dependent chain.
//
// Components mode (forward only) writes the two factors of S = l * cs as well:
// the per-octave stage of a multi-scale comparison consumes l, cs and S maps
// and their per-image means.
//
// Gradient mode has two uses:
//   training forward: the gradient fields of mean[n] itself (dL = 1) go to the
//                     caller's `saved` buffer, and the mean is reduced too;
//   recompute backward: the fields times dL[n] go to grad_img1 / grad_img2.
#include <cudaTypedefs.h>
#include <mutex>

#include <climits>

#include "common.cuh"
#include "ssim2d.cuh"

namespace gbssim {
namespace {

constexpr int NT = kThreads2d;         // threads per CTA
constexpr int SW = NT;                 // forward-only mode: statistic columns per strip
constexpr int GW = 116;                // gradient mode: gradient columns per strip
constexpr int SWG = GW + 10;           // gradient mode: statistic columns per strip (<= NT)
constexpr int GSHIFT = 2;              // gradient strips start at column GW * s - GSHIFT
constexpr int IWP = 140;               // float pitch of a staged input row (35 x 16 bytes)
constexpr int STEP = kTaps;            // rows per step = ring length
constexpr int RP = NT + 1;             // float4 pitch of a row of hb (one pad slot)
constexpr int HBUF = STEP * RP + 1;    // hb size in float4
constexpr int KA = 8;                  // columns per adjoint row-pass work item
constexpr int NGA = (GW + KA - 1) / KA;
constexpr int P2 = 130;                // float2 pitch of the adjoint pair planes
constexpr int P1 = 132;                // float pitch of the single adjoint plane
constexpr int CBP = 124;               // float pitch of the chain-rule pixel rows (16-byte rows)
constexpr int CBOFF = 2;               // gradient column jj sits at cb column jj + CBOFF
constexpr int NBUF = 2;                // input row blocks in flight
constexpr int XB = (STEP * IWP + 31) / 32 * 32;   // float stride of a staged block (128-byte multiple)
constexpr int CBB = (STEP * CBP + 31) / 32 * 32;  // float stride of a chain-rule pixel block
constexpr long long kWaitCycles = 1LL << 31;      // staging wait limit (about a second)
constexpr long long kDrainCycles = 1LL << 27;     // after a failed wait: copies still in flight

static_assert(SWG <= NT, "one thread per statistic column");
static_assert(IWP % 4 == 0 && IWP >= SW + 10 && IWP >= GW + 20, "input pitch");
static_assert((NGA - 1) * KA + KA + 9 < P2 && (NGA - 1) * KA + KA + 12 <= P1,
              "adjoint reads stay within a row");
static_assert(CBP % 4 == 0 && CBP >= NGA * KA + CBOFF, "chain-rule pixel pitch");
static_assert((GW - GSHIFT - CBOFF) % 4 == 0 && (GSHIFT + CBOFF) % 4 == 0,
              "chain-rule rows start on a 16-byte boundary (column j0 - CBOFF)");
static_assert((GW - GSHIFT - 10) % 4 == 0 && (GSHIFT + 10) % 4 == 0,
              "gradient strips stage from 16-byte aligned columns");

// Tensor staging.  On the aligned path one thread issues, per row block, two
// tensor copies (img1, img2) of STEP rows x IWP columns at (ic0, first row,
// plane); the copy unit writes zeros for every coordinate outside the image, so
// the halo needs no special case.  Completion is tracked by a transaction
// barrier per buffer (and one for the chain-rule pixels); every wait on one is
// bounded, and a block whose wait runs out stops, records the failure and
// returns NaN as its partial sum.
constexpr unsigned kBlockTx = 2u * STEP * IWP * sizeof(float);
constexpr unsigned kChainTx = 2u * STEP * CBP * sizeof(float);

__device__ unsigned g_staging_status;  // bit 0: a staging wait ran out of time

// Staged rows start at input column ic0, a multiple of 4 in both modes (the
// strips are shifted to make it so): then, when W % 4 == 0 and the images are
// 16-byte aligned, whole rows move as 16-byte cp.async chunks, entirely inside
// or entirely outside the image.  Otherwise a 4-byte path stages them.
__device__ __forceinline__ int stat_shift(int off) { return (4 - (off & 3)) & 3; }

// Shared memory (byte offsets):
//   xs, ys  [NBUF][XB] float               input rows: STEP rows of IWP floats
//   hb      [HBUF] float4                  row-blurred statistics (m1, m2, es, ed)
// gradient mode only:
//   va      [STEP][P2] float2              adjoint column sums (g_f1, g_es)
//   vb2     [STEP][P2] float2              (g_ed, g_f2)         [grad2]
//   vc      [STEP][P1] float               g_ed                 [grad1 only]
//   cbx,cby [CBB] float                    input pixels of this step's gradient rows,
//                                          STEP rows of CBP floats
// Every buffer starts on a 128-byte boundary (tensor-copy destinations).
// Work items of the row passes are numbered row-fastest (item = g * STEP + k),
// so the eight threads of a quarter warp mostly touch eight consecutive rows;
// the odd pitches (in 16-byte units: IWP 35, RP 129, P2 65, P1 33) put those in
// distinct bank groups, and every address inside an item is a base plus a
// compile-time offset.
constexpr size_t round128(size_t b) { return (b + 127) / 128 * 128; }
constexpr size_t kInBytes = size_t(2) * NBUF * XB * sizeof(float);
constexpr size_t kHbBytes = round128(size_t(HBUF) * sizeof(float4));
constexpr size_t kPairPlane = round128(size_t(STEP) * P2 * sizeof(float2));
constexpr size_t kOnePlane = round128(size_t(STEP) * P1 * sizeof(float));
constexpr size_t kCbBytes = size_t(2) * CBB * sizeof(float);

// Dynamic shared memory, plus 128 bytes to align its base.
__host__ __device__ constexpr size_t smem_bytes_for(bool grad, bool g2)
{
    return 128 + kInBytes + kHbBytes +
           (grad ? kPairPlane + (g2 ? kPairPlane : kOnePlane) + kCbBytes : 0);
}
// Three gradient CTAs per SM: 228 KB per SM, 1 KB reserved per CTA, ~0.2 KB static.
static_assert(3 * (smem_bytes_for(true, false) + 1024 + 256) <= 233472,
              "three grad_img1 CTAs fit in an SM's shared memory");

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }
__device__ __forceinline__ float2 splat(float w) { return make_float2(w, w); }
__device__ __forceinline__ float2 lo(const float4 &v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi(const float4 &v) { return make_float2(v.z, v.w); }

// sum_a w_a r[(N + 1 + a) % 11] (the oldest entry gets w_0) through the symmetry
// w_a = w_{10-a}: w_5 r_5 + sum_{a<5} w_a (r_a + r_{10-a}).
template <int N>
__device__ __forceinline__ float2 ring_sum2(const float2 (&r)[kTaps])
{
    float2 acc = __fmul2_rn(splat(tap(5)), r[(N + 6) % kTaps]);
#pragma unroll
    for (int a = 0; a < 5; ++a)
        acc = __ffma2_rn(splat(tap(a)), __fadd2_rn(r[(N + 1 + a) % kTaps], r[(N + 11 - a) % kTaps]),
                         acc);
    return acc;
}

template <int N>
__device__ __forceinline__ float ring_sum1(const float (&r)[kTaps])
{
    float acc = tap(5) * r[(N + 6) % kTaps];
#pragma unroll
    for (int a = 0; a < 5; ++a)
        acc = fmaf(tap(a), r[(N + 1 + a) % kTaps] + r[(N + 11 - a) % kTaps], acc);
    return acc;
}

// The work of block b.  Each plane has `per_plane` blocks over its column strips:
// strips [0, seg_extra) are cut into seg_base + 1 row segments, the others into
// seg_base (the rows split as evenly as integers allow).  Blocks are numbered
// longest segments first (all planes), then the shorter ones, so that the block
// scheduler starts the long ones first and spreads them over the SMs.  `slot`
// numbers the blocks plane by plane: the partial sums of one image are contiguous.
struct SegWork {
    int plane, strip, seg, r0, r1, slot;
};

__device__ __forceinline__ SegWork segment_of(const Ssim2dArgs &a, int b)
{
    const int base = a.seg_base, extra = a.seg_extra;
    const int nl = (a.strips - extra) * base;  // blocks with base segments, per plane
    const int ns = extra * (base + 1);         // blocks with base + 1 segments, per plane
    SegWork w;
    int r, nseg;
    if (b < a.long_blocks) {
        w.plane = b / nl;
        r = b - w.plane * nl;
        w.strip = extra + r / base;
        w.seg = r - (w.strip - extra) * base;
        nseg = base;
        w.slot = w.plane * a.per_plane + ns + r;
    } else {
        const int b2 = b - a.long_blocks;
        w.plane = b2 / ns;
        r = b2 - w.plane * ns;
        w.strip = r / (base + 1);
        w.seg = r - w.strip * (base + 1);
        nseg = base + 1;
        w.slot = w.plane * a.per_plane + r;
    }
    // boundaries on multiples of STEP rows: a segment's steps then fall on one
    // grid for the whole strip, so each 11-row band and its shifts, and with
    // them every pixel's result, are the same whatever the plan
    const int J = (a.rows + STEP - 1) / STEP;
    w.r0 = min(a.rows, STEP * int((long long)w.seg * J / nseg));
    w.r1 = min(a.rows, STEP * int((long long)(w.seg + 1) * J / nseg));
    return w;
}

// Resident CTAs per SM the kernel is built for: three for the forward-only and
// the grad_img1 kernels (75 KB of shared memory, <= 168 registers), two with grad_img2.
template <bool GRAD, bool G2>
constexpr int min_blocks() { return (GRAD && G2) ? 2 : 3; }

// The work of one block (block = its index in the launch's plan of `a`).  With
// MULTI the block's partial sums are written but the means are left to the
// caller (one finish for several octaves in one launch).
template <bool GRAD, bool G2, bool COMP, bool MULTI, bool DUMP = false>
__device__ __forceinline__ void stream_body(const Ssim2dArgs &a, int block)
{
    static_assert(!(COMP && GRAD), "components mode is forward only");
    static_assert(!DUMP || (GRAD && G2), "the statistics dump runs in gradient mode with grad2");
    // columns per row-pass work item: an item forms the shifted products of its
    // KH + 10 input columns once, so wider items repeat fewer of them (8: each
    // input's products are formed 2.25 times; 4: 3.5 times)
    constexpr int KH = 8;
    constexpr int NGH = SW / KH;
    static_assert(SW % KH == 0, "strip width must be a multiple of the row-pass block");

    extern __shared__ __align__(128) unsigned char smem_dyn[];
    unsigned char *smem_raw = smem_dyn + ((128 - (smem_u32(smem_dyn) & 127)) & 127);
    float *xs = reinterpret_cast<float *>(smem_raw);
    float *ys = xs + NBUF * XB;
    float4 *hb = reinterpret_cast<float4 *>(smem_raw + kInBytes);
    unsigned char *gbase = smem_raw + kInBytes + kHbBytes;
    float2 *va = reinterpret_cast<float2 *>(gbase);
    float2 *vb2 = reinterpret_cast<float2 *>(gbase + kPairPlane);
    float *vc = reinterpret_cast<float *>(gbase + kPairPlane);
    float *cbx = reinterpret_cast<float *>(gbase + kPairPlane + (G2 ? kPairPlane : kOnePlane));
    float *cby = cbx + CBB;
    __shared__ double red[COMP ? 3 : 1][NT / 32];
    __shared__ uint64_t bars[3];  // tensor staging: buffers 0 and 1, chain-rule pixels

    pdl_trigger();
    // launched early (per-octave stage): the kernel ahead wrote our inputs,
    // unless they are the caller's images (no_wait)
    if (!a.no_wait) pdl_wait();
    const int tid = threadIdx.x;
    const SegWork w = segment_of(a, block);
    const int strip = w.strip, seg = w.seg, plane = w.plane;
    const int n = plane / a.C;
    const size_t plane_off = size_t(plane) * size_t(a.H) * size_t(a.W);
    const float *__restrict__ xp = a.x + plane_off;
    const float *__restrict__ yp = a.y + plane_off;

    // Geometry of the walk.  Input row r completes statistic row p = r + off - 10;
    // in gradient mode statistic row p completes gradient row q = p - off = r - 10.
    int j0 = 0, sc0, ic0, R0, nrows, q0 = 0, q1 = 0;
    if (GRAD) {
        j0 = strip * GW - GSHIFT;
        q0 = w.r0;
        q1 = w.r1;
        sc0 = j0 + a.off - 10;
        ic0 = j0 - 10;
        R0 = q0 - 10;
        nrows = q1 - q0 + 20;
    } else {
        sc0 = strip * SW - stat_shift(a.off);
        const int r0 = w.r0, r1 = w.r1;
        ic0 = sc0 - a.off;
        R0 = r0 - a.off;
        nrows = r1 - r0 + 10;
    }
    const int steps = (nrows + STEP - 1) / STEP;
    const int Rend = R0 + nrows;

    // ---- staging of one block of STEP input rows into buffer t % NBUF (zeros outside)
    constexpr int NCOL = GRAD ? GW + 20 : SW + 10;  // input columns a strip needs
    constexpr int NCHK = (NCOL + 3) / 4;            // as 16-byte chunks
    const int cA = ic0 + tid, cB = ic0 + tid + NT;   // 4-byte path: columns tid, tid + NT
    const bool inA = (cA >= 0) && (cA < a.W);
    const bool hasB = (tid + NT) < NCOL;
    const bool inB = hasB && (cB >= 0) && (cB < a.W);
    auto load_block = [&](int t) {
        const int buf = t % NBUF;
        const int rbase = R0 + t * STEP;
        if (a.tma) {
            if (tid == 0) {
                mbar_arrive_expect_tx(&bars[buf], kBlockTx + a.tx_extra);
                tma_load_3d(xs + buf * XB, &a.tm_x, ic0, rbase, plane, &bars[buf]);
                tma_load_3d(ys + buf * XB, &a.tm_y, ic0, rbase, plane, &bars[buf]);
            }
            return;
        }
        if (a.vec16) {
            for (int e = tid; e < STEP * NCHK; e += NT) {
                const int ri = e / NCHK, ch = e - ri * NCHK;
                const int R = rbase + ri, Cc = ic0 + 4 * ch;
                const bool inb = (R >= 0) && (R < a.H) && (Cc >= 0) && (Cc < a.W);
                const size_t gi = inb ? size_t(R) * a.W + Cc : 0;
                const int si = buf * XB + ri * IWP + 4 * ch;
                cp_async16(xs + si, xp + gi, inb);
                cp_async16(ys + si, yp + gi, inb);
            }
            return;
        }
        float *dx = xs + buf * XB + tid;
        float *dy = ys + buf * XB + tid;
#pragma unroll
        for (int ri = 0; ri < STEP; ++ri) {
            const int R = rbase + ri;
            const bool rin = (R >= 0) && (R < a.H);
            const size_t roff = rin ? size_t(R) * a.W : 0;
            const bool okA = rin && inA;
            const size_t gA = okA ? roff + cA : 0;
            cp_async4(dx + ri * IWP, xp + gA, okA);
            cp_async4(dy + ri * IWP, yp + gA, okA);
            if (hasB) {
                const bool okB = rin && inB;
                const size_t gB = okB ? roff + cB : 0;
                cp_async4(dx + ri * IWP + NT, xp + gB, okB);
                cp_async4(dy + ri * IWP + NT, yp + gB, okB);
            }
        }
    };

    // ---- the input pixels of the gradient rows of step t: rows R0 + 11 t - 10 + k,
    //      gradient columns jj at cb column jj + CBOFF (zeros outside the image)
    auto load_chain = [&](int t) {
        const int qb = R0 + t * STEP - 10;
        if (a.tma) {
            if (tid == 0) {
                mbar_arrive_expect_tx(&bars[2], kChainTx + a.tx_extra);
                tma_load_3d(cbx, &a.tm_cx, j0 - CBOFF, qb, plane, &bars[2]);
                tma_load_3d(cby, &a.tm_cy, j0 - CBOFF, qb, plane, &bars[2]);
            }
            return;
        }
        if (a.vec16) {
            // 16-byte chunks from column j0 - CBOFF (a multiple of 4): each chunk
            // entirely inside or outside the image (W % 4 == 0)
            constexpr int NCH = (NGA * KA + CBOFF + 3) / 4;
            for (int e = tid; e < STEP * NCH; e += NT) {
                const int k = e / NCH, ch = e - k * NCH;
                const int q = qb + k, j = j0 - CBOFF + 4 * ch;
                const bool inb = (q >= 0) && (q < a.H) && (j >= 0) && (j < a.W);
                const size_t gi = inb ? size_t(q) * a.W + j : 0;
                cp_async16(cbx + k * CBP + 4 * ch, xp + gi, inb);
                cp_async16(cby + k * CBP + 4 * ch, yp + gi, inb);
            }
            return;
        }
        const int j = j0 + tid;
        const bool cin = (tid < GW) && (j >= 0) && (j < a.W);
        for (int k = 0; k < STEP; ++k) {
            const int q = qb + k;
            const bool inb = cin && (q >= 0) && (q < a.H);
            const size_t gi = inb ? size_t(q) * a.W + j : 0;
            if (tid < GW) {
                cp_async4(cbx + k * CBP + CBOFF + tid, xp + gi, inb);
                cp_async4(cby + k * CBP + CBOFF + tid, yp + gi, inb);
            }
        }
    };

    // ---- the shift (s, t) of the windows of row-pass group g whose statistics
    //      complete in step t: the pixel pair at the first row of block t and
    //      the middle column of the group's input columns, moved into the image
    //      (a block wholly outside the image, all zeros, takes 0).  Every window
    //      of the group that completes in this step lies around that pixel, so
    //      in a flat region the shifted values are close to zero.  H(t) and V(t)
    //      read the same staged element while block t is resident.  The value
    //      is clamped to [0, 1] (NaN gives 0): any shift is exact, and a finite
    //      one keeps a NaN or infinite pixel from reaching windows that do not
    //      contain it (through the ring's rebasing).
    auto shift_of = [&](int t, int g) -> float2 {
        const int rb = R0 + t * STEP;
        const int kk = min(max(rb, 0), a.H - 1) - rb;
        if (kk < 0 || kk >= STEP) return f2(0.f, 0.f);
        const int cc = min(max(ic0 + g * KH + (KH + 9) / 2, 0), a.W - 1) - ic0;
        const int i = (t % NBUF) * XB + kk * IWP + cc;
        return f2(fminf(fmaxf(xs[i], 0.f), 1.f), fminf(fmaxf(ys[i], 0.f), 1.f));
    };
    // Block t lies wholly below the image (only a walk's last block can): its
    // windows' in-image rows are the ones above it, so it keeps the shift of
    // block t - 1 (staged in the other buffer while H(t) runs; V holds it).
    auto below = [&](int t) { return R0 + t * STEP > a.H - 1; };

    // ---- row pass of the statistics: row k of block t, columns [KH g, KH g + KH)
    auto h_item = [&](int t, int item) {
        const int g = item / STEP, k = item - g * STEP;
        const int base = (t % NBUF) * XB + k * IWP + g * KH;  // float4-aligned
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
        const float2 sh = shift_of(below(t) ? t - 1 : t, g);
        float2 accA[KH], accB[KH];  // (m1, m2), (es, ed)
#pragma unroll
        for (int m = 0; m < KH + 10; ++m) {
            // two scalar subtractions: x and y come from different loads, and a
            // packed subtraction would first have to move them into one pair
            const float2 p = f2(xv[m] - sh.x, yv[m] - sh.y);
            const float2 sq = __fmul2_rn(p, p);
            const float dd = p.x - p.y;
            const float2 q = f2(sq.x + sq.y, dd * dd);
#pragma unroll
            for (int o = 0; o < KH; ++o) {
                const int b = m - o;
                if (b < 0 || b > 10) continue;
                const float2 w = splat(tap(b));
                if (b == 0) {
                    accA[o] = __fmul2_rn(w, p);
                    accB[o] = __fmul2_rn(w, q);
                } else {
                    accA[o] = __ffma2_rn(w, p, accA[o]);
                    accB[o] = __ffma2_rn(w, q, accB[o]);
                }
            }
        }
        float4 *dst = hb + k * RP + g * KH;
#pragma unroll
        for (int o = 0; o < KH; ++o)
            dst[o] = make_float4(accA[o].x, accA[o].y, accB[o].x, accB[o].y);
    };

    const float scale = (GRAD && a.dL) ? a.dL[n] * a.inv_count : a.inv_count;

    // ---- row pass of the adjoint for the gradient row of (step a_step, row k), the
    //      chain rule with the prefetched pixels, and the store of the gradient
    int a_step = 0;
    auto a_item = [&](int item) {
        const int g = item / STEP, k = item - g * STEP;
        const int q = R0 + (a_step * STEP) + k - 10;
        if (q < q0 || q >= q1) return;
        float2 accA[KA];             // (B^T g_f1, B^T g_es)
        float2 accB[KA];             // (B^T g_ed, B^T g_f2)    [G2]
        float accC[KA];              // B^T g_ed               [grad1 only]
        const float2 *pa = va + k * P2 + g * KA;   // 16-byte aligned (g * KA even)
#pragma unroll
        for (int m = 0; m < KA + 10; m += 2) {
            const float4 u = *reinterpret_cast<const float4 *>(pa + m);  // columns m, m+1
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float2 v = h ? hi(u) : lo(u);
#pragma unroll
                for (int o = 0; o < KA; ++o) {
                    const int b = m + h - o;
                    if (b < 0 || b > 10) continue;
                    const float2 w = splat(tap(b));
                    accA[o] = (b == 0) ? __fmul2_rn(w, v) : __ffma2_rn(w, v, accA[o]);
                }
            }
        }
        if (G2) {
            const float2 *pq = vb2 + k * P2 + g * KA;
#pragma unroll
            for (int m = 0; m < KA + 10; m += 2) {
                const float4 u = *reinterpret_cast<const float4 *>(pq + m);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float2 v = h ? hi(u) : lo(u);
#pragma unroll
                    for (int o = 0; o < KA; ++o) {
                        const int b = m + h - o;
                        if (b < 0 || b > 10) continue;
                        const float2 w = splat(tap(b));
                        accB[o] = (b == 0) ? __fmul2_rn(w, v) : __ffma2_rn(w, v, accB[o]);
                    }
                }
            }
        } else {
            const float *pc = vc + k * P1 + g * KA;  // 16-byte aligned
#pragma unroll
            for (int m = 0; m < KA + 12; m += 4) {
                const float4 u = *reinterpret_cast<const float4 *>(pc + m);
                const float uv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
#pragma unroll
                    for (int o = 0; o < KA; ++o) {
                        const int b = m + h - o;
                        if (b < 0 || b > 10) continue;
                        accC[o] = (b == 0) ? tap(b) * uv[h] : fmaf(tap(b), uv[h], accC[o]);
                    }
                }
            }
        }
        // chain rule with the prefetched pixels (cb columns jj + CBOFF: 8-byte
        // aligned).  Per window p (shift (s, t)) and pixel r the term is
        //   g_m1 + 2 (x - s) g_es + 2 ((x - s) - (y - t)) g_ed
        //     = g_f1 + 2 (x - 1/2) g_es + 2 (x - y) g_ed,
        // g_f1 being formed with the derivatives (MomentGrads), so the pixels
        // here need no shift.  In a flat window g_ed is of order 1 / C2 and meets x - y,
        // small where the two images agree; g_es is small there.
        const float *px = cbx + k * CBP + CBOFF + g * KA;
        const float *py = cby + k * CBP + CBOFF + g * KA;
        float r1[KA], r2[KA];
#pragma unroll
        for (int o = 0; o < KA; o += 2) {
            const float2 xx = *reinterpret_cast<const float2 *>(px + o);
            const float2 yy = *reinterpret_cast<const float2 *>(py + o);
            const float xv[2] = {xx.x, xx.y};
            const float yv[2] = {yy.x, yy.y};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int oo = o + h;
                const float ged = G2 ? accB[oo].x : accC[oo];
                const float dxy2 = 2.0f * (xv[h] - yv[h]);
                r1[oo] = scale * fmaf(dxy2, ged, fmaf(2.0f * (xv[h] - kShift), accA[oo].y, accA[oo].x));
                if (G2) r2[oo] = scale * fmaf(-dxy2, ged, fmaf(2.0f * (yv[h] - kShift), accA[oo].y, accB[oo].y));
            }
        }
        const size_t rowg = plane_off + size_t(q) * a.W;
        if (a.pair_out) {
            // j0 + KA g is even, W % 4 == 0 and the fields are 8-byte aligned: pairs
            // are 8-byte aligned, inside or outside the image together
#pragma unroll
            for (int o = 0; o < KA; o += 2) {
                const int jj = g * KA + o, j = j0 + jj;
                if (jj < GW && j >= 0 && j < a.W) {
                    *reinterpret_cast<float2 *>(a.out1 + rowg + j) = make_float2(r1[o], r1[o + 1]);
                    if (G2) *reinterpret_cast<float2 *>(a.out2 + rowg + j) = make_float2(r2[o], r2[o + 1]);
                }
            }
        } else {
#pragma unroll
            for (int o = 0; o < KA; ++o) {
                const int jj = g * KA + o, j = j0 + jj;
                if (jj < GW && j >= 0 && j < a.W) {
                    a.out1[rowg + j] = r1[o];
                    if (G2) a.out2[rowg + j] = r2[o];
                }
            }
        }
    };
    // ---- column pass state: registers of thread tid (statistic column sc0 + tid)
    float2 hA[STEP], hB[STEP];   // row-blurred (m1, m2), (es, ed)
    float2 gA[STEP];             // (g_f1, g_es)
    float2 gB[STEP];             // (g_ed, g_f2)    [G2]
    float gC[STEP];              // g_ed            [grad1 only]
#pragma unroll
    for (int k = 0; k < STEP; ++k) {
        hA[k] = hB[k] = gA[k] = gB[k] = f2(0.f, 0.f);
        gC[k] = 0.f;
    }
    const int pc = sc0 + tid;
    const bool col_ok = (tid < (GRAD ? SWG : SW)) && (pc >= 0) && (pc < a.Wo);
    const bool col_own = GRAD ? (tid >= 10 || strip == 0) : true;
    const bool want_mean = (a.partials != nullptr);
    float ssum = 0.0f;
    float lsum = 0.0f, csum = 0.0f;  // components mode: sums of l and cs
    // Columns the strip needs (the last strip of a plane is usually narrower):
    // statistic columns tid < nstat, gradient columns jj < ngrad.  Row-pass
    // groups and column-pass warps wholly beyond them are skipped; the entries
    // they would have written stay at the zeros set below.
    const int nstat = max(0, min(GRAD ? SWG : SW, a.Wo - sc0));
    const int ngrad = GRAD ? max(0, min(GW, a.W - j0)) : 0;
    const int ngh = min(NGH, (nstat + KH - 1) / KH);
    const int nga = min(NGA, (ngrad + KA - 1) / KA);
    const bool v_warp = (tid & ~31) < nstat;
    if (ngh < NGH || (GRAD && nga < NGA)) {
        // hb and the adjoint planes are contiguous
        constexpr int n4 = int((kHbBytes + (GRAD ? kPairPlane + (G2 ? kPairPlane : kOnePlane) : 0)) / 16);
        for (int i = tid; i < n4; i += NT) hb[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    int klo = 0, khi = 0, kown = 0;  // rows k of the current step: valid in [klo, khi), owned from kown
    float2 sh = f2(0.f, 0.f);        // shift of this column's windows completing in the current step

    // The ring's entries of the previous step were formed at that step's shift;
    // move them to the new one (d = old - new): with x' = x - s_old,
    //   E[x' + dx] = m1 + dx,
    //   E[(x' + dx)^2] + E[(y' + dy)^2] = es + dx (2 m1 + dx) + dy (2 m2 + dy),
    //   E[(x' - y' + dd)^2] = ed + dd (2 (m1 - m2) + dd),   dd = dx - dy,
    // exact because every row-pass window's weights sum to one.  The two
    // corrections of es are summed before es is touched: where the old shift was
    // far from the rows' values they nearly cancel es, and one rounding of es
    // plus a term of its size would double the error.  Entry 0 is overwritten by
    // the step's first row before any sum reads it.
    auto rebase_ring = [&](float2 d) {
#pragma unroll
        for (int k = 1; k < STEP; ++k) {
            const float2 m = hA[k];
            const float2 v = __fmul2_rn(__ffma2_rn(f2(2.f, 2.f), m, d), d);
            float2 e = hB[k];
            e.x = e.x + (v.x + v.y);
            const float dd = d.x - d.y;
            e.y = fmaf(dd, fmaf(2.0f, m.x - m.y, dd), e.y);
            hB[k] = e;
            hA[k] = __fadd2_rn(m, d);
        }
    };

    // ---- prologue
    if (a.tma) {
        if (tid == 0) {
            mbar_init(&bars[0], 1);
            mbar_init(&bars[1], 1);
            mbar_init(&bars[2], 1);
            mbar_init_fence();
        }
        __syncthreads();
    }
    int issued_blocks = 0, issued_chains = 0;  // tensor copies issued (uniform)
    load_block(0);
    ++issued_blocks;
    if (GRAD) {
        load_chain(0);
        ++issued_chains;
    }
    cp_async_commit();
    if (steps > 1) {
        load_block(1);
        ++issued_blocks;
    }
    cp_async_commit();
    bool ok = true;
    if (a.tma) ok = mbar_wait_bounded(&bars[0], 0, kWaitCycles);
    else cp_async_wait<0>();
    bool failed = __syncthreads_or(!ok);
    if (!failed) {
        for (int i = tid; i < STEP * ngh; i += NT) h_item(0, i);
        __syncthreads();
    }

    auto v_row = [&](auto K_, int t) {
        constexpr int k = decltype(K_)::value;
        const float4 h = hb[k * RP + tid];
        hA[k] = lo(h);
        hB[k] = hi(h);
        if (k < klo) {
            // warm-up row: its window is not complete; nothing downstream reads
            // its results, only the ring entries must be set
            gA[k] = gB[k] = f2(0.f, 0.f);
            gC[k] = 0.f;
            return;
        }
        const bool ok = col_ok && (k < khi);
        const int p = R0 + t * STEP + k + a.off - 10;
        const float2 M = ring_sum2<k>(hA);
        const float2 E = ring_sum2<k>(hB);
        const Moments mo{M.x, M.y, E.x, E.y};
        if (GRAD) {
            MomentGrads gg;
            const float S = ssim_and_grads<G2>(mo, sh, ok, gg);
            // the first maps come with the window's shift folded in (see
            // MomentGrads and the chain rule in the adjoint row pass)
            gA[k] = f2(gg.g_f1, gg.g_es);
            if (G2) gB[k] = f2(gg.g_ed, gg.g_f2);
            else gC[k] = gg.g_ed;
            const bool own = ok && col_own && (k >= kown);
            if (want_mean) {
                ssum += own ? S : 0.0f;
                if (a.map && own) a.map[(size_t(plane) * a.Ho + p) * a.Wo + pc] = S;
            }
            if (DUMP && own) {
                // the window's statistics and the derivatives of S with respect
                // to the unshifted moments mu1, mu2, E[x^2] (= E[y^2]), E[xy]
                const size_t o = (size_t(plane) * a.Ho + p) * a.Wo + pc;
                // (es and ed each hold E[x^2] + E[y^2] once; ed holds -2 E[xy])
                const float ss = mo.es - (mo.m1 * mo.m1 + mo.m2 * mo.m2);
                const float s12 = fmaf(-mo.m1, mo.m2, 0.5f * (mo.es - mo.ed));
                reinterpret_cast<float4 *>(a.dump_stats)[o] =
                    make_float4(mo.m1 + sh.x, mo.m2 + sh.y, ss, s12);
                // dS/dmu1 = g_f1 - g_es: the chain rule's per-pixel form
                // g_f1 + 2 (x - 1/2) g_es + 2 (x - y) g_ed against the textbook
                // dS/dmu1 + 2 x dS/dE[x^2] + y dS/dE[xy]
                reinterpret_cast<float4 *>(a.dump_grads)[o] =
                    make_float4(gg.g_f1 - gg.g_es, gg.g_f2 - gg.g_es, gg.g_es + gg.g_ed, -2.0f * gg.g_ed);
            }
            va[k * P2 + tid] = ring_sum2<k>(gA);
            if (G2) vb2[k * P2 + tid] = ring_sum2<k>(gB);
            else vc[k * P1 + tid] = ring_sum1<k>(gC);
        } else if (COMP) {
            const float2 lc = ssim_factors(mo, sh);
            const float S = lc.x * lc.y;
            lsum += ok ? lc.x : 0.0f;
            csum += ok ? lc.y : 0.0f;
            ssum += ok ? S : 0.0f;
            if (a.map && ok) {
                float *m = a.map + (size_t(plane) * a.Ho + p) * a.Wo + pc;
                m[0] = lc.x;
                m[a.map_stride] = lc.y;
                m[2 * a.map_stride] = S;
            }
        } else {
            const float S = ssim_value(mo, sh);
            ssum += ok ? S : 0.0f;
            if (a.map && ok) a.map[(size_t(plane) * a.Ho + p) * a.Wo + pc] = S;
        }
    };

    for (int t = 0; t < steps && !failed; ++t) {
        // rows of this step: r = rb + k, statistic row p = r + off - 10
        const int rb = R0 + t * STEP;
        const int pb = rb + a.off - 10;
        klo = max(max(0, R0 + 10 - rb), -pb);
        khi = min(min(STEP, Rend - rb), a.Ho - pb);
        kown = (GRAD && seg != 0) ? q0 + 10 - rb : 0;  // q = r - 10 >= q0
        // ---- V: column passes of step t, at the step's shift
        if (v_warp) {
            const float2 nsh = below(t) ? sh : shift_of(t, tid / KH);
            if (t > 0) rebase_ring(f2(sh.x - nsh.x, sh.y - nsh.y));
            sh = nsh;
            v_row(std::integral_constant<int, 0>{}, t);
            v_row(std::integral_constant<int, 1>{}, t);
            v_row(std::integral_constant<int, 2>{}, t);
            v_row(std::integral_constant<int, 3>{}, t);
            v_row(std::integral_constant<int, 4>{}, t);
            v_row(std::integral_constant<int, 5>{}, t);
            v_row(std::integral_constant<int, 6>{}, t);
            v_row(std::integral_constant<int, 7>{}, t);
            v_row(std::integral_constant<int, 8>{}, t);
            v_row(std::integral_constant<int, 9>{}, t);
            v_row(std::integral_constant<int, 10>{}, t);
        }
        // block t+1 and the chain-rule pixels of step t have landed
        if (a.tma) {
            ok = (t + 1 >= steps) || mbar_wait_bounded(&bars[(t + 1) & 1], ((t + 1) >> 1) & 1, kWaitCycles);
            if (GRAD && ok) ok = mbar_wait_bounded(&bars[2], t & 1, kWaitCycles);
        } else {
            cp_async_wait<0>();
        }
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        // ---- H of step t+1 and A of step t.  The row-pass items are counted in
        //      whole warps so that no warp runs both kinds in one round.
        const int nh = (t + 1 < steps) ? (STEP * ngh + 31) / 32 * 32 : 0;
        const int na = GRAD ? STEP * nga : 0;
        a_step = t;
        for (int i = tid; i < nh + na; i += NT) {
            if (i < nh) {
                if (i < STEP * ngh) h_item(t + 1, i);
            } else {
                a_item(i - nh);
            }
        }
        __syncthreads();
        // block t's buffer (read by H(t) long ago) and cb (just read by A(t)) are free
        if (t + 2 < steps) {
            load_block(t + 2);
            ++issued_blocks;
        }
        if (GRAD && t + 1 < steps) {
            load_chain(t + 1);
            ++issued_chains;
        }
        cp_async_commit();
    }
    cp_async_wait<0>();
    if (failed && tid == 0) {
        // let the tensor copies still in flight land (bounded), then record the failure
        const long long t0 = clock64();
        for (int b = 0; b < 3; ++b) {
            const int n = b < 2 ? (issued_blocks + 1 - b) / 2 : issued_chains;
            const long long left = kDrainCycles - (clock64() - t0);
            if (n > 0 && left > 0) mbar_wait_bounded(&bars[b], (n - 1) & 1, left);
        }
        atomicOr(&g_staging_status, 1u);
    }

    if (want_mean) {
        const double nan = __longlong_as_double(0x7ff8000000000000LL);
        if (COMP) {
            // three sums (l, cs, S); partials and means are [3][...]
            const double tl = block_sum<NT>(lsum, red[0]);
            const double tc = block_sum<NT>(csum, red[1]);
            const double ts = block_sum<NT>(ssum, red[2]);
            if (tid == 0) {
                a.partials[w.slot] = failed ? nan : tl;
                a.partials[a.segments + w.slot] = failed ? nan : tc;
                a.partials[2 * a.segments + w.slot] = failed ? nan : ts;
            }
            if (!MULTI)
                finish_means_k<NT, 3>(a.partials, a.segments, a.counter, a.mean, a.images,
                                      a.blocks_per_image, a.count);
        } else {
            const double tot = block_sum<NT>(ssum, red[0]);
            if (tid == 0) a.partials[w.slot] = failed ? nan : tot;
            finish_means<NT>(a.partials, a.counter, a.mean, a.images, a.blocks_per_image, a.count);
        }
    }
}

// ------------------------------------------------- forward-only split kernel
//
// The forward-only walk (mean and map; components mode: l, cs and S) with the
// two phases of a step on the two warpgroups of a 256-thread CTA, which run at
// the same time:
//   warpgroup 0 (V, one thread per statistic column): the column pass of step
//     t -- the statistic ring, SSIM (or l and cs), the sums and the maps;
//   warpgroup 1 (W): the row pass of step t+1; one of its threads issues the
//     tensor copies, all of them wait for the copies they read.
// One CTA barrier per step; the row-pass results (hb) and the shifts are
// double-buffered across it.  The column pass is a chain of dependent window
// sums and SSIM terms per row, the row pass many independent sums: run side by
// side they fill each other's idle issue slots, where the stream kernel runs
// them one after the other between barriers.  Needs tensor-copy staging (a.tma).
constexpr int NTF = 2 * NT;                                   // threads of a CTA
constexpr size_t kFInBytes = size_t(2) * NBUF * XB * sizeof(float);
constexpr size_t kFSplitSmem = 128 + kFInBytes + 2 * kHbBytes;  // + alignment slack
constexpr int kFSplitBlocks = 3;                              // resident CTAs per SM
static_assert(kFSplitBlocks * (kFSplitSmem + 1024 + 512) <= 233472,
              "three forward split CTAs fit in an SM's shared memory");

template <bool COMP, bool MULTI>
__device__ __forceinline__ void fsplit_body(const Ssim2dArgs &a, int block)
{
    constexpr int KH = 8;  // columns per row-pass work item
    constexpr int NGH = SW / KH;
    static_assert(STEP * NGH >= NT && 2 * (STEP * NGH - NT) <= NT,
                  "a step's row pass is one item per thread plus at most one half item");
    extern __shared__ __align__(128) unsigned char smem_fs[];
    unsigned char *base = smem_fs + ((128 - (smem_u32(smem_fs) & 127)) & 127);
    float *xs = reinterpret_cast<float *>(base);   // [2][XB], tensor-copy destinations
    float *ys = xs + NBUF * XB;                    // [2][XB]
    float4 *hbuf = reinterpret_cast<float4 *>(base + kFInBytes);  // [2][HBUF]
    __shared__ double red[COMP ? 3 : 1][NTF / 32];
    __shared__ uint64_t bars[2];
    __shared__ float2 shifts[2][NGH];

    pdl_trigger();
    if (!a.no_wait) pdl_wait();
    const int tid = threadIdx.x;
    const SegWork w = segment_of(a, block);
    const int plane = w.plane;
    // geometry of the forward walk (as in stream_body): input row r completes
    // statistic row p = r + off - 10
    const int sc0 = w.strip * SW - stat_shift(a.off);
    const int ic0 = sc0 - a.off;
    const int R0 = w.r0 - a.off;
    const int nrows = w.r1 - w.r0 + 10;
    const int steps = (nrows + STEP - 1) / STEP;
    const int Rend = R0 + nrows;
    const int nstat = max(0, min(SW, a.Wo - sc0));
    const int ngh = min(NGH, (nstat + KH - 1) / KH);

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_init_fence();
    }
    if (ngh < NGH) {  // columns no item writes read as zeros
        constexpr int n4 = int(2 * kHbBytes / 16);
        for (int i = tid; i < n4; i += NTF) hbuf[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (tid < 2 * NGH) shifts[tid / NGH][tid % NGH] = f2(0.f, 0.f);
    __syncthreads();

    bool failed = false;
    float ssum = 0.0f, lsum = 0.0f, csum = 0.0f;
    if (tid < NT) {
        // ================================================================ V
        float2 hA[STEP], hB[STEP];
#pragma unroll
        for (int k = 0; k < STEP; ++k) hA[k] = hB[k] = f2(0.f, 0.f);
        const int pc = sc0 + tid;
        const bool col_ok = (pc >= 0) && (pc < a.Wo);
        const bool v_warp = (tid & ~31) < nstat;
        float2 sh = f2(0.f, 0.f);
        int klo = 0, khi = 0;
        const float4 *hb = hbuf;
        auto v_row = [&](auto K_, int t) {
            constexpr int k = decltype(K_)::value;
            const float4 h = hb[k * RP + tid];
            hA[k] = lo(h);
            hB[k] = hi(h);
            if (k < klo) return;  // warm-up row: only the ring entries are needed
            const bool ok = col_ok && (k < khi);
            const int p = R0 + t * STEP + k + a.off - 10;
            const float2 M = ring_sum2<k>(hA);
            const float2 E = ring_sum2<k>(hB);
            const Moments mo{M.x, M.y, E.x, E.y};
            if (COMP) {
                const float2 lc = ssim_factors(mo, sh);
                const float S = lc.x * lc.y;
                lsum += ok ? lc.x : 0.0f;
                csum += ok ? lc.y : 0.0f;
                ssum += ok ? S : 0.0f;
                if (a.map && ok) {
                    float *m = a.map + (size_t(plane) * a.Ho + p) * a.Wo + pc;
                    m[0] = lc.x;
                    m[a.map_stride] = lc.y;
                    m[2 * a.map_stride] = S;
                }
            } else {
                const float S = ssim_value(mo, sh);
                ssum += ok ? S : 0.0f;
                if (a.map && ok) a.map[(size_t(plane) * a.Ho + p) * a.Wo + pc] = S;
            }
        };
        failed = __syncthreads_or(0);  // H(0) is in hb[0]
        for (int t = 0; t < steps && !failed; ++t) {
            if (v_warp) {
                const int rb = R0 + t * STEP;
                const int pb = rb + a.off - 10;
                klo = max(max(0, R0 + 10 - rb), -pb);
                khi = min(min(STEP, Rend - rb), a.Ho - pb);
                hb = hbuf + (t & 1) * (kHbBytes / 16);
                const float2 nsh = shifts[t & 1][tid / KH];
                if (t > 0) {
                    // the ring's entries of step t-1 to this step's shift (see stream_body)
                    const float2 d = f2(sh.x - nsh.x, sh.y - nsh.y);
#pragma unroll
                    for (int k = 1; k < STEP; ++k) {
                        const float2 m = hA[k];
                        const float2 v = __fmul2_rn(__ffma2_rn(f2(2.f, 2.f), m, d), d);
                        float2 e = hB[k];
                        e.x = e.x + (v.x + v.y);
                        const float dd = d.x - d.y;
                        e.y = fmaf(dd, fmaf(2.0f, m.x - m.y, dd), e.y);
                        hB[k] = e;
                        hA[k] = __fadd2_rn(m, d);
                    }
                }
                sh = nsh;
                v_row(std::integral_constant<int, 0>{}, t);
                v_row(std::integral_constant<int, 1>{}, t);
                v_row(std::integral_constant<int, 2>{}, t);
                v_row(std::integral_constant<int, 3>{}, t);
                v_row(std::integral_constant<int, 4>{}, t);
                v_row(std::integral_constant<int, 5>{}, t);
                v_row(std::integral_constant<int, 6>{}, t);
                v_row(std::integral_constant<int, 7>{}, t);
                v_row(std::integral_constant<int, 8>{}, t);
                v_row(std::integral_constant<int, 9>{}, t);
                v_row(std::integral_constant<int, 10>{}, t);
            }
            if (__syncthreads_or(0)) {
                failed = true;
                break;
            }
        }
    } else {
        // ================================================================ W
        const int wt = tid - NT;
        int issued = 0;
        auto load_block = [&](int t) {  // block t into buffer t % 2 (thread wt == 0)
            mbar_arrive_expect_tx(&bars[t & 1], kBlockTx + a.tx_extra);
            tma_load_3d(xs + (t & 1) * XB, &a.tm_x, ic0, R0 + t * STEP, plane, &bars[t & 1]);
            tma_load_3d(ys + (t & 1) * XB, &a.tm_y, ic0, R0 + t * STEP, plane, &bars[t & 1]);
            ++issued;
        };
        // the shift of group g for block t (see stream_body's shift_of)
        // (a block wholly below the image keeps the shift of block t - 1, kept
        // in shifts[(t - 1) % 2])
        auto shift_of = [&](int t, int g) -> float2 {
            const int rb = R0 + t * STEP;
            if (t > 0 && rb > a.H - 1) return shifts[(t - 1) & 1][g];
            const int kk = min(max(rb, 0), a.H - 1) - rb;
            if (kk < 0 || kk >= STEP) return f2(0.f, 0.f);
            const int cc = min(max(ic0 + g * KH + (KH + 9) / 2, 0), a.W - 1) - ic0;
            const int i = (t & 1) * XB + kk * IWP + cc;
            return f2(fminf(fmaxf(xs[i], 0.f), 1.f), fminf(fmaxf(ys[i], 0.f), 1.f));
        };
        // the row pass of KW columns from column c0 (a multiple of 4) of group g,
        // row k of block t
        auto h_cols = [&](auto KW_, int t, int g, int k, int c0) {
            constexpr int KW = decltype(KW_)::value;
            const int base_i = (t & 1) * XB + k * IWP + c0;
            float xv[KW + 10], yv[KW + 10];
#pragma unroll
            for (int m = 0; m < KW + 8; m += 4) {
                const float4 u = *reinterpret_cast<const float4 *>(xs + base_i + m);
                const float4 v = *reinterpret_cast<const float4 *>(ys + base_i + m);
                xv[m] = u.x; xv[m + 1] = u.y; xv[m + 2] = u.z; xv[m + 3] = u.w;
                yv[m] = v.x; yv[m + 1] = v.y; yv[m + 2] = v.z; yv[m + 3] = v.w;
            }
            {
                const float2 u = *reinterpret_cast<const float2 *>(xs + base_i + KW + 8);
                const float2 v = *reinterpret_cast<const float2 *>(ys + base_i + KW + 8);
                xv[KW + 8] = u.x; xv[KW + 9] = u.y;
                yv[KW + 8] = v.x; yv[KW + 9] = v.y;
            }
            const float2 sh = shift_of(t, g);
            if (k == 0 && c0 == g * KH) shifts[t & 1][g] = sh;
            float2 accA[KW], accB[KW];
#pragma unroll
            for (int m = 0; m < KW + 10; ++m) {
                const float2 p = f2(xv[m] - sh.x, yv[m] - sh.y);
                const float2 sq = __fmul2_rn(p, p);
                const float dd = p.x - p.y;
                const float2 q = f2(sq.x + sq.y, dd * dd);
#pragma unroll
                for (int o = 0; o < KW; ++o) {
                    const int b = m - o;
                    if (b < 0 || b > 10) continue;
                    const float2 wt2 = splat(tap(b));
                    if (b == 0) {
                        accA[o] = __fmul2_rn(wt2, p);
                        accB[o] = __fmul2_rn(wt2, q);
                    } else {
                        accA[o] = __ffma2_rn(wt2, p, accA[o]);
                        accB[o] = __ffma2_rn(wt2, q, accB[o]);
                    }
                }
            }
            float4 *dst = hbuf + (t & 1) * (kHbBytes / 16) + k * RP + c0;
#pragma unroll
            for (int o = 0; o < KW; ++o)
                dst[o] = make_float4(accA[o].x, accA[o].y, accB[o].x, accB[o].y);
        };
        // The row pass of block t: items of KH columns x 1 row, one per thread;
        // the items beyond the warpgroup's threads are done as two half items
        // each (4 columns), by threads that rotate with the step and the block,
        // so that the warps' shares of a step differ by half an item at most
        // and no scheduler partition holds the extra work every step.
        auto h_block = [&](int t) {
            const int n_items = STEP * ngh;
            if (wt < n_items) {
                const int g = wt / STEP;
                h_cols(std::integral_constant<int, KH>{}, t, g, wt - g * STEP, g * KH);
            }
            const int n_half = 2 * (n_items - NT);
            if (n_half > 0) {
                const int j = (wt + 32 * ((t + block) & 3)) & (NT - 1);
                if (j < n_half) {
                    const int item = NT + (j >> 1);
                    const int g = item / STEP;
                    h_cols(std::integral_constant<int, KH / 2>{}, t, g, item - g * STEP,
                           g * KH + (j & 1) * (KH / 2));
                }
            }
        };

        if (wt == 0) {
            load_block(0);
        }
        // block 1 goes out once block 0 has landed: issued together, the grid's
        // first two blocks share the HBM queue and block 0 arrives later
        bool ok = mbar_wait_bounded(&bars[0], 0, kWaitCycles);
        if (ok && wt == 0 && steps > 1) load_block(1);
        if (ok) h_block(0);
        failed = __syncthreads_or(!ok);  // H(0) is in hb[0]
        for (int t = 0; t < steps && !failed; ++t) {
            // block t + 2 goes into the buffer H(t) read in the last step
            if (ok && wt == 0 && t + 2 < steps) load_block(t + 2);
            if (ok && t + 1 < steps) {
                ok = mbar_wait_bounded(&bars[(t + 1) & 1], ((t + 1) >> 1) & 1, kWaitCycles);
                if (ok) h_block(t + 1);
            }
            if (__syncthreads_or(!ok)) {
                failed = true;
                break;
            }
        }
        if (failed && wt == 0) {
            // let the tensor copies in flight land (bounded), then record the failure
            const long long t0 = clock64();
            for (int b = 0; b < 2; ++b) {
                const int cnt = (issued + 1 - b) / 2;
                const long long left = kDrainCycles - (clock64() - t0);
                if (cnt > 0 && left > 0) mbar_wait_bounded(&bars[b], (cnt - 1) & 1, left);
            }
            atomicOr(&g_staging_status, 1u);
        }
    }

    if (a.partials != nullptr) {
        const double nan = __longlong_as_double(0x7ff8000000000000LL);
        if (COMP) {
            const double tl = block_sum<NTF>(lsum, red[0]);
            const double tc = block_sum<NTF>(csum, red[1]);
            const double ts = block_sum<NTF>(ssum, red[2]);
            if (tid == 0) {
                a.partials[w.slot] = failed ? nan : tl;
                a.partials[a.segments + w.slot] = failed ? nan : tc;
                a.partials[2 * a.segments + w.slot] = failed ? nan : ts;
            }
            if (!MULTI)
                finish_means_k<NTF, 3>(a.partials, a.segments, a.counter, a.mean, a.images,
                                       a.blocks_per_image, a.count);
        } else {
            const double tot = block_sum<NTF>(ssum, red[0]);
            if (tid == 0) a.partials[w.slot] = failed ? nan : tot;
            finish_means<NTF>(a.partials, a.counter, a.mean, a.images, a.blocks_per_image, a.count);
        }
    }
}

template <bool COMP>
__global__ void __launch_bounds__(NTF, kFSplitBlocks)
    ssim2d_fsplit_kernel(const __grid_constant__ Ssim2dArgs a)
{
    fsplit_body<COMP, false>(a, blockIdx.x);
}

// Components mode for several octaves in one launch (see the stream kernel's).
__global__ void __launch_bounds__(NTF, kFSplitBlocks)
    ssim2d_fsplit_multi_kernel(const __grid_constant__ Ssim2dMulti m)
{
    int o = 0;
    while (o + 1 < m.count && int(blockIdx.x) >= m.first[o + 1]) ++o;
    fsplit_body<true, true>(m.oct[o], int(blockIdx.x) - m.first[o]);
    if (!finish_ticket<NTF>(m.counter)) return;
    for (int k = 0; k < m.count; ++k) {
        const Ssim2dArgs &q = m.oct[k];
        reduce_means_k<NTF, 3>(q.partials, q.segments, q.mean, q.images, q.blocks_per_image,
                               q.count);
    }
    if (threadIdx.x == 0) *m.counter = 0u;
}

template <bool GRAD, bool G2, bool COMP = false>
__global__ void __launch_bounds__(NT, min_blocks<GRAD, G2>())
    ssim2d_stream_kernel(const __grid_constant__ Ssim2dArgs a)
{
    stream_body<GRAD, G2, COMP, false>(a, blockIdx.x);
}

#ifdef GBSSIM_TEST_HOOKS
__global__ void __launch_bounds__(NT, min_blocks<true, true>())
    ssim2d_dump_kernel(const __grid_constant__ Ssim2dArgs a)
{
    stream_body<true, true, false, false, true>(a, blockIdx.x);
}
#endif

// Components mode for several octaves in one launch: block b belongs to the
// octave o with first[o] <= b < first[o + 1]; the last block to finish reduces
// every octave's means.
__global__ void __launch_bounds__(NT, min_blocks<false, false>())
    ssim2d_components_multi_kernel(const __grid_constant__ Ssim2dMulti m)
{
    int o = 0;
    while (o + 1 < m.count && int(blockIdx.x) >= m.first[o + 1]) ++o;
    stream_body<false, false, true, true>(m.oct[o], int(blockIdx.x) - m.first[o]);
    if (!finish_ticket<NT>(m.counter)) return;
    for (int k = 0; k < m.count; ++k) {
        const Ssim2dArgs &q = m.oct[k];
        reduce_means_k<NT, 3>(q.partials, q.segments, q.mean, q.images, q.blocks_per_image, q.count);
    }
    if (threadIdx.x == 0) *m.counter = 0u;
}

// grad = field * dL[n] / count, elementwise; n = index / per_image.
// A field may be scaled in place (g == f).
__global__ void __launch_bounds__(256) scale_fields_vec4(const float4 *f1, const float4 *f2,
                                                         float4 *g1, float4 *g2,
                                                         const float *__restrict__ dL,
                                                         float inv_count, size_t per_image4,
                                                         size_t total4)
{
    pdl_wait();
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
    pdl_wait();
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += size_t(gridDim.x) * blockDim.x) {
        const float s = dL[i / per_image] * inv_count;
        g1[i] = f1[i] * s;
        if (g2) g2[i] = f2[i] * s;
    }
}

size_t smem_bytes(bool grad, bool g2) { return smem_bytes_for(grad, g2); }

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

// [planes][H][W] float32 at ptr; box of `rows` rows x `cols` columns of one plane;
// out-of-range elements read as zeros.
bool encode_rows_map(CUtensorMap &m, const float *ptr, long long planes, int H, int W, int cols,
                     int rows)
{
    const auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {cuuint64_t(W), cuuint64_t(H), cuuint64_t(planes)};
    const cuuint64_t strides[2] = {cuuint64_t(W) * sizeof(float),
                                   cuuint64_t(H) * cuuint64_t(W) * sizeof(float)};
    const cuuint32_t box[3] = {cuuint32_t(cols), cuuint32_t(rows), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool GRAD, bool G2, bool COMP = false>
cudaError_t launch_stream(const Ssim2dArgs &a, int blocks, cudaStream_t s, bool early = false)
{
    if (!early) {
        ssim2d_stream_kernel<GRAD, G2, COMP><<<blocks, NT, smem_bytes(GRAD, G2), s>>>(a);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = smem_bytes(GRAD, G2);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, ssim2d_stream_kernel<GRAD, G2, COMP>, a);
}

// Octaves lo + 1 .. lo + levels of both images from octave lo, levels <= 5:
// out(i, j) = mean of the in-range pixels of the 2x2 block at (2i, 2j) of the
// octave above (extents ceil(H / 2) x ceil(W / 2)), summed in the order
// (0,0), (0,1), (1,0), (1,1).  A block owns a kChainTile x kChainTile * kChainG
// tile of octave lo (rows and columns at multiples of the tile), so the tiles
// of every lower octave lie inside it: each thread forms kChainG pixels of
// octave lo + 1 straight from global memory, the later octaves are formed
// level by level in shared memory.  With wait_first the kernel ahead on the
// stream wrote octave lo; otherwise octave lo is an input and this launch runs
// beside the kernel ahead, its blocks taking the SM slots that kernel's blocks
// leave; block 0 alone waits for that kernel before it exits, so that this
// launch completes after it (the launch behind waits for this one) while the
// other blocks leave their slots as soon as their tiles are done.
// The (up to) four pixels of a 2x2 block of one image: q[0], q[1] of row r
// and q[2], q[3] of row r + 1; only in-range ones are loaded.
struct Quad {
    float v[4];
};

__device__ __forceinline__ Quad load_quad(const float *__restrict__ p, int W, int r, int c, bool r1,
                                          bool c1, bool pair)
{
    Quad q{{0.f, 0.f, 0.f, 0.f}};
    const float *a = p + size_t(r) * W + c;
    if (pair) {
        const float2 u = __ldg(reinterpret_cast<const float2 *>(a));
        q.v[0] = u.x; q.v[1] = u.y;
        if (r1) {
            const float2 w = __ldg(reinterpret_cast<const float2 *>(a + W));
            q.v[2] = w.x; q.v[3] = w.y;
        }
        return q;
    }
    q.v[0] = __ldg(a);
    if (c1) q.v[1] = __ldg(a + 1);
    if (r1) {
        q.v[2] = __ldg(a + W);
        if (c1) q.v[3] = __ldg(a + W + 1);
    }
    return q;
}

// Sum in the order (0,0), (0,1), (1,0), (1,1) of the in-range pixels.
__device__ __forceinline__ float quad_sum(const Quad &q, bool r1, bool c1)
{
    float s = q.v[0];
    if (c1) s += q.v[1];
    if (r1) {
        s += q.v[2];
        if (c1) s += q.v[3];
    }
    return s;
}

__global__ void __launch_bounds__(256) octave_chain_kernel(const __grid_constant__ OctaveChainArgs m)
{
    constexpr int R1 = kChainTile / 2, C1 = kChainTile * kChainG / 2;  // octave lo + 1 tile
    __shared__ float buf[2][2][R1][C1 + 1];                            // [ping][image][row][col]
    // the launch behind may start once every block is past this point, i.e.
    // after the kernel ahead completed (with wait_first)
    if (m.wait_first) pdl_wait();
    pdl_trigger();
    const int tiles = m.tiles_x * m.tiles_y;
    const long long plane = blockIdx.x / tiles;
    const int t = int(blockIdx.x - plane * tiles);
    const int ty = t / m.tiles_x, tx = t - ty * m.tiles_x;
    {
        const int H0 = m.H[0], W0 = m.W[0], H1 = m.H[1], W1 = m.W[1];
        const float *__restrict__ px = m.x + size_t(plane) * H0 * W0;
        const float *__restrict__ py = m.y + size_t(plane) * H0 * W0;
        const bool even = (W0 % 2 == 0) && ((reinterpret_cast<uintptr_t>(m.x) |
                                              reinterpret_cast<uintptr_t>(m.y)) % 8 == 0);
        const int i = threadIdx.x / 16, gi = ty * R1 + i;
        // every load of the thread first, then the sums and stores
        Quad qx[kChainG], qy[kChainG];
#pragma unroll
        for (int k = 0; k < kChainG; ++k) {
            const int gj = tx * C1 + threadIdx.x % 16 + 16 * k;
            const bool in = (gi < H1) && (gj < W1);
            const bool r1 = 2 * gi + 1 < H0, c1 = 2 * gj + 1 < W0;
            qx[k] = in ? load_quad(px, W0, 2 * gi, 2 * gj, r1, c1, even && c1) : Quad{{0.f, 0.f, 0.f, 0.f}};
            qy[k] = in ? load_quad(py, W0, 2 * gi, 2 * gj, r1, c1, even && c1) : Quad{{0.f, 0.f, 0.f, 0.f}};
        }
#pragma unroll
        for (int k = 0; k < kChainG; ++k) {
            const int j = threadIdx.x % 16 + 16 * k;
            const int gj = tx * C1 + j;
            float sx = 0.0f, sy = 0.0f;
            if (gi < H1 && gj < W1) {
                const bool r1 = 2 * gi + 1 < H0, c1 = 2 * gj + 1 < W0;
                const float inv = (r1 && c1) ? 0.25f : ((r1 || c1) ? 0.5f : 1.0f);
                sx = quad_sum(qx[k], r1, c1) * inv;
                sy = quad_sum(qy[k], r1, c1) * inv;
                const size_t gidx = (size_t(plane) * H1 + gi) * W1 + gj;
                m.ox[0][gidx] = sx;
                m.oy[0][gidx] = sy;
            }
            buf[0][0][i][j] = sx;
            buf[0][1][i][j] = sy;
        }
    }
    __syncthreads();
    int cur = 0;
    for (int l = 2; l <= m.levels; ++l) {
        const int nr = R1 >> (l - 1), nc = C1 >> (l - 1);  // tile extent at level l
        const int Hp = m.H[l - 1], Wp = m.W[l - 1], Hl = m.H[l], Wl = m.W[l];
        float *ox = m.ox[l - 1], *oy = m.oy[l - 1];
        for (int e = threadIdx.x; e < nr * nc; e += blockDim.x) {
            const int i = e / nc, j = e - i * nc;
            const int gi = ty * nr + i, gj = tx * nc + j;
            float sx = 0.0f, sy = 0.0f;
            if (gi < Hl && gj < Wl) {
                const int r0 = 2 * i, c0 = 2 * j;
                const bool r1 = 2 * gi + 1 < Hp, c1 = 2 * gj + 1 < Wp;
                sx = buf[cur][0][r0][c0];
                sy = buf[cur][1][r0][c0];
                if (c1) { sx += buf[cur][0][r0][c0 + 1]; sy += buf[cur][1][r0][c0 + 1]; }
                if (r1) {
                    sx += buf[cur][0][r0 + 1][c0]; sy += buf[cur][1][r0 + 1][c0];
                    if (c1) { sx += buf[cur][0][r0 + 1][c0 + 1]; sy += buf[cur][1][r0 + 1][c0 + 1]; }
                }
                const float inv = (r1 && c1) ? 0.25f : ((r1 || c1) ? 0.5f : 1.0f);
                sx *= inv;
                sy *= inv;
                const size_t gidx = (size_t(plane) * Hl + gi) * Wl + gj;
                ox[gidx] = sx;
                oy[gidx] = sy;
            }
            buf[cur ^ 1][0][i][j] = sx;
            buf[cur ^ 1][1][i][j] = sy;
        }
        __syncthreads();
        cur ^= 1;
    }
    if (m.wait_first || blockIdx.x == 0) pdl_wait();
}

}  // namespace

size_t ssim2d_smem_bytes(bool grad, bool g2) { return smem_bytes(grad, g2); }

int g_staging_mode = 0;

void ssim2d_prepare_staging(Ssim2dArgs &a, long long planes, bool grad)
{
    // the maps need 16-byte aligned bases and row pitches (a.vec16) and strides
    // below 2^40 bytes
    const unsigned long long plane_bytes = (unsigned long long)a.H * a.W * sizeof(float);
    bool ok = g_staging_mode != 1 && a.vec16 && plane_bytes < (1ULL << 40) && planes < (1LL << 31);
    ok = ok && encode_rows_map(a.tm_x, a.x, planes, a.H, a.W, IWP, STEP) &&
         encode_rows_map(a.tm_y, a.y, planes, a.H, a.W, IWP, STEP);
    if (ok && grad)
        ok = encode_rows_map(a.tm_cx, a.x, planes, a.H, a.W, CBP, STEP) &&
             encode_rows_map(a.tm_cy, a.y, planes, a.H, a.W, CBP, STEP);
    a.tma = ok ? 1 : 0;
    a.tx_extra = (ok && g_staging_mode == 2) ? 16u : 0u;
}

void ssim2d_set_staging_mode(int mode) { g_staging_mode = (mode >= 0 && mode <= 2) ? mode : 0; }

int staging_mode() { return g_staging_mode; }

bool encode_tiled_f32(CUtensorMap &m, const void *ptr, int rank, const unsigned long long *dims,
                      const unsigned long long *strides, const unsigned *box)
{
    const auto enc = tensor_map_encoder();
    if (!enc || rank < 1 || rank > 5) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], e[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        e[i] = 1;
        if (i + 1 < rank) st[i] = strides[i];
    }
    return enc(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, cuuint32_t(rank), const_cast<void *>(ptr), d,
               st, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t ssim2d_staging_status(unsigned *flags, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_staging_status, sizeof(unsigned));
    if (e == cudaSuccess && clear) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_staging_status, &zero, sizeof(unsigned));
    }
    return e;
}

int ssim2d_strips(bool grad, int W, int Wo, int off)
{
    if (grad) return (W + GSHIFT + GW - 1) / GW;
    const int shift = (4 - (off & 3)) & 3;
    return (Wo + shift + SW - 1) / SW;
}

const void *ssim2d_kernel_ptr(bool grad, bool g2)
{
    if (!grad) return reinterpret_cast<const void *>(ssim2d_stream_kernel<false, false>);
    return g2 ? reinterpret_cast<const void *>(ssim2d_stream_kernel<true, true>)
              : reinterpret_cast<const void *>(ssim2d_stream_kernel<true, false>);
}

cudaError_t ssim2d_components_launch(const Ssim2dArgs &a, int blocks, cudaStream_t s, bool early)
{
    return launch_stream<false, false, true>(a, blocks, s, early);
}

const void *ssim2d_components_kernel_ptr()
{
    return reinterpret_cast<const void *>(ssim2d_stream_kernel<false, false, true>);
}

cudaError_t octave_chain_launch(const OctaveChainArgs &m, cudaStream_t s)
{
    const long long blocks = m.planes * m.tiles_x * m.tiles_y;
    if (blocks > INT_MAX) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, octave_chain_kernel, m);
}

cudaError_t ssim2d_components_multi_launch(const Ssim2dMulti &m, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(m.first[m.count]));
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = smem_bytes(false, false);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, ssim2d_components_multi_kernel, m);
}

const void *ssim2d_components_multi_kernel_ptr()
{
    return reinterpret_cast<const void *>(ssim2d_components_multi_kernel);
}

#ifdef GBSSIM_TEST_HOOKS
cudaError_t ssim2d_dump_launch(const Ssim2dArgs &a, int blocks, cudaStream_t s)
{
    const size_t smem = smem_bytes(true, true);
    const cudaError_t e =
        cudaFuncSetAttribute(ssim2d_dump_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    ssim2d_dump_kernel<<<blocks, NT, smem, s>>>(a);
    return cudaGetLastError();
}
#endif

size_t ssim2d_fsplit_smem_bytes() { return kFSplitSmem; }

const void *ssim2d_fsplit_kernel_ptr(int kind)
{
    if (kind == 0) return reinterpret_cast<const void *>(ssim2d_fsplit_kernel<false>);
    if (kind == 1) return reinterpret_cast<const void *>(ssim2d_fsplit_kernel<true>);
    return reinterpret_cast<const void *>(ssim2d_fsplit_multi_kernel);
}

cudaError_t ssim2d_fsplit_launch(const Ssim2dArgs &a, bool comp, int blocks, cudaStream_t s,
                                 bool early)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(NTF);
    cfg.dynamicSmemBytes = kFSplitSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 1 : 0;
    return comp ? cudaLaunchKernelEx(&cfg, ssim2d_fsplit_kernel<true>, a)
                : cudaLaunchKernelEx(&cfg, ssim2d_fsplit_kernel<false>, a);
}

cudaError_t ssim2d_fsplit_multi_launch(const Ssim2dMulti &m, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(m.first[m.count]));
    cfg.blockDim = dim3(NTF);
    cfg.dynamicSmemBytes = kFSplitSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, ssim2d_fsplit_multi_kernel, m);
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
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (vec)
        return cudaLaunchKernelEx(&cfg, scale_fields_vec4, reinterpret_cast<const float4 *>(f1),
                                  reinterpret_cast<const float4 *>(f2), reinterpret_cast<float4 *>(g1),
                                  reinterpret_cast<float4 *>(g2), dL, inv_count, per_image / 4,
                                  total / 4);
    return cudaLaunchKernelEx(&cfg, scale_fields_scalar, f1, f2, g1, g2, dL, inv_count, per_image,
                              total);
}

}  // namespace gbssim
