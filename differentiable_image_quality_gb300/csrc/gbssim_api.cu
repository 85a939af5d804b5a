// The C ABI (include/gbssim.h): argument checks, launch planning, dispatch.
// Host code only; every step of the computation runs in the kernels.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <mutex>
#include <queue>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "gbssim.h"
#include "common.cuh"
#include "ssim2d.cuh"
#include "ssim3d.cuh"

namespace {

using namespace gbssim;

constexpr int kMaxDevices = 64;
constexpr int kMinSegRows = 22;    // shortest row segment of a gradient-mode plan
constexpr int kMinSegRowsFwd = 11; // ... and of a forward-only plan (small images: more blocks)
constexpr size_t kCounterBytes = 256;  // completion counter, then the partial sums

struct DeviceInfo {
    bool ready = false;
    int sm_count = 0;
    int occ2d[3] = {0, 0, 0};  // resident CTAs per SM: forward, gradient, gradient + grad2
    int occ_comp = 0;          // components mode of the forward
    int occ_multi = 0;         // ... several octaves in one launch
    int occ_fsplit[3] = {0, 0, 0};  // forward split kernels: forward, components, several octaves
    int occ3d[5] = {0, 0, 0, 0, 0};  // 3D: xy; z forward, gradient, + grad2; adjoint
};

// An NVTX range named after the entry point, open for the call's host-side work
// (argument checks, planning, launches), so that a profiler's timeline shows
// which call issued which kernels.  With no profiler attached both NVTX calls
// return at once.
struct CallRange {
    explicit CallRange(const char *name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
    CallRange(const CallRange &) = delete;
    CallRange &operator=(const CallRange &) = delete;
};

std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];
int g_seg_rows_override = 0;  // tuning: 0 = planner's choice

int cuda_fail(cudaError_t e)
{
    (void)cudaGetLastError();  // clear a sticky launch error so the next call starts clean
    return e == cudaSuccess ? GBSSIM_OK : GBSSIM_ECUDA;
}

// Per-device launch facts, filled once per device with that device current.
int device_info(DeviceInfo **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return cuda_fail(cudaErrorInvalidDevice);
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return cuda_fail(cudaErrorInvalidDevice);
        const bool grad[3] = {false, true, true}, g2[3] = {false, false, true};
        for (int i = 0; i < 3; ++i) {
            const void *k = ssim2d_kernel_ptr(grad[i], g2[i]);
            const size_t smem = ssim2d_smem_bytes(grad[i], g2[i]);
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 int(smem));
            if (e != cudaSuccess) return cuda_fail(e);
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.occ2d[i], k, kThreads2d, smem);
            if (e != cudaSuccess) return cuda_fail(e);
            if (d.occ2d[i] < 1) return cuda_fail(cudaErrorInvalidConfiguration);
        }
        for (int multi = 0; multi < 2; ++multi) {
            const void *k = multi ? ssim2d_components_multi_kernel_ptr()
                                  : ssim2d_components_kernel_ptr();
            const size_t smem = ssim2d_smem_bytes(false, false);
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 int(smem));
            if (e != cudaSuccess) return cuda_fail(e);
            int occ = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kThreads2d, smem);
            if (e != cudaSuccess) return cuda_fail(e);
            if (occ < 1) return cuda_fail(cudaErrorInvalidConfiguration);
            (multi ? d.occ_multi : d.occ_comp) = occ;
        }
        for (int kind = 0; kind < 3; ++kind) {
            const void *k = ssim2d_fsplit_kernel_ptr(kind);
            const size_t smem = ssim2d_fsplit_smem_bytes();
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 int(smem));
            if (e != cudaSuccess) return cuda_fail(e);
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.occ_fsplit[kind], k,
                                                              kThreads2dFsplit, smem);
            if (e != cudaSuccess) return cuda_fail(e);
            if (d.occ_fsplit[kind] < 1) return cuda_fail(cudaErrorInvalidConfiguration);
        }
        const cudaError_t e3 = ssim3d_prepare(d.occ3d);
        if (e3 != cudaSuccess) return cuda_fail(e3);
        d.ready = true;
    }
    *out = &d;
    return GBSSIM_OK;
}

int check_in(const void *p)
{
    if (!p) return GBSSIM_EINVAL;
    if (reinterpret_cast<uintptr_t>(p) % 4 != 0) return GBSSIM_EALIGN;
    return GBSSIM_OK;
}

int check_opt(const void *p) { return p ? check_in(p) : GBSSIM_OK; }

int extent_ok(int n, int padding)
{
    if (padding == GBSSIM_VALID) return n >= kTaps;
    if (padding == GBSSIM_SAME_ZERO) return n >= 1;
    return 0;
}

int out_extent(int n, int padding) { return padding == GBSSIM_VALID ? n - (kTaps - 1) : n; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    if (!a || !b) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// Launch plan of the 2D streaming kernel: per plane, `per_plane` blocks over the
// column strips; strips [0, extra) get base + 1 row segments, the rest base.
struct Plan2d {
    int strips = 0, per_plane = 0, base = 0, extra = 0;
    long long blocks = 0, long_blocks = 0;
};

// Relative SM throughput with k resident CTAs (k = 1, 2, 3, 4+), measured on the
// 1080p workload: one 4-warp CTA alone leaves the SM about half idle.
double occupancy_eff(int k)
{
    static const double e[4] = {0.5, 0.8, 1.0, 1.05};
    return e[k < 1 ? 0 : (k > 4 ? 3 : k - 1)];
}

// Time of `blocks` equal CTAs of `steps` row steps each, in units of one
// CTA-step at full occupancy: the grid runs in waves of SMs x occ CTAs; a wave
// whose busiest SM holds k CTAs takes k (steps + 1) / eff(k) (the +1 is a CTA's
// fixed start-up and finish).
double wave_cost(long long blocks, long long steps, int sm_count, int occ)
{
    const long long slots = (long long)sm_count * occ;
    double cost = 0.0;
    while (blocks > 0) {
        const long long in_wave = blocks < slots ? blocks : slots;
        const int k = int(ceil_div(in_wave, sm_count));
        cost += double(k) * double(steps + 1) / occupancy_eff(k);
        blocks -= in_wave;
    }
    return cost;
}

// Same units for CTAs of two lengths that fit in one wave (blocks <= SMs x occ):
// the long ones are issued first, one per SM in turn, then each short one goes
// to the least loaded SM (the block scheduler fills free slots in order).
double one_wave_cost(long long n_long, long long s_long, long long n_short, long long s_short,
                     int sm_count)
{
    std::vector<long long> load(size_t(sm_count), 0), cnt(size_t(sm_count), 0);
    for (long long i = 0; i < n_long; ++i) {
        load[size_t(i % sm_count)] += s_long + 1;
        ++cnt[size_t(i % sm_count)];
    }
    // (load, SM) min-heap: ties go to the lower-numbered SM
    using Entry = std::pair<long long, int>;
    std::priority_queue<Entry, std::vector<Entry>, std::greater<Entry>> heap;
    for (int j = 0; j < sm_count; ++j) heap.push({load[size_t(j)], j});
    for (long long i = 0; i < n_short; ++i) {
        const Entry e = heap.top();
        heap.pop();
        load[size_t(e.second)] += s_short + 1;
        ++cnt[size_t(e.second)];
        heap.push({load[size_t(e.second)], e.second});
    }
    double worst = 0.0;
    for (size_t j = 0; j < load.size(); ++j)
        if (cnt[j]) worst = std::max(worst, double(load[j]) / occupancy_eff(int(cnt[j])));
    return worst;
}

long long seg_steps(int rows, int nseg, int halo)
{
    return ceil_div(ceil_div(rows, nseg) + halo, kTaps);
}

// Pick the segmentation.  Candidates: every strip with s segments (s = 1 ..
// rows / kMinSegRows), costed by the wave model; and the largest per-plane count
// that still fits one wave, with the strips' segment counts differing by one
// (the last strip of a plane, usually the narrowest, gets the fewer), costed by
// one_wave_cost.  A gradient-mode segment walks its rows + 20, a forward-only
// one its rows + 10.
Plan2d plan2d(long long planes, int H, int W, int Ho, int Wo, int off, bool grad, int sm_count,
              int occ)
{
    Plan2d p;
    const int rows = grad ? H : Ho;
    const int halo = grad ? 20 : 10;
    const int S = ssim2d_strips(grad, W, Wo, off);
    p.strips = S;
    const int max_segs = std::max(1, rows / (grad ? kMinSegRows : kMinSegRowsFwd));
    auto take = [&](int per_plane) {
        p.per_plane = per_plane;
        p.base = per_plane / S;
        p.extra = per_plane % S;
        p.blocks = planes * per_plane;
        p.long_blocks = planes * (S - p.extra) * p.base;
    };
    if (g_seg_rows_override > 0) {
        take(S * int(ceil_div(rows, std::min(g_seg_rows_override, rows))));
        return p;
    }
    double best = -1.0;
    long long best_work = 0;
    int best_k = S;
    for (int s = 1; s <= max_segs; ++s) {
        const long long blocks = (long long)S * planes * s;
        const long long steps = seg_steps(rows, s, halo);
        const double cost = wave_cost(blocks, steps, sm_count, occ);
        const long long work = blocks * steps;
        if (best < 0 || cost < best - 1e-9 || (cost <= best + 1e-9 && work < best_work)) {
            best = cost;
            best_work = work;
            best_k = S * s;
        }
    }
    const long long slots = (long long)sm_count * occ;
    const long long fill = slots / planes;  // blocks per plane that fill one wave
    if (fill > S && fill < (long long)S * max_segs && fill % S != 0) {
        const int k = int(fill), base = k / S, extra = k % S;
        const double cost = one_wave_cost(planes * (S - extra) * base, seg_steps(rows, base, halo),
                                          planes * extra * (base + 1),
                                          seg_steps(rows, base + 1, halo), sm_count);
        if (cost < best - 1e-9) best_k = k;
    }
    take(best_k);
    return p;
}

// A forward-mode plan of about `target` blocks: every strip of every plane cut
// into the same number of row segments (within the planner's limits).
Plan2d plan2d_blocks(long long planes, int Ho, int Wo, int off, long long target)
{
    Plan2d p;
    const int S = ssim2d_strips(false, 0, Wo, off);  // forward strips depend on Wo only
    p.strips = S;
    const int max_segs = std::max(1, Ho / kMinSegRowsFwd);
    long long per_plane = target / planes;
    per_plane = std::max<long long>(S, std::min<long long>(per_plane, (long long)S * max_segs));
    p.per_plane = int(per_plane);
    p.base = p.per_plane / S;
    p.extra = p.per_plane % S;
    p.blocks = planes * p.per_plane;
    p.long_blocks = planes * (S - p.extra) * p.base;
    return p;
}

// The planner's results for recent shapes (it runs a small simulation): a
// direct-mapped cache keyed by everything plan2d reads.
struct PlanKey {
    long long planes;
    int H, W, Ho, Wo, off, grad, sm_count, occ, override_rows;
    bool operator==(const PlanKey &o) const
    {
        return planes == o.planes && H == o.H && W == o.W && Ho == o.Ho && Wo == o.Wo &&
               off == o.off && grad == o.grad && sm_count == o.sm_count && occ == o.occ &&
               override_rows == o.override_rows;
    }
};

Plan2d cached_plan2d(long long planes, int H, int W, int Ho, int Wo, int off, bool grad,
                     int sm_count, int occ)
{
    constexpr int kSlots = 32;
    static PlanKey keys[kSlots];
    static Plan2d plans[kSlots];
    static bool used[kSlots] = {};
    static std::mutex m;
    const int mode = grad ? 1 : 0;
    const PlanKey k{planes, H, W, Ho, Wo, off, mode, sm_count, occ, g_seg_rows_override};
    const size_t h = (size_t(planes) * 1000003u + size_t(H) * 10007u + size_t(W) * 101u +
                      size_t(off) * 7u + size_t(mode) * 3u + size_t(occ)) % kSlots;
    {
        std::lock_guard<std::mutex> lock(m);
        if (used[h] && keys[h] == k) return plans[h];
    }
    const Plan2d p = plan2d(planes, H, W, Ho, Wo, off, grad, sm_count, occ);
    std::lock_guard<std::mutex> lock(m);
    keys[h] = k;
    plans[h] = p;
    used[h] = true;
    return p;
}

void set_segments(Ssim2dArgs &a, const Plan2d &p, int rows)
{
    a.strips = p.strips;
    a.rows = rows;
    a.per_plane = p.per_plane;
    a.seg_base = p.base;
    a.seg_extra = p.extra;
    a.long_blocks = int(p.long_blocks);
}

bool g_fsplit_enabled = true;  // test build: the stream kernel can be forced for the forward

// The gradient-mode launch of a 2D call whose arguments are filled in except
// the segmentation.  With a.partials set, the workspace must hold the plan's
// partial sums.
int launch_grad2d(Ssim2dArgs &a, const DeviceInfo *d, int N, bool g2, size_t workspace_bytes,
                  cudaStream_t s)
{
    const long long planes = (long long)N * a.C;
    a.pair_out = a.vec16 && (reinterpret_cast<uintptr_t>(a.out1) % 8 == 0) &&
                 (reinterpret_cast<uintptr_t>(a.out2) % 8 == 0);
    const Plan2d p = cached_plan2d(planes, a.H, a.W, a.Ho, a.Wo, a.off, true, d->sm_count,
                                   d->occ2d[g2 ? 2 : 1]);
    if (p.blocks > INT_MAX) return GBSSIM_ESHAPE;
    if (a.partials && workspace_bytes < kCounterBytes + size_t(p.blocks) * sizeof(double))
        return GBSSIM_EWORKSPACE;
    set_segments(a, p, a.H);
    a.images = N;
    a.blocks_per_image = int(p.blocks / N);
    return cuda_fail(ssim2d_launch(a, true, g2, int(p.blocks), s));
}

// Upper bound of blocks over every plan (segments never shorter than the minima).
long long max_blocks2d(long long planes, int H, int W, int Ho, int Wo, int off)
{
    const long long g = ssim2d_strips(true, W, Wo, off) * ceil_div(H, kMinSegRows);
    const long long f = ssim2d_strips(false, W, Wo, off) * ceil_div(Ho, kMinSegRowsFwd);
    return planes * (g > f ? g : f);
}

bool shape2d_ok(int N, int C, int H, int W, int padding)
{
    if (N < 1 || C < 1) return false;
    if (padding != GBSSIM_VALID && padding != GBSSIM_SAME_ZERO) return false;
    if (!extent_ok(H, padding) || !extent_ok(W, padding)) return false;
    if ((long long)N * C > INT_MAX) return false;
    if (H > (1 << 28) || W > (1 << 28)) return false;
    return true;
}

// ---- 3D

constexpr int kMinZSeg = 12;      // shortest z segment of the z kernel
constexpr int kMinSliceSeg = 4;   // ... and of the two slice kernels

bool shape3d_ok(int N, int C, int D, int H, int W, int padding)
{
    if (N < 1 || C < 1) return false;
    if (padding != GBSSIM_VALID && padding != GBSSIM_SAME_ZERO) return false;
    if (!extent_ok(D, padding) || !extent_ok(H, padding) || !extent_ok(W, padding)) return false;
    if ((long long)N * C > INT_MAX) return false;
    if (D > (1 << 20) || H > (1 << 20) || W > (1 << 20)) return false;
    if ((long long)H * W > (1LL << 30)) return false;
    return true;
}

struct Plan3d {
    int tiles_x = 0, tiles_y = 0, col_blocks = 0, zsegs = 0, zseg_len = 0;
    long long blocks = 0;
};

// z segments over zlen for per_z blocks of block_warps warps per z range, each
// segment costing `warm` steps beyond its length.  Per SM: the blocks run in
// waves of at most occ; a wave of k blocks takes `steps` step times scaled by
// k / sat when it holds more than sat blocks (an SM is taken as saturated at 16
// resident warps), else the same as sat blocks would (latency-bound).
void plan_z(Plan3d &p, long long per_z, int zlen, int warm, int min_seg, int block_warps,
            int sm_count, int occ)
{
    const int full = std::max(1, 16 / block_warps);
    const int sat = occ < full ? occ : full;
    const int max_segs = int(ceil_div(zlen, min_seg));
    double best = -1.0;
    long long best_work = 0;
    for (int s = 1; s <= max_segs; ++s) {
        const int len = int(ceil_div(zlen, s));
        const int segs = int(ceil_div(zlen, len));
        const long long blocks = per_z * segs;
        const long long steps = len + warm;
        long long left = ceil_div(blocks, (long long)sm_count);
        double cost = 0.0;
        while (left > 0) {
            const long long k = left < occ ? left : occ;
            cost += double(steps) * (k > sat ? double(k) / sat : 1.0);
            left -= k;
        }
        const long long work = blocks * steps;
        if (best < 0 || cost < best - 1e-9 || (cost <= best + 1e-9 && work < best_work)) {
            best = cost;
            best_work = work;
            p.zsegs = segs;
            p.zseg_len = len;
            p.blocks = blocks;
        }
    }
}

// A slice kernel: tiles of 16 x tile_x over (rows, cols), every slice of the
// volume walked once (a segment's only extra cost is its pipeline fill).
Plan3d plan_slices(long long planes, int D, int rows, int cols, int tile_x, int sm_count, int occ)
{
    Plan3d p;
    p.tiles_x = int(ceil_div(cols, tile_x));
    p.tiles_y = int(ceil_div(rows, kTile3dY));
    plan_z(p, planes * p.tiles_x * p.tiles_y, D, 2, kMinSliceSeg, kTile3dY * tile_x / 32,
           sm_count, occ);
    return p;
}

// The z kernel: blocks of kZThreads output columns; zlen = D with gradients
// (20 slices of warm-up), Do without (10).
Plan3d plan_columns(long long planes, int zlen, long long columns, bool grad, int sm_count, int occ)
{
    Plan3d p;
    p.col_blocks = int(ceil_div(columns, (long long)kZThreads));
    plan_z(p, planes * p.col_blocks, zlen, grad ? 20 : 10, kMinZSeg, kZThreads / 32, sm_count, occ);
    return p;
}

// Workspace of the 3D calls: the completion counter, the z kernel's partial
// sums, then the statistics field and the derivative field, float4 per
// (plane, slice, output column) each, 256-byte aligned.
struct Layout3d {
    size_t t_off, u_off, total;
};

Layout3d layout3d(int N, int C, int D, int H, int W, int padding)
{
    const long long planes = (long long)N * C;
    const long long cols = (long long)out_extent(H, padding) * out_extent(W, padding);
    const long long maxb = planes * ceil_div(cols, (long long)kZThreads) * ceil_div(D, kMinZSeg);
    const size_t field = size_t(planes) * D * size_t(cols) * sizeof(float4);
    Layout3d l;
    l.t_off = size_t(ceil_div((long long)(kCounterBytes + maxb * sizeof(double)), 256)) * 256;
    l.u_off = l.t_off + (field + 255) / 256 * 256;
    l.total = l.u_off + field;
    return l;
}

// ---- per-octave maps

constexpr int kMaxOctaves = 32;

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

// Workspace of ssim_pyramid: the completion counter, the partial sums (3 per
// block of every octave: they are planned into one launch), then the
// downscaled pair of each octave >= 1 (every image 256-byte aligned).
struct PyrLayout {
    int octaves = 0;
    int H[kMaxOctaves], W[kMaxOctaves];
    size_t x_off[kMaxOctaves], y_off[kMaxOctaves];
    size_t map_floats = 0, total = 0;
};

bool pyramid_layout(int N, int C, int H, int W, int padding, int octaves, PyrLayout &L)
{
    if (octaves < 1 || octaves > kMaxOctaves || !shape2d_ok(N, C, H, W, padding)) return false;
    const long long planes = (long long)N * C;
    const int off = padding == GBSSIM_VALID ? 0 : kRadius;
    long long first_blocks = 0, later_blocks = 0;
    int h = H, w = W;
    L.octaves = octaves;
    L.map_floats = 0;
    for (int o = 0; o < octaves; ++o) {
        if (!extent_ok(h, padding) || !extent_ok(w, padding)) return false;
        L.H[o] = h;
        L.W[o] = w;
        const int ho = out_extent(h, padding), wo = out_extent(w, padding);
        (o == 0 ? first_blocks : later_blocks) += max_blocks2d(planes, h, w, ho, wo, off);
        L.map_floats += 3 * size_t(planes) * size_t(ho) * size_t(wo);
        h = (h + 1) / 2;
        w = (w + 1) / 2;
    }
    const long long max_blocks = first_blocks + later_blocks;  // one launch, every octave
    size_t pos = round256(kCounterBytes + 3 * size_t(max_blocks) * sizeof(double));
    L.x_off[0] = L.y_off[0] = 0;
    for (int o = 1; o < octaves; ++o) {
        const size_t img = round256(size_t(planes) * L.H[o] * L.W[o] * sizeof(float));
        L.x_off[o] = pos;
        L.y_off[o] = pos + img;
        pos += 2 * img;
    }
    L.total = pos;
    return true;
}

}  // namespace

extern "C" {

int gbssim_abi_version(void) { return GBSSIM_ABI_VERSION; }

const char *gbssim_strerror(int status)
{
    switch (status) {
    case GBSSIM_OK: return "ok";
    case GBSSIM_EINVAL: return "invalid argument (null pointer, bad padding or overlapping buffers)";
    case GBSSIM_ESHAPE: return "invalid shape (N or C < 1, an extent below the window, or too large)";
    case GBSSIM_EALIGN: return "misaligned pointer (float32 buffers need 4-byte alignment)";
    case GBSSIM_EWORKSPACE: return "workspace or saved buffer missing or too small";
    case GBSSIM_ECUDA: return "a CUDA runtime call or kernel launch failed";
    case GBSSIM_ETOOLARGE:
        return "problem too large for the fixed scratch of ssim_fwd_noalloc (use ssim_fwd)";
    default: return "unknown status";
    }
}

void gbssim_window(float w[11])
{
    if (!w) return;
    for (int k = 0; k < kTaps; ++k) w[k] = tap(k);
}

int gbssim_device_status(unsigned *flags_out)
{
    if (!flags_out) return GBSSIM_EINVAL;
    *flags_out = 0;
    unsigned f3 = 0;
    const cudaError_t e = ssim2d_staging_status(flags_out, true);
    if (e != cudaSuccess) return cuda_fail(e);
    const cudaError_t e3 = ssim3d_staging_status(&f3, true);
    *flags_out |= f3;
    return cuda_fail(e3);
}

size_t gbssim_workspace_bytes(int N, int C, int H, int W, int padding)
{
    if (!shape2d_ok(N, C, H, W, padding)) return 0;
    const long long b = max_blocks2d((long long)N * C, H, W, out_extent(H, padding),
                                     out_extent(W, padding), padding == GBSSIM_VALID ? 0 : kRadius);
    return kCounterBytes + size_t(b) * sizeof(double);
}

size_t gbssim_saved_bytes(int N, int C, int H, int W, int want_grad2)
{
    if (N < 1 || C < 1 || H < 1 || W < 1) return 0;
    const size_t field = size_t(N) * C * H * W * sizeof(float);
    return want_grad2 ? 2 * field : field;
}

int ssim_fwd(const float *img1, const float *img2, int N, int C, int H, int W, int padding,
             float *out_mean, float *out_map_or_null, float *saved_or_null, size_t saved_bytes,
             int want_grad2, void *workspace, size_t workspace_bytes, void *stream)
{
    const CallRange range("ssim_fwd");
    int rc;
    if ((rc = check_in(img1)) || (rc = check_in(img2)) || (rc = check_in(out_mean)) ||
        (rc = check_opt(out_map_or_null)) || (rc = check_opt(saved_or_null)))
        return rc;
    if (padding != GBSSIM_VALID && padding != GBSSIM_SAME_ZERO) return GBSSIM_EINVAL;
    if (!shape2d_ok(N, C, H, W, padding)) return GBSSIM_ESHAPE;
    if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return GBSSIM_EWORKSPACE;
    const bool grad = saved_or_null != nullptr;
    const size_t img_bytes = size_t(N) * C * H * W * sizeof(float);
    if (grad && saved_bytes < gbssim_saved_bytes(N, C, H, W, want_grad2))
        return GBSSIM_EWORKSPACE;
    const int Ho = out_extent(H, padding), Wo = out_extent(W, padding);
    const size_t map_bytes = size_t(N) * C * Ho * Wo * sizeof(float);
    if (grad && (overlaps(saved_or_null, saved_bytes, img1, img_bytes) ||
                 overlaps(saved_or_null, saved_bytes, img2, img_bytes) ||
                 overlaps(saved_or_null, saved_bytes, out_map_or_null, map_bytes)))
        return GBSSIM_EINVAL;

    DeviceInfo *d = nullptr;
    if ((rc = device_info(&d))) return rc;
    const int off = padding == GBSSIM_VALID ? 0 : kRadius;
    Ssim2dArgs a{};
    a.x = img1; a.y = img2;
    a.H = H; a.W = W; a.Ho = Ho; a.Wo = Wo;
    a.off = off;
    a.C = C;
    a.vec16 = (W % 4 == 0) && (reinterpret_cast<uintptr_t>(img1) % 16 == 0) &&
              (reinterpret_cast<uintptr_t>(img2) % 16 == 0);
    ssim2d_prepare_staging(a, (long long)N * C, grad);
    a.out1 = grad ? saved_or_null : nullptr;
    a.out2 = (grad && want_grad2) ? saved_or_null + size_t(N) * C * H * W : nullptr;
    a.dL = nullptr;
    a.inv_count = float(1.0 / (double(C) * double(Ho) * double(Wo)));
    a.map = out_map_or_null;
    a.counter = static_cast<unsigned *>(workspace);
    a.partials = reinterpret_cast<double *>(static_cast<unsigned char *>(workspace) + kCounterBytes);
    a.mean = out_mean;
    a.count = double(C) * double(Ho) * double(Wo);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (grad) return launch_grad2d(a, d, N, want_grad2 != 0, workspace_bytes, s);
    // forward only: the split kernel where the inputs are staged by tensor copies
    const bool fs = a.tma && g_fsplit_enabled;
    const Plan2d p = cached_plan2d((long long)N * C, H, W, Ho, Wo, off, false, d->sm_count,
                                   fs ? d->occ_fsplit[0] : d->occ2d[0]);
    if (p.blocks > INT_MAX) return GBSSIM_ESHAPE;
    if (workspace_bytes < kCounterBytes + size_t(p.blocks) * sizeof(double))
        return GBSSIM_EWORKSPACE;
    set_segments(a, p, Ho);
    a.images = N;
    a.blocks_per_image = int(p.blocks / N);
    if (fs) return cuda_fail(ssim2d_fsplit_launch(a, false, int(p.blocks), s, false));
    return cuda_fail(ssim2d_launch(a, false, false, int(p.blocks), s));
}

int ssim_bwd(const float *dL, const float *img1, const float *img2, int N, int C, int H, int W,
             int padding, const float *saved_or_null, size_t saved_bytes, float *grad_img1,
             float *grad_img2_or_null, void *stream)
{
    const CallRange range("ssim_bwd");
    int rc;
    if ((rc = check_in(dL)) || (rc = check_in(img1)) || (rc = check_in(img2)) ||
        (rc = check_in(grad_img1)) || (rc = check_opt(grad_img2_or_null)) ||
        (rc = check_opt(saved_or_null)))
        return rc;
    if (padding != GBSSIM_VALID && padding != GBSSIM_SAME_ZERO) return GBSSIM_EINVAL;
    if (!shape2d_ok(N, C, H, W, padding)) return GBSSIM_ESHAPE;
    const size_t total = size_t(N) * C * H * W;
    const size_t img_bytes = total * sizeof(float);
    const bool g2 = grad_img2_or_null != nullptr;
    // gradients may not overlap the images, dL or each other
    if (overlaps(grad_img1, img_bytes, img1, img_bytes) ||
        overlaps(grad_img1, img_bytes, img2, img_bytes) ||
        overlaps(grad_img1, img_bytes, dL, size_t(N) * sizeof(float)) ||
        (g2 && (overlaps(grad_img2_or_null, img_bytes, img1, img_bytes) ||
                overlaps(grad_img2_or_null, img_bytes, img2, img_bytes) ||
                overlaps(grad_img2_or_null, img_bytes, dL, size_t(N) * sizeof(float)) ||
                overlaps(grad_img2_or_null, img_bytes, grad_img1, img_bytes))))
        return GBSSIM_EINVAL;

    const float *f1 = saved_or_null, *f2 = (saved_or_null && g2) ? saved_or_null + total : nullptr;
    if (saved_or_null) {
        if (saved_bytes < gbssim_saved_bytes(N, C, H, W, g2)) return GBSSIM_EWORKSPACE;
        // a gradient may be the saved field itself (scaled in place), but not a shifted overlap
        if ((overlaps(grad_img1, img_bytes, saved_or_null, saved_bytes) && grad_img1 != f1) ||
            (g2 && overlaps(grad_img2_or_null, img_bytes, saved_or_null, saved_bytes) &&
             grad_img2_or_null != f2))
            return GBSSIM_EINVAL;
    }

    DeviceInfo *d = nullptr;
    if ((rc = device_info(&d))) return rc;
    const int Ho = out_extent(H, padding), Wo = out_extent(W, padding);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (saved_or_null)
        return cuda_fail(scale_fields_launch(f1, f2, grad_img1, grad_img2_or_null, dL, 1.0f,
                                             size_t(C) * H * W, total, d->sm_count, s));
    const int off = padding == GBSSIM_VALID ? 0 : kRadius;
    Ssim2dArgs a{};
    a.x = img1; a.y = img2;
    a.H = H; a.W = W; a.Ho = Ho; a.Wo = Wo;
    a.off = off;
    a.C = C;
    a.vec16 = (W % 4 == 0) && (reinterpret_cast<uintptr_t>(img1) % 16 == 0) &&
              (reinterpret_cast<uintptr_t>(img2) % 16 == 0);
    ssim2d_prepare_staging(a, (long long)N * C, true);
    a.out1 = grad_img1;
    a.out2 = grad_img2_or_null;
    a.dL = dL;
    a.inv_count = float(1.0 / (double(C) * double(Ho) * double(Wo)));
    a.map = nullptr;
    a.partials = nullptr;
    a.counter = nullptr;
    a.mean = nullptr;
    a.count = double(C) * double(Ho) * double(Wo);
    return launch_grad2d(a, d, N, g2, 0, s);
}


size_t gbssim_pyramid_workspace_bytes(int N, int C, int H, int W, int padding, int octaves)
{
    PyrLayout L;
    return pyramid_layout(N, C, H, W, padding, octaves, L) ? L.total : 0;
}

size_t gbssim_pyramid_map_floats(int N, int C, int H, int W, int padding, int octaves)
{
    PyrLayout L;
    return pyramid_layout(N, C, H, W, padding, octaves, L) ? L.map_floats : 0;
}

int ssim_pyramid(const float *img1, const float *img2, int N, int C, int H, int W, int padding,
                 int octaves, float *out_means, float *maps_or_null, void *workspace,
                 size_t workspace_bytes, void *stream)
{
    const CallRange range("ssim_pyramid");
    int rc;
    if ((rc = check_in(img1)) || (rc = check_in(img2)) || (rc = check_in(out_means)) ||
        (rc = check_opt(maps_or_null)))
        return rc;
    if (padding != GBSSIM_VALID && padding != GBSSIM_SAME_ZERO) return GBSSIM_EINVAL;
    PyrLayout L;
    if (!pyramid_layout(N, C, H, W, padding, octaves, L)) return GBSSIM_ESHAPE;
    if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256 != 0 ||
        workspace_bytes < L.total)
        return GBSSIM_EWORKSPACE;
    const long long planes = (long long)N * C;
    const size_t img_bytes = size_t(planes) * H * W * sizeof(float);
    const size_t map_bytes = L.map_floats * sizeof(float);
    const size_t mean_bytes = size_t(octaves) * 3 * N * sizeof(float);
    if (overlaps(maps_or_null, map_bytes, img1, img_bytes) ||
        overlaps(maps_or_null, map_bytes, img2, img_bytes) ||
        overlaps(maps_or_null, map_bytes, out_means, mean_bytes) ||
        overlaps(out_means, mean_bytes, img1, img_bytes) ||
        overlaps(out_means, mean_bytes, img2, img_bytes) ||
        overlaps(workspace, workspace_bytes, img1, img_bytes) ||
        overlaps(workspace, workspace_bytes, img2, img_bytes) ||
        overlaps(workspace, workspace_bytes, out_means, mean_bytes) ||
        overlaps(workspace, workspace_bytes, maps_or_null, map_bytes))
        return GBSSIM_EINVAL;

    DeviceInfo *d = nullptr;
    if ((rc = device_info(&d))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    const int off = padding == GBSSIM_VALID ? 0 : kRadius;
    unsigned *counter = reinterpret_cast<unsigned *>(ws);
    double *partials = reinterpret_cast<double *>(ws + kCounterBytes);
    // the components-mode arguments of octave o; its partial sums at `part`
    auto octave_args = [&](int o, double *part, size_t map_pos, int occ, long long target,
                           Ssim2dArgs &a, long long &blocks) -> int {
        const int h = L.H[o], w = L.W[o];
        const float *cx = o ? reinterpret_cast<const float *>(ws + L.x_off[o]) : img1;
        const float *cy = o ? reinterpret_cast<const float *>(ws + L.y_off[o]) : img2;
        const int ho = out_extent(h, padding), wo = out_extent(w, padding);
        const Plan2d p = target > 0 ? plan2d_blocks(planes, ho, wo, off, target)
                                    : cached_plan2d(planes, h, w, ho, wo, off, false, d->sm_count, occ);
        if (p.blocks > INT_MAX) return GBSSIM_ESHAPE;
        a = Ssim2dArgs{};
        a.x = cx; a.y = cy;
        a.H = h; a.W = w; a.Ho = ho; a.Wo = wo;
        a.off = off;
        a.C = C;
        set_segments(a, p, ho);
        a.vec16 = (w % 4 == 0) && (reinterpret_cast<uintptr_t>(cx) % 16 == 0) &&
                  (reinterpret_cast<uintptr_t>(cy) % 16 == 0);
        ssim2d_prepare_staging(a, planes, false);
        a.inv_count = float(1.0 / (double(C) * double(ho) * double(wo)));
        a.map = maps_or_null ? maps_or_null + map_pos : nullptr;
        a.map_stride = size_t(planes) * ho * wo;
        a.segments = int(p.blocks);
        a.counter = counter;
        a.partials = part;
        a.mean = out_means + size_t(o) * 3 * N;
        a.images = N;
        a.blocks_per_image = int(p.blocks / N);
        a.count = double(C) * double(ho) * double(wo);
        blocks = p.blocks;
        return GBSSIM_OK;
    };
    // the forward split kernel where every octave's images allow tensor copies
    // (16-byte aligned, W_o % 4 == 0; the downscaled ones are 256-byte aligned)
    bool fs = g_fsplit_enabled && staging_mode() != 1 &&
              (reinterpret_cast<uintptr_t>(img1) % 16 == 0) &&
              (reinterpret_cast<uintptr_t>(img2) % 16 == 0);
    for (int o = 0; o < octaves; ++o) fs = fs && (L.W[o] % 4 == 0);
    cudaError_t e;
    if (fs && octaves > 1) {
        // Octave 0 alone first (it reads the caller's images); the octave chain
        // runs beside it, its blocks taking the slots octave 0's blocks leave at
        // the end of their walks; then the other octaves in one wave (waiting
        // for the chain, whose completion implies octave 0's).
        Ssim2dArgs a0;
        long long b0 = 0;
        if ((rc = octave_args(0, partials, 0, d->occ_fsplit[1], 0, a0, b0))) return rc;
        if (a0.tma) {
            if ((e = ssim2d_fsplit_launch(a0, true, int(b0), s, false)) != cudaSuccess)
                return cuda_fail(e);
            for (int lo = 0; lo + 1 < octaves; lo += kChainLevels) {
                OctaveChainArgs m{};
                m.levels = std::min(kChainLevels, octaves - 1 - lo);
                m.x = lo ? reinterpret_cast<const float *>(ws + L.x_off[lo]) : img1;
                m.y = lo ? reinterpret_cast<const float *>(ws + L.y_off[lo]) : img2;
                for (int l = 0; l <= m.levels; ++l) {
                    m.H[l] = L.H[lo + l];
                    m.W[l] = L.W[lo + l];
                    if (l > 0) {
                        m.ox[l - 1] = reinterpret_cast<float *>(ws + L.x_off[lo + l]);
                        m.oy[l - 1] = reinterpret_cast<float *>(ws + L.y_off[lo + l]);
                    }
                }
                m.tiles_x = int(ceil_div(L.W[lo], kChainTile * kChainG));
                m.tiles_y = int(ceil_div(L.H[lo], kChainTile));
                m.planes = planes;
                m.wait_first = lo > 0 ? 1 : 0;
                if ((e = octave_chain_launch(m, s)) != cudaSuccess) return cuda_fail(e);
            }
            double *part = partials + 3 * b0;
            size_t map_pos = 3 * a0.map_stride;
            for (int o0 = 1; o0 < octaves; o0 += kMaxMulti) {
                Ssim2dMulti m{};
                m.count = std::min(kMaxMulti, octaves - o0);
                m.counter = counter;
                long long total = 0;
                double work = 0.0;
                for (int k = 0; k < m.count; ++k)
                    work += double(out_extent(L.H[o0 + k], padding)) * out_extent(L.W[o0 + k], padding);
                for (int k = 0; k < m.count; ++k) {
                    long long blocks = 0;
                    const double share = double(out_extent(L.H[o0 + k], padding)) *
                                         out_extent(L.W[o0 + k], padding) / work;
                    const int occ = d->occ_fsplit[2];
                    const long long target = std::max(1LL, (long long)(share * d->sm_count * occ + 0.5));
                    if ((rc = octave_args(o0 + k, part, map_pos, occ, target, m.oct[k], blocks)))
                        return rc;
                    m.oct[k].no_wait = 0;
                    m.first[k] = int(total);
                    total += blocks;
                    if (total > INT_MAX) return GBSSIM_ESHAPE;
                    part += 3 * blocks;
                    map_pos += 3 * m.oct[k].map_stride;
                }
                m.first[m.count] = int(total);
                bool all_tma = true;
                for (int k = 0; k < m.count; ++k) all_tma = all_tma && m.oct[k].tma;
                e = all_tma ? ssim2d_fsplit_multi_launch(m, s) : ssim2d_components_multi_launch(m, s);
                if (e != cudaSuccess) return cuda_fail(e);
            }
            return GBSSIM_OK;
        }
    }
    if (octaves == 1) {
        Ssim2dArgs a0;
        long long b0 = 0;
        if ((rc = octave_args(0, partials, 0, fs ? d->occ_fsplit[1] : d->occ_comp, 0, a0, b0)))
            return rc;
        if (fs && a0.tma) return cuda_fail(ssim2d_fsplit_launch(a0, true, int(b0), s, false));
        return cuda_fail(ssim2d_components_launch(a0, int(b0), s, false));
    }
    // the downscaled octaves first, up to kChainLevels per launch (each waits
    // for the kernel ahead before its blocks let the launch behind start)
    for (int lo = 0; lo + 1 < octaves; lo += kChainLevels) {
        OctaveChainArgs m{};
        m.levels = std::min(kChainLevels, octaves - 1 - lo);
        m.x = lo ? reinterpret_cast<const float *>(ws + L.x_off[lo]) : img1;
        m.y = lo ? reinterpret_cast<const float *>(ws + L.y_off[lo]) : img2;
        for (int l = 0; l <= m.levels; ++l) {
            m.H[l] = L.H[lo + l];
            m.W[l] = L.W[lo + l];
            if (l > 0) {
                m.ox[l - 1] = reinterpret_cast<float *>(ws + L.x_off[lo + l]);
                m.oy[l - 1] = reinterpret_cast<float *>(ws + L.y_off[lo + l]);
            }
        }
        m.tiles_x = int(ceil_div(L.W[lo], kChainTile * kChainG));
        m.tiles_y = int(ceil_div(L.H[lo], kChainTile));
        m.planes = planes;
        m.wait_first = 1;
        if ((e = octave_chain_launch(m, s)) != cudaSuccess) return cuda_fail(e);
    }
    // then the statistics of every octave, up to kMaxMulti octaves per launch;
    // a launch's blocks fill the GPU's resident slots once, shared among its
    // octaves by output pixels, so that its blocks end close together
    size_t map_pos = 0;
    for (int o0 = 0; o0 < octaves; o0 += kMaxMulti) {
        Ssim2dMulti m{};
        m.count = std::min(kMaxMulti, octaves - o0);
        m.counter = counter;
        double *part = partials;
        long long total = 0;
        double work = 0.0;
        for (int k = 0; k < m.count; ++k)
            work += double(out_extent(L.H[o0 + k], padding)) * out_extent(L.W[o0 + k], padding);
        for (int k = 0; k < m.count; ++k) {
            long long blocks = 0;
            const double share = double(out_extent(L.H[o0 + k], padding)) *
                                 out_extent(L.W[o0 + k], padding) / work;
            const int occ = fs ? d->occ_fsplit[2] : d->occ_multi;
            const long long target = std::max(1LL, (long long)(share * d->sm_count * occ + 0.5));
            if ((rc = octave_args(o0 + k, part, map_pos, occ, target, m.oct[k], blocks)))
                return rc;
            // octave 0 reads the caller's images: its blocks need not wait for the
            // octave chain ahead (which itself waited for the work before it)
            m.oct[k].no_wait = (o0 + k == 0) ? 1 : 0;
            m.first[k] = int(total);
            total += blocks;
            if (total > INT_MAX) return GBSSIM_ESHAPE;
            part += 3 * blocks;
            map_pos += 3 * m.oct[k].map_stride;
        }
        m.first[m.count] = int(total);
        bool all_tma = fs;
        for (int k = 0; k < m.count; ++k) all_tma = all_tma && m.oct[k].tma;
        e = all_tma ? ssim2d_fsplit_multi_launch(m, s) : ssim2d_components_multi_launch(m, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return GBSSIM_OK;
}

size_t gbssim3d_workspace_bytes(int N, int C, int D, int H, int W, int padding)
{
    if (!shape3d_ok(N, C, D, H, W, padding)) return 0;
    return layout3d(N, C, D, H, W, padding).total;
}

size_t gbssim3d_saved_bytes(int N, int C, int D, int H, int W, int want_grad2)
{
    if (N < 1 || C < 1 || D < 1 || H < 1 || W < 1) return 0;
    const size_t field = size_t(N) * C * D * H * W * sizeof(float);
    return want_grad2 ? 2 * field : field;
}

static void fill3d(Ssim3dArgs &a, const float *x, const float *y, int N, int C, int D, int H,
                   int W, int padding, void *workspace)
{
    a.x = x; a.y = y;
    a.D = D; a.H = H; a.W = W;
    a.Do = out_extent(D, padding); a.Ho = out_extent(H, padding); a.Wo = out_extent(W, padding);
    a.off = padding == GBSSIM_VALID ? 0 : kRadius;
    a.C = C;
    // 16-byte staging of the xy kernel: tile origins (multiples of 8 minus off)
    // on 16-byte boundaries, 16-byte row pitch, aligned volumes
    a.vec16 = (a.off % 4 == 0) && (W % 4 == 0) && (reinterpret_cast<uintptr_t>(x) % 16 == 0) &&
              (reinterpret_cast<uintptr_t>(y) % 16 == 0);
    const Layout3d l = layout3d(N, C, D, H, W, padding);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    a.counter = reinterpret_cast<unsigned *>(ws);
    a.partials = reinterpret_cast<double *>(ws + kCounterBytes);
    a.tfield = reinterpret_cast<float4 *>(ws + l.t_off);
    a.ufield = reinterpret_cast<float4 *>(ws + l.u_off);
    a.inv_count = float(1.0 / (double(C) * a.Do * a.Ho * a.Wo));
    a.count = double(C) * a.Do * a.Ho * a.Wo;
    a.images = N;
    ssim3d_prepare_staging(a, (long long)N * C);
}

static void apply_plan(Ssim3dArgs &a, const Plan3d &p)
{
    a.tiles_x = p.tiles_x; a.tiles_y = p.tiles_y; a.col_blocks = p.col_blocks;
    a.zsegs = p.zsegs; a.zseg_len = p.zseg_len;
}

// The passes of one 3D call on stream s: xy, z (mean into `mean` unless null,
// map unless null; derivatives when grad), then with grad the adjoint kernel
// writing out1 (and out2 when g2), scaled by dL[n] (1 when null) / count.
static int run3d(const DeviceInfo *d, Ssim3dArgs &a, int N, float *mean, float *map, bool grad,
                 bool g2, float *out1, float *out2, const float *dL, cudaStream_t s)
{
    const long long planes = (long long)N * a.C;
    const Plan3d px = plan_slices(planes, a.D, a.Ho, a.Wo, kXy3dX, d->sm_count, d->occ3d[0]);
    const Plan3d pz = plan_columns(planes, grad ? a.D : a.Do, (long long)a.Ho * a.Wo, grad,
                                   d->sm_count, d->occ3d[grad ? (g2 ? 3 : 2) : 1]);
    Plan3d pa;
    if (grad) pa = plan_slices(planes, a.D, a.H, a.W, kAdj3dX, d->sm_count, d->occ3d[4]);
    if (px.blocks > INT_MAX || pz.blocks > INT_MAX || pa.blocks > INT_MAX) return GBSSIM_ESHAPE;
    apply_plan(a, px);
    cudaError_t e = ssim3d_xy_launch(a, int(px.blocks), s);
    if (e != cudaSuccess) return cuda_fail(e);
    apply_plan(a, pz);
    if (!mean) a.partials = nullptr;
    a.mean = mean;
    a.map = map;
    a.blocks_per_image = int(pz.blocks / N);
    e = ssim3d_z_launch(a, grad, g2, int(pz.blocks), s);
    if (e != cudaSuccess || !grad) return cuda_fail(e);
    apply_plan(a, pa);
    a.out1 = out1;
    a.out2 = out2;
    a.dL = dL;
    return cuda_fail(ssim3d_adjoint_launch(a, g2, int(pa.blocks), s));
}

int ssim3d_fwd(const float *img1, const float *img2, int N, int C, int D, int H, int W,
               int padding, float *out_mean, float *out_map_or_null, float *saved_or_null,
               size_t saved_bytes, int want_grad2, void *workspace, size_t workspace_bytes,
               void *stream)
{
    const CallRange range("ssim3d_fwd");
    int rc;
    if ((rc = check_in(img1)) || (rc = check_in(img2)) || (rc = check_in(out_mean)) ||
        (rc = check_opt(out_map_or_null)) || (rc = check_opt(saved_or_null)))
        return rc;
    if (padding != GBSSIM_VALID && padding != GBSSIM_SAME_ZERO) return GBSSIM_EINVAL;
    if (!shape3d_ok(N, C, D, H, W, padding)) return GBSSIM_ESHAPE;
    if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return GBSSIM_EWORKSPACE;
    if (workspace_bytes < gbssim3d_workspace_bytes(N, C, D, H, W, padding)) return GBSSIM_EWORKSPACE;
    const bool grad = saved_or_null != nullptr;
    const size_t img_bytes = size_t(N) * C * D * H * W * sizeof(float);
    if (grad && saved_bytes < gbssim3d_saved_bytes(N, C, D, H, W, want_grad2))
        return GBSSIM_EWORKSPACE;
    if (grad && (overlaps(saved_or_null, saved_bytes, img1, img_bytes) ||
                 overlaps(saved_or_null, saved_bytes, img2, img_bytes) ||
                 overlaps(saved_or_null, saved_bytes, workspace, workspace_bytes)))
        return GBSSIM_EINVAL;

    DeviceInfo *d = nullptr;
    if ((rc = device_info(&d))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Ssim3dArgs a{};
    fill3d(a, img1, img2, N, C, D, H, W, padding, workspace);
    float *f2 = (grad && want_grad2) ? saved_or_null + size_t(N) * C * D * H * W : nullptr;
    return run3d(d, a, N, out_mean, out_map_or_null, grad, grad && want_grad2, saved_or_null, f2,
                 nullptr, s);
}

int ssim3d_bwd(const float *dL, const float *img1, const float *img2, int N, int C, int D,
               int H, int W, int padding, const float *saved_or_null, size_t saved_bytes,
               float *grad_img1, float *grad_img2_or_null, void *workspace,
               size_t workspace_bytes, void *stream)
{
    const CallRange range("ssim3d_bwd");
    int rc;
    if ((rc = check_in(dL)) || (rc = check_in(img1)) || (rc = check_in(img2)) ||
        (rc = check_in(grad_img1)) || (rc = check_opt(grad_img2_or_null)) ||
        (rc = check_opt(saved_or_null)))
        return rc;
    if (padding != GBSSIM_VALID && padding != GBSSIM_SAME_ZERO) return GBSSIM_EINVAL;
    if (!shape3d_ok(N, C, D, H, W, padding)) return GBSSIM_ESHAPE;
    const size_t total = size_t(N) * C * D * H * W;
    const size_t img_bytes = total * sizeof(float);
    const bool g2 = grad_img2_or_null != nullptr;
    if (overlaps(grad_img1, img_bytes, img1, img_bytes) ||
        overlaps(grad_img1, img_bytes, img2, img_bytes) ||
        overlaps(grad_img1, img_bytes, dL, size_t(N) * sizeof(float)) ||
        (g2 && (overlaps(grad_img2_or_null, img_bytes, img1, img_bytes) ||
                overlaps(grad_img2_or_null, img_bytes, img2, img_bytes) ||
                overlaps(grad_img2_or_null, img_bytes, dL, size_t(N) * sizeof(float)) ||
                overlaps(grad_img2_or_null, img_bytes, grad_img1, img_bytes))))
        return GBSSIM_EINVAL;
    const float *f1 = saved_or_null, *f2 = (saved_or_null && g2) ? saved_or_null + total : nullptr;
    if (saved_or_null) {
        if (saved_bytes < gbssim3d_saved_bytes(N, C, D, H, W, g2)) return GBSSIM_EWORKSPACE;
        if ((overlaps(grad_img1, img_bytes, saved_or_null, saved_bytes) && grad_img1 != f1) ||
            (g2 && overlaps(grad_img2_or_null, img_bytes, saved_or_null, saved_bytes) &&
             grad_img2_or_null != f2))
            return GBSSIM_EINVAL;
    } else {
        if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256 != 0 ||
            workspace_bytes < gbssim3d_workspace_bytes(N, C, D, H, W, padding))
            return GBSSIM_EWORKSPACE;
        if (overlaps(grad_img1, img_bytes, workspace, workspace_bytes) ||
            (g2 && overlaps(grad_img2_or_null, img_bytes, workspace, workspace_bytes)))
            return GBSSIM_EINVAL;
    }

    DeviceInfo *d = nullptr;
    if ((rc = device_info(&d))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (saved_or_null)
        return cuda_fail(scale_fields_launch(f1, f2, grad_img1, grad_img2_or_null, dL, 1.0f,
                                             size_t(C) * D * H * W, total, d->sm_count, s));
    Ssim3dArgs a{};
    fill3d(a, img1, img2, N, C, D, H, W, padding, workspace);
    return run3d(d, a, N, nullptr, nullptr, true, g2, grad_img1, grad_img2_or_null, dL, s);
}


int ssim_fwd_bwd(const float *img1, const float *img2, int N, int C, int H, int W, int padding,
                 const float *dL, float *out_mean, float *out_map_or_null, float *grad_img1,
                 float *grad_img2_or_null, void *workspace, size_t workspace_bytes, void *stream)
{
    const CallRange range("ssim_fwd_bwd");
    int rc;
    if ((rc = check_in(img1)) || (rc = check_in(img2)) || (rc = check_in(dL)) ||
        (rc = check_in(out_mean)) || (rc = check_opt(out_map_or_null)) ||
        (rc = check_in(grad_img1)) || (rc = check_opt(grad_img2_or_null)))
        return rc;
    if (padding != GBSSIM_VALID && padding != GBSSIM_SAME_ZERO) return GBSSIM_EINVAL;
    if (!shape2d_ok(N, C, H, W, padding)) return GBSSIM_ESHAPE;
    if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return GBSSIM_EWORKSPACE;
    const size_t img_bytes = size_t(N) * C * H * W * sizeof(float);
    const bool g2 = grad_img2_or_null != nullptr;
    const int Ho = out_extent(H, padding), Wo = out_extent(W, padding);
    const size_t map_bytes = size_t(N) * C * Ho * Wo * sizeof(float);
    if (overlaps(grad_img1, img_bytes, img1, img_bytes) ||
        overlaps(grad_img1, img_bytes, img2, img_bytes) ||
        overlaps(grad_img1, img_bytes, out_map_or_null, map_bytes) ||
        overlaps(grad_img1, img_bytes, dL, size_t(N) * sizeof(float)) ||
        (g2 && (overlaps(grad_img2_or_null, img_bytes, img1, img_bytes) ||
                overlaps(grad_img2_or_null, img_bytes, img2, img_bytes) ||
                overlaps(grad_img2_or_null, img_bytes, grad_img1, img_bytes) ||
                overlaps(grad_img2_or_null, img_bytes, out_map_or_null, map_bytes) ||
                overlaps(grad_img2_or_null, img_bytes, dL, size_t(N) * sizeof(float)))))
        return GBSSIM_EINVAL;

    DeviceInfo *d = nullptr;
    if ((rc = device_info(&d))) return rc;
    const int off = padding == GBSSIM_VALID ? 0 : kRadius;
    Ssim2dArgs a{};
    a.x = img1; a.y = img2;
    a.H = H; a.W = W; a.Ho = Ho; a.Wo = Wo;
    a.off = off;
    a.C = C;
    a.vec16 = (W % 4 == 0) && (reinterpret_cast<uintptr_t>(img1) % 16 == 0) &&
              (reinterpret_cast<uintptr_t>(img2) % 16 == 0);
    ssim2d_prepare_staging(a, (long long)N * C, true);
    a.out1 = grad_img1;
    a.out2 = grad_img2_or_null;
    a.dL = dL;
    a.inv_count = float(1.0 / (double(C) * double(Ho) * double(Wo)));
    a.map = out_map_or_null;
    a.counter = static_cast<unsigned *>(workspace);
    a.partials = reinterpret_cast<double *>(static_cast<unsigned char *>(workspace) + kCounterBytes);
    a.mean = out_mean;
    a.count = double(C) * double(Ho) * double(Wo);
    return launch_grad2d(a, d, N, g2, workspace_bytes, static_cast<cudaStream_t>(stream));
}

int ssim3d_fwd_bwd(const float *img1, const float *img2, int N, int C, int D, int H, int W,
                   int padding, const float *dL, float *out_mean, float *out_map_or_null,
                   float *grad_img1, float *grad_img2_or_null, void *workspace,
                   size_t workspace_bytes, void *stream)
{
    const CallRange range("ssim3d_fwd_bwd");
    int rc;
    if ((rc = check_in(img1)) || (rc = check_in(img2)) || (rc = check_in(dL)) ||
        (rc = check_in(out_mean)) || (rc = check_opt(out_map_or_null)) ||
        (rc = check_in(grad_img1)) || (rc = check_opt(grad_img2_or_null)))
        return rc;
    if (padding != GBSSIM_VALID && padding != GBSSIM_SAME_ZERO) return GBSSIM_EINVAL;
    if (!shape3d_ok(N, C, D, H, W, padding)) return GBSSIM_ESHAPE;
    if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256 != 0 ||
        workspace_bytes < gbssim3d_workspace_bytes(N, C, D, H, W, padding))
        return GBSSIM_EWORKSPACE;
    const size_t img_bytes = size_t(N) * C * D * H * W * sizeof(float);
    const bool g2 = grad_img2_or_null != nullptr;
    if (overlaps(grad_img1, img_bytes, img1, img_bytes) ||
        overlaps(grad_img1, img_bytes, img2, img_bytes) ||
        overlaps(grad_img1, img_bytes, workspace, workspace_bytes) ||
        overlaps(grad_img1, img_bytes, dL, size_t(N) * sizeof(float)) ||
        (g2 && (overlaps(grad_img2_or_null, img_bytes, img1, img_bytes) ||
                overlaps(grad_img2_or_null, img_bytes, img2, img_bytes) ||
                overlaps(grad_img2_or_null, img_bytes, grad_img1, img_bytes) ||
                overlaps(grad_img2_or_null, img_bytes, workspace, workspace_bytes) ||
                overlaps(grad_img2_or_null, img_bytes, dL, size_t(N) * sizeof(float)))))
        return GBSSIM_EINVAL;

    DeviceInfo *d = nullptr;
    if ((rc = device_info(&d))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Ssim3dArgs a{};
    fill3d(a, img1, img2, N, C, D, H, W, padding, workspace);
    return run3d(d, a, N, out_mean, out_map_or_null, true, g2, grad_img1, grad_img2_or_null, dL, s);
}

#ifdef GBSSIM_TEST_HOOKS
// ---- test build only (csrc/gbssim_test_hooks.h)

// Make the 2D planner cut every strip into ceil(rows / `rows`) equal row
// segments (0 restores the planner; lengths below the planner's minimum are
// raised to it).  Results do not depend on it.
void gbssim_tune_seg_rows(int rows)
{
    g_seg_rows_override = rows > 0 ? (rows < kMinSegRows ? kMinSegRows : rows) : 0;
}

// Staging of the 2D and 3D kernels: 0 tensor copies where the images allow
// them (the product behaviour), 1 cp.async copies only, 2 tensor copies whose
// waits are made to run out (exercises the bounded-wait failure path).
void gbssim_tune_staging(int mode) { ssim2d_set_staging_mode(mode); }

// Force the stream kernel for every later forward-only and per-octave launch
// (on = 0), or let the forward split kernel run where it applies (on = 1, the
// product behaviour).
void gbssim_tune_fwd_split(int on) { g_fsplit_enabled = on != 0; }

// One run of the gradient-mode kernel of ssim_fwd's stored variant with grad2,
// writing besides the two gradient fields of the means (dL = 1) the window
// statistics and the derivatives of S of every output pixel: stage-by-stage
// parity.
int gbssim_test_stage_dump2d(const float *img1, const float *img2, int N, int C, int H, int W,
                             int padding, float *out_stats, float *out_grads, float *field1,
                             float *field2, void *stream)
{
    int rc;
    if ((rc = check_in(img1)) || (rc = check_in(img2)) || (rc = check_in(out_stats)) ||
        (rc = check_in(out_grads)) || (rc = check_in(field1)) || (rc = check_in(field2)))
        return rc;
    if (padding != GBSSIM_VALID && padding != GBSSIM_SAME_ZERO) return GBSSIM_EINVAL;
    if (!shape2d_ok(N, C, H, W, padding)) return GBSSIM_ESHAPE;
    if ((reinterpret_cast<uintptr_t>(out_stats) | reinterpret_cast<uintptr_t>(out_grads)) % 16)
        return GBSSIM_EALIGN;
    DeviceInfo *d = nullptr;
    if ((rc = device_info(&d))) return rc;
    const int Ho = out_extent(H, padding), Wo = out_extent(W, padding);
    const int off = padding == GBSSIM_VALID ? 0 : kRadius;
    Ssim2dArgs a{};
    a.x = img1; a.y = img2;
    a.H = H; a.W = W; a.Ho = Ho; a.Wo = Wo;
    a.off = off;
    a.C = C;
    a.vec16 = (W % 4 == 0) && (reinterpret_cast<uintptr_t>(img1) % 16 == 0) &&
              (reinterpret_cast<uintptr_t>(img2) % 16 == 0);
    ssim2d_prepare_staging(a, (long long)N * C, true);
    a.out1 = field1;
    a.out2 = field2;
    a.pair_out = a.vec16 && (reinterpret_cast<uintptr_t>(a.out1) % 8 == 0) &&
                 (reinterpret_cast<uintptr_t>(a.out2) % 8 == 0);
    const Plan2d p = cached_plan2d((long long)N * C, H, W, Ho, Wo, off, true, d->sm_count,
                                   d->occ2d[2]);
    if (p.blocks > INT_MAX) return GBSSIM_ESHAPE;
    set_segments(a, p, H);
    a.inv_count = float(1.0 / (double(C) * double(Ho) * double(Wo)));
    a.dump_stats = out_stats;
    a.dump_grads = out_grads;
    a.images = N;
    a.blocks_per_image = int(p.blocks / N);
    a.count = double(C) * double(Ho) * double(Wo);
    return cuda_fail(ssim2d_dump_launch(a, int(p.blocks), static_cast<cudaStream_t>(stream)));
}
#endif

}  // extern "C"
