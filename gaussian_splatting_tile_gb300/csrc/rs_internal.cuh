// Internal declarations of the sm_103a rasteriser library: constants of the method, the packed
// per-Gaussian record and the kernel launchers behind the C ABI in include/rs.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <utility>

#include "rs.h"

namespace rs {

// Launches `kernel` on `s` with programmatic stream serialization (see RS_PDL_ENTER).
template <typename... Params, typename... Args>
inline cudaError_t pdl_launch(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Constants of the method (rigel README "Projection", "Rasterization"; learn-gs "11 - Tiles",
// constants cell).
// Programmatic dependent launch (Hopper and later): kernels of the frame are launched with
// programmatic stream serialization, so a kernel's blocks are scheduled while its predecessor
// drains.  Every kernel of the library begins with RS_PDL_ENTER(): it waits until the kernels
// before it in the stream have completed and their writes are visible (so a kernel never reads
// a predecessor's output early, and completion stays transitive along the stream), then lets
// its own dependents be scheduled.  In a kernel launched without the attribute both are no-ops.
#define RS_PDL_ENTER()                                              \
    do {                                                            \
        asm volatile("griddepcontrol.wait;" ::: "memory");          \
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); \
    } while (0)

constexpr int kTile = RS_TILE;
constexpr int kTilePixels = kTile * kTile;
constexpr float kDilation = 0.3f;      // EWA low-pass added to the 2D covariance diagonal
constexpr float kZNear = 0.05f;        // near-plane cull
constexpr float kClampFrac = 1.3f;     // x/z, y/z clamp, in units of the frustum half-width
constexpr float kLambdaFloor = 0.1f;   // floor on the eigenvalue discriminant
constexpr float kAlphaMax = 0.99f;
constexpr float kAlphaMin = 1.0f / 255.0f;
constexpr float kTStop = 1e-4f;
constexpr float kLog2e = 1.4426950408889634f;

// Packed record the projection writes once per Gaussian and both rasterisers gather per list
// entry.  Three 16-byte words:
//   p = (u, v, opacity, ext_x)    position, opacity, half-width of the alpha >= 1/255 region
//   q = (qa, qb, qc, ext_y)       power in log2 units: power2 = qa dx^2 + qb dx dy + qc dy^2
//                                 with qa = -A/2 log2(e), qb = -B log2(e), qc = -C/2 log2(e);
//                                 half-height of the alpha >= 1/255 region
//   c = (r, g, b, 1/opacity)      colour; the reciprocal for the opacity gradient
// Storing the log2-scaled quadratic lets the rasterisers evaluate exp(power) as one ex2 on the
// multi-function unit; forward and backward read the same words, so both evaluate alpha with
// bit-identical arithmetic.  The extents (negative: never reaches 1/255) let a warp skip entries
// that cannot pass the alpha threshold anywhere in its pixels; skipping such an entry is exactly
// what evaluating it and failing the threshold would do.
struct __align__(16) Record {
    float4 p;
    float4 q;
    float4 c;
};
static_assert(sizeof(Record) == RS_RECORD_BYTES, "record size");

struct CameraF {
    float R[9];
    float t[3];
    float fx, fy, cx, cy;
    int W, H;
    int TX, TY;
};

inline CameraF make_camera(const rs_camera& c) {
    CameraF o;
    for (int i = 0; i < 9; ++i) o.R[i] = c.R[i];
    for (int i = 0; i < 3; ++i) o.t[i] = c.t[i];
    o.fx = c.fx; o.fy = c.fy; o.cx = c.cx; o.cy = c.cy;
    o.W = c.width; o.H = c.height;
    o.TX = (c.width + kTile - 1) / kTile;
    o.TY = (c.height + kTile - 1) / kTile;
    return o;
}

// ex2.approx.ftz: the multi-function unit's base-2 exponential (PTX ISA), relative error about
// 2^-22; arguments below -126 give 0, which the alpha threshold then skips.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 1 / x by the approximate reciprocal instruction (PTX rcp.approx.ftz.f32: relative error below
// 2^-23 for normal x; the compositing backward's divisor 1 - alpha lies in [0.01, 1]).
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// alpha of one list entry at pixel (px, py), shared by the forward and the backward so both
// take identical skip, clamp and stop decisions (rigel README "Rasterization":
// alpha = min(0.99, opacity exp(power)), power = -1/2 (A dx^2 + C dy^2) - B dx dy, here in log2
// units).  Returns alpha; `G` = exp(power), `raw` = opacity * G before the clamp.
// The quadratic is evaluated as dy (qc dy + qb dx) + (qa dx) dx, so that pixels sharing a column
// (the backward's two pixels per lane) share the dx terms: entry_alpha_col gives each of them
// exactly what entry_alpha gives.
__device__ __forceinline__ float entry_alpha(const float4& p, const float4& q, float px, float py,
                                             float& dx, float& dy, float& G, float& raw) {
    dx = px - p.x;
    dy = py - p.y;
    const float power2 = fmaf(dy, fmaf(q.z, dy, q.y * dx), (q.x * dx) * dx);
    G = ex2_approx(power2);
    raw = p.z * G;
    return fminf(kAlphaMax, raw);
}

// entry_alpha at (px, py0) and (px, py1), bit-identical to two calls.
__device__ __forceinline__ void entry_alpha_col(const float4& p, const float4& q, float px, float py0, float py1,
                                                float& dx, float& dy0, float& dy1, float& a0, float& raw0,
                                                float& a1, float& raw1) {
    dx = px - p.x;
    dy0 = py0 - p.y;
    dy1 = py1 - p.y;
    const float bx = q.y * dx, axx = (q.x * dx) * dx;
    raw0 = p.z * ex2_approx(fmaf(dy0, fmaf(q.z, dy0, bx), axx));
    raw1 = p.z * ex2_approx(fmaf(dy1, fmaf(q.z, dy1, bx), axx));
    a0 = fminf(kAlphaMax, raw0);
    a1 = fminf(kAlphaMax, raw1);
}

// Tile span bound of a splat's bounding square (learn-gs "11 - Tiles", tile_spans):
// floor((p - r) / 16) for the lower bound, floor((p + r) / 16) + 1 for the upper, clamped to
// [0, n_tiles] in float before the conversion so any finite or infinite p is safe.  The
// projection (tiles_touched) and the expansion (keys) both call this, so they always agree.
__device__ __forceinline__ int span_bound(float p, float r, int n_tiles, bool upper) {
    float f = floorf((upper ? p + r : p - r) * (1.0f / kTile));
    if (upper) f += 1.0f;
    f = fminf(fmaxf(f, 0.0f), float(n_tiles));
    return int(f);
}

// Tile coverage of the ellipse test (RS_TILE_TEST_ELLIPSE): the tiles of the radius square whose
// pixel-centre squares [16 tx, 16 tx + 15] x [16 ty, 16 ty + 15] meet the ellipse d^T Q d <= k
// (Q = (A, B; B, C) the conic, d = pixel - mean).  The ellipse is convex, so each tile row meets
// it in a run of columns, found from the ellipse's x-extent over the row's band of y: the
// extreme point of the left (right) boundary x = -(B/A) dy -+ sqrt(A k - det dy^2) / A, at
// dy = +-B sqrt(k / (det C)) with x = -+sqrt(C k / det), if it lies in the band, else the nearer
// band edge.  Widened by 0.01 px.  Every operation is an explicitly rounded IEEE single-precision
// operation (no fused multiply-add; divisions and square roots correctly rounded), so any
// implementation that performs the same operations takes the same integer decisions.  The
// per-splat part (divisions included) is computed once; a row costs two square roots.
struct EllipseTiles {
    float u, v;
    float nb, inva, ak, det;  // B / A, 1 / A, A k, A C - B^2
    float eyc, ex, dyl;       // y half-extent, x half-extent, dy of the leftmost point
    int ylo, yhi;             // tile rows, inclusive (none when ylo > yhi)
    int xl, xh;               // the radius square's columns [xl, xh)
};

// rect = the radius square's tile span {xl, xh, yl, yh} (half-open): the test keeps a subset of
// it, so the rendered footprint stays the square test's.
__device__ __forceinline__ bool ellipse_tiles_init(float u, float v, float A, float B, float C, float k,
                                                   const int (&rect)[4], int TY, EllipseTiles& e) {
    e.u = u; e.v = v;
    e.xl = rect[0];
    e.xh = rect[1];
    e.ylo = 0; e.yhi = -1;
    if (!(k > 0.f) || !(A > 0.f) || !(C > 0.f)) return false;
    e.det = __fsub_rn(__fmul_rn(A, C), __fmul_rn(B, B));
    if (!(e.det > 0.f)) return false;
    e.inva = __fdiv_rn(1.f, A);
    e.nb = __fmul_rn(B, e.inva);
    e.ak = __fmul_rn(A, k);
    e.eyc = __fsqrt_rn(__fdiv_rn(e.ak, e.det));
    e.ex = __fsqrt_rn(__fdiv_rn(__fmul_rn(C, k), e.det));
    e.dyl = __fmul_rn(B, __fsqrt_rn(__fdiv_rn(k, __fmul_rn(e.det, C))));
    const float ey = __fadd_rn(e.eyc, 0.01f);
    float lo = ceilf(__fmul_rn(__fsub_rn(__fsub_rn(v, ey), 15.f), 0.0625f));
    float hi = floorf(__fmul_rn(__fadd_rn(v, ey), 0.0625f));
    lo = fminf(fmaxf(lo, 0.f), float(TY));
    hi = fmaxf(fminf(hi, float(TY - 1)), -1.f);
    e.ylo = max(int(lo), rect[2]);
    e.yhi = min(int(hi), rect[3] - 1);
    return e.ylo <= e.yhi;
}

// Columns [xlo, xhi] (inclusive; none when xlo > xhi) of tile row ty.
__device__ __forceinline__ void ellipse_row(const EllipseTiles& e, int ty, int TX, int& xlo, int& xhi) {
    const float y0 = fminf(fmaxf(__fsub_rn(float(16 * ty), e.v), -e.eyc), e.eyc);
    const float y1 = fminf(fmaxf(__fsub_rn(float(16 * ty + 15), e.v), -e.eyc), e.eyc);
    // boundary at the band edges: centre -(B/A) y, half-width sqrt(A k - det y^2) / A
    const float c0 = -__fmul_rn(e.nb, y0), c1 = -__fmul_rn(e.nb, y1);
    const float h0 = __fmul_rn(__fsqrt_rn(fmaxf(__fsub_rn(e.ak, __fmul_rn(e.det, __fmul_rn(y0, y0))), 0.f)), e.inva);
    const float h1 = __fmul_rn(__fsqrt_rn(fmaxf(__fsub_rn(e.ak, __fmul_rn(e.det, __fmul_rn(y1, y1))), 0.f)), e.inva);
    const float xmin = (y0 <= e.dyl && e.dyl <= y1) ? -e.ex : fminf(__fsub_rn(c0, h0), __fsub_rn(c1, h1));
    const float dyr = -e.dyl;
    const float xmax = (y0 <= dyr && dyr <= y1) ? e.ex : fmaxf(__fadd_rn(c0, h0), __fadd_rn(c1, h1));
    float lo = ceilf(__fmul_rn(__fsub_rn(__fadd_rn(e.u, xmin), 15.01f), 0.0625f));
    float hi = floorf(__fmul_rn(__fadd_rn(__fadd_rn(e.u, xmax), 0.01f), 0.0625f));
    lo = fminf(fmaxf(lo, 0.f), float(TX));
    hi = fmaxf(fminf(hi, float(TX - 1)), -1.f);
    xlo = max(int(lo), e.xl);
    xhi = min(int(hi), e.xh - 1);
}

// The per-splat part as 11 words (expansion staging): u, v, nb, inva, ak, det, eyc, ex, dyl,
// ylo | yhi << 16, xl | xh << 16 (tile indices fit 16 bits: at most 2048 columns or rows).
constexpr int kEllWords = 11;
static_assert(kEllWords + 1 == RS_ELLIPSE_WORDS, "k, then the packed setup");
__device__ __forceinline__ void ellipse_pack(const EllipseTiles& e, float (&w)[kEllWords]) {
    w[0] = e.u; w[1] = e.v; w[2] = e.nb; w[3] = e.inva; w[4] = e.ak; w[5] = e.det;
    w[6] = e.eyc; w[7] = e.ex; w[8] = e.dyl;
    w[9] = __uint_as_float(uint32_t(e.ylo & 0xffff) | (uint32_t(e.yhi & 0xffff) << 16));
    w[10] = __uint_as_float(uint32_t(e.xl & 0xffff) | (uint32_t(e.xh & 0xffff) << 16));
}
__device__ __forceinline__ void ellipse_unpack(const float* w, int stride, EllipseTiles& e) {
    e.u = w[0]; e.v = w[stride]; e.nb = w[2 * stride]; e.inva = w[3 * stride]; e.ak = w[4 * stride];
    e.det = w[5 * stride]; e.eyc = w[6 * stride]; e.ex = w[7 * stride]; e.dyl = w[8 * stride];
    const uint32_t y = __float_as_uint(w[9 * stride]), x = __float_as_uint(w[10 * stride]);
    e.ylo = int(int16_t(y & 0xffff)); e.yhi = int(int16_t(y >> 16));
    e.xl = int(int16_t(x & 0xffff)); e.xh = int(int16_t(x >> 16));
}

// k of the ellipse test for an opacity (0 when it can never reach alpha 1/255).
__device__ __forceinline__ float alpha_k_of(float o) {
    const float o255 = 255.f * o;
    return o255 > 1.f ? 2.002f * logf(o255) : 0.f;
}

// Launchers (each returns the cudaError_t of its launches).
cudaError_t launch_project(const CameraF& cam, const rs_gaussians& g, const rs_projected& out,
                           cudaStream_t s);
cudaError_t launch_project_bwd(const CameraF& cam, const rs_gaussians& g, const rs_projected& p,
                               const float* dm2, const float* dcon, const float* dcol,
                               float* dmeans, float* dscales, float* dquats, float* dsh,
                               cudaStream_t s);

struct BinPlan {
    int32_t n;
    int n_tiles;
    int tile_bits;         // ceil(log2(n_tiles)), at least 1
    int tile_passes;       // ceil(tile_bits / 8)
    size_t capacity;
    size_t depth_tiles, tile_tiles;  // sort tiles of the depth sort and of the tile sort
    size_t slice_blocks;             // blocks of the slice scan (1024 Gaussians each)
    size_t chunks;                   // 1024-entry chunks of the capacity (expansion blocks)
    // workspace layout (byte offsets)
    size_t off_dkeys, off_dvals, off_tiles_sorted, off_start, off_rect, off_owner, off_tkeys, off_tvals;
    size_t off_ctl, off_result, off_counters, off_ghist_depth, off_ghist_tile, off_status_slices,
        off_status_depth, off_status_tile, ctl_bytes, total_bytes;
};
BinPlan plan_bin(int32_t n, const CameraF& cam, size_t capacity);
// Enqueues the whole binning: depth sort of the Gaussians, scan of their tile counts, expansion
// in depth order, stable sort by tile, ranges.  Afterwards ws + off_result holds
// {E (uint64), error (uint32)}: E is the entry count (nothing past the capacity is written when
// E > capacity) and error is nonzero when a bounded wait of the sort gave up.
cudaError_t launch_bin(const BinPlan& plan, const CameraF& cam, const rs_projected& p, uint8_t* ws,
                       uint64_t* keys_out, uint32_t* point_list, uint32_t* tile_ranges, cudaStream_t s);

// Compositing workspace: chunk -> tile map and the forward's per-pixel state at chunk boundaries.
// Writes the binning's {E, error} (the workspace's result block) to `host` (a device-visible
// pointer to pinned host memory) from a one-thread kernel.
cudaError_t launch_report(const uint8_t* result_block, uint64_t* host, cudaStream_t s);
size_t raster_workspace_bytes(size_t capacity, size_t n_tiles);
cudaError_t launch_raster_fwd(const CameraF& cam, int32_t n, const Record* rec, const uint32_t* ranges,
                              const uint32_t* list, size_t capacity, float3 bg, float* image, float* final_T,
                              uint32_t* n_contrib, void* ws, cudaStream_t s);
cudaError_t launch_raster_bwd(const CameraF& cam, int32_t n, const Record* rec,
                              const uint32_t* ranges, const uint32_t* list, size_t capacity, float3 bg,
                              const float* final_T, const uint32_t* n_contrib, void* ws,
                              const float* dL_dimage, float* dm2, float* dcon, float* dop, float* dcol,
                              cudaStream_t s);
// Fill a background image (n = 0 or no entries): image = bg, final_T = 1, n_contrib = 0.
cudaError_t launch_fill_background(const CameraF& cam, float3 bg, float* image, float* final_T,
                                   uint32_t* n_contrib, cudaStream_t s);
cudaError_t launch_zero_grads(float* dm2, float* dcon, float* dop, float* dcol, size_t n,
                              cudaStream_t s);

// Appearance MLP (hidden 32 or 64, latent_dim + 3 <= 32) and the L1 loss gradient.
cudaError_t launch_appearance_fwd(const CameraF& cam, int n, const float* means, const float* latents,
                                  const rs_mlp& m, float* colors, cudaStream_t s);
cudaError_t launch_appearance_bwd(const CameraF& cam, int n, const float* means, const float* latents,
                                  const rs_mlp& m, const float* dcolors, float* dlatents,
                                  const rs_mlp_grads& gr, cudaStream_t s);
cudaError_t launch_l1(size_t count, const float* img, const float* tgt, float scale, float* dimg,
                      float* loss, cudaStream_t s);
// L1 + D-SSIM loss and gradient; the workspace holds 3 C H W floats and two sums.
// 1 if a tensor-core wait gave up since the last call (the flag is cleared), 0 if not, -1 on a
// CUDA error.
int take_device_error();
// The same for the projection's bounded waits on its staged copies.
int take_projection_error();
// 1 if a compositing kernel found a point-list entry >= n or a tile range past the capacity since
// the last call (the flag is cleared), 0 if not, -1 on a CUDA error.
int take_raster_check();
size_t ssim_workspace_bytes(int C, int H, int W);
cudaError_t launch_l1_dssim(int C, int H, int W, const float* img, const float* tgt, float lambda, float scale,
                            float* dimg, float* loss, void* ws, cudaStream_t s);

// Fused Adam over parameter groups and the densification statistics.
cudaError_t launch_adam(const rs_adam_segment* segs, int n, double beta1, double beta2, double eps, int step,
                        cudaStream_t s);
cudaError_t launch_densify_stats(int n, const float* dm2, const int* radius, float* accum, float* count,
                                 cudaStream_t s);

}  // namespace rs
