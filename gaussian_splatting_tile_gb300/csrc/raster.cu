// [3] forward compositing and [4] its backward: one block per 16x16 tile (the forward 256
// threads, one pixel each; the backward 128 threads, two pixels each), the tile's depth-sorted
// list staged through shared memory 256 entries at a time.
//
// Forward: rigel README "Rasterization"; learn-gs "11 - Tiles", "The kernel" (cooperative
// fetch, __syncthreads_count vote: the block leaves once all 256 pixels are saturated).
// Backward: rigel README "Backward": walk each tile back to front from final_T and n_contrib,
// T_i = T_{i+1} / (1 - a_i), the colour behind carried as a running blend; per-pixel
// contributions are summed over the warp (a shuffle reduce-scatter) and over the tile
// (shared-memory accumulators, one slot per staged entry) before one global atomic per entry,
// component and tile -- the reduction rigel's README names as missing from its backward.
//
// The forward gives each warp an 8x4 pixel rectangle, the backward an 8x8 square; after a batch
// is staged, each warp compacts the entries whose alpha >= 1/255 box (from the record) meets its
// rectangle: the other
// entries would be examined and skipped at every pixel of the warp, so they are skipped without
// being evaluated.  n_contrib is kept as a position in the list (one past the entry that stopped
// the pixel, or the list length), which is exactly the count of examined entries.
#include "rs_internal.cuh"

namespace rs {
namespace {

constexpr int kBatch = kTilePixels;  // 256 entries staged per round, one per thread
constexpr int kWarps = kTilePixels / 32;
constexpr unsigned kFull = 0xffffffffu;

// Resident blocks per SM the compositing kernels are compiled for (register budget per thread =
// 65536 / (256 x blocks)).
#ifndef RS_FWD_MIN_BLOCKS
#define RS_FWD_MIN_BLOCKS 6
#endif
#ifndef RS_BWD_MIN_BLOCKS
#define RS_BWD_MIN_BLOCKS 8  // blocks of 128 threads
#endif

// Pixel of this thread: warp w owns the 8x4 sub-rectangle at columns (w & 1) * 8 and rows
// (w >> 1) * 4 of the tile; lane l is pixel (l & 7, l >> 3) inside it.
__device__ __forceinline__ void tile_pixel(const CameraF& cam, int tile, int& tx0, int& ty0, int& px,
                                           int& py) {
    tx0 = (tile % cam.TX) * kTile;
    ty0 = (tile / cam.TX) * kTile;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    px = tx0 + (warp & 1) * 8 + (lane & 7);
    py = ty0 + (warp >> 1) * 4 + (lane >> 3);
}

// Bit w is set when warp w's 8x4 pixel rectangle meets the entry's alpha >= 1/255 box
// [u - ext_x, u + ext_x] x [v - ext_y, v + ext_y]; pixels outside the box cannot pass the alpha
// threshold, so a warp whose bit is clear would skip the entry at every one of its pixels.
__device__ __forceinline__ uint32_t warp_mask(const float4& p, const float4& q, int tx0, int ty0) {
    if (!(p.w >= 0.f)) return 0u;
    const float xl = p.x - p.w - float(tx0), xh = p.x + p.w - float(tx0);
    const float yl = p.y - q.w - float(ty0), yh = p.y + q.w - float(ty0);
    const bool c0 = xl <= 7.f && xh >= 0.f;
    const bool c1 = xl <= 15.f && xh >= 8.f;
    uint32_t m = 0u;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const bool row = yl <= float(4 * r + 3) && yh >= float(4 * r);
        m |= (row && c0 ? 1u : 0u) << (2 * r);
        m |= (row && c1 ? 1u : 0u) << (2 * r + 1);
    }
    return m;
}

// Compacts, in order, the staged entries j (< 256) for which `hit` holds into `list`; returns
// the count.  Warp-cooperative: every lane of the warp must call it.
template <typename Hit>
__device__ __forceinline__ int compact_warp(uint8_t* list, Hit hit) {
    const unsigned lane = threadIdx.x & 31;
    const uint32_t lt = (1u << lane) - 1u;
    int n = 0;
#pragma unroll
    for (int c = 0; c < kBatch / 32; ++c) {
        const int j = c * 32 + int(lane);
        const bool h = hit(j);
        const uint32_t b = __ballot_sync(kFull, h);
        if (h) list[n + __popc(b & lt)] = uint8_t(j);
        n += __popc(b);
    }
    __syncwarp();
    return n;
}

__global__ void __launch_bounds__(kTilePixels, RS_FWD_MIN_BLOCKS) k_raster_fwd(CameraF cam, const Record* __restrict__ rec,
                                                           const uint2* __restrict__ ranges,
                                                           const uint32_t* __restrict__ list,
                                                           float3 bg, float* __restrict__ image,
                                                           float* __restrict__ final_T,
                                                           uint32_t* __restrict__ n_contrib) {
    __shared__ float4 s_p[kBatch], s_q[kBatch], s_c[kBatch];
    __shared__ uint32_t s_mask[kBatch];
    __shared__ uint8_t s_list[kWarps][kBatch];
    const int tile = blockIdx.x;
    const int warp = threadIdx.x >> 5;
    int tx0, ty0, px, py;
    tile_pixel(cam, tile, tx0, ty0, px, py);
    const bool inside = px < cam.W && py < cam.H;
    const uint2 range = ranges[tile];
    const float fx = float(px), fy = float(py);
    float T = 1.f, C0 = 0.f, C1 = 0.f, C2 = 0.f;
    uint32_t stop = range.y;  // one past the last entry this pixel examined
    bool done = !inside;
    const uint32_t wbit = 1u << warp;
    uint8_t* my_list = s_list[warp];
    for (uint32_t base = range.x; base < range.y; base += kBatch) {
        // every thread reaches this barrier; the block leaves once all 256 pixels are done
        if (__syncthreads_count(done) == kBatch) break;
        const uint32_t e = base + threadIdx.x;
        uint32_t m = 0u;
        if (e < range.y) {
            const Record& r = rec[list[e]];
            s_p[threadIdx.x] = r.p;
            s_q[threadIdx.x] = r.q;
            s_c[threadIdx.x] = r.c;
            m = warp_mask(r.p, r.q, tx0, ty0);
        }
        s_mask[threadIdx.x] = m;
        __syncthreads();
        if (__all_sync(kFull, done)) continue;
        const int nl = compact_warp(my_list, [&](int j) { return (s_mask[j] & wbit) != 0u; });
        if (done) continue;
        for (int k = 0; k < nl; ++k) {
            const int j = my_list[k];
            float dx, dy, G, raw;
            const float alpha = entry_alpha(s_p[j], s_q[j], fx, fy, dx, dy, G, raw);
            if (alpha < kAlphaMin) continue;
            const float4 c = s_c[j];
            const float w = alpha * T;
            C0 = fmaf(c.x, w, C0);
            C1 = fmaf(c.y, w, C1);
            C2 = fmaf(c.z, w, C2);
            T = fmaf(-T, alpha, T);
            if (T < kTStop) {
                done = true;
                stop = base + uint32_t(j) + 1u;
                break;
            }
        }
    }
    if (inside) {
        const size_t HW = size_t(cam.W) * cam.H, pix = size_t(py) * cam.W + px;
        image[pix] = fmaf(T, bg.x, C0);
        image[HW + pix] = fmaf(T, bg.y, C1);
        image[2 * HW + pix] = fmaf(T, bg.z, C2);
        final_T[pix] = T;
        n_contrib[pix] = stop - range.x;
    }
}

// Reduce-scatter of nine per-lane values over the warp in five xor-shuffle steps (9 -> 5 -> 3
// -> 2 -> 1 -> 1), each lane sending the half of its vector that its partner keeps.  Afterwards
// lane L holds the warp's sum of value sum_slot(L) (lanes L and L^1 hold the same sum): 46
// instructions instead of 9 x 5 shuffle-add pairs.
__device__ __forceinline__ float butterfly9(const float (&v)[9], unsigned lane) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
    float a[5];
#pragma unroll
    for (int k = 0; k < 5; ++k) {
        const float lo = v[k], hi = k + 5 < 9 ? v[k + 5] : 0.f;
        a[k] = (b4 ? hi : lo) + __shfl_xor_sync(kFull, b4 ? lo : hi, 16);
    }
    float b[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const float lo = a[k], hi = k + 3 < 5 ? a[k + 3] : 0.f;
        b[k] = (b3 ? hi : lo) + __shfl_xor_sync(kFull, b3 ? lo : hi, 8);
    }
    float c[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const float lo = b[k], hi = k + 2 < 3 ? b[k + 2] : 0.f;
        c[k] = (b2 ? hi : lo) + __shfl_xor_sync(kFull, b2 ? lo : hi, 4);
    }
    float d = (b1 ? c[1] : c[0]) + __shfl_xor_sync(kFull, b1 ? c[0] : c[1], 2);
    return d + __shfl_xor_sync(kFull, d, 1);
}

// Which of the nine sums lane L holds after butterfly9 (-1: padding or the odd twin).
__device__ __forceinline__ int sum_slot(unsigned lane) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
    if ((lane & 1) || (b2 && b1) || (b3 && b2) || (b4 && b3 && b1)) return -1;
    const int v = 5 * b4 + 3 * b3 + 2 * b2 + b1;
    return v < 9 ? v : -1;
}

constexpr int kSums = 9;          // per entry: gp dx, gp dy, gp dx^2, gp dx dy, gp dy^2, gp, w G_rgb
constexpr int kAccStride = kBatch + 1;  // padding keeps the nine slots of one entry in nine banks

// The backward runs 128 threads per tile: warp w owns the 8x8 square at columns (w & 1) * 8 and
// rows (w >> 1) * 8, and lane l the two pixels (l & 7, l >> 3) and (l & 7, (l >> 3) + 4) of it.
// Each warp-level reduction then covers 64 pixels, and the two pixels of a lane share their
// column, so their nine sums fold before the shuffles.
constexpr int kBwdThreads = 128;
constexpr int kBwdWarps = kBwdThreads / 32;

// Bit w is set when warp w's 8x8 square meets the entry's alpha >= 1/255 box.
__device__ __forceinline__ uint32_t square_mask(const float4& p, const float4& q, int tx0, int ty0) {
    if (!(p.w >= 0.f)) return 0u;
    const float xl = p.x - p.w - float(tx0), xh = p.x + p.w - float(tx0);
    const float yl = p.y - q.w - float(ty0), yh = p.y + q.w - float(ty0);
    const bool c0 = xl <= 7.f && xh >= 0.f, c1 = xl <= 15.f && xh >= 8.f;
    const bool r0 = yl <= 7.f && yh >= 0.f, r1 = yl <= 15.f && yh >= 8.f;
    return (r0 && c0 ? 1u : 0u) | (r0 && c1 ? 2u : 0u) | (r1 && c0 ? 4u : 0u) | (r1 && c1 ? 8u : 0u);
}

// Per-pixel state of the reverse walk.
struct BwdPixel {
    float T, SG, G0, G1, G2;
    uint32_t end;  // one past the last entry the pixel examined
};

// One entry at one pixel: updates the pixel's state; returns gp = dL/dpower (0 if clamped) and
// w = alpha T_j, or false if the entry is skipped there.
__device__ __forceinline__ bool bwd_step(BwdPixel& px, float alpha, float raw, const float4& c, float& gp,
                                         float& w) {
    const float one_m = 1.f - alpha;
    const float Tj = __fdividef(px.T, one_m);
    w = alpha * Tj;
    const float cG = fmaf(c.x, px.G0, fmaf(c.y, px.G1, c.z * px.G2));
    const float dalpha = Tj * (cG - px.SG);
    px.SG = fmaf(alpha, cG, one_m * px.SG);
    px.T = Tj;
    gp = raw <= kAlphaMax ? alpha * dalpha : 0.f;  // not clamped: alpha = opacity * exp(power)
    return true;
}

__global__ void __launch_bounds__(kBwdThreads, RS_BWD_MIN_BLOCKS) k_raster_bwd(
    CameraF cam, int n, const Record* __restrict__ rec, const uint2* __restrict__ ranges,
    const uint32_t* __restrict__ list, float3 bg, const float* __restrict__ final_T,
    const uint32_t* __restrict__ n_contrib, const float* __restrict__ dL_dimage,
    float* __restrict__ dm2, float* __restrict__ dcon, float* __restrict__ dop,
    float* __restrict__ dcol) {
    __shared__ float4 s_p[kBatch], s_q[kBatch], s_c[kBatch];
    __shared__ uint32_t s_g[kBatch];
    __shared__ uint8_t s_mask[kBatch];
    __shared__ uint8_t s_list[kBwdWarps][kBatch];
    __shared__ float s_acc[kSums * kAccStride];
    __shared__ uint32_t s_wmax[kBwdWarps];
    const int tile = blockIdx.x;
    const int warp = threadIdx.x >> 5;
    const unsigned lane = threadIdx.x & 31;
    const int tx0 = (tile % cam.TX) * kTile, ty0 = (tile / cam.TX) * kTile;
    const int px = tx0 + (warp & 1) * 8 + int(lane & 7);
    const int py0 = ty0 + (warp >> 1) * 8 + int(lane >> 3);
    const uint2 range = ranges[tile];
    const uint32_t len = range.y - range.x;
    const size_t HW = size_t(cam.W) * cam.H;
    BwdPixel P[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int py = py0 + 4 * h;
        const bool inside = px < cam.W && py < cam.H;
        const size_t pix = inside ? size_t(py) * cam.W + px : 0;
        // n_contrib never exceeds the list length when it comes from rs_rasterize_fwd; the min()
        // keeps inconsistent caller data inside the tile's list
        P[h].end = range.x + (inside ? min(n_contrib[pix], len) : 0u);
        P[h].T = inside ? final_T[pix] : 1.f;
        P[h].G0 = inside ? dL_dimage[pix] : 0.f;
        P[h].G1 = inside ? dL_dimage[HW + pix] : 0.f;
        P[h].G2 = inside ? dL_dimage[2 * HW + pix] : 0.f;
        // the colour behind an entry (per unit T) only enters the gradient through its dot
        // product with dL/dC, so that scalar is carried instead of the colour
        P[h].SG = bg.x * P[h].G0 + bg.y * P[h].G1 + bg.z * P[h].G2;
    }
    for (int i = threadIdx.x; i < kSums * kAccStride; i += kBwdThreads) s_acc[i] = 0.f;
    const uint32_t warp_end = __reduce_max_sync(kFull, max(P[0].end, P[1].end));
    if (lane == 0) s_wmax[warp] = warp_end;
    __syncthreads();
    uint32_t walk_end = s_wmax[0];
#pragma unroll
    for (int w = 1; w < kBwdWarps; ++w) walk_end = max(walk_end, s_wmax[w]);
    const float fx = float(px), fy0 = float(py0), fy1 = float(py0 + 4);
    const uint32_t wbit = 1u << warp;
    const int slot = sum_slot(lane);
    uint8_t* my_list = s_list[warp];
    for (uint32_t batch_end = walk_end; batch_end > range.x;) {
        const uint32_t batch_start = batch_end - range.x > uint32_t(kBatch) ? batch_end - kBatch : range.x;
        const int cnt = int(batch_end - batch_start);
#pragma unroll
        for (int r = 0; r < kBatch / kBwdThreads; ++r) {
            const int t = r * kBwdThreads + int(threadIdx.x);
            uint32_t m = 0u;
            if (t < cnt) {
                const uint32_t g = list[batch_start + t];
                const Record& rr = rec[g];
                s_g[t] = g;
                s_p[t] = rr.p;
                s_q[t] = rr.q;
                s_c[t] = rr.c;
                m = square_mask(rr.p, rr.q, tx0, ty0);
            }
            s_mask[t] = uint8_t(m);
        }
        __syncthreads();
        const int nl = compact_warp(my_list, [&](int j) {
            return (s_mask[j] & wbit) != 0u && batch_start + uint32_t(j) < warp_end;
        });
        for (int k = nl - 1; k >= 0; --k) {
            const int j = my_list[k];
            const uint32_t e = batch_start + uint32_t(j);
            const float4 p = s_p[j], q = s_q[j];
            float dx, dy0, dy1, G, raw0, raw1;
            const float a0 = entry_alpha(p, q, fx, fy0, dx, dy0, G, raw0);
            const float a1 = entry_alpha(p, q, fx, fy1, dx, dy1, G, raw1);
            const bool act0 = e < P[0].end && a0 >= kAlphaMin;
            const bool act1 = e < P[1].end && a1 >= kAlphaMin;
            float gp0 = 0.f, gp1 = 0.f, w0 = 0.f, w1 = 0.f;
            if (act0 || act1) {
                const float4 c = s_c[j];
                if (act0) bwd_step(P[0], a0, raw0, c, gp0, w0);
                if (act1) bwd_step(P[1], a1, raw1, c, gp1, w1);
            }
            if (__any_sync(kFull, act0 || act1)) {
                // the two pixels share dx: fold their sums, then reduce over the warp
                const float sg = gp0 + gp1;
                const float sgy = fmaf(gp1, dy1, gp0 * dy0);
                float v[kSums];
                v[0] = sg * dx;
                v[1] = sgy;
                v[2] = v[0] * dx;
                v[3] = sgy * dx;
                v[4] = fmaf(gp1 * dy1, dy1, (gp0 * dy0) * dy0);
                v[5] = sg;
                v[6] = fmaf(w1, P[1].G0, w0 * P[0].G0);
                v[7] = fmaf(w1, P[1].G1, w0 * P[0].G1);
                v[8] = fmaf(w1, P[1].G2, w0 * P[0].G2);
                const float sum = butterfly9(v, lane);
                if (slot >= 0) atomicAdd(&s_acc[slot * kAccStride + j], sum);
            }
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < kBatch / kBwdThreads; ++r) {
            const int t = r * kBwdThreads + int(threadIdx.x);
            if (t < cnt) {
                // per-entry tile sums -> gradients of the entry's Gaussian:
                //   du = A sum(gp dx) + B sum(gp dy), dv = B sum(gp dx) + C sum(gp dy),
                //   dA = -sum(gp dx^2)/2, dB = -sum(gp dx dy), dC = -sum(gp dy^2)/2,
                //   dopacity = sum(gp)/opacity (gp = opacity exp(power) dL/dalpha),
                //   dcolour = sum(w G)
                float a[kSums];
                bool any = false;
#pragma unroll
                for (int k = 0; k < kSums; ++k) {
                    a[k] = s_acc[k * kAccStride + t];
                    s_acc[k * kAccStride + t] = 0.f;
                    any |= a[k] != 0.f;
                }
                if (any) {
                    const uint32_t g = s_g[t];
                    const size_t N = size_t(n);
                    const float4 p = s_p[t], q = s_q[t];
                    constexpr float kLn2 = 0.6931471805599453f;
                    const float A = -2.f * kLn2 * q.x, B = -kLn2 * q.y, C = -2.f * kLn2 * q.z;
                    atomicAdd(dm2 + g, fmaf(A, a[0], B * a[1]));
                    atomicAdd(dm2 + N + g, fmaf(B, a[0], C * a[1]));
                    atomicAdd(dcon + g, -0.5f * a[2]);
                    atomicAdd(dcon + N + g, -a[3]);
                    atomicAdd(dcon + 2 * N + g, -0.5f * a[4]);
                    atomicAdd(dop + g, a[5] / p.z);
                    atomicAdd(dcol + g, a[6]);
                    atomicAdd(dcol + N + g, a[7]);
                    atomicAdd(dcol + 2 * N + g, a[8]);
                }
            }
        }
        __syncthreads();
        batch_end = batch_start;
    }
}

__global__ void k_fill_background(CameraF cam, float3 bg, float* image, float* final_T,
                                  uint32_t* n_contrib) {
    const size_t HW = size_t(cam.W) * cam.H;
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < HW; i += size_t(gridDim.x) * blockDim.x) {
        image[i] = bg.x;
        image[HW + i] = bg.y;
        image[2 * HW + i] = bg.z;
        final_T[i] = 1.f;
        n_contrib[i] = 0;
    }
}

// Zeroes the four gradient outputs of the compositing backward in one launch.
struct ZeroSpans {
    float* p[4];
    size_t count[4];
};

__global__ void k_zero4(ZeroSpans z) {
    const size_t stride = size_t(gridDim.x) * blockDim.x;
#pragma unroll
    for (int k = 0; k < 4; ++k)
        for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < z.count[k]; i += stride)
            z.p[k][i] = 0.f;
}

}  // namespace

cudaError_t launch_raster_fwd(const CameraF& cam, const Record* rec, const uint32_t* ranges,
                              const uint32_t* list, float3 bg, float* image, float* final_T,
                              uint32_t* n_contrib, cudaStream_t s) {
    const int tiles = cam.TX * cam.TY;
    k_raster_fwd<<<tiles, kTilePixels, 0, s>>>(cam, rec, reinterpret_cast<const uint2*>(ranges), list,
                                               bg, image, final_T, n_contrib);
    return cudaGetLastError();
}

cudaError_t launch_raster_bwd(const CameraF& cam, int32_t n, const Record* rec,
                              const uint32_t* ranges, const uint32_t* list, float3 bg,
                              const float* final_T, const uint32_t* n_contrib,
                              const float* dL_dimage, float* dm2, float* dcon, float* dop,
                              float* dcol, cudaStream_t s) {
    const int tiles = cam.TX * cam.TY;
    k_raster_bwd<<<tiles, kBwdThreads, 0, s>>>(cam, n, rec, reinterpret_cast<const uint2*>(ranges),
                                               list, bg, final_T, n_contrib, dL_dimage, dm2, dcon,
                                               dop, dcol);
    return cudaGetLastError();
}

cudaError_t launch_fill_background(const CameraF& cam, float3 bg, float* image, float* final_T,
                                   uint32_t* n_contrib, cudaStream_t s) {
    const size_t HW = size_t(cam.W) * cam.H;
    const unsigned blocks = unsigned(std::min<size_t>((HW + 255) / 256, 152 * 16));
    k_fill_background<<<blocks, 256, 0, s>>>(cam, bg, image, final_T, n_contrib);
    return cudaGetLastError();
}

cudaError_t launch_zero_grads(float* dm2, float* dcon, float* dop, float* dcol, size_t n,
                              cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    ZeroSpans z{{dm2, dcon, dop, dcol}, {2 * n, 3 * n, n, 3 * n}};
    const unsigned blocks = unsigned(std::min<size_t>((3 * n + 255) / 256, 152 * 8));
    k_zero4<<<blocks, 256, 0, s>>>(z);
    return cudaGetLastError();
}

}  // namespace rs
