// [3] forward compositing and [4] its backward: one 256-thread block per 16x16 tile, one pixel
// per thread, the tile's depth-sorted list staged through shared memory 256 entries at a time.
//
// Forward: rigel README "Rasterization"; learn-gs "11 - Tiles", "The kernel" (cooperative
// fetch, __syncthreads_count vote: the block leaves once all 256 pixels are saturated).
// Backward: rigel README "Backward": walk each tile back to front from final_T and n_contrib,
// T_i = T_{i+1} / (1 - a_i), the colour behind carried as a running blend; per-pixel
// contributions are summed over the warp (shuffles) and over the tile (shared-memory
// accumulators, one slot per staged entry) before one global atomic per entry, component and
// tile -- the reduction rigel's README names as missing from its rasteriser backward.
#include "rs_internal.cuh"

namespace rs {
namespace {

constexpr int kBatch = kTilePixels;  // 256 entries staged per round, one per thread

__device__ __forceinline__ void tile_pixel(const CameraF& cam, int tile, int& px, int& py) {
    const int tx = tile % cam.TX, ty = tile / cam.TX;
    px = tx * kTile + (threadIdx.x & (kTile - 1));
    py = ty * kTile + (threadIdx.x / kTile);
}

__global__ void __launch_bounds__(kTilePixels) k_raster_fwd(CameraF cam, const Record* __restrict__ rec,
                                                           const uint2* __restrict__ ranges,
                                                           const uint32_t* __restrict__ list,
                                                           float3 bg, float* __restrict__ image,
                                                           float* __restrict__ final_T,
                                                           uint32_t* __restrict__ n_contrib) {
    __shared__ float4 s_p[kBatch], s_q[kBatch], s_c[kBatch];
    const int tile = blockIdx.x;
    int px, py;
    tile_pixel(cam, tile, px, py);
    const bool inside = px < cam.W && py < cam.H;
    const uint2 range = ranges[tile];
    const float fx = float(px), fy = float(py);
    float T = 1.f, C0 = 0.f, C1 = 0.f, C2 = 0.f;
    uint32_t count = 0;
    bool done = !inside;
    for (uint32_t base = range.x; base < range.y; base += kBatch) {
        // every thread reaches this barrier; the block leaves once all 256 pixels are done
        if (__syncthreads_count(done) == kBatch) break;
        const uint32_t e = base + threadIdx.x;
        if (e < range.y) {
            const Record& r = rec[list[e]];
            s_p[threadIdx.x] = r.p;
            s_q[threadIdx.x] = r.q;
            s_c[threadIdx.x] = r.c;
        }
        __syncthreads();
        if (!done) {
            const int cnt = int(min(uint32_t(kBatch), range.y - base));
            for (int j = 0; j < cnt; ++j) {
                ++count;
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
                    break;
                }
            }
        }
    }
    if (inside) {
        const size_t HW = size_t(cam.W) * cam.H, pix = size_t(py) * cam.W + px;
        image[pix] = fmaf(T, bg.x, C0);
        image[HW + pix] = fmaf(T, bg.y, C1);
        image[2 * HW + pix] = fmaf(T, bg.z, C2);
        final_T[pix] = T;
        n_contrib[pix] = count;
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

constexpr int kGrads = 9;  // du, dv, dA, dB, dC, dopacity, dr, dg, db

__global__ void __launch_bounds__(kTilePixels) k_raster_bwd(
    CameraF cam, int n, const Record* __restrict__ rec, const uint2* __restrict__ ranges,
    const uint32_t* __restrict__ list, float3 bg, const float* __restrict__ final_T,
    const uint32_t* __restrict__ n_contrib, const float* __restrict__ dL_dimage,
    float* __restrict__ dm2, float* __restrict__ dcon, float* __restrict__ dop,
    float* __restrict__ dcol) {
    __shared__ float4 s_p[kBatch], s_q[kBatch], s_c[kBatch];
    __shared__ uint32_t s_g[kBatch];
    __shared__ float s_acc[kGrads][kBatch];
    __shared__ uint32_t s_max;
    const int tile = blockIdx.x;
    int px, py;
    tile_pixel(cam, tile, px, py);
    const bool inside = px < cam.W && py < cam.H;
    const uint2 range = ranges[tile];
    const size_t HW = size_t(cam.W) * cam.H, pix = inside ? size_t(py) * cam.W + px : 0;
    const uint32_t my_n = inside ? n_contrib[pix] : 0u;
    float T = inside ? final_T[pix] : 1.f;
    const float G0 = inside ? dL_dimage[pix] : 0.f;
    const float G1 = inside ? dL_dimage[HW + pix] : 0.f;
    const float G2 = inside ? dL_dimage[2 * HW + pix] : 0.f;
    float S0 = bg.x, S1 = bg.y, S2 = bg.z;  // colour behind the current entry, per unit T
    if (threadIdx.x == 0) s_max = 0;
    __syncthreads();
    const uint32_t wmax = __reduce_max_sync(0xffffffffu, my_n);
    if ((threadIdx.x & 31) == 0) atomicMax(&s_max, wmax);
    __syncthreads();
    // n_contrib never exceeds the list length when it comes from rs_rasterize_fwd; the min()
    // keeps inconsistent caller data inside the tile's list
    const uint32_t len = range.y - range.x;
    const uint32_t my_end = range.x + min(my_n, len);
    const uint32_t walk_end = range.x + min(s_max, len);
    const float fx = float(px), fy = float(py);
    const unsigned lane = threadIdx.x & 31;
    for (uint32_t batch_end = walk_end; batch_end > range.x;) {
        const uint32_t batch_start = batch_end - range.x > uint32_t(kBatch) ? batch_end - kBatch : range.x;
        const int cnt = int(batch_end - batch_start);
        if (int(threadIdx.x) < cnt) {
            const uint32_t g = list[batch_start + threadIdx.x];
            const Record& r = rec[g];
            s_g[threadIdx.x] = g;
            s_p[threadIdx.x] = r.p;
            s_q[threadIdx.x] = r.q;
            s_c[threadIdx.x] = r.c;
        }
#pragma unroll
        for (int k = 0; k < kGrads; ++k) s_acc[k][threadIdx.x] = 0.f;
        __syncthreads();
        for (int j = cnt - 1; j >= 0; --j) {
            float gr[kGrads];
#pragma unroll
            for (int k = 0; k < kGrads; ++k) gr[k] = 0.f;
            bool act = false;
            if (batch_start + uint32_t(j) < my_end) {
                const float4 p = s_p[j], q = s_q[j];
                float dx, dy, G, raw;
                const float alpha = entry_alpha(p, q, fx, fy, dx, dy, G, raw);
                if (alpha >= kAlphaMin) {
                    act = true;
                    const float4 c = s_c[j];
                    const float one_m = 1.f - alpha;
                    const float Tj = __fdividef(T, one_m);
                    const float w = alpha * Tj;
                    gr[6] = w * G0;
                    gr[7] = w * G1;
                    gr[8] = w * G2;
                    const float dalpha = Tj * ((c.x - S0) * G0 + (c.y - S1) * G1 + (c.z - S2) * G2);
                    S0 = fmaf(alpha, c.x, one_m * S0);
                    S1 = fmaf(alpha, c.y, one_m * S1);
                    S2 = fmaf(alpha, c.z, one_m * S2);
                    T = Tj;
                    if (raw <= kAlphaMax) {  // not clamped: alpha = opacity * exp(power)
                        gr[5] = G * dalpha;
                        const float gp = alpha * dalpha;  // dL/dpower
                        gr[2] = -0.5f * dx * dx * gp;
                        gr[3] = -dx * dy * gp;
                        gr[4] = -0.5f * dy * dy * gp;
                        gr[0] = gp * fmaf(p.w, dx, q.w * dy);  // A dx + B dy
                        gr[1] = gp * fmaf(c.w, dy, q.w * dx);  // C dy + B dx
                    }
                }
            }
            if (__any_sync(0xffffffffu, act)) {
#pragma unroll
                for (int k = 0; k < kGrads; ++k) {
                    const float v = warp_sum(gr[k]);
                    if (lane == 0 && v != 0.f) atomicAdd(&s_acc[k][j], v);
                }
            }
        }
        __syncthreads();
        if (int(threadIdx.x) < cnt) {
            const uint32_t g = s_g[threadIdx.x];
            const size_t N = size_t(n);
            float v;
            if ((v = s_acc[0][threadIdx.x]) != 0.f) atomicAdd(dm2 + g, v);
            if ((v = s_acc[1][threadIdx.x]) != 0.f) atomicAdd(dm2 + N + g, v);
            if ((v = s_acc[2][threadIdx.x]) != 0.f) atomicAdd(dcon + g, v);
            if ((v = s_acc[3][threadIdx.x]) != 0.f) atomicAdd(dcon + N + g, v);
            if ((v = s_acc[4][threadIdx.x]) != 0.f) atomicAdd(dcon + 2 * N + g, v);
            if ((v = s_acc[5][threadIdx.x]) != 0.f) atomicAdd(dop + g, v);
            if ((v = s_acc[6][threadIdx.x]) != 0.f) atomicAdd(dcol + g, v);
            if ((v = s_acc[7][threadIdx.x]) != 0.f) atomicAdd(dcol + N + g, v);
            if ((v = s_acc[8][threadIdx.x]) != 0.f) atomicAdd(dcol + 2 * N + g, v);
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
    k_raster_bwd<<<tiles, kTilePixels, 0, s>>>(cam, n, rec, reinterpret_cast<const uint2*>(ranges),
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
