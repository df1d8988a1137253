// [3] forward compositing and [4] its backward.  The forward runs one block of 128 threads per
// half of a 16x16 tile, one pixel per thread, the tile's depth-sorted list staged through shared
// memory 256 entries at a time; the backward runs persistent one-warp blocks, each taking 8x8
// squares of 256-entry chunks of the point list, two pixels per lane.
//
// Forward: rigel README "Rasterization"; learn-gs "11 - Tiles", "The kernel" (cooperative
// fetch, __syncthreads_count vote: the block leaves once all its pixels are saturated).
// Backward: rigel README "Backward": walk each tile back to front from final_T and n_contrib,
// T_i = T_{i+1} / (1 - a_i), the colour behind carried as a running blend; per-pixel
// contributions are summed over a warp's 64 pixels (buffered in shared memory and summed by four
// lanes per entry) before one global atomic per entry, component and warp -- the reduction
// rigel's README names as missing from its backward.
//
// The forward gives each warp an 8x4 pixel rectangle, the backward an 8x8 square.  The forward
// skips, per warp, the staged entries whose alpha >= 1/255 region cannot reach its rectangle, and
// records which warps composited each entry; the backward evaluates an entry only in the squares
// where the forward composited it.  Skipping such an entry is exactly what evaluating it and
// failing the threshold at every pixel would do.  n_contrib is kept as a position in the list (one
// past the entry that stopped the pixel, or the list length), which is exactly the count of
// examined entries.
#include <type_traits>

#include "rs_internal.cuh"

namespace rs {
namespace {

// Raised when a compositing kernel meets a point-list entry >= n or a tile range past the list's
// capacity (caller data): the entry or the tile is skipped instead of read out of bounds.
__device__ unsigned int g_raster_check;

constexpr int kBatch = kTilePixels;  // 256 entries staged per round
constexpr uint32_t kChunk = RS_RASTER_CHUNK;  // backward task length and checkpoint spacing
static_assert(kChunk == uint32_t(kBatch), "a forward batch ends at every chunk boundary");
// The forward's block: 1, half a tile (16x8 pixels, 128 threads, two blocks per tile, each
// staging the tile's batches for its own four warps); 0, the whole tile (256 threads).  A batch
// waits at the block barrier for its slowest warp; with four warps instead of eight the slowest
// one carries 1.34 instead of 1.64 times the mean work (counted with the oracle on the 160k
// 1080p view): 0.131 -> 0.128 ms, issue 75% -> 79% of cycles for 1% more instructions.
#ifndef RS_FWD_HALF
#define RS_FWD_HALF 1
#endif
constexpr int kFwdHalves = RS_FWD_HALF ? 2 : 1;
constexpr int kFwdThreads = kTilePixels / kFwdHalves;
constexpr int kFwdWarps = kFwdThreads / 32;
constexpr int kFwdRows = kTile / kFwdHalves;  // pixel rows of a forward block
constexpr unsigned kFull = 0xffffffffu;

// Resident blocks per SM the compositing kernels are compiled for (register budget per thread =
// 65536 / (threads per block x blocks)).
#ifndef RS_FWD_MIN_BLOCKS
#define RS_FWD_MIN_BLOCKS (RS_FWD_HALF ? 12 : 6)
#endif
// backward, in groups of four one-warp blocks (one tile's squares): 7 (72 registers; 6 and 5
// measured the same on the 160k 1080p orbit view, 8 at 64 registers slower)
#ifndef RS_BWD_MIN_BLOCKS
#define RS_BWD_MIN_BLOCKS 7
#endif

// Pixel of this thread: warp w owns the 8x4 sub-rectangle at columns (w & 1) * 8 and rows
// (w >> 1) * 4 of the block's region, which starts at row ry0 = ty0 + kFwdRows * half of the
// tile; lane l is pixel (l & 7, l >> 3) inside it.
__device__ __forceinline__ void tile_pixel(const CameraF& cam, int tile, int half, int& tx0, int& ty0, int& ry0,
                                           int& px, int& py) {
    tx0 = (tile % cam.TX) * kTile;
    ty0 = (tile / cam.TX) * kTile;
    ry0 = ty0 + kFwdRows * half;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    px = tx0 + (warp & 1) * 8 + (lane & 7);
    py = ry0 + (warp >> 1) * 4 + (lane >> 3);
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
    for (int r = 0; r < kFwdWarps / 2; ++r) {
        const bool row = yl <= float(4 * r + 3) && yh >= float(4 * r);
        m |= (row && c0 ? 1u : 0u) << (2 * r);
        m |= (row && c1 ? 1u : 0u) << (2 * r + 1);
    }
    return m;
}

// The warps of mask m (from warp_mask) whose 8x4 rectangle the entry's alpha >= 1/255 ellipse can
// reach: the largest exponent over the rectangle (pixel centres relaxed to the continuous
// rectangle, so nothing that passes is dropped) is compared with log2(1 / (255 opacity)), less a
// margin that covers the rounding of both this test and the compositing's own evaluation.  The
// exponent is concave, so outside its peak its largest value on a rectangle lies on the edge(s)
// facing the peak; on an edge it is a parabola whose vertex is clamped to the edge.
#ifndef RS_FWD_EXACT_MASK
#define RS_FWD_EXACT_MASK 1
#endif
__device__ __forceinline__ float edge_peak(float qa, float qb, float qc, float fixed, float lo, float hi, float r2a) {
    // max over t in [lo, hi] of qa t^2 + qb fixed t + qc fixed^2 (qa < 0); r2a = 1 / (2 qa)
    const float t = fminf(fmaxf(-qb * fixed * r2a, lo), hi);
    return fmaf(t, fmaf(qa, t, qb * fixed), (qc * fixed) * fixed);
}

__device__ __forceinline__ uint32_t warp_mask_exact(uint32_t m, const float4& p, const float4& q, const float4& c,
                                                    int tx0, int ty0) {
    constexpr float kLog2_255 = 7.994353436858858f;
    constexpr float kMargin = 0.02f;  // log2 units: 1.4% of alpha
    const float thr = __log2f(c.w) - kLog2_255 - kMargin;  // c.w = 1 / opacity
    const float rx = rcp_approx(2.f * q.x), rz = rcp_approx(2.f * q.z);
    uint32_t keep = 0u;
    for (uint32_t mm = m; mm;) {
        const int r = __ffs(mm) - 1;
        mm &= mm - 1u;
        const float X0 = float(tx0 + (r & 1) * 8) - p.x, X1 = X0 + 7.f;   // dx range
        const float Y0 = float(ty0 + (r >> 1) * 4) - p.y, Y1 = Y0 + 3.f;  // dy range
        float best = -INFINITY;
        const bool inx = X0 <= 0.f && X1 >= 0.f, iny = Y0 <= 0.f && Y1 >= 0.f;
        if (inx && iny) best = 0.f;
        if (!inx) best = fmaxf(best, edge_peak(q.z, q.y, q.x, X0 > 0.f ? X0 : X1, Y0, Y1, rz));
        if (!iny) best = fmaxf(best, edge_peak(q.x, q.y, q.z, Y0 > 0.f ? Y0 : Y1, X0, X1, rx));
        if (best >= thr) keep |= 1u << r;
    }
    return keep;
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

// Shared staging of the forward: one batch of 256 entries.
struct FwdSmem {
    float4 p[kBatch], q[kBatch], c[kBatch];
    uint32_t mask[kBatch];
    uint8_t list[kFwdWarps][kBatch];
    uint8_t comp[kFwdWarps][kBatch];  // 1 where some pixel of the warp composited the entry
};

// Entry j of the staged batch: bit w set when warp w composited it at some pixel.
__device__ __forceinline__ uint8_t comp_byte(const FwdSmem& sm, int j) {
    uint32_t b = 0u;
#pragma unroll
    for (int w = 0; w < kFwdWarps; ++w) b |= uint32_t(sm.comp[w][j]) << w;
    return uint8_t(b);
}

// The forward of one tile.  SPLIT: the tile's list crosses a chunk boundary of the point list,
// so each pixel also sums the colour of every stretch between boundaries and records its state
// there for the backward; other tiles skip that work.  Measured and not kept: a branch-free blend
// (alpha taken as 0 where the pixel is done or below the threshold, a warp vote to leave the
// batch: 2% more instructions and no faster); each batch's list entries loaded while the batch
// before it is composited (2% more instructions, spills, 0.128 -> 0.130 ms).
template <bool SPLIT>
__device__ __forceinline__ void raster_fwd_tile(const CameraF& cam, uint32_t n, const Record* __restrict__ rec,
                                                uint32_t tile, uint2 range,
                                                const uint32_t* __restrict__ list, float3 bg,
                                                float* __restrict__ image, float* __restrict__ final_T,
                                                uint32_t* __restrict__ n_contrib, float4* __restrict__ ckpt,
                                                uint32_t slots, uint8_t* __restrict__ comp, int half, FwdSmem& sm) {
    const int warp = threadIdx.x >> 5;
    int tx0, ty0, ry0, px, py;
    tile_pixel(cam, int(tile), half, tx0, ty0, ry0, px, py);
    const bool inside = px < cam.W && py < cam.H;
    const float fx = float(px), fy = float(py);
    float T = 1.f, C0 = 0.f, C1 = 0.f, C2 = 0.f;
    float D0 = 0.f, D1 = 0.f, D2 = 0.f;  // colour added since the last chunk boundary (SPLIT)
    uint32_t stop = range.y;  // one past the last entry this pixel examined
    bool done = !inside;
    const uint32_t wbit = 1u << warp;
    uint8_t* my_list = sm.list[warp];
    const int lidx = (py - ty0) * kTile + (px - tx0);
    // batches end at the chunk boundaries of the point list; at each boundary inside the list a
    // pixel still going records T and the colour its previous stretch added
    uint32_t pbase = 0u, pend = 0u;  // the previous batch, whose composited flags go out next
    for (uint32_t base = range.x, bend; base < range.y; base = bend) {
        bend = min(range.y, (base / kChunk + 1) * kChunk);
        if (SPLIT && base != range.x && !done) {
            if (base / kChunk < slots) ckpt[size_t(base / kChunk) * kTilePixels + lidx] = make_float4(D0, D1, D2, T);
            // the finished stretch joins the colour in front
            C0 += D0;
            C1 += D1;
            C2 += D2;
            D0 = D1 = D2 = 0.f;
        }
        // every thread reaches this barrier; the block leaves once all its pixels are done
        const int ndone = __syncthreads_count(done);
#pragma unroll
        for (int t = threadIdx.x; t < kBatch; t += kFwdThreads)
            if (pbase + uint32_t(t) < pend) comp[pbase + t] = comp_byte(sm, t);
        pbase = base;
        pend = 0u;
        if (ndone == kFwdThreads) break;
        pend = bend;
#pragma unroll
        for (int t = threadIdx.x; t < kBatch; t += kFwdThreads) {
            const uint32_t e = base + uint32_t(t);
            uint32_t m = 0u;
            if (e < bend) {
                const uint32_t g = list[e];
                if (g >= n) {
                    atomicOr(&g_raster_check, 1u);  // caller data out of range: the entry is skipped
                } else {
                    const Record& r = rec[g];
                    sm.p[t] = r.p;
                    sm.q[t] = r.q;
                    sm.c[t] = r.c;
                    m = warp_mask(r.p, r.q, tx0, ry0);
#if RS_FWD_EXACT_MASK
                    if (m) m = warp_mask_exact(m, r.p, r.q, r.c, tx0, ry0);
#endif
                }
            }
            sm.mask[t] = m;
        }
        __syncthreads();
        // this warp's composited flags for the batch (the previous batch's were gathered before
        // the barrier above)
        reinterpret_cast<uint2*>(sm.comp[warp])[threadIdx.x & 31] = make_uint2(0u, 0u);
        __syncwarp();
        if (__all_sync(kFull, done)) continue;
        const int nl = compact_warp(my_list, [&](int j) { return (sm.mask[j] & wbit) != 0u; });
        if (done) continue;
        // entry j composited at this pixel; returns true when the pixel is done
        auto blend = [&](int j, float alpha) {
            sm.comp[warp][j] = 1u;  // every lane that composites stores the same flag
            const float4 c = sm.c[j];
            const float w = alpha * T;
            // a tile whose list crosses chunk boundaries sums the current stretch only (it joins
            // the colour in front at the stretch's end)
            if (SPLIT) {
                D0 = fmaf(c.x, w, D0);
                D1 = fmaf(c.y, w, D1);
                D2 = fmaf(c.z, w, D2);
            } else {
                C0 = fmaf(c.x, w, C0);
                C1 = fmaf(c.y, w, C1);
                C2 = fmaf(c.z, w, C2);
            }
            T = fmaf(-T, alpha, T);
            if (T < kTStop) {
                done = true;
                stop = base + uint32_t(j) + 1u;
            }
            return done;
        };
        // two entries per step: one list load, and the second alpha evaluated while the first
        // blends (the blends stay in list order)
        int k = 0;
        for (; k + 1 < nl; k += 2) {
            const uint32_t jj = *reinterpret_cast<const uint16_t*>(my_list + k);
            const int j0 = int(jj & 0xffu), j1 = int(jj >> 8);
            float dx, dy, G, raw;
            const float a0 = entry_alpha(sm.p[j0], sm.q[j0], fx, fy, dx, dy, G, raw);
            const float a1 = entry_alpha(sm.p[j1], sm.q[j1], fx, fy, dx, dy, G, raw);
            if (a0 >= kAlphaMin && blend(j0, a0)) break;
            if (a1 >= kAlphaMin && blend(j1, a1)) break;
        }
        if (k < nl && !done) {
            const int j = my_list[k];
            float dx, dy, G, raw;
            const float a = entry_alpha(sm.p[j], sm.q[j], fx, fy, dx, dy, G, raw);
            if (a >= kAlphaMin) blend(j, a);
        }
    }
    __syncthreads();
#pragma unroll
    for (int t = threadIdx.x; t < kBatch; t += kFwdThreads)
        if (pbase + uint32_t(t) < pend) comp[pbase + t] = comp_byte(sm, t);
    if (inside) {
        const size_t HW = size_t(cam.W) * cam.H, pix = size_t(py) * cam.W + px;
        // (D is the last stretch's colour with SPLIT, else 0)
        image[pix] = fmaf(T, bg.x, C0 + D0);
        image[HW + pix] = fmaf(T, bg.y, C1 + D1);
        image[2 * HW + pix] = fmaf(T, bg.z, C2 + D2);
        final_T[pix] = T;
        n_contrib[pix] = stop - range.x;
        // the backward resumes at each recorded boundary b with the colour behind it,
        // sum over entries from b on of colour alpha T, plus T bg: summed back to front from the
        // stretches' own sums (a difference of running totals would lose the small tail)
        if (SPLIT && stop > range.x) {
            float b0 = fmaf(T, bg.x, D0), b1 = fmaf(T, bg.y, D1), b2 = fmaf(T, bg.z, D2);
            for (uint32_t b = ((stop - 1u) / kChunk) * kChunk; b > range.x; b -= kChunk) {
                if (b / kChunk >= slots) continue;
                float4& f = ckpt[size_t(b / kChunk) * kTilePixels + lidx];
                const float4 d = f;
                f = make_float4(b0, b1, b2, d.w);
                b0 += d.x;
                b1 += d.y;
                b2 += d.z;
            }
        }
    }
}

__global__ void __launch_bounds__(kFwdThreads, RS_FWD_MIN_BLOCKS) k_raster_fwd(CameraF cam, uint32_t n, uint32_t cap,
                                                           const Record* __restrict__ rec,
                                                           const uint2* __restrict__ ranges,
                                                           const uint32_t* __restrict__ list,
                                                           float3 bg, float* __restrict__ image,
                                                           float* __restrict__ final_T,
                                                           uint32_t* __restrict__ n_contrib,
                                                           uint32_t* __restrict__ chunk_tile,
                                                           float4* __restrict__ ckpt, uint32_t slots,
                                                           const uint32_t* __restrict__ order,
                                                           uint8_t* __restrict__ comp, size_t comp_stride) {
    RS_PDL_ENTER();
    __shared__ FwdSmem sm;
    // blocks take the tiles in order, a tile's halves one after the other; half h writes its
    // composited flags to its own array (comp + h comp_stride)
    const uint32_t tile = order[blockIdx.x / uint32_t(kFwdHalves)];
    const int half = int(blockIdx.x % uint32_t(kFwdHalves));
    comp += size_t(half) * comp_stride;
    uint2 range = ranges[tile];
    if (range.y > cap || range.x > range.y) {
        // caller data out of range: the tile is drawn empty
        if (threadIdx.x == 0) atomicOr(&g_raster_check, 1u);
        range = make_uint2(0u, 0u);
    }
    // the tile's list positions that are multiples of the chunk size are the backward's task
    // starts: record which tile holds them
    if (half == 0)
        for (uint32_t c = (range.x + kChunk - 1) / kChunk + threadIdx.x;
             c < (range.y + kChunk - 1) / kChunk && c < slots; c += kFwdThreads)
            chunk_tile[c] = tile;
    if (range.y > range.x && (range.y - 1u) / kChunk > range.x / kChunk)
        raster_fwd_tile<true>(cam, n, rec, tile, range, list, bg, image, final_T, n_contrib, ckpt, slots, comp, half,
                              sm);
    else
        raster_fwd_tile<false>(cam, n, rec, tile, range, list, bg, image, final_T, n_contrib, ckpt, slots, comp, half,
                               sm);
}

// The backward's unit of work is one 8x8 square of one 256-entry chunk of the point list,
// [256 c, 256 c + 256), which may hold the end of one tile's list and several short lists after
// it (pieces).  A piece that stops at the chunk's end while its tile's list goes on starts each
// pixel from the state the forward recorded there, so a long list is walked by as many warps per
// square as it has chunks.  Each block is one warp, persistent: it takes work items (chunk,
// square) from a counter until the list ends.  Square s covers columns (s & 1) * 8 and rows
// (s >> 1) * 8 of the piece's tile, and lane l the two pixels (l & 7, l >> 3) and
// (l & 7, (l >> 3) + 4) of it.  A warp walks each piece back to front, 32 entries at a time: each
// lane reads one entry's composited flags from the forward and, where one of the two forward
// warps inside the square composited it (a hit), loads its record into the warp's shared-memory
// slots; the hits are evaluated one after another by all 64 pixels.  Each hit's nine sums over
// the square (dL/dpower times 1, dx, dy, dx^2, dx dy, dy^2, and alpha T_j times dL/dC) are
// deferred: the per-pixel dL/dpower and alpha T_j go to a shared-memory buffer of eight hits, and
// when it is full or the piece ends four lanes per hit add up its 64 pixels as moments, turn them
// into the Gaussian's gradient values and reduce-scatter those between them; one lane per value
// adds it to the Gaussian's gradient with a global atomic.  There are no block-wide barriers.
// Measured and not kept (160k 1080p orbit view): the nine sums of each hit (or of two hits at
// once) reduced over the whole warp with shuffles (0.220 ms against 0.192 for the deferred sums);
// four pixels per lane on 8x16 areas; four-warp blocks, one per chunk (0.195 against 0.177 ms for
// one-warp persistent blocks: a block's warps finish at different times and its slot waits for
// the last); a third form of the step for entries below every pixel's end (no end test: 126.2
// against 125.0 M instructions, no faster); a piece's pixel inputs (n_contrib, dL/dC, final_T
// and the checkpoint) all loaded at once instead of after n_contrib (0.159 -> 0.161 ms); the two
// pixels' arithmetic and the buffer sums in
// paired fp32 instructions (f32x2:
// 9% fewer instructions, but issue fell from 74% to 65% of cycles and the kernel took 187 against
// 176 us; the buffer sums alone: 6% fewer, the same time); the items taken heaviest first (a
// kernel between forward and backward filing each item in one of seven classes by the count of
// its composited entries: 0.182 against 0.178 ms, the heavy items of the dense regions running all
// at once).
constexpr int kBwdPx = 2;                        // pixels per lane, 4 rows apart in one column
constexpr int kSqH = 4 * kBwdPx;                 // rows of a square (8 columns wide)
constexpr int kBwdWarps = 2 * (kTile / kSqH);    // squares per tile
constexpr int kBwdThreads = 32;                  // one warp per block
// Hits buffered per warp before they are summed, and the buffer's row stride in float4 (33: the
// four lanes of a hit read lane slots 8r + i of rows h = 0..7 in one step, and the odd stride
// puts the eight rows on distinct banks).
constexpr int kHitBuf = 8;
constexpr int kHitStride = 33;
constexpr int kSlots = 32 + kHitBuf;  // record slots of the staged hits

// Per-pixel state of the reverse walk.
struct BwdPixel {
    float T, SG, G0, G1, G2;
    uint32_t end;  // one past the last entry of the piece the pixel examined
};

// One entry at one pixel: updates the pixel's state; returns gp = dL/dpower (0 if clamped) and
// w = alpha T_j.  Branch-free: a pixel the entry does not reach (act false) takes alpha as 0, so
// SG + 0 d = SG and w = gp = 0, and keeps T through the select; an active pixel gets exactly the
// arithmetic of the recurrence.  CLAMP false: the caller knows raw < kAlphaMax (see
// kNoClampOpacity), so no clamp test.
template <bool CLAMP>
__device__ __forceinline__ void bwd_step(BwdPixel& px, bool act, float alpha, float raw, const float4& c,
                                         float& gp, float& w) {
    const float a = act ? alpha : 0.f;
    const float Tj = act ? px.T * rcp_approx(1.f - alpha) : px.T;
    w = a * Tj;
    const float cG = fmaf(c.x, px.G0, fmaf(c.y, px.G1, c.z * px.G2));
    // dL/dalpha = Tj (cG - SG), and the entry's own colour joins SG: SG + alpha (cG - SG)
    const float d = cG - px.SG;
    px.SG = fmaf(a, d, px.SG);
    px.T = Tj;
    // alpha dL/dalpha where not clamped (alpha = opacity exp(power))
    gp = !CLAMP || raw <= kAlphaMax ? w * d : 0.f;
}

// An entry of opacity at most this cannot reach the 0.99 clamp at any pixel: opacity exp(power)
// with power <= 0 stays below it even when rounding leaves the evaluated exponent slightly
// positive (by less than log2(0.99 / 0.98) = 0.0146), so min(0.99, raw) = raw there, as in the
// forward, and the clamp test can be skipped.
constexpr float kNoClampOpacity = 0.98f;

__global__ void __launch_bounds__(kBwdThreads, RS_BWD_MIN_BLOCKS * kBwdWarps) k_raster_bwd(
    CameraF cam, int n, const Record* __restrict__ rec, const uint2* __restrict__ ranges,
    const uint32_t* __restrict__ list, float3 bg,
    const float* __restrict__ final_T, const uint32_t* __restrict__ n_contrib,
    const uint32_t* __restrict__ chunk_tile, const float4* __restrict__ ckpt, uint32_t slots,
    const uint8_t* __restrict__ comp, size_t comp_stride, uint32_t cap, const float* __restrict__ dL_dimage,
    float* __restrict__ dm2, float* __restrict__ dcon, float* __restrict__ dop, float* __restrict__ dcol,
    uint32_t* __restrict__ work) {
    RS_PDL_ENTER();
    // staged hits: up to kHitBuf - 1 carried over from the previous batch, then this batch's
    __shared__ float4 s_p[kSlots], s_q[kSlots], s_c[kSlots];
    // per buffered hit h and lane L: (dL/dpower, alpha T_j) at the lane's two pixels
    __shared__ float4 s_buf[kHitBuf][kHitStride];
    // dL/dC at lane L's two pixels: (G0, G1, G2 of the first, G0 of the second), (G1, G2 of it)
    __shared__ float4 s_ga[32];
    __shared__ float2 s_gb[32];
    const uint32_t n_tiles = uint32_t(cam.TX) * uint32_t(cam.TY);
    const unsigned lane = threadIdx.x;
    const size_t HW = size_t(cam.W) * cam.H;
    const size_t N = size_t(n);
    constexpr float kLn2 = 0.6931471805599453f;
    // Summing buffered hits, lane L serves hit L & 7 and the lane slots 8r .. 8r + 7 (pixel rows r
    // and r + 4 of the square, columns 0..7), r = L >> 3; after the reduce-scatter over the hit's
    // four lanes it holds the gradient values below and adds them to:
    //   r = 0: dmeans2d.x, dconic.C, dcolor.b     r = 1: dmeans2d.y, dopacity
    //   r = 2: dconic.A, dcolor.r                  r = 3: dconic.B, dcolor.g
    const int sr = int(lane >> 3), sh = int(lane & 7);
    // Persistent warps: warp w starts with (chunk, square) item w and, each time it finishes one,
    // takes the next in increasing order from work[0] (offset by the grid's warp count) until it
    // meets a chunk past the list's end; every later item is past it too.  An item is claimed only
    // when a warp is free for it (claimed ahead, it would wait behind the claimant's current item
    // while other warps idle at the end: 0.200 against 0.177 ms).  The last warp to leave resets
    // the counter.
    const uint32_t n_warps = gridDim.x;
    uint32_t item = blockIdx.x;
    for (;; item = __shfl_sync(kFull, lane == 0 ? n_warps + atomicAdd(work, 1u) : 0u, 0)) {
        const uint32_t chunk = item / uint32_t(kBwdWarps);
        const int sq = int(item % uint32_t(kBwdWarps));
        if (chunk >= slots) break;
        const uint32_t a0 = chunk * kChunk, a1 = a0 + kChunk;
        // the tile holding position a0; a chunk past the end of the list has none
        uint32_t tile = chunk_tile[chunk];
        if (tile >= n_tiles) break;
        uint2 range = ranges[tile];
        if (!(range.x <= a0 && a0 < range.y)) break;
        if (range.y > cap) {
            // caller data out of range (the forward drew this tile empty)
            if (lane == 0) atomicOr(&g_raster_check, 1u);
            continue;
        }
        uint32_t pa = a0;
        while (true) {
            // the piece [pa, pb) of this tile's list
            const uint32_t pb = min(range.y, a1);
            const int tx0 = int(tile % uint32_t(cam.TX)) * kTile, ty0 = int(tile / uint32_t(cam.TX)) * kTile;
            const int sx = tx0 + (sq & 1) * 8, sy = ty0 + (sq >> 1) * kSqH;
            const int px = sx + int(lane & 7);
            const int py0 = sy + int(lane >> 3);
            const uint32_t len = range.y - range.x;
            BwdPixel P[kBwdPx];
#pragma unroll
            for (int h = 0; h < kBwdPx; ++h) {
                const int py = py0 + 4 * h;
                const bool inside = px < cam.W && py < cam.H;
                const size_t pix = inside ? size_t(py) * cam.W + px : 0;
                // n_contrib never exceeds the list length when it comes from rs_rasterize_fwd; the
                // min() keeps inconsistent caller data inside the tile's list
                const uint32_t end = range.x + (inside ? min(n_contrib[pix], len) : 0u);
                P[h].end = min(end, pb);
                P[h].G0 = P[h].G1 = P[h].G2 = 0.f;
                P[h].T = 1.f;
                P[h].SG = 0.f;
                if (end > pa) {
                    P[h].G0 = dL_dimage[pix];
                    P[h].G1 = dL_dimage[HW + pix];
                    P[h].G2 = dL_dimage[2 * HW + pix];
                    const uint32_t ck = pb / kChunk;
                    if (end > pb && ck < slots) {
                        // the pixel goes on past the chunk: resume from the forward's state at pb,
                        // (colour behind pb, T); the colour behind per unit T enters as its dot
                        // product with dL/dC
                        const float4 f = ckpt[size_t(ck) * kTilePixels + (py - ty0) * kTile + (px - tx0)];
                        P[h].T = f.w;
                        P[h].SG = __fdividef(fmaf(P[h].G0, f.x, fmaf(P[h].G1, f.y, P[h].G2 * f.z)), f.w);
                    } else {
                        // the colour behind an entry (per unit T) only enters the gradient through
                        // its dot product with dL/dC, so that scalar is carried instead of the colour
                        P[h].T = final_T[pix];
                        P[h].SG = bg.x * P[h].G0 + bg.y * P[h].G1 + bg.z * P[h].G2;
                    }
                }
            }
            // the sums of the buffered hits read every lane's dL/dC (the previous piece's last read of
            // these ended with a warp barrier)
            s_ga[lane] = make_float4(P[0].G0, P[0].G1, P[0].G2, P[1].G0);
            s_gb[lane] = make_float2(P[1].G1, P[1].G2);
            uint32_t lane_end = P[0].end;
#pragma unroll
            for (int h = 1; h < kBwdPx; ++h) lane_end = max(lane_end, P[h].end);
            const uint32_t warp_end = __reduce_max_sync(kFull, lane_end);
            const float fx = float(px), fy0 = float(py0);
            // the forward's warps (8x4 pixels) inside this warp's area, numbered within the forward
            // block's region (the square's half of the tile with half-tile blocks): an entry none
            // of them composited has no active pixel here
            const int fr0 = (sy - ty0) / 4 - (RS_FWD_HALF ? 2 * (sq >> 1) : 0);
            const uint8_t* const compq = comp + (RS_FWD_HALF ? size_t(sq >> 1) * comp_stride : size_t(0));
            uint32_t fwarps = 0u;
#pragma unroll
            for (int r = 0; r < kSqH / 4; ++r) fwarps |= 1u << ((fr0 + r) * 2 + (sq & 1));
            // The buffered hits' sums.  Lane (hit sh, row sr) adds up its eight lane slots as
            // moments about the square's middle column (dx = bx + i - 3.5 at column i, dy = by0 or
            // by1 on its two pixel rows), turns them into the hit's gradient values, and the
            // hit's four lanes reduce-scatter those (xor 16, then xor 8) before the atomics.
            auto flush = [&](int cnt, int r0) {
                __syncwarp();
                const float4* b = s_buf[sh] + 8 * sr;
                const float4* ga = s_ga + 8 * sr;
                const float2* gb = s_gb + 8 * sr;
                float S0 = 0.f, S1 = 0.f, X0 = 0.f, X1 = 0.f, XX = 0.f, C0 = 0.f, C1 = 0.f, C2 = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float xi = float(i) - 3.5f;
                    const float4 v = b[i];  // (gp, gp', w, w') at the slot's two pixels
                    const float4 g4 = ga[i];
                    const float2 g2 = gb[i];
                    S0 += v.x;
                    S1 += v.y;
                    X0 = fmaf(v.x, xi, X0);
                    X1 = fmaf(v.y, xi, X1);
                    XX = fmaf(v.x + v.y, xi * xi, XX);
                    C0 = fmaf(v.z, g4.x, fmaf(v.w, g4.w, C0));
                    C1 = fmaf(v.z, g4.y, fmaf(v.w, g2.x, C1));
                    C2 = fmaf(v.z, g4.z, fmaf(v.w, g2.y, C2));
                }
                // lanes past the buffered count compute on stale slots and add nothing
                const int j = min(r0 + sh, kSlots - 1);
                const float4 p = s_p[j], q = s_q[j];
                const float iop = s_c[j].w;
                const float bx = (float(sx) + 3.5f) - p.x;
                const float by0 = float(sy + sr) - p.y, by1 = float(sy + sr + 4) - p.y;
                const float S = S0 + S1, X = X0 + X1;
                const float Sdx = fmaf(bx, S, X);          // sum gp dx
                const float Sdx2 = fmaf(bx, Sdx + X, XX);  // sum gp dx^2
                const float u0 = by0 * S0, u1 = by1 * S1;
                const float Sdy = u0 + u1;                 // sum gp dy
                const float Sdy2 = fmaf(by0, u0, by1 * u1);  // sum gp dy^2
                const float Sdxdy = fmaf(by0, fmaf(bx, S0, X0), by1 * fmaf(bx, S1, X1));
                // the conic from the record's log2-scaled quadratic: A = -2 ln2 qa, B = -ln2 qb, ...
                const float A = -2.f * kLn2 * q.x, B = -kLn2 * q.y, C = -2.f * kLn2 * q.z;
                // (du, dv, dA, dB, dC, dopacity, dcolour): split into the values rows 0 and 1 keep
                // (du, dv, dC, dopacity, db) and those rows 2 and 3 keep (dA, dB, dr, dg)
                const float lo[5] = {fmaf(A, Sdx, B * Sdy), fmaf(C, Sdy, B * Sdx), -0.5f * Sdy2, iop * S, C2};
                const float hi[5] = {-0.5f * Sdx2, -Sdxdy, C0, C1, 0.f};
                const bool r1 = sr & 2, r0b = sr & 1;
                float a[5];
#pragma unroll
                for (int k = 0; k < 5; ++k)
                    a[k] = (r1 ? hi[k] : lo[k]) + __shfl_xor_sync(kFull, r1 ? lo[k] : hi[k], 16);
                const float v0 = (r0b ? a[1] : a[0]) + __shfl_xor_sync(kFull, r0b ? a[0] : a[1], 8);
                const float v1 = (r0b ? a[3] : a[2]) + __shfl_xor_sync(kFull, r0b ? a[2] : a[3], 8);
                const float v2 = (r0b ? 0.f : a[4]) + __shfl_xor_sync(kFull, r0b ? a[4] : 0.f, 8);
                if (sh < cnt) {
                    const size_t gi = __float_as_uint(p.w);
                    float* const dst0 = sr == 0 ? dm2 : sr == 1 ? dm2 + N : sr == 2 ? dcon : dcon + N;
                    float* const dst1 = sr == 0 ? dcon + 2 * N : sr == 1 ? dop : sr == 2 ? dcol : dcol + N;
                    atomicAdd(dst0 + gi, v0);
                    atomicAdd(dst1 + gi, v1);
                    if (sr == 0) atomicAdd(dcol + 2 * N + gi, v2);
                }
                __syncwarp();  // the buffer is read before the next hits overwrite it
            };
            // the buffered hits: slots r0 .. r0 + cnt - 1, buffer rows 0 .. cnt - 1; a buffer not
            // yet full at a batch's end is carried into the next batch
            int cnt = 0, r0 = 0;
            // each batch's list entries and composited flags are loaded one batch ahead
            uint32_t g_next = 0u, f_next = 0u;
            if (warp_end > pa) {
                const uint32_t lo1 = warp_end - pa > 32u ? warp_end - 32u : pa;
                if (lo1 + lane < warp_end) {
                    g_next = list[lo1 + lane];
                    f_next = compq[lo1 + lane];
                }
            }
            for (uint32_t hi = warp_end; hi > pa;) {
                const uint32_t lo = hi - pa > 32u ? hi - 32u : pa;
                const uint32_t e = lo + lane;
                const uint32_t g_cur = g_next, f_cur = f_next;
                g_next = f_next = 0u;
                if (lo > pa) {
                    const uint32_t lo2 = lo - pa > 32u ? lo - 32u : pa;
                    if (lo2 + lane < lo) {
                        g_next = list[lo2 + lane];
                        f_next = compq[lo2 + lane];
                    }
                }
                if (r0 > 0 && cnt > 0) {
                    // the carried hits move to the front slots (r0 >= kHitBuf > cnt: no overlap)
                    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a, c = a;
                    if (int(lane) < cnt) {
                        a = s_p[r0 + lane];
                        b = s_q[r0 + lane];
                        c = s_c[r0 + lane];
                    }
                    __syncwarp();
                    if (int(lane) < cnt) {
                        s_p[lane] = a;
                        s_q[lane] = b;
                        s_c[lane] = c;
                    }
                    __syncwarp();
                }
                r0 = 0;
                bool hit = false;
                uint32_t g = 0u;
                if (e < hi) {
                    // an entry some forward warp of this area composited (its alpha >= 1/255 box
                    // meets the area then too): only those records are loaded
                    g = g_cur;
                    hit = (f_cur & fwarps) != 0u;
                    if (hit && g >= uint32_t(n)) {
                        atomicOr(&g_raster_check, 1u);  // caller data out of range: the entry is skipped
                        hit = false;
                    }
                }
                const uint32_t m = __ballot_sync(kFull, hit);
                const int nh = __popc(m);
                if (hit) {
                    // the hits are taken back to front and staged in that order after the carried
                    // ones: slot cnt + r holds the hit with r hits above it, so that a buffer's hits
                    // sit in consecutive slots
                    const int r = cnt + __popc(m & (0xfffffffeu << lane));
                    const Record& rc = rec[g];
                    const float4 p = rc.p, q = rc.q, c = rc.c;
                    // the backward uses neither extent: p.w carries the Gaussian's index, q.w the
                    // entry's list position
                    s_p[r] = make_float4(p.x, p.y, p.z, __uint_as_float(g));
                    s_q[r] = make_float4(q.x, q.y, q.z, __uint_as_float(e));
                    s_c[r] = c;
                }
                __syncwarp();
                // the hit in slot j at the lane's pixels: updates their state
                auto step = [&](int j, float& dx, float (&dy)[kBwdPx], float (&gp)[kBwdPx], float (&w)[kBwdPx]) {
                    const float4 p = s_p[j], q = s_q[j];
                    const uint32_t ej = __float_as_uint(q.w);
                    // the lane's pixels share a column: dx and its terms are common (the same
                    // arithmetic as entry_alpha, pixel by pixel)
                    dx = fx - p.x;
                    const float bx = q.y * dx, axx = (q.x * dx) * dx;
                    const float4 c = s_c[j];
                    auto pixels = [&](auto clamp) {
#pragma unroll
                        for (int h = 0; h < kBwdPx; ++h) {
                            dy[h] = (fy0 + float(4 * h)) - p.y;
                            const float raw = p.z * ex2_approx(fmaf(dy[h], fmaf(q.z, dy[h], bx), axx));
                            const float al = decltype(clamp)::value ? fminf(kAlphaMax, raw) : raw;
                            bwd_step<decltype(clamp)::value>(P[h], ej < P[h].end && al >= kAlphaMin, al, raw, c,
                                                             gp[h], w[h]);
                        }
                    };
                    // the branch is the same for the whole warp (one entry)
                    if (p.z <= kNoClampOpacity) pixels(std::false_type{});
                    else pixels(std::true_type{});
                };
                // every hit has a composited pixel in this area (the forward's flags); back to front,
                // each hit's per-pixel values go to the buffer, which is summed when full (a partial
                // buffer is carried to the next batch, and summed at the piece's end)
                for (int j = 0; j < nh; ++j) {
                    float dx, dy[kBwdPx], gp[kBwdPx], w[kBwdPx];
                    step(r0 + cnt, dx, dy, gp, w);
                    s_buf[cnt][lane] = make_float4(gp[0], gp[1], w[0], w[1]);
                    if (++cnt == kHitBuf) {
                        flush(cnt, r0);
                        r0 += cnt;
                        cnt = 0;
                    }
                }
                __syncwarp();  // the slots are read before the next batch overwrites them
                hi = lo;
            }
            // the piece's last hits (their sums use this piece's pixels)
            if (cnt > 0) flush(cnt, r0);
            if (pb >= a1) break;
            // this tile's list ended inside the chunk: the next non-empty list starts at pb (unless
            // pb is the end of the point list)
            uint32_t nt = n_tiles;
            for (uint32_t u = tile + 1; u < n_tiles; u += 32) {
                const uint32_t t = u + lane;
                const uint2 r = t < n_tiles ? ranges[t] : make_uint2(0u, 0u);
                const uint32_t b = __ballot_sync(kFull, r.y > r.x);
                if (b) {
                    nt = u + uint32_t(__ffs(b) - 1);
                    break;
                }
            }
            if (nt >= n_tiles) break;
            tile = nt;
            range = ranges[tile];
            if (range.x != pb || range.y > cap) break;
            pa = pb;
        }
    }
    if (lane == 0 && atomicAdd(work + 1, 1u) == n_warps - 1u) {
        work[0] = 0u;
        work[1] = 0u;
    }
}

__global__ void k_fill_background(CameraF cam, float3 bg, float* image, float* final_T,
                                  uint32_t* n_contrib) {
    RS_PDL_ENTER();
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
    RS_PDL_ENTER();
    const size_t stride = size_t(gridDim.x) * blockDim.x;
#pragma unroll
    for (int k = 0; k < 4; ++k)
        for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < z.count[k]; i += stride)
            z.p[k][i] = 0.f;
}

}  // namespace

namespace {
struct RasterWs {
    uint32_t* chunk_tile;   // [slots] tile holding list position 256 c
    float4* ckpt;           // [slots][256] the forward's state at position 256 c
    uint32_t* order;        // [n_tiles] tiles in the forward's order
    uint8_t* comp;          // [halves][comp_stride] per entry: the forward warps (8x4 pixels) that composited it
    size_t comp_stride;     // the capacity rounded up to 256
    uint32_t* work;         // [2] the backward's next work item and count of finished warps
    uint32_t slots;
};
size_t align256z(size_t x) { return (x + 255) & ~size_t(255); }
RasterWs raster_ws(void* ws, size_t capacity, size_t n_tiles, size_t* bytes = nullptr) {
    const size_t slots = capacity / kChunk + 1;
    uint8_t* b = static_cast<uint8_t*>(ws);
    size_t o = 0;
    RasterWs w;
    w.chunk_tile = reinterpret_cast<uint32_t*>(b + o);
    o = align256z(o + slots * sizeof(uint32_t));
    w.order = reinterpret_cast<uint32_t*>(b + o);
    o = align256z(o + n_tiles * sizeof(uint32_t));
    w.ckpt = reinterpret_cast<float4*>(b + o);
    o = align256z(o + slots * kTilePixels * sizeof(float4));
    w.comp = b + o;
    w.comp_stride = align256z(capacity);
    o += size_t(kFwdHalves) * w.comp_stride;
    w.work = reinterpret_cast<uint32_t*>(b + o);
    o += 2 * sizeof(uint32_t);
    w.slots = uint32_t(slots);
    if (bytes) *bytes = o;
    return w;
}

// Tiles in decreasing order of list length, in six classes (>= 1024, 512, 256, 128, 32 entries,
// shorter): the forward's blocks take tiles in this order, so the longest lists start first and
// the short ones fill in around them (the hardware hands out blocks in index order as earlier
// ones finish).  One block; a warp ranks its tiles per class with ballots, the warps' class
// counts are scanned class-major, and every tile is written to its slot (deterministic).
constexpr int kOrderThreads = 1024;
constexpr int kOrderWarps = kOrderThreads / 32;
constexpr int kOrderPer = 8;  // tiles per thread per round (8160 tiles at 1080p: one round)
constexpr int kClasses = 6;  // fewer measured slower: 2 classes 0.156 ms, 3 0.140, 4 0.132, 6 0.133
__device__ __forceinline__ int tile_class(uint2 r) {
    const uint32_t len = r.y > r.x ? r.y - r.x : 0u;
    return len >= 1024u ? 0 : len >= 512u ? 1 : len >= 256u ? 2 : len >= 128u ? 3 : len >= 32u ? 4 : 5;
}

__global__ void __launch_bounds__(kOrderThreads) k_tile_order(const uint2* __restrict__ ranges, uint32_t n_tiles,
                                                             uint32_t* __restrict__ order,
                                                             uint32_t* __restrict__ work) {
    RS_PDL_ENTER();
    // the backward's work counter starts at zero after every forward (each backward leaves it there)
    if (threadIdx.x == 0) {
        work[0] = 0u;
        work[1] = 0u;
    }
    __shared__ uint32_t s_cnt[kClasses][kOrderWarps];
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5, lt = (1u << lane) - 1u;
    // 1. per warp and class: the number of tiles
    uint32_t cnt[kClasses] = {};
    for (uint32_t base = 0; base < n_tiles; base += kOrderThreads * kOrderPer) {
#pragma unroll
        for (int k = 0; k < kOrderPer; ++k) {
            const uint32_t t = base + k * kOrderThreads + threadIdx.x;
            const int c = t < n_tiles ? tile_class(ranges[t]) : kClasses;
#pragma unroll
            for (int j = 0; j < kClasses; ++j) cnt[j] += __popc(__ballot_sync(kFull, c == j));
        }
    }
    if (lane == 0)
#pragma unroll
        for (int j = 0; j < kClasses; ++j) s_cnt[j][warp] = cnt[j];
    __syncthreads();
    // 2. exclusive scan in (class, warp) order by one warp
    if (warp == 0) {
        uint32_t carry = 0u;
        for (int j = 0; j < kClasses; ++j) {
            const uint32_t v = s_cnt[j][lane];
            uint32_t x = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(kFull, x, o);
                if (lane >= uint32_t(o)) x += y;
            }
            s_cnt[j][lane] = carry + x - v;
            carry += __shfl_sync(kFull, x, 31);
        }
    }
    __syncthreads();
    // 3. every tile to its slot: warp offset + earlier tiles of its class in the warp
    uint32_t run[kClasses];
#pragma unroll
    for (int j = 0; j < kClasses; ++j) run[j] = s_cnt[j][warp];
    for (uint32_t base = 0; base < n_tiles; base += kOrderThreads * kOrderPer) {
#pragma unroll
        for (int k = 0; k < kOrderPer; ++k) {
            const uint32_t t = base + k * kOrderThreads + threadIdx.x;
            const int c = t < n_tiles ? tile_class(ranges[t]) : kClasses;
#pragma unroll
            for (int j = 0; j < kClasses; ++j) {
                const uint32_t m = __ballot_sync(kFull, c == j);
                if (c == j) order[run[j] + uint32_t(__popc(m & lt))] = t;
                run[j] += __popc(m);
            }
        }
    }
}
}  // namespace

int take_raster_check() {
    unsigned int v = 0u;
    if (cudaMemcpyFromSymbol(&v, g_raster_check, sizeof(v)) != cudaSuccess) return -1;
    if (v == 0u) return 0;
    const unsigned int zero = 0u;
    if (cudaMemcpyToSymbol(g_raster_check, &zero, sizeof(zero)) != cudaSuccess) return -1;
    return 1;
}

size_t raster_workspace_bytes(size_t capacity, size_t n_tiles) {
    size_t bytes = 0;
    raster_ws(nullptr, capacity, n_tiles, &bytes);
    return bytes;
}

cudaError_t launch_raster_fwd(const CameraF& cam, int32_t n, const Record* rec, const uint32_t* ranges,
                              const uint32_t* list, size_t capacity, float3 bg, float* image, float* final_T,
                              uint32_t* n_contrib, void* ws, cudaStream_t s) {
    const int tiles = cam.TX * cam.TY;
    const RasterWs w = raster_ws(ws, capacity, size_t(tiles));
    pdl_launch(k_tile_order, 1, kOrderThreads, 0, s, reinterpret_cast<const uint2*>(ranges), uint32_t(tiles), w.order,
               w.work);
    pdl_launch(k_raster_fwd, unsigned(tiles * kFwdHalves), kFwdThreads, 0, s, cam, uint32_t(n), uint32_t(capacity),
               rec, reinterpret_cast<const uint2*>(ranges), list, bg, image, final_T, n_contrib, w.chunk_tile, w.ckpt,
               w.slots, w.order, w.comp, w.comp_stride);
    return cudaGetLastError();
}

cudaError_t launch_raster_bwd(const CameraF& cam, int32_t n, const Record* rec,
                              const uint32_t* ranges, const uint32_t* list, size_t capacity, float3 bg,
                              const float* final_T, const uint32_t* n_contrib, void* ws,
                              const float* dL_dimage, float* dm2, float* dcon, float* dop, float* dcol,
                              cudaStream_t s) {
    const RasterWs w = raster_ws(ws, capacity, size_t(cam.TX) * cam.TY);
    // one-warp blocks, as many as fit on the GPU at once (at most one per item of the capacity),
    // each taking (chunk, square) items until the list ends
    const size_t chunks = (capacity + kChunk - 1) / kChunk;
    if (chunks == 0) return cudaSuccess;
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_raster_bwd, kBwdThreads, 0);
    if (e != cudaSuccess) return e;
    const size_t blocks = std::min(chunks * size_t(kBwdWarps), size_t(std::max(sms, 1)) * size_t(std::max(per_sm, 1)));
    pdl_launch(k_raster_bwd, unsigned(blocks), kBwdThreads, 0, s, cam, n, rec, reinterpret_cast<const uint2*>(ranges),
               list, bg, final_T, n_contrib, w.chunk_tile, w.ckpt, w.slots, w.comp, w.comp_stride,
               uint32_t(capacity), dL_dimage, dm2, dcon, dop, dcol, w.work);
    return cudaGetLastError();
}

cudaError_t launch_fill_background(const CameraF& cam, float3 bg, float* image, float* final_T,
                                   uint32_t* n_contrib, cudaStream_t s) {
    const size_t HW = size_t(cam.W) * cam.H;
    const unsigned blocks = unsigned(std::min<size_t>((HW + 255) / 256, 152 * 16));
    pdl_launch(k_fill_background, blocks, 256, 0, s, cam, bg, image, final_T, n_contrib);
    return cudaGetLastError();
}

cudaError_t launch_zero_grads(float* dm2, float* dcon, float* dop, float* dcol, size_t n,
                              cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    ZeroSpans z{{dm2, dcon, dop, dcol}, {2 * n, 3 * n, n, 3 * n}};
    const unsigned blocks = unsigned(std::min<size_t>((3 * n + 255) / 256, 152 * 8));
    pdl_launch(k_zero4, blocks, 256, 0, s, z);
    return cudaGetLastError();
}

}  // namespace rs
