// [2] binning: exclusive scan of tiles_touched, load-balanced expansion into 64-bit keys, a
// stable LSD radix sort over the bits the tile count needs, and tile-range extraction.
//
// rigel README "Binning" (key = (tile_id << 32) | float_bits(depth), a sort restricted to the
// occupied bits, a range kernel); "3D Gaussian Splatting ビューワを作る" 4.1 (exclusive scan
// giving each Gaussian a private slice), 4.2 (duplicate), 4.3 (8-bit digits, per-block
// histograms, bin offsets from a scan over (digit, block), in-bin ranks, ping-pong buffers),
// 4.4 (ranges; empty tiles cleared to (0, 0)).
//
// GB300 design: every kernel is a plain grid over the data with no inter-block waiting (the
// sort is reduce-then-scan, not a chained look-back), so no launch can stall on another block.
// Working sets of the headline workloads (a few million 12-byte entries) sit in the 126 MB L2.
#include "rs_internal.cuh"

namespace rs {
namespace {

constexpr int kScanThreads = 256;
constexpr int kScanItems = 8;
constexpr int kScanChunk = kScanThreads * kScanItems;  // 2048 elements per block

constexpr int kSortThreads = 256;
constexpr int kSortIters = 16;
constexpr int kSortTile = kSortThreads * kSortIters;  // 4096 keys per block
constexpr int kRadixBits = 8;
constexpr int kRadix = 1 << kRadixBits;

size_t ceil_div(size_t a, size_t b) { return (a + b - 1) / b; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ---------------------------------------------------------------- device-wide exclusive scan
// Three phases per level: per-chunk sums, a scan of those sums (recursively), then a per-chunk
// scan seeded with its chunk's offset.

__device__ __forceinline__ uint64_t block_exclusive_scan(uint64_t v, uint64_t* s_warp, uint64_t& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint64_t w = lane < (kScanThreads / 32) ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < (kScanThreads / 32)) s_warp[lane] = w;
    }
    __syncthreads();
    total = s_warp[kScanThreads / 32 - 1];
    const uint64_t before = warp > 0 ? s_warp[warp - 1] : 0;
    __syncthreads();
    return before + x - v;
}

template <typename In>
__global__ void __launch_bounds__(kScanThreads) k_scan_reduce(const In* __restrict__ in, size_t n,
                                                              uint64_t* __restrict__ sums) {
    __shared__ uint64_t s_warp[kScanThreads / 32];
    const size_t base = size_t(blockIdx.x) * kScanChunk;
    uint64_t acc = 0;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        const size_t i = base + size_t(k) * kScanThreads + threadIdx.x;
        if (i < n) acc += uint64_t(in[i]);
    }
    uint64_t total;
    block_exclusive_scan(acc, s_warp, total);
    if (threadIdx.x == 0) sums[blockIdx.x] = total;
}

// Scans [0, n) of `in` into `out` (exclusive), adding offsets[blockIdx.x] (if given); if
// `total_out` is given, the grand total is written there by the last block.
template <typename In, typename Out>
__global__ void __launch_bounds__(kScanThreads) k_scan_down(const In* __restrict__ in, size_t n,
                                                            const uint64_t* __restrict__ offsets,
                                                            Out* __restrict__ out,
                                                            uint64_t* __restrict__ total_out) {
    __shared__ uint64_t s_data[kScanChunk];
    __shared__ uint64_t s_warp[kScanThreads / 32];
    const size_t base = size_t(blockIdx.x) * kScanChunk;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        const int j = k * kScanThreads + threadIdx.x;
        const size_t i = base + j;
        s_data[j] = i < n ? uint64_t(in[i]) : 0;
    }
    __syncthreads();
    uint64_t local[kScanItems];
    uint64_t acc = 0;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        local[k] = acc;
        acc += s_data[threadIdx.x * kScanItems + k];
    }
    uint64_t total;
    const uint64_t pre = block_exclusive_scan(acc, s_warp, total);
    const uint64_t off = offsets ? offsets[blockIdx.x] : 0;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) s_data[threadIdx.x * kScanItems + k] = off + pre + local[k];
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        const int j = k * kScanThreads + threadIdx.x;
        const size_t i = base + j;
        if (i < n) out[i] = Out(s_data[j]);
    }
    if (total_out && blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) *total_out = off + total;
}

size_t scan_tmp_elems(size_t n) {
    size_t t = 0;
    while (n > size_t(kScanChunk)) {
        n = ceil_div(n, kScanChunk);
        t += n;
    }
    return t;
}

// Exclusive scan of n elements into out; `tmp` holds scan_tmp_elems(n) uint64_t.
template <typename In, typename Out>
cudaError_t device_exclusive_scan(const In* in, size_t n, Out* out, uint64_t* total,
                                  uint64_t* tmp, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const size_t blocks = ceil_div(n, kScanChunk);
    if (blocks == 1) {
        k_scan_down<In, Out><<<1, kScanThreads, 0, s>>>(in, n, nullptr, out, total);
        return cudaGetLastError();
    }
    uint64_t* sums = tmp;
    k_scan_reduce<In><<<unsigned(blocks), kScanThreads, 0, s>>>(in, n, sums);
    // scan the block sums in place (exclusive), recursively
    cudaError_t e = device_exclusive_scan<uint64_t, uint64_t>(sums, blocks, sums, nullptr,
                                                              tmp + blocks, s);
    if (e != cudaSuccess) return e;
    k_scan_down<In, Out><<<unsigned(blocks), kScanThreads, 0, s>>>(in, n, sums, out, total);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- ranges
__global__ void k_clear_ranges(uint32_t* ranges, int n_tiles) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t < n_tiles) reinterpret_cast<uint2*>(ranges)[t] = make_uint2(0u, 0u);
}

__global__ void k_ranges(const uint64_t* __restrict__ keys, uint32_t E, uint32_t n_tiles,
                         uint32_t* ranges) {
    const uint32_t e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    const uint32_t tile = uint32_t(keys[e] >> 32);
    if (tile >= n_tiles) return;  // unreachable for keys made by k_expand; keeps writes in bounds
    if (e == 0 || uint32_t(keys[e - 1] >> 32) != tile) ranges[2 * size_t(tile)] = e;
    if (e == E - 1 || uint32_t(keys[e + 1] >> 32) != tile) ranges[2 * size_t(tile) + 1] = e + 1;
}

// ---------------------------------------------------------------- expansion
// One thread per entry: the owning Gaussian is the last g with offsets[g] <= e (offsets holds
// n+1 values, offsets[n] = E); the entry's position inside the Gaussian's span, row-major
// (tile rows outer, columns inner), gives its tile.
__global__ void __launch_bounds__(256) k_expand(CameraF cam, int n, uint32_t E,
                                                const uint64_t* __restrict__ offsets,
                                                const float* __restrict__ means2d,
                                                const float* __restrict__ depth,
                                                const int* __restrict__ radius,
                                                uint64_t* __restrict__ keys,
                                                uint32_t* __restrict__ vals) {
    const uint32_t e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    int lo = 0, hi = n;  // invariant: offsets[lo] <= e < offsets[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (offsets[mid] <= e) lo = mid; else hi = mid;
    }
    const int g = lo;
    const uint32_t k = e - uint32_t(offsets[g]);
    const float u = means2d[g], v = means2d[size_t(n) + g];
    const float r = float(radius[g]);
    const int xl = span_bound(u, r, cam.TX, false), xh = span_bound(u, r, cam.TX, true);
    const int yl = span_bound(v, r, cam.TY, false);
    // sx >= 1 whenever tiles_touched[g] > 0 came from rs_project (same span arithmetic); the
    // max() only keeps inconsistent caller data from dividing by zero
    const uint32_t sx = uint32_t(max(xh - xl, 1));
    const uint32_t tx = uint32_t(xl) + k % sx, ty = uint32_t(yl) + k / sx;
    const uint64_t tile = uint64_t(ty) * uint64_t(cam.TX) + tx;
    keys[e] = (tile << 32) | uint64_t(__float_as_uint(depth[g]));
    vals[e] = uint32_t(g);
}

// ---------------------------------------------------------------- radix sort (one 8-bit digit)
// Per-block digit histogram, written digit-major: hist[d * blocks + b].
__global__ void __launch_bounds__(kSortThreads) k_radix_hist(const uint64_t* __restrict__ keys,
                                                             uint32_t E, int shift,
                                                             uint32_t* __restrict__ hist) {
    __shared__ uint32_t s_hist[kRadix];
    s_hist[threadIdx.x] = 0;
    __syncthreads();
    const uint32_t lane = threadIdx.x & 31;
    const size_t base = size_t(blockIdx.x) * kSortTile;
    for (int it = 0; it < kSortIters; ++it) {
        const size_t i = base + size_t(it) * kSortThreads + threadIdx.x;
        const bool valid = i < E;
        const uint32_t d = valid ? uint32_t(keys[i] >> shift) & (kRadix - 1) : kRadix;
        const uint32_t peers = __match_any_sync(0xffffffffu, d);
        if (valid && lane == uint32_t(__ffs(peers) - 1)) atomicAdd(&s_hist[d], uint32_t(__popc(peers)));
    }
    __syncthreads();
    hist[size_t(threadIdx.x) * gridDim.x + blockIdx.x] = s_hist[threadIdx.x];
}

// Stable scatter of one digit.  Within a block, keys are taken 256 at a time in index order; a
// key's destination is the global offset of (digit, block) plus the count of equal digits
// before it in this block: earlier rounds (s_base), earlier warps (per-warp counts scanned
// over warps) and earlier lanes (popcount of the matching-digit lane mask).
__global__ void __launch_bounds__(kSortThreads) k_radix_scatter(
    const uint64_t* __restrict__ keys_in, const uint32_t* __restrict__ vals_in, uint32_t E,
    int shift, const uint32_t* __restrict__ hist_scanned, uint64_t* __restrict__ keys_out,
    uint32_t* __restrict__ vals_out) {
    constexpr int kWarps = kSortThreads / 32;
    __shared__ uint32_t s_wcount[2][kWarps][kRadix];
    __shared__ uint32_t s_base[kRadix];
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    s_base[threadIdx.x] = hist_scanned[size_t(threadIdx.x) * gridDim.x + blockIdx.x];
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        s_wcount[0][w][threadIdx.x] = 0;
        s_wcount[1][w][threadIdx.x] = 0;
    }
    __syncthreads();
    const uint32_t lt_mask = (1u << lane) - 1u;
    const size_t base = size_t(blockIdx.x) * kSortTile;
    for (int it = 0; it < kSortIters; ++it) {
        const int buf = it & 1;
        const size_t i = base + size_t(it) * kSortThreads + threadIdx.x;
        const bool valid = i < E;
        uint64_t key = 0;
        uint32_t val = 0;
        if (valid) {
            key = keys_in[i];
            val = vals_in[i];
        }
        const uint32_t d = valid ? uint32_t(key >> shift) & (kRadix - 1) : kRadix;
        const uint32_t peers = __match_any_sync(0xffffffffu, d);
        const uint32_t rank = __popc(peers & lt_mask);
        if (valid && rank == 0) s_wcount[buf][warp][d] = __popc(peers);
        __syncthreads();
        {  // thread t owns digit t: exclusive scan over warps, seeded by the running base
            uint32_t run = s_base[threadIdx.x];
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const uint32_t c = s_wcount[buf][w][threadIdx.x];
                s_wcount[buf][w][threadIdx.x] = run;
                run += c;
            }
            s_base[threadIdx.x] = run;
        }
        __syncthreads();
        if (valid) {
            const uint32_t pos = s_wcount[buf][warp][d] + rank;
            keys_out[pos] = key;
            vals_out[pos] = val;
        }
        __syncthreads();
        // reset this round's counts; the next round uses the other buffer, which was cleared
        // one round earlier, behind at least one barrier
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s_wcount[buf][w][threadIdx.x] = 0;
    }
}

}  // namespace

BinPlan plan_bin(int32_t n, const CameraF& cam, size_t capacity) {
    BinPlan p{};
    p.n = n;
    p.n_tiles = cam.TX * cam.TY;
    int tile_bits = 0;
    while ((1ll << tile_bits) < (long long)p.n_tiles) ++tile_bits;
    p.key_bits = 32 + tile_bits;
    p.passes = (p.key_bits + kRadixBits - 1) / kRadixBits;
    p.capacity = capacity;
    const size_t sort_blocks = ceil_div(std::max<size_t>(capacity, 1), kSortTile);
    const size_t hist_elems = sort_blocks * kRadix;
    p.scan_tmp_elems = scan_tmp_elems(size_t(n) + 1);
    p.hist_tmp_elems = scan_tmp_elems(hist_elems);
    size_t o = 0;
    p.off_offsets = o;   o = align256(o + (size_t(n) + 1) * sizeof(uint64_t));
    p.off_scan_tmp = o;  o = align256(o + std::max<size_t>(p.scan_tmp_elems, 1) * sizeof(uint64_t));
    p.off_total = o;     o = align256(o + sizeof(uint64_t));
    p.off_keys = o;      o = align256(o + capacity * sizeof(uint64_t));
    p.off_keys2 = o;     o = align256(o + capacity * sizeof(uint64_t));
    p.off_vals = o;      o = align256(o + capacity * sizeof(uint32_t));
    p.off_vals2 = o;     // unused: the caller's point list is the second value buffer
    p.off_hist = o;      o = align256(o + hist_elems * sizeof(uint32_t));
    p.off_hist_tmp = o;  o = align256(o + std::max<size_t>(p.hist_tmp_elems, 1) * sizeof(uint64_t));
    p.total_bytes = o;
    return p;
}

// tiles_touched (n values, plus a zero for index n) -> offsets[0..n]; offsets[n] = E.
cudaError_t launch_bin_scan(const BinPlan& plan, const CameraF& cam, const rs_projected& p,
                            uint8_t* ws, uint32_t* tile_ranges, cudaStream_t s) {
    (void)cam;
    k_clear_ranges<<<unsigned(ceil_div(plan.n_tiles, 256)), 256, 0, s>>>(tile_ranges, plan.n_tiles);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    uint64_t* offsets = reinterpret_cast<uint64_t*>(ws + plan.off_offsets);
    uint64_t* total = reinterpret_cast<uint64_t*>(ws + plan.off_total);
    uint64_t* tmp = reinterpret_cast<uint64_t*>(ws + plan.off_scan_tmp);
    if (plan.n == 0) return cudaMemsetAsync(total, 0, sizeof(uint64_t), s);
    e = device_exclusive_scan<uint32_t, uint64_t>(p.d_tiles_touched, size_t(plan.n), offsets, total,
                                                  tmp, s);
    if (e != cudaSuccess) return e;
    // offsets[n] = E, so the expansion's binary search has a sentinel
    return cudaMemcpyAsync(offsets + plan.n, total, sizeof(uint64_t), cudaMemcpyDeviceToDevice, s);
}

cudaError_t launch_bin_sort(const BinPlan& plan, const CameraF& cam, const rs_projected& p,
                            uint8_t* ws, uint64_t E64, uint64_t* keys_out, uint32_t* point_list,
                            uint32_t* tile_ranges, cudaStream_t s) {
    if (E64 == 0) return cudaSuccess;
    const uint32_t E = uint32_t(E64);
    const uint64_t* offsets = reinterpret_cast<const uint64_t*>(ws + plan.off_offsets);
    // ping-pong: buffer 0 is the caller's (keys_out or workspace keys2, point_list), buffer 1 is
    // the workspace; expand into the buffer that makes the last pass land in buffer 0
    uint64_t* K[2] = {keys_out ? keys_out : reinterpret_cast<uint64_t*>(ws + plan.off_keys2),
                      reinterpret_cast<uint64_t*>(ws + plan.off_keys)};
    uint32_t* V[2] = {point_list, reinterpret_cast<uint32_t*>(ws + plan.off_vals)};
    int cur = plan.passes % 2;
    k_expand<<<unsigned(ceil_div(E, 256)), 256, 0, s>>>(cam, plan.n, E, offsets, p.d_means2d,
                                                        p.d_depth, p.d_radius, K[cur], V[cur]);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const unsigned blocks = unsigned(ceil_div(E, kSortTile));
    uint32_t* hist = reinterpret_cast<uint32_t*>(ws + plan.off_hist);
    uint64_t* htmp = reinterpret_cast<uint64_t*>(ws + plan.off_hist_tmp);
    for (int pass = 0; pass < plan.passes; ++pass) {
        const int shift = pass * kRadixBits;
        k_radix_hist<<<blocks, kSortThreads, 0, s>>>(K[cur], E, shift, hist);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        e = device_exclusive_scan<uint32_t, uint32_t>(hist, size_t(blocks) * kRadix, hist, nullptr,
                                                      htmp, s);
        if (e != cudaSuccess) return e;
        k_radix_scatter<<<blocks, kSortThreads, 0, s>>>(K[cur], V[cur], E, shift, hist,
                                                        K[cur ^ 1], V[cur ^ 1]);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        cur ^= 1;
    }
    k_ranges<<<unsigned(ceil_div(E, 256)), 256, 0, s>>>(K[0], E, uint32_t(plan.n_tiles), tile_ranges);
    return cudaGetLastError();
}

}  // namespace rs
