// [2] binning: entries keyed (tile_id << 32) | float_bits(depth), sorted stably, and the tile
// ranges of the sorted list.
//
// The 64-bit stable sort is done as two 32-bit stable sorts: the Gaussians are first sorted by
// depth (their index order breaks ties), the entries are then produced Gaussian by Gaussian in
// that depth order, and finally sorted stably by tile id alone.  Within a tile each Gaussian has
// one entry, so the result is ordered by (tile, depth, index): exactly the stable sort of the
// 64-bit keys produced in index order, with 4 radix passes over N Gaussians and
// ceil(log2(tiles)/8) passes over the E entries instead of ceil((32 + log2(tiles))/8) passes
// over E.
//
// rigel README "Binning" (key = (tile_id << 32) | float_bits(depth), a sort restricted to the
// occupied bits, a range kernel); "3D Gaussian Splatting ビューワを作る" 4.1 (exclusive scan
// giving each Gaussian a private slice), 4.2 (duplicate), 4.3 (8-bit digits, per-block
// histograms, bin offsets from a scan over (digit, block), in-bin ranks, ping-pong buffers),
// 4.4 (ranges; empty tiles cleared to (0, 0)).
//
// GB300 design: each radix pass is one kernel ("one sweep"): a histogram kernel counts the
// digits of every pass up front, then in a pass kernel each block takes the next tile id from an
// atomic counter, ranks its keys, publishes its digit counts and reads its predecessors' counts
// with a decoupled look-back.  A block only ever waits for tiles with smaller ids, which were
// taken by blocks already running, so every wait ends; each wait is still bounded, and a timeout
// sets an error word (reported as RS_ERR_DEVICE_TIMEOUT) instead of spinning on.  Kernels after
// the scan read the entry count E from device memory (grids sized for the capacity), so the host
// enqueues the whole binning at once and reads E back a single time at the end.
// Working sets of the headline workloads (a few million 8-byte entries) sit in the 126 MB L2.
#include "rs_internal.cuh"

namespace rs {
namespace {

constexpr int kScanThreads = 256;
constexpr int kScanItems = 8;
constexpr int kScanChunk = kScanThreads * kScanItems;  // 2048 elements per block

constexpr int kRsThreads = 256;
constexpr int kRsWarps = kRsThreads / 32;
constexpr int kDepthItems = 8;                          // depth sort: 2048 keys per block
constexpr int kTileItems = 16;                          // tile sort: 4096 keys per block
constexpr unsigned kFull = 0xffffffffu;

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

// ---------------------------------------------------------------- one-sweep LSD radix sort
constexpr uint32_t kFlagAgg = 1u << 30;    // status word: this tile's own digit count
constexpr uint32_t kFlagIncl = 2u << 30;   // status word: count of this and every earlier tile
constexpr uint32_t kFlagMask = 3u << 30;
constexpr uint32_t kCountMask = (1u << 30) - 1u;
constexpr int kMaxSpins = 1 << 20;         // bound on one look-back wait (then give up, flag it)
constexpr int kWindow = 8;                 // predecessors whose status words are read together

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed(uint32_t* p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Number of keys: a host value, or the device entry count (0 when it exceeds the capacity, so
// nothing is written past the caller's buffers).
struct Count {
    uint32_t host;
    const uint64_t* dev;
    uint32_t cap;
    __device__ __forceinline__ uint32_t get() const {
        if (!dev) return host;
        const uint64_t v = *dev;
        return v > uint64_t(cap) ? 0u : uint32_t(v);
    }
};

struct SortCtl {
    uint32_t* counter;   // [passes] next tile id
    uint32_t* ghist;     // [passes][256] digit totals over all keys
    uint32_t* status;    // [passes][max_tiles][256] look-back words
    uint32_t* error;     // set when a look-back wait gave up
    uint32_t max_tiles;
};

struct DepthKeySource {
    const float* depth;   // key = float bits of depth for visible Gaussians, all ones otherwise
    const int* radius;    // value = Gaussian index
};

template <bool FROM_DEPTH>
__device__ __forceinline__ void rs_load(const uint32_t* __restrict__ keys, const uint32_t* __restrict__ vals,
                                        const DepthKeySource& src, uint32_t i, uint32_t& key,
                                        uint32_t& val) {
    if (FROM_DEPTH) {
        key = src.radius[i] > 0 ? __float_as_uint(src.depth[i]) : 0xffffffffu;
        val = i;
    } else {
        key = keys[i];
        val = vals ? vals[i] : 0u;
    }
}

// Digit totals of every pass at once: ghist[p][d] += #keys whose digit p is d.
template <int RBITS, int ITEMS, int PASSES, bool FROM_DEPTH>
__global__ void __launch_bounds__(kRsThreads) k_sweep_hist(const uint32_t* __restrict__ keys,
                                                          DepthKeySource src, Count count, int digit_bits,
                                                          uint32_t* __restrict__ ghist) {
    constexpr int R = 1 << RBITS;
    __shared__ uint32_t s_h[PASSES][R];
    for (int i = threadIdx.x; i < PASSES * R; i += kRsThreads) (&s_h[0][0])[i] = 0u;
    __syncthreads();
    const uint32_t n = count.get();
    const uint32_t base = blockIdx.x * (kRsThreads * ITEMS);
    if (base >= n) return;
    const uint32_t lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
        const uint32_t i = base + k * kRsThreads + threadIdx.x;
        uint32_t key = 0u, val;
        if (i < n) rs_load<FROM_DEPTH>(keys, nullptr, src, i, key, val);
#pragma unroll
        for (int p = 0; p < PASSES; ++p) {
            const uint32_t d = i < n ? (key >> (p * digit_bits)) & uint32_t(R - 1) : uint32_t(R);
            const uint32_t peers = __match_any_sync(kFull, d);
            if (d < uint32_t(R) && lane == uint32_t(__ffs(peers) - 1)) atomicAdd(&s_h[p][d], uint32_t(__popc(peers)));
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < PASSES * R; i += kRsThreads) {
        const uint32_t c = (&s_h[0][0])[i];
        if (c) atomicAdd(ghist + (i / R) * 256 + (i % R), c);
    }
}

// Exclusive scan of one value per thread over the first 256 threads (others pass 0).
__device__ __forceinline__ uint32_t block_exclusive_scan_256(uint32_t v, uint32_t* s_w) {
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, x, o);
        if (lane >= uint32_t(o)) x += y;
    }
    if (lane == 31) s_w[warp] = x;
    __syncthreads();
    uint32_t before = 0u;
    for (uint32_t w = 0; w < warp; ++w) before += s_w[w];
    return before + x - v;
}

// One stable pass over the digit at `shift`.  A block owns ITEMS x 256 consecutive keys of its
// tile; warp w owns the w-th contiguous 32 x ITEMS of them and walks them 32 at a time in index
// order, ranking equal digits with match masks and per-warp running counts.  A key goes to
// (keys of smaller digits) + (same digit in earlier tiles, from the look-back)
// + (same digit in earlier warps of the tile) + (its rank in its warp).
template <int RBITS, int ITEMS, bool FROM_DEPTH, bool GATHER_TILES>
__global__ void __launch_bounds__(kRsThreads) k_sweep_pass(
    const uint32_t* __restrict__ keys_in, const uint32_t* __restrict__ vals_in, DepthKeySource src,
    Count count, int shift, int pass, SortCtl ctl, uint32_t* __restrict__ keys_out,
    uint32_t* __restrict__ vals_out, const uint32_t* __restrict__ tiles_in,
    uint32_t* __restrict__ tiles_out) {
    constexpr int R = 1 << RBITS;
    constexpr uint32_t TILE = kRsThreads * ITEMS;
    __shared__ uint32_t s_cnt[kRsWarps][R];
    __shared__ uint32_t s_off[R];
    __shared__ uint32_t s_w[kRsWarps];
    __shared__ uint32_t s_tile;
    if (threadIdx.x == 0) s_tile = atomicAdd(ctl.counter + pass, 1u);
    for (int i = threadIdx.x; i < kRsWarps * R; i += kRsThreads) (&s_cnt[0][0])[i] = 0u;
    __syncthreads();
    const uint32_t n = count.get();
    const uint32_t tile = s_tile;
    if (tile >= (n + TILE - 1) / TILE) return;  // uniform: nothing to do (and nobody waits on it)
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t lt = (1u << lane) - 1u;
    const uint32_t base = tile * TILE + warp * (32 * ITEMS);
    uint32_t key[ITEMS], val[ITEMS], d[ITEMS], rank[ITEMS];
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
        const uint32_t i = base + k * 32 + lane;
        key[k] = 0u;
        val[k] = 0u;
        if (i < n) rs_load<FROM_DEPTH>(keys_in, vals_in, src, i, key[k], val[k]);
        d[k] = i < n ? (key[k] >> shift) & uint32_t(R - 1) : uint32_t(R);
    }
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
        const uint32_t peers = __match_any_sync(kFull, d[k]);
        const uint32_t leader = uint32_t(__ffs(peers) - 1);
        const bool lead = lane == leader && d[k] < uint32_t(R);
        uint32_t before = lead ? s_cnt[warp][d[k]] : 0u;
        before = __shfl_sync(kFull, before, leader);
        rank[k] = before + uint32_t(__popc(peers & lt));
        if (lead) s_cnt[warp][d[k]] = before + uint32_t(__popc(peers));
        __syncwarp();
    }
    __syncthreads();
    uint32_t* status = ctl.status + size_t(pass) * ctl.max_tiles * 256;
    const uint32_t t = threadIdx.x;
    uint32_t excl = 0u, gtotal = 0u;
    if (t < uint32_t(R)) {
        uint32_t run = 0u;  // per-warp offsets inside the tile; run ends as the tile's count
#pragma unroll
        for (int w = 0; w < kRsWarps; ++w) {
            const uint32_t c = s_cnt[w][t];
            s_cnt[w][t] = run;
            run += c;
        }
        uint32_t* mine = status + size_t(tile) * 256 + t;
        if (tile == 0) {
            st_relaxed(mine, kFlagIncl | run);
        } else {
            st_relaxed(mine, kFlagAgg | run);
            // look back over up to kWindow predecessors at a time: the window's status words are
            // loaded together, then consumed nearest first; only a word not yet published is
            // re-read (bounded)
            int pt = int(tile) - 1;
            bool found = false;
            while (!found && pt >= 0) {
                const int nwin = min(kWindow, pt + 1);
                uint32_t v[kWindow];
#pragma unroll
                for (int j = 0; j < kWindow; ++j)
                    v[j] = j < nwin ? ld_relaxed(status + size_t(pt - j) * 256 + t) : 0u;
#pragma unroll
                for (int j = 0; j < kWindow; ++j) {
                    if (found || j >= nwin) break;
                    uint32_t w = v[j];
                    int spins = 0;
                    while ((w & kFlagMask) == 0u) {
                        ++spins;
                        if ((spins & 255) == 0 && (spins >= kMaxSpins || ld_relaxed(ctl.error) != 0u)) {
                            atomicOr(ctl.error, 1u);
                            w = kFlagIncl;  // give up: the sort is reported as failed
                            break;
                        }
                        __nanosleep(32);
                        w = ld_relaxed(status + size_t(pt - j) * 256 + t);
                    }
                    excl += w & kCountMask;
                    found = (w & kFlagMask) == kFlagIncl;
                }
                pt -= nwin;
            }
            st_relaxed(mine, kFlagIncl | (excl + run));
        }
        gtotal = ctl.ghist[pass * 256 + t];
    }
    const uint32_t dbase = block_exclusive_scan_256(t < uint32_t(R) ? gtotal : 0u, s_w);
    if (t < uint32_t(R)) s_off[t] = dbase + excl;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
        if (d[k] < uint32_t(R)) {
            const uint32_t pos = s_off[d[k]] + s_cnt[warp][d[k]] + rank[k];
            keys_out[pos] = key[k];
            vals_out[pos] = val[k];
            if (GATHER_TILES) tiles_out[pos] = tiles_in[val[k]];
        }
    }
}

// ---------------------------------------------------------------- clearing, ranges
// Zeroes the tile ranges and the sort's control words (counters, histograms, look-back status,
// result block) in one launch.
__global__ void k_clear(uint32_t* __restrict__ ranges, uint32_t range_words, uint32_t* __restrict__ ctl,
                        size_t ctl_words) {
    const size_t stride = size_t(gridDim.x) * blockDim.x;
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < range_words; i += stride) ranges[i] = 0u;
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < ctl_words; i += stride) ctl[i] = 0u;
}

// Ranges from the sorted tile ids; also writes the 64-bit keys when asked.
__global__ void k_ranges(const uint32_t* __restrict__ tiles, const uint32_t* __restrict__ vals,
                         const float* __restrict__ depth, Count count, uint32_t n_tiles,
                         uint32_t* __restrict__ ranges, uint64_t* __restrict__ keys_out) {
    const uint32_t E = count.get();
    const uint32_t e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    const uint32_t tile = tiles[e];
    if (keys_out) keys_out[e] = (uint64_t(tile) << 32) | uint64_t(__float_as_uint(depth[vals[e]]));
    if (tile >= n_tiles) return;  // unreachable for ids made by k_expand; keeps writes in bounds
    if (e == 0 || tiles[e - 1] != tile) ranges[2 * size_t(tile)] = e;
    if (e == E - 1 || tiles[e + 1] != tile) ranges[2 * size_t(tile) + 1] = e + 1;
}

// ---------------------------------------------------------------- expansion in depth order
// Block b produces entries [1024 b, 1024 b + 1024).  offsets[i] (i in depth order; E past the
// end) starts Gaussian perm[i]'s slice.  Every Gaussian before the culled tail of the depth order
// has at least one entry, so the owners of 1024 consecutive entries are at most 1024 consecutive
// depth positions: the block finds the first owner with a warp-parallel search, stages the
// 1025 offsets after it in shared memory and searches there per entry.  Tiles of a Gaussian are
// taken row by row (tile rows outer, columns inner).
constexpr int kExpThreads = 256;
constexpr int kExpTile = 1024;

__global__ void __launch_bounds__(kExpThreads) k_expand(CameraF cam, int n, Count count,
                                                       const uint64_t* __restrict__ offsets,
                                                       const uint32_t* __restrict__ perm,
                                                       const float* __restrict__ means2d,
                                                       const int* __restrict__ radius,
                                                       uint32_t* __restrict__ tile_keys,
                                                       uint32_t* __restrict__ vals) {
    __shared__ uint64_t s_off[kExpTile + 1];
    __shared__ int s_i0;
    const uint32_t E = count.get();
    const uint32_t e0 = blockIdx.x * kExpTile;
    if (e0 >= E) return;
    if (threadIdx.x < 32) {
        // last i with offsets[i] <= e0; invariant offsets[lo] <= e0 < offsets[hi] (offsets[n] = E)
        const unsigned lane = threadIdx.x;
        int lo = 0, hi = n;
        while (hi - lo > 1) {
            const int step = (hi - lo + 31) / 32;
            const int p = lo + int(lane + 1) * step;
            const bool le = p < hi && offsets[p] <= e0;
            const int c = __popc(__ballot_sync(kFull, le));
            lo += c * step;
            hi = min(hi, lo + step);
        }
        if (lane == 0) s_i0 = lo;
    }
    __syncthreads();
    const int i0 = s_i0;
    const int window = min(kExpTile + 1, n + 1 - i0);
    for (int j = threadIdx.x; j < window; j += kExpThreads)
        s_off[j] = i0 + j < n ? offsets[i0 + j] : uint64_t(E);
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kExpTile / kExpThreads; ++k) {
        const uint32_t e = e0 + k * kExpThreads + threadIdx.x;
        if (e >= E) break;
        int lo = 0, hi = window - 1;  // s_off[lo] <= e < s_off[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_off[mid] <= e) lo = mid; else hi = mid;
        }
        const uint32_t g = perm[i0 + lo];
        const uint32_t kk = e - uint32_t(s_off[lo]);
        const float u = means2d[g], v = means2d[size_t(n) + g];
        const float r = float(radius[g]);
        const int xl = span_bound(u, r, cam.TX, false), xh = span_bound(u, r, cam.TX, true);
        const int yl = span_bound(v, r, cam.TY, false);
        // sx >= 1 whenever tiles_touched[g] > 0 came from rs_project (same span arithmetic); the
        // max() only keeps inconsistent caller data from dividing by zero
        const uint32_t sx = uint32_t(max(xh - xl, 1));
        const uint32_t tx = uint32_t(xl) + kk % sx, ty = uint32_t(yl) + kk / sx;
        tile_keys[e] = ty * uint32_t(cam.TX) + tx;
        vals[e] = g;
    }
}

template <int RBITS>
void tile_sort_launch(const uint32_t* kin, const uint32_t* vin, Count count, int digit, int pass,
                      const SortCtl& ctl, unsigned blocks, uint32_t* kout, uint32_t* vout, cudaStream_t s) {
    k_sweep_pass<RBITS, kTileItems, false, false><<<blocks, kRsThreads, 0, s>>>(
        kin, vin, DepthKeySource{}, count, pass * digit, pass, ctl, kout, vout, nullptr, nullptr);
}

template <int RBITS>
void tile_hist_launch(const uint32_t* keys, Count count, int digit, int passes, unsigned blocks,
                      uint32_t* ghist, cudaStream_t s) {
    if (passes == 1)
        k_sweep_hist<RBITS, kTileItems, 1, false><<<blocks, kRsThreads, 0, s>>>(keys, DepthKeySource{}, count, digit, ghist);
    else
        k_sweep_hist<RBITS, kTileItems, 2, false><<<blocks, kRsThreads, 0, s>>>(keys, DepthKeySource{}, count, digit, ghist);
}

}  // namespace

BinPlan plan_bin(int32_t n, const CameraF& cam, size_t capacity) {
    BinPlan p{};
    p.n = n;
    p.n_tiles = cam.TX * cam.TY;
    int tile_bits = 0;
    while ((1ll << tile_bits) < (long long)p.n_tiles) ++tile_bits;
    p.tile_bits = std::max(tile_bits, 1);
    p.tile_passes = (p.tile_bits + 7) / 8;
    p.capacity = capacity;
    const size_t N = size_t(n);
    p.depth_tiles = ceil_div(std::max<size_t>(N, 1), size_t(kRsThreads) * kDepthItems);
    p.tile_tiles = ceil_div(std::max<size_t>(capacity, 1), size_t(kRsThreads) * kTileItems);
    p.scan_tmp_elems = scan_tmp_elems(N);
    size_t o = 0;
    p.off_dkeys = o;      o = align256(o + 2 * N * sizeof(uint32_t));   // depth keys, 2 buffers
    p.off_dvals = o;      o = align256(o + 2 * N * sizeof(uint32_t));   // Gaussian ids, 2 buffers
    p.off_tiles_sorted = o; o = align256(o + N * sizeof(uint32_t));     // tiles_touched, depth order
    p.off_offsets = o;    o = align256(o + std::max<size_t>(N, 1) * sizeof(uint64_t));
    p.off_scan_tmp = o;   o = align256(o + std::max<size_t>(p.scan_tmp_elems, 1) * sizeof(uint64_t));
    p.off_tkeys = o;      o = align256(o + 2 * capacity * sizeof(uint32_t));  // tile ids, 2 buffers
    p.off_tvals = o;      o = align256(o + capacity * sizeof(uint32_t));      // + the caller's list
    // control words, zeroed by one kernel at the start of every call:
    // result {E (u64), error (u32), pad}, counters, digit totals, look-back status
    p.off_ctl = o;
    p.off_result = o;               o += 16;
    p.off_counters = o;             o += 8 * sizeof(uint32_t);
    p.off_ghist_depth = o;          o += 4 * 256 * sizeof(uint32_t);
    p.off_ghist_tile = o;           o += 2 * 256 * sizeof(uint32_t);
    p.off_status_depth = o;         o += 4 * p.depth_tiles * 256 * sizeof(uint32_t);
    p.off_status_tile = o;          o += size_t(p.tile_passes) * p.tile_tiles * 256 * sizeof(uint32_t);
    p.ctl_bytes = o - p.off_ctl;
    o = align256(o);
    p.total_bytes = o;
    return p;
}

cudaError_t launch_bin(const BinPlan& plan, const CameraF& cam, const rs_projected& p, uint8_t* ws,
                       uint64_t* keys_out, uint32_t* point_list, uint32_t* tile_ranges, cudaStream_t s) {
    uint32_t* ctl_words = reinterpret_cast<uint32_t*>(ws + plan.off_ctl);
    {
        const size_t words = plan.ctl_bytes / 4 + 2u * uint32_t(plan.n_tiles);
        const unsigned blocks = unsigned(std::min<size_t>(ceil_div(words, 256), 152 * 8));
        k_clear<<<blocks, 256, 0, s>>>(tile_ranges, 2u * uint32_t(plan.n_tiles), ctl_words, plan.ctl_bytes / 4);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || plan.n == 0) return e;
    const uint32_t n = uint32_t(plan.n);
    uint64_t* result = reinterpret_cast<uint64_t*>(ws + plan.off_result);  // result[0] = E
    uint32_t* error = reinterpret_cast<uint32_t*>(ws + plan.off_result + 8);
    uint32_t* counters = reinterpret_cast<uint32_t*>(ws + plan.off_counters);

    // 1. depth sort of the Gaussians (4 passes of 8 bits; culled ones last)
    uint32_t* dk = reinterpret_cast<uint32_t*>(ws + plan.off_dkeys);
    uint32_t* dv = reinterpret_cast<uint32_t*>(ws + plan.off_dvals);
    uint32_t* DK[2] = {dk, dk + n};
    uint32_t* DV[2] = {dv, dv + n};
    uint32_t* tiles_sorted = reinterpret_cast<uint32_t*>(ws + plan.off_tiles_sorted);
    const DepthKeySource src{p.d_depth, p.d_radius};
    const Count cn{n, nullptr, n};
    const SortCtl dctl{counters, reinterpret_cast<uint32_t*>(ws + plan.off_ghist_depth),
                       reinterpret_cast<uint32_t*>(ws + plan.off_status_depth), error,
                       uint32_t(plan.depth_tiles)};
    const unsigned dblocks = unsigned(plan.depth_tiles);
    k_sweep_hist<8, kDepthItems, 4, true><<<dblocks, kRsThreads, 0, s>>>(nullptr, src, cn, 8, dctl.ghist);
    k_sweep_pass<8, kDepthItems, true, false><<<dblocks, kRsThreads, 0, s>>>(
        nullptr, nullptr, src, cn, 0, 0, dctl, DK[0], DV[0], nullptr, nullptr);
    k_sweep_pass<8, kDepthItems, false, false><<<dblocks, kRsThreads, 0, s>>>(
        DK[0], DV[0], src, cn, 8, 1, dctl, DK[1], DV[1], nullptr, nullptr);
    k_sweep_pass<8, kDepthItems, false, false><<<dblocks, kRsThreads, 0, s>>>(
        DK[1], DV[1], src, cn, 16, 2, dctl, DK[0], DV[0], nullptr, nullptr);
    k_sweep_pass<8, kDepthItems, false, true><<<dblocks, kRsThreads, 0, s>>>(
        DK[0], DV[0], src, cn, 24, 3, dctl, DK[1], DV[1], p.d_tiles_touched, tiles_sorted);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const uint32_t* perm = DV[1];

    // 2. offsets of each Gaussian's entries, in depth order; E lands in result[0]
    uint64_t* offsets = reinterpret_cast<uint64_t*>(ws + plan.off_offsets);
    uint64_t* tmp = reinterpret_cast<uint64_t*>(ws + plan.off_scan_tmp);
    e = device_exclusive_scan<uint32_t, uint64_t>(tiles_sorted, size_t(n), offsets, result, tmp, s);
    if (e != cudaSuccess || plan.capacity == 0) return e;

    // 3. entries in depth order, then a stable sort by tile id
    const Count ce{0u, result, uint32_t(plan.capacity)};
    uint32_t* tk = reinterpret_cast<uint32_t*>(ws + plan.off_tkeys);
    uint32_t* TK[2] = {tk, tk + plan.capacity};
    uint32_t* TV[2] = {point_list, reinterpret_cast<uint32_t*>(ws + plan.off_tvals)};
    int cur = plan.tile_passes % 2;  // the last pass lands in buffer 0 (the caller's list)
    k_expand<<<unsigned(ceil_div(plan.capacity, kExpTile)), kExpThreads, 0, s>>>(
        cam, plan.n, ce, offsets, perm, p.d_means2d, p.d_radius, TK[cur], TV[cur]);
    const int digit = (plan.tile_bits + plan.tile_passes - 1) / plan.tile_passes;  // <= 8
    const SortCtl tctl{counters + 4, reinterpret_cast<uint32_t*>(ws + plan.off_ghist_tile),
                       reinterpret_cast<uint32_t*>(ws + plan.off_status_tile), error,
                       uint32_t(plan.tile_tiles)};
    const unsigned tblocks = unsigned(plan.tile_tiles);
    const int rbits = digit <= 4 ? 4 : digit <= 6 ? 6 : digit == 7 ? 7 : 8;
    switch (rbits) {
        case 4: tile_hist_launch<4>(TK[cur], ce, digit, plan.tile_passes, tblocks, tctl.ghist, s); break;
        case 6: tile_hist_launch<6>(TK[cur], ce, digit, plan.tile_passes, tblocks, tctl.ghist, s); break;
        case 7: tile_hist_launch<7>(TK[cur], ce, digit, plan.tile_passes, tblocks, tctl.ghist, s); break;
        default: tile_hist_launch<8>(TK[cur], ce, digit, plan.tile_passes, tblocks, tctl.ghist, s); break;
    }
    for (int pass = 0; pass < plan.tile_passes; ++pass) {
        switch (rbits) {
            case 4: tile_sort_launch<4>(TK[cur], TV[cur], ce, digit, pass, tctl, tblocks, TK[cur ^ 1], TV[cur ^ 1], s); break;
            case 6: tile_sort_launch<6>(TK[cur], TV[cur], ce, digit, pass, tctl, tblocks, TK[cur ^ 1], TV[cur ^ 1], s); break;
            case 7: tile_sort_launch<7>(TK[cur], TV[cur], ce, digit, pass, tctl, tblocks, TK[cur ^ 1], TV[cur ^ 1], s); break;
            default: tile_sort_launch<8>(TK[cur], TV[cur], ce, digit, pass, tctl, tblocks, TK[cur ^ 1], TV[cur ^ 1], s); break;
        }
        cur ^= 1;
    }
    k_ranges<<<unsigned(ceil_div(plan.capacity, 256)), 256, 0, s>>>(TK[0], TV[0], p.d_depth, ce,
                                                                   uint32_t(plan.n_tiles), tile_ranges, keys_out);
    return cudaGetLastError();
}

}  // namespace rs
