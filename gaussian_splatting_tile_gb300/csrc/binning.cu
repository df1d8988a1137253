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

constexpr int kRsThreads = 256;
constexpr int kRsWarps = kRsThreads / 32;
// keys per thread of the sort passes (a block holds 256 x that many keys)
#ifndef RS_DEPTH_ITEMS
#define RS_DEPTH_ITEMS 8
#endif
#ifndef RS_TILE_ITEMS
#define RS_TILE_ITEMS 20
#endif
constexpr int kDepthItems = RS_DEPTH_ITEMS;             // depth sort: 2048 keys per block
constexpr int kTileItems = RS_TILE_ITEMS;               // tile sort: 5120 keys per block
// Tile-sort blocks resident per SM: two blocks of 5120 keys hold 1.56 M entries on the 152 SMs in
// one wave (a pass whose blocks do not all fit waits a second block latency for the last ones).
#ifndef RS_TILE_MIN_BLOCKS
#define RS_TILE_MIN_BLOCKS 2
#endif
constexpr int kTileMinBlocks = RS_TILE_MIN_BLOCKS;
constexpr int kDepthHistItems = 2;                      // depth digit counts: 512 keys per block
constexpr unsigned kFull = 0xffffffffu;

size_t ceil_div(size_t a, size_t b) { return (a + b - 1) / b; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ---------------------------------------------------------------- one-sweep LSD radix sort
constexpr uint32_t kFlagAgg = 1u << 30;    // status word: this tile's own digit count
constexpr uint32_t kFlagIncl = 2u << 30;   // status word: count of this and every earlier tile
constexpr uint32_t kFlagMask = 3u << 30;
constexpr uint32_t kCountMask = (1u << 30) - 1u;
constexpr int kMaxSpins = 1 << 20;         // bound on one look-back wait (then give up, flag it)
#ifndef RS_LOOKBACK_WINDOW
#define RS_LOOKBACK_WINDOW 32
#endif
constexpr int kWindow = RS_LOOKBACK_WINDOW;  // predecessors whose status words are read together

// Lanes of the warp holding the same value d as this lane, for 0 <= d <= R = 2^RBITS (R marks
// "no key").  1: one ballot per bit of d (RBITS + 1 ballots and selects); 0: the match
// instruction.  Both give the same mask; the match instruction's latency bounded the ranking and
// digit-counting loops (at 10 M entries a tile-id pass took 129 us with it, 98 us with ballots;
// the expansion 102 and 92 us).
#ifndef RS_RANK_BALLOT
#define RS_RANK_BALLOT 1
#endif
template <int RBITS>
__device__ __forceinline__ uint32_t same_digit_lanes(uint32_t d) {
#if RS_RANK_BALLOT
    uint32_t m = 0xffffffffu;
#pragma unroll
    for (int b = 0; b <= RBITS; ++b) {
        const bool bit = (d >> b) & 1u;
        const uint32_t bal = __ballot_sync(0xffffffffu, bit);
        m &= bit ? bal : ~bal;
    }
    return m;
#else
    return __match_any_sync(0xffffffffu, d);
#endif
}

// Adds this lane's digit d to the histogram h (d == R: no key): the whole warp in one atomic when
// every lane holds the same digit (the high digits of neighbouring keys), else one shared-memory
// atomic per lane (the hardware serialises lanes that meet on one counter).  Counting needs no
// ranks, so this replaces the equal-digit masks in the histogram loops.
template <int R>
__device__ __forceinline__ void count_digit(uint32_t* h, uint32_t d) {
    const uint32_t d0 = __shfl_sync(0xffffffffu, d, 0);
    if (__all_sync(0xffffffffu, d == d0)) {
        if ((threadIdx.x & 31) == 0 && d0 < uint32_t(R)) atomicAdd(&h[d0], 32u);
    } else if (d < uint32_t(R)) {
        atomicAdd(&h[d], 1u);
    }
}

// q = n / d and r = n % d for 1 <= d and n < 2^24 (an entry's index within its Gaussian's tile
// rectangle, which is below the tile count, and the rectangle's width): the quotient estimated
// in float with the approximate reciprocal is within one of the exact one for these sizes, and
// comparing n - q d with 0 and d corrects it.
__device__ __forceinline__ void div_small(uint32_t n, uint32_t d, uint32_t& q, uint32_t& r) {
    uint32_t qe = __float2uint_rz(__uint2float_rn(n) * rcp_approx(__uint2float_rn(d)));
    int32_t rr = int32_t(n) - int32_t(qe * d);
    while (rr < 0) {
        --qe;
        rr += int32_t(d);
    }
    while (rr >= int32_t(d)) {
        ++qe;
        rr -= int32_t(d);
    }
    q = qe;
    r = uint32_t(rr);
}

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
        // both loads issued together (a depth load behind the radius test would wait for it)
        const int r = src.radius[i];
        const uint32_t d = __float_as_uint(src.depth[i]);
        key = r > 0 ? d : 0xffffffffu;
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
    RS_PDL_ENTER();
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
            count_digit<R>(s_h[p], i < n ? (key >> (p * digit_bits)) & uint32_t(R - 1) : uint32_t(R));
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < PASSES * R; i += kRsThreads) {
        const uint32_t c = (&s_h[0][0])[i];
        if (c) atomicAdd(ghist + (i / R) * 256 + (i % R), c);
    }
}

// Exclusive scan of one value per thread over the block's 256 threads.
__device__ __forceinline__ uint32_t block_exclusive_scan_256(uint32_t a, uint32_t* s_w) {
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = a;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, x, o);
        if (lane >= uint32_t(o)) x += y;
    }
    if (lane == 31) s_w[warp] = x;
    __syncthreads();
    uint32_t before = 0u;
    for (uint32_t w = 0; w < warp; ++w) before += s_w[w];
    return before + x - a;
}

// One stable pass over the digit at `shift`.  A block owns ITEMS x 256 consecutive keys of its
// tile; warp w owns the w-th contiguous 32 x ITEMS of them and walks them 32 at a time in index
// order, ranking equal digits with masks of the lanes that hold them and per-warp running counts.  A key goes to
// (keys of smaller digits) + (same digit in earlier tiles, from the look-back)
// + (same digit in earlier warps of the tile) + (its rank in its warp).  The tile's keys are
// first put in that order in shared memory, so the global writes of one digit are consecutive.
// With KEYS64 (last pass of the tile sort) the 64-bit keys (tile << 32) | float_bits(depth) are
// written as well when `keys64` is given.
template <int RBITS, int ITEMS, bool FROM_DEPTH, bool GATHER_TILES, bool KEYS64 = false, int MINB = 1>
__global__ void __launch_bounds__(kRsThreads, MINB) k_sweep_pass(
    const uint32_t* __restrict__ keys_in, const uint32_t* __restrict__ vals_in, DepthKeySource src,
    Count count, int shift, int pass, SortCtl ctl, uint32_t* __restrict__ keys_out,
    uint32_t* __restrict__ vals_out, const uint32_t* __restrict__ tiles_in,
    uint32_t* __restrict__ tiles_out, uint64_t* __restrict__ keys64) {
    RS_PDL_ENTER();
    constexpr int R = 1 << RBITS;
    constexpr uint32_t TILE = kRsThreads * ITEMS;
    __shared__ uint32_t s_cnt[kRsWarps][R];
    __shared__ uint32_t s_lstart[R];  // first slot of each digit in the tile's reordered keys
    __shared__ uint32_t s_delta[R];   // global position - slot, per digit
    __shared__ uint32_t s_w[kRsWarps];
    __shared__ uint32_t s_k[TILE], s_v[TILE];
    __shared__ uint32_t s_tile;
    if (threadIdx.x == 0) s_tile = atomicAdd(ctl.counter + pass, 1u);
    for (int i = threadIdx.x; i < kRsWarps * R; i += kRsThreads) (&s_cnt[0][0])[i] = 0u;
    __syncthreads();
    const uint32_t n = count.get();
    const uint32_t tile = s_tile;
    if (tile >= (n + TILE - 1) / TILE) return;  // uniform: nothing to do (and nobody waits on it)
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t lt = (1u << lane) - 1u;
    const uint32_t t = threadIdx.x;
    uint32_t* status = ctl.status + size_t(pass) * ctl.max_tiles * 256;
    // the digit totals (complete since the histogram kernel), loaded now to overlap the ranking
    const uint32_t gtotal = t < uint32_t(R) ? ctl.ghist[pass * 256 + t] : 0u;
    uint32_t run = 0u, lstart;
    {
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
            const uint32_t peers = same_digit_lanes<RBITS>(d[k]);
            const uint32_t leader = uint32_t(__ffs(peers) - 1);
            const bool lead = lane == leader && d[k] < uint32_t(R);
            uint32_t before = lead ? s_cnt[warp][d[k]] : 0u;
            before = __shfl_sync(kFull, before, leader);
            rank[k] = before + uint32_t(__popc(peers & lt));
            if (lead) s_cnt[warp][d[k]] = before + uint32_t(__popc(peers));
            __syncwarp();
        }
        __syncthreads();
        if (t < uint32_t(R)) {
            // per-warp offsets inside the tile; run ends as the tile's count of digit t, which is
            // published at once so that later tiles can go on looking back
#pragma unroll
            for (int w = 0; w < kRsWarps; ++w) {
                const uint32_t c = s_cnt[w][t];
                s_cnt[w][t] = run;
                run += c;
            }
            st_relaxed(status + size_t(tile) * 256 + t, (tile == 0 ? kFlagIncl : kFlagAgg) | run);
        }
        lstart = block_exclusive_scan_256(t < uint32_t(R) ? run : 0u, s_w);
        if (t < uint32_t(R)) s_lstart[t] = lstart;
        __syncthreads();
#pragma unroll
        for (int k = 0; k < ITEMS; ++k) {
            if (d[k] < uint32_t(R)) {
                const uint32_t slot = s_lstart[d[k]] + s_cnt[warp][d[k]] + rank[k];
                s_k[slot] = key[k];
                s_v[slot] = val[k];
            }
        }
    }
    uint32_t excl = 0u;
    if (t < uint32_t(R)) {
        if (tile != 0) {
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
            st_relaxed(status + size_t(tile) * 256 + t, kFlagIncl | (excl + run));
        }
    }
    const uint32_t dbase = block_exclusive_scan_256(t < uint32_t(R) ? gtotal : 0u, s_w);
    if (t < uint32_t(R)) s_delta[t] = dbase + excl - lstart;
    __syncthreads();
    const uint32_t in_tile = min(TILE, n - tile * TILE);
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
        const uint32_t j = uint32_t(k) * kRsThreads + t;
        if (j < in_tile) {
            const uint32_t kk = s_k[j], vv = s_v[j];
            const uint32_t pos = s_delta[(kk >> shift) & uint32_t(R - 1)] + j;
            keys_out[pos] = kk;
            vals_out[pos] = vv;
            if (GATHER_TILES) tiles_out[pos] = tiles_in[vv];
            if (KEYS64 && keys64) keys64[pos] = (uint64_t(kk) << 32) | uint64_t(__float_as_uint(src.depth[vv]));
        }
    }
}

// ---------------------------------------------------------------- clearing, ranges
// Zeroes the tile ranges and the sort's control words (counters, histograms, look-back status,
// result block) in one launch.
__global__ void k_clear(uint32_t* __restrict__ ranges, uint32_t range_words, uint32_t* __restrict__ ctl,
                        size_t ctl_words) {
    RS_PDL_ENTER();
    const size_t stride = size_t(gridDim.x) * blockDim.x;
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < range_words; i += stride) ranges[i] = 0u;
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < ctl_words; i += stride) ctl[i] = 0u;
}

// Ranges from the sorted tile ids.
__global__ void k_ranges(const uint32_t* __restrict__ tiles, Count count, uint32_t n_tiles,
                         uint32_t* __restrict__ ranges) {
    RS_PDL_ENTER();
    constexpr uint32_t kNone = 0xffffffffu;  // never a tile id
    const uint32_t E = count.get();
    const uint32_t quads = (E + 3u) / 4u;
    const uint32_t stride = gridDim.x * blockDim.x;
    // four consecutive entries per thread (one 16-byte load) and their two neighbours
    for (uint32_t q = blockIdx.x * blockDim.x + threadIdx.x; q < quads; q += stride) {
        const uint32_t e0 = 4u * q;
        uint32_t t[6];  // tiles[e0 - 1 .. e0 + 4], kNone outside [0, E)
        if (e0 + 4u <= E) {
            const uint4 v = *reinterpret_cast<const uint4*>(tiles + e0);
            t[1] = v.x;
            t[2] = v.y;
            t[3] = v.z;
            t[4] = v.w;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) t[1 + j] = e0 + uint32_t(j) < E ? tiles[e0 + j] : kNone;
        }
        t[0] = e0 > 0u ? tiles[e0 - 1u] : kNone;
        t[5] = e0 + 4u < E ? tiles[e0 + 4u] : kNone;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t e = e0 + uint32_t(j), tile = t[1 + j];
            if (e >= E || tile >= n_tiles) continue;  // ids made by the expansion are always below n_tiles
            if (t[j] != tile) ranges[2 * size_t(tile)] = e;
            if (t[j + 2] != tile) ranges[2 * size_t(tile) + 1] = e + 1u;
        }
    }
}

// ---------------------------------------------------------------- slices and expansion in depth order
// k_slices gives every Gaussian its slice of the entry list: block b (ids taken from an atomic
// counter, as in the sort passes) owns Gaussians [1024 b, 1024 b + 1024) of the depth order,
// scans their tile counts locally and gets the entries of all earlier blocks with a decoupled
// look-back over 64-bit status words.  It stores each slice start, the Gaussian's tile rectangle
// (first column | first row << 16, columns) and, for every 1024-entry chunk of the list, the
// Gaussian owning the chunk's first entry; the last block stores the total E.
// k_expand then writes 1024 entries per block (tiles of a Gaussian row by row: rows outer,
// columns inner) and counts the digits of the tile ids for every pass of the tile sort.
constexpr int kSlThreads = 256;
constexpr int kSlItems = 4;                          // Gaussians per thread
constexpr int kSlGauss = kSlThreads * kSlItems;      // Gaussians per block
constexpr int kExpThreads = 256;
constexpr int kExpChunk = 1024;                      // entries per expansion block
constexpr unsigned long long kSlAgg = 1ull << 62;    // status: this block's entry count
constexpr unsigned long long kSlIncl = 2ull << 62;   // status: entries of this and earlier blocks
constexpr unsigned long long kSlFlags = 3ull << 62;

__device__ __forceinline__ unsigned long long ld_relaxed64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

struct SliceOut {
    uint64_t* start;      // [n] first entry of each Gaussian's slice (depth order)
    uint2* rect;          // [n] tile rectangle of each Gaussian (depth order)
    uint32_t* owner;      // [chunks] depth position owning entry 1024 c
    uint32_t chunks;      // ceil(capacity / 1024)
    const float* ell;     // ellipse test only: the projection's words, [RS_ELLIPSE_WORDS][n] by
                          // Gaussian (row 0 k, rows 1.. the per-splat setup)
};

__global__ void __launch_bounds__(kSlThreads) k_slices(CameraF cam, uint32_t n, const uint32_t* __restrict__ perm,
                                                      const uint32_t* __restrict__ tiles_sorted,
                                                      const float* __restrict__ means2d,
                                                      const int* __restrict__ radius, uint32_t* counter,
                                                      unsigned long long* status, uint32_t* error,
                                                      uint64_t* total_out, SliceOut out) {
    RS_PDL_ENTER();
    __shared__ uint64_t s_w[kSlThreads / 32];
    __shared__ uint64_t s_prefix;
    __shared__ uint32_t s_blk;
    if (threadIdx.x == 0) s_blk = atomicAdd(counter, 1u);
    __syncthreads();
    const uint32_t blk = s_blk;
    const uint32_t nblk = (n + kSlGauss - 1) / kSlGauss;
    if (blk >= nblk) return;  // uniform; the grid has exactly nblk blocks, so never taken
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t i0 = blk * kSlGauss + threadIdx.x * kSlItems;
    uint32_t cnt[kSlItems];
    uint2 rect[kSlItems];
    uint64_t run = 0;
#pragma unroll
    for (int k = 0; k < kSlItems; ++k) {
        cnt[k] = i0 + k < n ? tiles_sorted[i0 + k] : 0u;
        run += cnt[k];
    }
    // the tile rectangles (gathers through the depth order) before the look-back, so that their
    // loads overlap it
#pragma unroll
    for (int k = 0; k < kSlItems; ++k) {
        rect[k] = make_uint2(0u, 1u);
        if (cnt[k]) {
            const uint32_t g = perm[i0 + k];
            const float u = means2d[g], v = means2d[size_t(n) + g];
            const float rad = float(radius[g]);
            const int xl = span_bound(u, rad, cam.TX, false), xh = span_bound(u, rad, cam.TX, true);
            const int yl = span_bound(v, rad, cam.TY, false);
            // >= 1 whenever tiles_touched > 0 came from the projection (same span arithmetic)
            rect[k] = make_uint2(uint32_t(xl) | (uint32_t(yl) << 16), uint32_t(max(xh - xl, 1)));
        }
    }
    uint64_t x = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(kFull, x, o);
        if (lane >= uint32_t(o)) x += y;
    }
    if (lane == 31) s_w[warp] = x;
    __syncthreads();
    uint64_t before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kSlThreads / 32; ++w) {
        const uint64_t c = s_w[w];
        before += uint32_t(w) < warp ? c : 0;
        total += c;
    }
    if (warp == 0) {
        // publish, then look back over 32 predecessors at a time (one per lane)
        if (lane == 0) st_relaxed64(status + blk, (blk == 0 ? kSlIncl : kSlAgg) | total);
        uint64_t excl = 0;
        int pt = int(blk) - 1;
        bool found = blk == 0;
        while (!found) {
            const int q = pt - int(lane);
            unsigned long long w = q >= 0 ? ld_relaxed64(status + q) : kSlIncl;
            int spins = 0;
            while ((w & kSlFlags) == 0ull) {
                ++spins;
                if ((spins & 255) == 0 && (spins >= kMaxSpins || ld_relaxed(error) != 0u)) {
                    atomicOr(error, 1u);
                    w = kSlIncl;  // give up: the binning is reported as failed
                    break;
                }
                __nanosleep(32);
                w = ld_relaxed64(status + q);
            }
            const uint32_t incl = __ballot_sync(kFull, (w & kSlFlags) == kSlIncl);
            // nearest inclusive word at lane f: sum lanes 0..f; otherwise all 32 and go on
            const int f = incl ? __ffs(incl) - 1 : 31;
            uint64_t c = uint32_t(lane) <= uint32_t(f) ? uint64_t(w & ~kSlFlags) : 0ull;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(kFull, c, o);
            excl += c;
            found = incl != 0u;
            pt -= 32;
        }
        if (lane == 0) {
            if (blk != 0) st_relaxed64(status + blk, kSlIncl | (excl + total));
            if (blk == nblk - 1) *total_out = excl + total;
            s_prefix = excl;
        }
    }
    __syncthreads();
    uint64_t start = s_prefix + before + x - run;
#pragma unroll
    for (int k = 0; k < kSlItems; ++k) {
        const uint32_t i = i0 + k;
        if (i < n) {
            out.start[i] = start;
            if (cnt[k]) {
                // chunks whose first entry falls in this slice
                const uint64_t end = start + cnt[k];
                for (uint64_t c = (start + kExpChunk - 1) / kExpChunk; c * kExpChunk < end && c < out.chunks; ++c)
                    out.owner[c] = i;
            }
            out.rect[i] = rect[k];
        }
        start += cnt[k];
    }
}


// The ellipse test's tile runs of a window's Gaussians, built once per chunk, one row per
// thread: row r of window Gaussian j is table entry rowstart[j] + r, holding the window's
// entries before that row (counted from the first Gaussian's slice start), the row's first tile
// and j; an entry then finds its row with one binary search.  Chunks whose Gaussians have more
// rows than the table holds walk the rows per entry.
constexpr int kRowCap = 2048;

template <int RBITS, bool ELL>
__global__ void __launch_bounds__(kExpThreads) k_expand(CameraF cam, uint32_t n, Count count,
                                                       const uint32_t* __restrict__ perm, SliceOut sl,
                                                       int digit_bits, int passes, uint32_t* __restrict__ ghist,
                                                       uint32_t* __restrict__ tile_keys,
                                                       uint32_t* __restrict__ vals) {
    RS_PDL_ENTER();
    constexpr int R = 1 << RBITS;
    constexpr int ROWS = ELL ? kRowCap : 1;
    // entries per block: 2048 for the square test (752 blocks of 5 per SM hold a 1080p frame's
    // 1.54 M entries in one wave), 1024 with the ellipse test's row tables; the slice scan
    // records the owner of every 1024th entry
    constexpr int CH = ELL ? kExpChunk : 2 * kExpChunk;
    constexpr int OWN = CH / kExpChunk;
    __shared__ uint64_t s_start[CH + 1];
    __shared__ uint2 s_rect[ELL ? 1 : CH];
    __shared__ uint32_t s_rowstart[ELL ? kExpChunk + 1 : 1];
    __shared__ uint32_t s_w[kExpThreads / 32];
    // ellipse mode, dynamic: the window's tile rows (ylo | yhi << 16) [kExpChunk], then the row
    // table: the window's entries before each row [ROWS], the row's first tile [ROWS] and its
    // Gaussian [ROWS] (16 bits); the other ellipse words are read from the slice output
    extern __shared__ __align__(16) float s_dyn[];
    float* s_e = s_dyn;
    uint32_t* s_rowcum = reinterpret_cast<uint32_t*>(s_dyn + (ELL ? kExpChunk : 0));
    uint32_t* s_rowtile = s_rowcum + ROWS;
    uint16_t* s_rowg = reinterpret_cast<uint16_t*>(s_rowtile + ROWS);  // window index of the row's Gaussian
    __shared__ uint32_t s_g[CH];
    __shared__ uint32_t s_h[3][R];
    const uint32_t E = count.get();
    const uint32_t chunks = (E + CH - 1) / CH;
    if (blockIdx.x >= chunks) return;
    for (int i = threadIdx.x; i < 3 * R; i += kExpThreads) (&s_h[0][0])[i] = 0u;
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t tiles_total = uint32_t(cam.TX) * uint32_t(cam.TY);
    for (uint32_t c = blockIdx.x; c < chunks; c += gridDim.x) {
        const uint32_t e0 = c * CH;
        // owners of the chunk's entries: depth positions i0 ..= i1.  Every Gaussian before the
        // culled tail of the depth order has at least one entry, so there are at most 1024 of
        // them; the slice after i1 starts past the chunk.
        const uint32_t i0 = sl.owner[OWN * c];
        const uint32_t i1 = c + 1 < chunks ? sl.owner[OWN * (c + 1)] : min(i0 + uint32_t(CH) - 1u, n - 1u);
        const int w = int(min(i1 - i0 + 1u, uint32_t(CH)));
        __syncthreads();  // the previous chunk is done with the window
        for (int j = threadIdx.x; j <= w; j += kExpThreads) {
            const uint32_t i = i0 + uint32_t(j);
            s_start[j] = i < n ? sl.start[i] : uint64_t(0xffffffffffffffffull);
            if (j < w) {
                const uint32_t g = perm[i];
                s_g[j] = g;
                if (ELL) {
                    // rows ylo | yhi << 16; a Gaussian without entries has none
                    const bool has = (i + 1 < n ? sl.start[i + 1] : uint64_t(E)) > sl.start[i];
                    s_e[j] = has ? sl.ell[10 * size_t(n) + g] : __uint_as_float(0xffff0000u);
                } else {
                    s_rect[j] = sl.rect[i];
                }
            }
        }
        bool table = false;
        if (ELL) {
            __syncthreads();
            // rows of the window's Gaussians (thread t: Gaussians 4t .. 4t + 3), their prefix
            uint32_t nr[kExpChunk / kExpThreads], sum = 0;
#pragma unroll
            for (int q = 0; q < kExpChunk / kExpThreads; ++q) {
                const int j = int(threadIdx.x) * (kExpChunk / kExpThreads) + q;
                nr[q] = 0u;
                if (j < w) {
                    const uint32_t y = __float_as_uint(s_e[j]);
                    const int ylo = int(int16_t(y & 0xffff)), yhi = int(int16_t(y >> 16));
                    nr[q] = yhi >= ylo ? uint32_t(yhi - ylo + 1) : 0u;
                }
                sum += nr[q];
            }
            uint32_t base = block_exclusive_scan_256(sum, s_w);
#pragma unroll
            for (int q = 0; q < kExpChunk / kExpThreads; ++q) {
                const int j = int(threadIdx.x) * (kExpChunk / kExpThreads) + q;
                if (j < w) s_rowstart[j] = base;
                base += nr[q];
            }
            if (threadIdx.x == kExpThreads - 1) s_rowstart[w] = base;  // total rows
            __syncthreads();
            const uint32_t rows = s_rowstart[w];
            table = rows <= uint32_t(kRowCap);
            if (table) {
                // one row per thread: its Gaussian (the last whose first row is at most o), its
                // run of columns; widths into s_rowcum, then their prefix over the window
                uint32_t wsum = 0;
                constexpr int RPT = kRowCap / kExpThreads;  // rows per thread in the prefix
                for (int o = int(threadIdx.x); o < int(rows); o += kExpThreads) {
                    int a = 0, b = w;  // s_rowstart[a] <= o < s_rowstart[b]
                    while (b - a > 1) {
                        const int mid = (a + b) >> 1;
                        if (s_rowstart[mid] <= uint32_t(o)) a = mid; else b = mid;
                    }
                    EllipseTiles el;
                    ellipse_unpack(sl.ell + size_t(n) + s_g[a], int(n), el);
                    const int ty = el.ylo + (o - int(s_rowstart[a]));
                    int xlo, xhi;
                    ellipse_row(el, ty, cam.TX, xlo, xhi);
                    s_rowcum[o] = xhi >= xlo ? uint32_t(xhi - xlo + 1) : 0u;
                    s_rowtile[o] = uint32_t(ty) * uint32_t(cam.TX) + uint32_t(max(xlo, 0));
                    s_rowg[o] = uint16_t(a);
                }
                __syncthreads();
                // exclusive prefix of the widths: thread t owns rows RPT t .. RPT t + RPT - 1
                uint32_t loc[RPT];
#pragma unroll
                for (int q = 0; q < RPT; ++q) {
                    const int o = int(threadIdx.x) * RPT + q;
                    loc[q] = o < int(rows) ? s_rowcum[o] : 0u;
                    wsum += loc[q];
                }
                uint32_t run = block_exclusive_scan_256(wsum, s_w);
                __syncthreads();  // every row's width was read before it is overwritten
#pragma unroll
                for (int q = 0; q < RPT; ++q) {
                    const int o = int(threadIdx.x) * RPT + q;
                    if (o < int(rows)) s_rowcum[o] = run;
                    run += loc[q];
                }
            }
        }
        __syncthreads();
        // the square test: warp v takes the chunk's entries [v CH/8, (v + 1) CH/8) 32 at a time
        // (lane l on entry 32 k + l of its run, so the stores stay consecutive); a lane finds the
        // owner of its first entry by binary search and then walks it forward past the few
        // Gaussians whose slices start between its successive entries.  The ellipse path keeps the
        // interleaved order (entry k 256 + t) of its row tables.
        const uint32_t run0 = ELL ? e0 + threadIdx.x : e0 + (threadIdx.x >> 5) * uint32_t(CH / (kExpThreads / 32)) + lane;
        int owner = -1;
#pragma unroll
        for (int k = 0; k < CH / kExpThreads; ++k) {
            const uint32_t e = ELL ? run0 + uint32_t(k * kExpThreads) : run0 + uint32_t(32 * k);
            const bool valid = e < E;
            uint32_t tile = 0u;
            uint32_t gid = 0u;
            if (valid && !ELL) {
                if (owner < 0) {
                    int lo = 0, hi = w;  // s_start[lo] <= e < s_start[hi]
                    while (hi - lo > 1) {
                        const int mid = (lo + hi) >> 1;
                        if (s_start[mid] <= e) lo = mid; else hi = mid;
                    }
                    owner = lo;
                } else {
                    while (s_start[owner + 1] <= e) ++owner;  // s_start[w] lies past the chunk
                }
                const uint32_t kk = uint32_t(uint64_t(e) - s_start[owner]);
                gid = s_g[owner];
                const uint2 r = s_rect[owner];
                uint32_t q, rem;
                div_small(kk, r.y, q, rem);
                tile = ((r.x >> 16) + q) * uint32_t(cam.TX) + (r.x & 0xffffu) + rem;
            } else if (valid && ELL && table) {
                // the window's rows in entry order: the last row starting at or before e
                const uint32_t off = uint32_t(uint64_t(e) - s_start[0]);
                int a = 0, b = int(s_rowstart[w]);
                while (b - a > 1) {
                    const int mid = (a + b) >> 1;
                    if (s_rowcum[mid] <= off) a = mid; else b = mid;
                }
                tile = s_rowtile[a] + (off - s_rowcum[a]);
                gid = s_g[s_rowg[a]];
            } else if (valid) {
                int lo = 0, hi = w;  // s_start[lo] <= e < s_start[hi]
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if (s_start[mid] <= e) lo = mid; else hi = mid;
                }
                const uint32_t kk = uint32_t(uint64_t(e) - s_start[lo]);
                gid = s_g[lo];
                if (ELL) {
                    // the kk-th tile of the splat's rows of column runs, walked row by row
                    tile = tiles_total;  // unreachable for consistent inputs; k_ranges skips it
                    EllipseTiles el;
                    ellipse_unpack(sl.ell + size_t(n) + s_g[lo], int(n), el);
                    if (el.ylo <= el.yhi) {
                        uint32_t cum = 0u;
                        for (int ty = el.ylo; ty <= el.yhi; ++ty) {
                            int xlo, xhi;
                            ellipse_row(el, ty, cam.TX, xlo, xhi);
                            const uint32_t wd = xhi >= xlo ? uint32_t(xhi - xlo + 1) : 0u;
                            if (kk < cum + wd) {
                                tile = uint32_t(ty) * uint32_t(cam.TX) + uint32_t(xlo) + (kk - cum);
                                break;
                            }
                            cum += wd;
                        }
                    }
                } else {
                    const uint2 r = s_rect[lo];
                    const uint32_t ty = (r.x >> 16) + kk / r.y, tx = (r.x & 0xffffu) + kk % r.y;
                    tile = ty * uint32_t(cam.TX) + tx;
                }
            }
            if (valid) {
                tile_keys[e] = tile;
                vals[e] = gid;
            }
            for (int p = 0; p < passes; ++p) {
                count_digit<R>(s_h[p], valid ? (tile >> (p * digit_bits)) & uint32_t(R - 1) : uint32_t(R));
            }
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < passes * R; i += kExpThreads) {
        const uint32_t cnt = (&s_h[0][0])[i];
        if (cnt) atomicAdd(ghist + (i / R) * 256 + (i % R), cnt);
    }
}

template <int RBITS>
void tile_sort_launch(const uint32_t* kin, const uint32_t* vin, Count count, int digit, int pass, bool last,
                      const float* depth, uint64_t* keys64, const SortCtl& ctl, unsigned blocks, uint32_t* kout,
                      uint32_t* vout, cudaStream_t s) {
    if (last && keys64)
        pdl_launch(k_sweep_pass<RBITS, kTileItems, false, false, true, kTileMinBlocks>, blocks, kRsThreads, 0, s,
            kin, vin, DepthKeySource{depth, nullptr}, count, pass * digit, pass, ctl, kout, vout, nullptr,
            nullptr, keys64);
    else
        pdl_launch(k_sweep_pass<RBITS, kTileItems, false, false, false, kTileMinBlocks>, blocks, kRsThreads, 0, s,
            kin, vin, DepthKeySource{}, count, pass * digit, pass, ctl, kout, vout, nullptr, nullptr, nullptr);
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
    p.slice_blocks = ceil_div(std::max<size_t>(N, 1), size_t(kSlGauss));
    p.chunks = ceil_div(std::max<size_t>(capacity, 1), size_t(kExpChunk));
    size_t o = 0;
    p.off_dkeys = o;      o = align256(o + 2 * N * sizeof(uint32_t));   // depth keys, 2 buffers
    p.off_dvals = o;      o = align256(o + 2 * N * sizeof(uint32_t));   // Gaussian ids, 2 buffers
    p.off_tiles_sorted = o; o = align256(o + N * sizeof(uint32_t));     // tiles_touched, depth order
    p.off_start = o;      o = align256(o + N * sizeof(uint64_t));     // slice starts, depth order
    p.off_rect = o;       o = align256(o + N * sizeof(uint2));        // tile rectangles, depth order
    p.off_owner = o;      o = align256(o + p.chunks * sizeof(uint32_t));  // owner of each chunk
    p.off_tkeys = o;      o = align256(o + 2 * capacity * sizeof(uint32_t));  // tile ids, 2 buffers
    p.off_tvals = o;      o = align256(o + capacity * sizeof(uint32_t));      // + the caller's list
    // control words, zeroed by one kernel at the start of every call:
    // result {E (u64), error (u32), pad}, counters, digit totals, look-back status
    p.off_ctl = o;
    p.off_result = o;               o += 16;
    p.off_counters = o;             o += 8 * sizeof(uint32_t);
    p.off_ghist_depth = o;          o += 4 * 256 * sizeof(uint32_t);
    p.off_ghist_tile = o;           o += 3 * 256 * sizeof(uint32_t);
    p.off_status_slices = o;        o += p.slice_blocks * sizeof(uint64_t);
    p.off_status_depth = o;         o += 4 * p.depth_tiles * 256 * sizeof(uint32_t);
    p.off_status_tile = o;          o += size_t(p.tile_passes) * p.tile_tiles * 256 * sizeof(uint32_t);
    p.ctl_bytes = o - p.off_ctl;
    o = align256(o);
    p.total_bytes = o;
    return p;
}

__global__ void k_report(const uint64_t* __restrict__ result, uint64_t* __restrict__ host) {
    RS_PDL_ENTER();
    host[0] = result[0];                                   // E
    host[1] = uint64_t(reinterpret_cast<const uint32_t*>(result + 1)[0]);  // look-back timeout flag
}

template <int RBITS>
void expand_launch(const CameraF& cam, uint32_t n, Count ce, const uint32_t* perm, const SliceOut& sl, int digit,
                   int passes, uint32_t* ghist, uint32_t* tk, uint32_t* tv, const rs_projected& p, cudaStream_t s) {
    const size_t per = p.tile_test == RS_TILE_TEST_ELLIPSE ? 1 : 2;  // 1024-entry chunks per block
    const unsigned blocks = unsigned(std::min<size_t>((sl.chunks + per - 1) / per, 152 * 8));
    if (p.tile_test == RS_TILE_TEST_ELLIPSE) {
        constexpr size_t smem = (kExpChunk + 2 * kRowCap) * sizeof(float) + kRowCap * sizeof(uint16_t);
        if (cudaFuncSetAttribute(k_expand<RBITS, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
            cudaSuccess)
            return;  // that error stays the last error, which launch_bin returns
        pdl_launch(k_expand<RBITS, true>, blocks, kExpThreads, smem, s, cam, n, ce, perm, sl, digit, passes, ghist, tk, tv);
    }
    else
        pdl_launch(k_expand<RBITS, false>, blocks, kExpThreads, 0, s, cam, n, ce, perm, sl, digit, passes, ghist, tk, tv);
}

cudaError_t launch_report(const uint8_t* result_block, uint64_t* host, cudaStream_t s) {
    pdl_launch(k_report, 1, 1, 0, s, reinterpret_cast<const uint64_t*>(result_block), host);
    return cudaGetLastError();
}

cudaError_t launch_bin(const BinPlan& plan, const CameraF& cam, const rs_projected& p, uint8_t* ws,
                       uint64_t* keys_out, uint32_t* point_list, uint32_t* tile_ranges, cudaStream_t s) {
    uint32_t* ctl_words = reinterpret_cast<uint32_t*>(ws + plan.off_ctl);
    {
        const size_t words = plan.ctl_bytes / 4 + 2u * uint32_t(plan.n_tiles);
        const unsigned blocks = unsigned(std::min<size_t>(ceil_div(words, 256), 152 * 8));
        pdl_launch(k_clear, blocks, 256, 0, s, tile_ranges, 2u * uint32_t(plan.n_tiles), ctl_words, plan.ctl_bytes / 4);
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
    pdl_launch(k_sweep_hist<8, kDepthHistItems, 4, true>, unsigned(ceil_div(n, kRsThreads * kDepthHistItems)), kRsThreads, 0, s,
        nullptr, src, cn, 8, dctl.ghist);
    pdl_launch(k_sweep_pass<8, kDepthItems, true, false>, dblocks, kRsThreads, 0, s,
        nullptr, nullptr, src, cn, 0, 0, dctl, DK[0], DV[0], nullptr, nullptr, nullptr);
    pdl_launch(k_sweep_pass<8, kDepthItems, false, false>, dblocks, kRsThreads, 0, s,
        DK[0], DV[0], src, cn, 8, 1, dctl, DK[1], DV[1], nullptr, nullptr, nullptr);
    pdl_launch(k_sweep_pass<8, kDepthItems, false, false>, dblocks, kRsThreads, 0, s,
        DK[1], DV[1], src, cn, 16, 2, dctl, DK[0], DV[0], nullptr, nullptr, nullptr);
    pdl_launch(k_sweep_pass<8, kDepthItems, false, true>, dblocks, kRsThreads, 0, s,
        DK[0], DV[0], src, cn, 24, 3, dctl, DK[1], DV[1], p.d_tiles_touched, tiles_sorted, nullptr);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const uint32_t* perm = DV[1];

    // 2. slices (E lands in result[0]), then the entries in depth order and the digit totals of
    //    their tile ids
    const int digit = (plan.tile_bits + plan.tile_passes - 1) / plan.tile_passes;  // <= 8
    const int rbits = digit <= 4 ? 4 : digit <= 6 ? 6 : digit == 7 ? 7 : 8;
    uint32_t* tk = reinterpret_cast<uint32_t*>(ws + plan.off_tkeys);
    uint32_t* TK[2] = {tk, tk + plan.capacity};
    uint32_t* TV[2] = {point_list, reinterpret_cast<uint32_t*>(ws + plan.off_tvals)};
    int cur = plan.tile_passes % 2;  // the last pass lands in buffer 0 (the caller's list)
    const bool ell = p.tile_test == RS_TILE_TEST_ELLIPSE;
    const SliceOut sl{reinterpret_cast<uint64_t*>(ws + plan.off_start), reinterpret_cast<uint2*>(ws + plan.off_rect),
                      reinterpret_cast<uint32_t*>(ws + plan.off_owner), uint32_t(plan.chunks),
                      ell ? p.d_ellipse : nullptr};
    pdl_launch(k_slices, unsigned(plan.slice_blocks), kSlThreads, 0, s,
        cam, n, perm, tiles_sorted, p.d_means2d, p.d_radius, counters + 7,
        reinterpret_cast<unsigned long long*>(ws + plan.off_status_slices), error, result, sl);
    e = cudaGetLastError();
    if (e != cudaSuccess || plan.capacity == 0) return e;
    const Count ce{0u, result, uint32_t(plan.capacity)};
    uint32_t* ghist_tile = reinterpret_cast<uint32_t*>(ws + plan.off_ghist_tile);
    switch (rbits) {
        case 4: expand_launch<4>(cam, n, ce, perm, sl, digit, plan.tile_passes, ghist_tile, TK[cur], TV[cur], p, s); break;
        case 6: expand_launch<6>(cam, n, ce, perm, sl, digit, plan.tile_passes, ghist_tile, TK[cur], TV[cur], p, s); break;
        case 7: expand_launch<7>(cam, n, ce, perm, sl, digit, plan.tile_passes, ghist_tile, TK[cur], TV[cur], p, s); break;
        default: expand_launch<8>(cam, n, ce, perm, sl, digit, plan.tile_passes, ghist_tile, TK[cur], TV[cur], p, s); break;
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    // 3. stable sort of the entries by tile id, then the ranges
    const SortCtl tctl{counters + 4, reinterpret_cast<uint32_t*>(ws + plan.off_ghist_tile),
                       reinterpret_cast<uint32_t*>(ws + plan.off_status_tile), error,
                       uint32_t(plan.tile_tiles)};
    const unsigned tblocks = unsigned(plan.tile_tiles);
    for (int pass = 0; pass < plan.tile_passes; ++pass) {
        switch (rbits) {
            case 4: tile_sort_launch<4>(TK[cur], TV[cur], ce, digit, pass, pass == plan.tile_passes - 1, p.d_depth, keys_out, tctl, tblocks, TK[cur ^ 1], TV[cur ^ 1], s); break;
            case 6: tile_sort_launch<6>(TK[cur], TV[cur], ce, digit, pass, pass == plan.tile_passes - 1, p.d_depth, keys_out, tctl, tblocks, TK[cur ^ 1], TV[cur ^ 1], s); break;
            case 7: tile_sort_launch<7>(TK[cur], TV[cur], ce, digit, pass, pass == plan.tile_passes - 1, p.d_depth, keys_out, tctl, tblocks, TK[cur ^ 1], TV[cur ^ 1], s); break;
            default: tile_sort_launch<8>(TK[cur], TV[cur], ce, digit, pass, pass == plan.tile_passes - 1, p.d_depth, keys_out, tctl, tblocks, TK[cur ^ 1], TV[cur ^ 1], s); break;
        }
        cur ^= 1;
    }
    {
        const unsigned rb = unsigned(std::min<size_t>(ceil_div(plan.capacity, 1024), 152 * 16));
        pdl_launch(k_ranges, rb, 256, 0, s, TK[0], ce, uint32_t(plan.n_tiles), tile_ranges);
    }
    return cudaGetLastError();
}

}  // namespace rs
