// Appearance MLP (rigel README "Appearance MLP") and the L1 loss gradient of the training step.
//
// Per Gaussian and view: x = [latent ; unit view direction], h = relu(W1 x + b1),
// colour = sigmoid(W2 h + b2).  The page runs one thread per Gaussian with the weights in shared
// memory.  All products keep float32 accuracy with split TF32 operands: a = a_hi + a_lo with both
// parts TF32, and a.b ~ a_hi b_hi + a_hi b_lo + a_lo b_hi.
//
// The forward runs the first layer on the fifth-generation tensor cores (tcgen05.mma, 128
// Gaussians x HID per CTA, the accumulator in tensor memory) and the thin second layer (three
// outputs) in float32 on the CUDA cores while reading the accumulator back.
//
// The backward runs on the tensor cores too (tcgen05.mma into tensor memory): per 128-Gaussian
// tile it recomputes the first layer, forms dL/dz2, dL/dz1 and dL/dlatent in float32 on the CUDA
// cores (two threads per Gaussian, one per half of the hidden units), and gets every weight
// gradient from one product per tile, [dZ1 | H]^T [X | dZ2 | 1], accumulated in tensor memory over
// all of a CTA's tiles and flushed with one global atomic per weight per CTA (the reduction
// pattern the page describes for its MLP backward).  View directions are constants: no gradient
// reaches the means.
#include "rs_internal.cuh"

namespace rs {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ uint32_t tf32_of(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// head and tail of x, both TF32 (the tail is the rounding error of the head, rounded again)
__device__ __forceinline__ void split(float x, uint32_t& hi, uint32_t& lo) {
    hi = tf32_of(x);
    lo = tf32_of(x - __uint_as_float(hi));
}

struct MlpArgs {
    CameraF cam;
    int n, L, D;                       // Gaussians, latent width, input width L + 3
    const float* means;
    const float* latents;
    const float* W1;
    const float* b1;
    const float* W2;
    const float* b2;
};

__device__ __forceinline__ float sigmoidf(float z) { return 1.0f / (1.0f + expf(-z)); }

// ---------------------------------------------------------------- forward on the tensor cores (tcgen05)
// A CTA of 128 threads takes 128 Gaussians at a time (thread r = row r = TMEM lane r).  Layer 1,
// Z = X W1^T [128 x HID] (X's columns: the view direction, then the latents; W1's columns staged
// in the same order), runs as tcgen05.mma kind::tf32 (M = 128, N = HID, K = 8 per
// instruction) with split operands, Z = Xh W1h + Xh W1l + Xl W1h (the three products that keep
// float32 accuracy), accumulated in tensor memory.  X and W1 sit in shared memory in the
// no-swizzle K-major layout of the PTX ISA's tcgen05 matrix descriptors: 8-row x 16-byte core
// matrices of 128 contiguous bytes, the next core matrix along K 128 bytes on (leading byte
// offset), the next 8-row group 2 KS x 128 bytes on (stride byte offset).  Each warp then reads
// its 32 rows of Z from tensor memory (tcgen05.ld 32x32b), adds b1, applies relu and forms the
// three outputs of the thin second layer (N = 3) in float32 before the sigmoid.
__device__ unsigned int g_tc_error;  // set when a bounded tensor-core wait gave up

constexpr int kTcRows = 128;
constexpr uint32_t kTcWaitLimit = 1u << 22;  // mbarrier polls before a wait is given up

template <int HID, int KS>
struct TcFwdSmem {
    static constexpr int kCore = 128;                       // bytes per core matrix
    static constexpr int kACores = (kTcRows / 8) * 2 * KS;  // X: 16 row groups x 2 KS core columns
    static constexpr int kBCores = (HID / 8) * 2 * KS;      // W1: HID / 8 row groups
    alignas(1024) uint8_t a_hi[kACores * kCore], a_lo[kACores * kCore];
    alignas(128) uint8_t b_hi[kBCores * kCore], b_lo[kBCores * kCore];
    alignas(16) float w2[3][HID];
    alignas(16) float b1[HID];
    float b2[4];
    alignas(8) uint64_t mbar;
    uint32_t tmem;
};

// Byte offset of element (row, k) in a K-major no-swizzle operand with 2 KS core columns.
template <int KS>
__device__ __forceinline__ int tc_kmajor_offset(int row, int k) {
    return ((row >> 3) * (2 * KS) + (k >> 2)) * 128 + (row & 7) * 16 + (k & 3) * 4;
}

// tcgen05 shared-memory matrix descriptor (PTX ISA "Matrix Descriptors"): start address, leading
// and stride byte offsets (all >> 4), the fixed 0b001 at bits 46-48, no swizzle.
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t(lbo >> 4) << 16) | (uint64_t(sbo >> 4) << 32) |
           (uint64_t(1) << 46);
}

// Instruction descriptor of kind::tf32 (PTX ISA "Instruction descriptor"): D float32 (bits 4-5 = 1),
// A and B TF32 (bits 7-9 and 10-12 = 2), both K-major, N >> 3 at bits 17-22, M >> 4 at 24-28.
template <int N>
__host__ __device__ constexpr uint32_t tc_idesc_tf32() {
    return (1u << 4) | (2u << 7) | (2u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(kTcRows >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc ? 1u : 0u));
}

__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity) {
    for (uint32_t i = 0; i < kTcWaitLimit; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(mbar), "r"(parity)
            : "memory");
        if (ok) return true;
    }
    return false;
}

// 32 consecutive tensor-memory columns of the warp's 32 lanes (tcgen05.ld 32x32b.x32): lane t
// gets row (lane base + t), columns taddr .. taddr + 31.
template <int COLS>
__device__ __forceinline__ void tc_ld_rows(uint32_t taddr, float (&v)[COLS]);

template <>
__device__ __forceinline__ void tc_ld_rows<32>(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

template <int HID, int KS>
__global__ void __launch_bounds__(kTcRows) k_mlp_fwd_tc(MlpArgs a, float* __restrict__ colors) {
    RS_PDL_ENTER();
    using Smem = TcFwdSmem<HID, KS>;
    extern __shared__ __align__(1024) unsigned char tc_smem_raw[];
    // the operands' 1 KB alignment, whatever the dynamic region's base (1 KB of slack is allocated)
    const uint32_t raw = static_cast<uint32_t>(__cvta_generic_to_shared(tc_smem_raw));
    Smem& sm = *reinterpret_cast<Smem*>(tc_smem_raw + ((1024u - (raw & 1023u)) & 1023u));
    const int r = threadIdx.x, warp = r >> 5;
    constexpr int K = KS * 8;
    // W1 as TF32 heads and tails in the K-major layout, its columns in X's order (the view
    // direction first, then the latents; zeros past D), W2 and the biases
    for (int e = r; e < HID * K; e += kTcRows) {
        const int j = e / K, k = e % K;
        const int src = k < 3 ? a.L + k : k - 3;
        const float v = k < a.D ? a.W1[j * a.D + src] : 0.f;
        uint32_t h, l;
        split(v, h, l);
        const int o = tc_kmajor_offset<KS>(j, k);
        *reinterpret_cast<uint32_t*>(sm.b_hi + o) = h;
        *reinterpret_cast<uint32_t*>(sm.b_lo + o) = l;
    }
    for (int e = r; e < 3 * HID; e += kTcRows) sm.w2[e / HID][e % HID] = a.W2[e];
    for (int e = r; e < HID; e += kTcRows) sm.b1[e] = a.b1[e];
    if (r < 3) sm.b2[r] = a.b2[r];
    const uint32_t mbar = static_cast<uint32_t>(__cvta_generic_to_shared(&sm.mbar));
    if (r == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(mbar) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == 0) {
        const uint32_t slot = static_cast<uint32_t>(__cvta_generic_to_shared(&sm.tmem));
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(slot), "r"(HID)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
    const uint32_t tmem = sm.tmem;
    const uint32_t a_hi = static_cast<uint32_t>(__cvta_generic_to_shared(sm.a_hi));
    const uint32_t a_lo = static_cast<uint32_t>(__cvta_generic_to_shared(sm.a_lo));
    const uint32_t b_hi = static_cast<uint32_t>(__cvta_generic_to_shared(sm.b_hi));
    const uint32_t b_lo = static_cast<uint32_t>(__cvta_generic_to_shared(sm.b_lo));
    constexpr uint32_t kSbo = 2 * KS * 128;
    constexpr uint32_t idesc = tc_idesc_tf32<HID>();
    // camera centre C = -R^T t
    const CameraF& cam = a.cam;
    const float C0 = -(cam.R[0] * cam.t[0] + cam.R[3] * cam.t[1] + cam.R[6] * cam.t[2]);
    const float C1 = -(cam.R[1] * cam.t[0] + cam.R[4] * cam.t[1] + cam.R[7] * cam.t[2]);
    const float C2 = -(cam.R[2] * cam.t[0] + cam.R[5] * cam.t[1] + cam.R[8] * cam.t[2]);
    const int tiles = (a.n + kTcRows - 1) / kTcRows;
    uint32_t phase = 0;
    bool failed = false;
    // this thread's row of X for a tile: the unit view direction, then the latents (zeros past D);
    // the next tile's row is loaded while the current tile's products and epilogue run
    float x[K - 3], d[3];
    auto load_row = [&](int tile) {
        const int i = tile * kTcRows + r;
        const bool in = tile < tiles && i < a.n;
#pragma unroll
        for (int k = 0; k < K - 3; ++k) x[k] = in && k < a.L ? a.latents[size_t(k) * a.n + i] : 0.f;
        d[0] = in ? a.means[i] - C0 : 0.f;
        d[1] = in ? a.means[size_t(a.n) + i] - C1 : 0.f;
        d[2] = in ? a.means[2 * size_t(a.n) + i] - C2 : 0.f;
    };
    load_row(blockIdx.x);
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int i = tile * kTcRows + r;
        const bool in = i < a.n;
        {
            const float len = sqrtf(d[0] * d[0] + d[1] * d[1] + d[2] * d[2]);
            const float il = len > 0.f ? 1.0f / len : 0.f;
            const float dn[3] = {d[0] * il, d[1] * il, d[2] * il};
#pragma unroll
            for (int k = 0; k < K; k += 4) {
                uint32_t h[4], l[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int kk = k + q;
                    split(kk < 3 ? dn[kk] : x[kk - 3], h[q], l[q]);
                }
                const int o = tc_kmajor_offset<KS>(r, k);
                *reinterpret_cast<uint4*>(sm.a_hi + o) = make_uint4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<uint4*>(sm.a_lo + o) = make_uint4(l[0], l[1], l[2], l[3]);
            }
        }
        // the operands are visible to the tensor cores, and every warp is done reading the
        // previous tile's tensor memory
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
        __syncthreads();
        asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
        if (r == 0) {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const uint32_t off = uint32_t(ks) * 2u * 128u;  // two core columns per K = 8 step
                const uint64_t ah = tc_desc(a_hi + off, 128, kSbo), al = tc_desc(a_lo + off, 128, kSbo);
                const uint64_t bh = tc_desc(b_hi + off, 128, kSbo), bl = tc_desc(b_lo + off, 128, kSbo);
                tc_mma_tf32(tmem, ah, bh, idesc, ks > 0);
                tc_mma_tf32(tmem, ah, bl, idesc, true);
                tc_mma_tf32(tmem, al, bh, idesc, true);
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(mbar)
                         : "memory");
        }
        load_row(tile + int(gridDim.x));
        // the products are done (or every thread gives up together: the warp-wide loads and the
        // barriers below need the whole CTA)
        const bool ok = __syncthreads_and(mbar_wait(mbar, phase));
        phase ^= 1u;
        asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
        if (!ok) {
            // give up on this CTA: flag it, and let the output show it
            atomicOr(&g_tc_error, 1u);
            failed = true;
            if (in)
                for (int c = 0; c < 3; ++c) colors[size_t(c) * a.n + i] = __int_as_float(0x7fc00000);
            break;
        }
        // relu(Z + b1) and the second layer, 32 hidden units at a time
        float o0 = sm.b2[0], o1 = sm.b2[1], o2 = sm.b2[2];
#pragma unroll
        for (int half = 0; half < HID / 32; ++half) {
            float z[32];
            tc_ld_rows<32>(tmem + (uint32_t(warp * 32) << 16) + uint32_t(32 * half), z);
#pragma unroll
            for (int jj = 0; jj < 32; jj += 4) {
                const int j = 32 * half + jj;
                const float4 bb = *reinterpret_cast<const float4*>(&sm.b1[j]);
                const float4 u0 = *reinterpret_cast<const float4*>(&sm.w2[0][j]);
                const float4 u1 = *reinterpret_cast<const float4*>(&sm.w2[1][j]);
                const float4 u2 = *reinterpret_cast<const float4*>(&sm.w2[2][j]);
                const float h0 = fmaxf(z[jj] + bb.x, 0.f), h1 = fmaxf(z[jj + 1] + bb.y, 0.f);
                const float h2 = fmaxf(z[jj + 2] + bb.z, 0.f), h3 = fmaxf(z[jj + 3] + bb.w, 0.f);
                o0 = fmaf(u0.x, h0, o0); o0 = fmaf(u0.y, h1, o0); o0 = fmaf(u0.z, h2, o0); o0 = fmaf(u0.w, h3, o0);
                o1 = fmaf(u1.x, h0, o1); o1 = fmaf(u1.y, h1, o1); o1 = fmaf(u1.z, h2, o1); o1 = fmaf(u1.w, h3, o1);
                o2 = fmaf(u2.x, h0, o2); o2 = fmaf(u2.y, h1, o2); o2 = fmaf(u2.z, h2, o2); o2 = fmaf(u2.w, h3, o2);
            }
        }
        if (in) {
            colors[i] = sigmoidf(o0);
            colors[size_t(a.n) + i] = sigmoidf(o1);
            colors[2 * size_t(a.n) + i] = sigmoidf(o2);
        }
    }
    // tensor memory goes back once no warp reads it and no product is in flight
    if (failed) (void)mbar_wait(mbar, phase ^ 1u);
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(HID) : "memory");
}

// ---------------------------------------------------------------- backward on the tensor cores (tcgen05)
// A CTA of 128 threads takes 128 Gaussians at a time (thread r = row r = TMEM lane r):
//  1. Z1 = X W1^T on the tensor cores, as in the forward (tensor memory columns [0, HID)).
//  2. Thread r reads its row of Z1 back and forms, in float32 on the CUDA cores,
//     h = relu(z1 + b1), z2 = W2 h + b2, s = sigmoid(z2), dz2 = dL/dcolour s (1 - s),
//     dz1 = (W2^T dz2) where z1 > 0, and dL/dlatent = W1^T dz1 (the latent columns of W1).
//  3. The tile's weight gradients are one product on the tensor cores,
//     G = [dZ1 | H]^T [X | dZ2 | 1] (M = 128: rows h of dZ1^T, then rows 64 + h of H^T; N = NW:
//     the columns of X, then dz2 (3), then ones; K = the tile's 128 Gaussians), accumulated in
//     tensor memory columns [HID, HID + NW) over all of the CTA's tiles.  Its blocks give
//     dW1 = dZ1^T X, db1 = dZ1^T 1 and dW2^T = H^T dZ2; the others are not used.
//  4. At the end every weight's CTA sum goes to global memory with one atomic (the reduction the
//     page describes for its MLP backward, per CTA), and db2 with a block reduction.
// Both operands of the product are the transposes of what the threads hold (row r of the tile),
// stored K-major without swizzle: thread r writes column r.  In the core-matrix layout the bank
// of element (m, r) is (m mod 8) * 4 + (r mod 4), so a warp writing one row m for its 32 Gaussians
// would hit 4 banks; instead lane L writes, at step j, row 8 g + ((L / 4 + j) mod 8) of each group
// g of eight rows -- 32 distinct banks -- after rotating its eight values of the group by L / 4.
template <int KS>
constexpr int tc_bwd_nw() { return ((8 * KS + 4 + 15) / 16) * 16; }

template <int HID, int KS>
struct TcBwdSmem {
    static constexpr int NW = tc_bwd_nw<KS>();
    static constexpr int kCore = 128;
    static constexpr int kXCores = (kTcRows / 8) * 2 * KS;   // X [128 x 8 KS]
    static constexpr int kWCores = (HID / 8) * 2 * KS;       // W1 [HID x 8 KS]
    static constexpr int kGCores = (kTcRows / 8) * 32;       // [dZ1 | H]^T [128 x 128 Gaussians]
    static constexpr int kRCores = (NW / 8) * 32;            // [X | dZ2 | 1]^T [NW x 128 Gaussians]
    alignas(1024) uint8_t x_hi[kXCores * kCore], x_lo[kXCores * kCore];
    alignas(128) uint8_t w_hi[kWCores * kCore], w_lo[kWCores * kCore];
    alignas(128) uint8_t g_hi[kGCores * kCore], g_lo[kGCores * kCore];
    alignas(128) uint8_t r_hi[kRCores * kCore], r_lo[kRCores * kCore];
    // W1 in float32, row-major [HID][8 KS], for dL/dx where it fits (else W1 = head + tail)
    static constexpr bool kW1f = KS <= 3;
    alignas(16) float w1f[kW1f ? HID * 8 * KS : 4];
    alignas(16) float w2[3][HID];
    alignas(16) float b1[HID];
    float b2[4];
    float db2[4][4];
    alignas(8) uint64_t mbar_z, mbar_g;
    uint32_t tmem;
};

// Byte offset of element (row, k) of a K-major no-swizzle operand whose K extent is KC core
// columns (4 elements each).
template <int KC>
__device__ __forceinline__ int tc_offset(int row, int k) {
    return ((row >> 3) * KC + (k >> 2)) * 128 + (row & 7) * 16 + (k & 3) * 4;
}

// v rotated by s (0..7) positions: out[i] = v[(i + s) mod 8], in three select stages.
__device__ __forceinline__ void rotate8(float (&v)[8], int s) {
    float t[8];
    if (s & 1) {
#pragma unroll
        for (int i = 0; i < 8; ++i) t[i] = v[(i + 1) & 7];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = t[i];
    }
    if (s & 2) {
#pragma unroll
        for (int i = 0; i < 8; ++i) t[i] = v[(i + 2) & 7];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = t[i];
    }
    if (s & 4) {
#pragma unroll
        for (int i = 0; i < 8; ++i) t[i] = v[(i + 4) & 7];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = t[i];
    }
}

// tcgen05.ld 32x32b.x8 without the wait: the registers are valid only after tc_ld_wait.
__device__ __forceinline__ void tc_ld8_async(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
}
// Waits for this thread's tensor-memory loads; the registers pass through an empty asm so that
// no use of them is scheduled before the wait.
__device__ __forceinline__ void tc_ld_wait(uint32_t (&r)[8]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) asm volatile("" : "+r"(r[i]));
}

template <>
__device__ __forceinline__ void tc_ld_rows<16>(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Split into a TF32 head (x with its low 13 mantissa bits cleared) and the exact remainder; the
// tensor cores read a TF32 operand from the top 19 bits of its word, so the remainder's own low
// bits are dropped there: the pair still carries x to about 2^-21.
__device__ __forceinline__ void split_trunc(float x, uint32_t& hi, uint32_t& lo) {
    hi = __float_as_uint(x) & 0xffffe000u;
    lo = __float_as_uint(x - __uint_as_float(hi));
}

// Column k (this thread's Gaussian) of rows 8 grp .. 8 grp + 7 of a transposed operand with 32
// core columns of K, as TF32 heads and tails (truncating split), written in the conflict-free
// rotated order.
__device__ __forceinline__ void store_col8_t(uint8_t* hi, uint8_t* lo, int grp, int k, float (&v)[8], int lane) {
    const int s = lane >> 2;
    rotate8(v, s);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t h, l;
        split_trunc(v[j], h, l);
        const int o = tc_offset<32>(8 * grp + ((s + j) & 7), k);
        *reinterpret_cast<uint32_t*>(hi + o) = h;
        *reinterpret_cast<uint32_t*>(lo + o) = l;
    }
}

constexpr int kTcBwdThreads = 2 * kTcRows;  // two threads per Gaussian row: one per half of the hidden units

// tcgen05.st 32x32b.x32: 32 consecutive tensor-memory columns of this warp's 32 lanes.
__device__ __forceinline__ void tc_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
        "tcgen05.wait::st.sync.aligned;\n" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
        "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
        "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])),
        "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
        "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])),
        "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

template <int HID, int KS>
__global__ void __launch_bounds__(kTcBwdThreads) k_mlp_bwd_tc(MlpArgs a, const float* __restrict__ dcolors,
                                                               float* __restrict__ dlatents, float* __restrict__ dW1,
                                                               float* __restrict__ db1, float* __restrict__ dW2,
                                                               float* __restrict__ db2) {
    RS_PDL_ENTER();
    using Smem = TcBwdSmem<HID, KS>;
    constexpr int NW = Smem::NW;
    constexpr int K = KS * 8;
    constexpr int kOnes = K + 3;       // the column of ones in [X | dZ2 | 1]
    constexpr int HH = HID / 2;        // hidden units per half
    extern __shared__ __align__(1024) unsigned char tc_smem_raw[];
    const uint32_t raw = static_cast<uint32_t>(__cvta_generic_to_shared(tc_smem_raw));
    Smem& sm = *reinterpret_cast<Smem*>(tc_smem_raw + ((1024u - (raw & 1023u)) & 1023u));
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int r = t & (kTcRows - 1);   // this thread's row (Gaussian) of the tile = tensor-memory lane
    const int half = t >> 7;           // which half of the hidden units: [half HH, half HH + HH)
    // W1 (split, K-major, columns in X's order: the view direction, then the latents), W2, biases;
    // the transposed weight-gradient operand starts at zero (rows past HID in either half are
    // never written)
    for (int e = t; e < HID * K; e += kTcBwdThreads) {
        const int j = e / K, k = e % K;
        const int src = k < 3 ? a.L + k : k - 3;
        const float v = k < a.D ? a.W1[j * a.D + src] : 0.f;
        uint32_t h, l;
        split(v, h, l);
        const int o = tc_offset<2 * KS>(j, k);
        *reinterpret_cast<uint32_t*>(sm.w_hi + o) = h;
        *reinterpret_cast<uint32_t*>(sm.w_lo + o) = l;
        if constexpr (Smem::kW1f) sm.w1f[j * K + k] = v;
    }
    for (int e = t; e < int(sizeof(sm.g_hi) / 16); e += kTcBwdThreads) {
        reinterpret_cast<uint4*>(sm.g_hi)[e] = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint4*>(sm.g_lo)[e] = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int e = t; e < 3 * HID; e += kTcBwdThreads) sm.w2[e / HID][e % HID] = a.W2[e];
    for (int e = t; e < HID; e += kTcBwdThreads) sm.b1[e] = a.b1[e];
    if (t < 3) sm.b2[t] = a.b2[t];
    const uint32_t mbar_z = static_cast<uint32_t>(__cvta_generic_to_shared(&sm.mbar_z));
    const uint32_t mbar_g = static_cast<uint32_t>(__cvta_generic_to_shared(&sm.mbar_g));
    if (t == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(mbar_z) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(mbar_g) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    // tensor memory: Z1 [0, HID), G [HID, HID + NW), the second half's partial dL/dx
    // [HID + NW, HID + NW + 32)
    constexpr uint32_t kTmemCols = 256;
    constexpr uint32_t kDlCol = HID + NW;
    static_assert(kDlCol + 32 <= kTmemCols, "tensor memory");
    if (warp == 0) {
        const uint32_t slot = static_cast<uint32_t>(__cvta_generic_to_shared(&sm.tmem));
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(slot),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
    const uint32_t tmem = sm.tmem;
    const uint32_t trow = tmem + (uint32_t((warp & 3) * 32) << 16);  // this warp's 32 lanes
    const uint32_t x_hi = static_cast<uint32_t>(__cvta_generic_to_shared(sm.x_hi));
    const uint32_t x_lo = static_cast<uint32_t>(__cvta_generic_to_shared(sm.x_lo));
    const uint32_t w_hi = static_cast<uint32_t>(__cvta_generic_to_shared(sm.w_hi));
    const uint32_t w_lo = static_cast<uint32_t>(__cvta_generic_to_shared(sm.w_lo));
    const uint32_t g_hi = static_cast<uint32_t>(__cvta_generic_to_shared(sm.g_hi));
    const uint32_t g_lo = static_cast<uint32_t>(__cvta_generic_to_shared(sm.g_lo));
    const uint32_t r_hi = static_cast<uint32_t>(__cvta_generic_to_shared(sm.r_hi));
    const uint32_t r_lo = static_cast<uint32_t>(__cvta_generic_to_shared(sm.r_lo));
    constexpr uint32_t kSboX = 2 * KS * 128, kSboG = 32 * 128;
    constexpr uint32_t idesc_z = tc_idesc_tf32<HID>(), idesc_g = tc_idesc_tf32<NW>();
    const CameraF& cam = a.cam;
    const float C0 = -(cam.R[0] * cam.t[0] + cam.R[3] * cam.t[1] + cam.R[6] * cam.t[2]);
    const float C1 = -(cam.R[1] * cam.t[0] + cam.R[4] * cam.t[1] + cam.R[7] * cam.t[2]);
    const float C2 = -(cam.R[2] * cam.t[0] + cam.R[5] * cam.t[1] + cam.R[8] * cam.t[2]);
    const int tiles = (a.n + kTcRows - 1) / kTcRows;
    uint32_t phase_z = 0, phase_g = 0;
    bool failed = false, g_pending = false;
    float db2_acc[3] = {0.f, 0.f, 0.f};
    // the first half loads this row's latents and view direction; both load dL/dcolour
    float x[K - 3], d[3], dc[3];
    auto load_row = [&](int tile) {
        const int i = tile * kTcRows + r;
        const bool in = tile < tiles && i < a.n;
        if (half == 0) {
#pragma unroll
            for (int k = 0; k < K - 3; ++k) x[k] = in && k < a.L ? a.latents[size_t(k) * a.n + i] : 0.f;
            d[0] = in ? a.means[i] - C0 : 0.f;
            d[1] = in ? a.means[size_t(a.n) + i] - C1 : 0.f;
            d[2] = in ? a.means[2 * size_t(a.n) + i] - C2 : 0.f;
        }
#pragma unroll
        for (int c = 0; c < 3; ++c) dc[c] = in ? dcolors[size_t(c) * a.n + i] : 0.f;
    };
    load_row(blockIdx.x);
    int done = 0;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++done) {
        const int i = tile * kTcRows + r;
        const bool in = i < a.n;
        float xr[K];  // (first half) this row of X: the unit view direction, the latents, zeros
        if (half == 0) {
            const float len = sqrtf(d[0] * d[0] + d[1] * d[1] + d[2] * d[2]);
            const float il = len > 0.f ? 1.0f / len : 0.f;
#pragma unroll
            for (int k = 0; k < K; ++k) xr[k] = k < 3 ? d[k] * il : x[k - 3];
#pragma unroll
            for (int k = 0; k < K; k += 4) {
                uint32_t h[4], l[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) split_trunc(xr[k + q], h[q], l[q]);
                const int o = tc_offset<2 * KS>(r, k);
                *reinterpret_cast<uint4*>(sm.x_hi + o) = make_uint4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<uint4*>(sm.x_lo + o) = make_uint4(l[0], l[1], l[2], l[3]);
            }
        }
        const float g0 = dc[0], g1 = dc[1], g2 = dc[2];
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
        __syncthreads();
        asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
        if (t == kTcRows) {  // a thread of the second half, which stages no X
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const uint32_t off = uint32_t(ks) * 256u;
                const uint64_t ah = tc_desc(x_hi + off, 128, kSboX), al = tc_desc(x_lo + off, 128, kSboX);
                const uint64_t bh = tc_desc(w_hi + off, 128, kSboX), bl = tc_desc(w_lo + off, 128, kSboX);
                tc_mma_tf32(tmem, ah, bh, idesc_z, ks > 0);
                tc_mma_tf32(tmem, ah, bl, idesc_z, true);
                tc_mma_tf32(tmem, al, bh, idesc_z, true);
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(mbar_z)
                         : "memory");
        }
        load_row(tile + int(gridDim.x));
        bool ok = mbar_wait(mbar_z, phase_z);
        phase_z ^= 1u;
        // the previous tile's weight-gradient product has read its operands before they are
        // rewritten below
        if (g_pending) {
            ok = mbar_wait(mbar_g, phase_g) && ok;
            phase_g ^= 1u;
            g_pending = false;
        }
        ok = __syncthreads_and(ok);
        asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
        if (!ok) {
            atomicOr(&g_tc_error, 1u);
            failed = true;
            break;
        }
        // this half's share of the second layer from its columns of Z1, exchanged with the other
        // half's through shared memory
        float z2[3] = {0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < HH / 16; ++c) {
            float z[16];
            tc_ld_rows<16>(trow + uint32_t(half * HH + 16 * c), z);
#pragma unroll
            for (int q = 0; q < 16; q += 4) {
                const int u = half * HH + 16 * c + q;
                const float4 bb = *reinterpret_cast<const float4*>(&sm.b1[u]);
                const float4 u0 = *reinterpret_cast<const float4*>(&sm.w2[0][u]);
                const float4 u1 = *reinterpret_cast<const float4*>(&sm.w2[1][u]);
                const float4 u2 = *reinterpret_cast<const float4*>(&sm.w2[2][u]);
                const float h0 = fmaxf(z[q] + bb.x, 0.f), h1 = fmaxf(z[q + 1] + bb.y, 0.f);
                const float h2 = fmaxf(z[q + 2] + bb.z, 0.f), h3 = fmaxf(z[q + 3] + bb.w, 0.f);
                z2[0] = fmaf(u0.x, h0, fmaf(u0.y, h1, fmaf(u0.z, h2, fmaf(u0.w, h3, z2[0]))));
                z2[1] = fmaf(u1.x, h0, fmaf(u1.y, h1, fmaf(u1.z, h2, fmaf(u1.w, h3, z2[1]))));
                z2[2] = fmaf(u2.x, h0, fmaf(u2.y, h1, fmaf(u2.z, h2, fmaf(u2.w, h3, z2[2]))));
            }
        }
        // the exchange goes through the X operand's buffer: the product that read it is done,
        // and the next tile's X is written only after the barrier before the next product
        float* const zx = reinterpret_cast<float*>(sm.x_hi);
        static_assert(sizeof(sm.x_hi) >= 2 * kTcRows * 3 * sizeof(float), "exchange space");
        zx[(half * kTcRows + r) * 3 + 0] = z2[0];
        zx[(half * kTcRows + r) * 3 + 1] = z2[1];
        zx[(half * kTcRows + r) * 3 + 2] = z2[2];
        __syncthreads();
        float dz2[3];
        const float gc[3] = {g0, g1, g2};
#pragma unroll
        for (int c = 0; c < 3; ++c) {
            const float zz = zx[r * 3 + c] + zx[(kTcRows + r) * 3 + c] + sm.b2[c];
            const float sg = sigmoidf(zz);
            dz2[c] = gc[c] * sg * (1.f - sg);
            if (half == 0) db2_acc[c] += dz2[c];
        }
        // this half's hidden units, eight at a time: h, dz1 = (W2^T dz2) where z1 > 0, their
        // columns of the transposed operand, and its share of dL/dx = W1^T dz1 (latent columns)
        float dl[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) dl[k] = 0.f;
        const int kd = (a.D + 3) & ~3;  // the inputs' columns, rounded up to groups of four
        uint32_t zc[8], zn[8];
        tc_ld8_async(trow + uint32_t(half * HH), zc);
        tc_ld_wait(zc);
#pragma unroll 1
        for (int gq = 0; gq < HH / 8; ++gq) {
            const int grp = half * (HH / 8) + gq;
            if (gq + 1 < HH / 8) tc_ld8_async(trow + uint32_t(8 * (grp + 1)), zn);
            float vd[8], vh[8];
#pragma unroll
            for (int q = 0; q < 8; q += 4) {
                const int u = 8 * grp + q;
                const float4 bb = *reinterpret_cast<const float4*>(&sm.b1[u]);
                const float4 u0 = *reinterpret_cast<const float4*>(&sm.w2[0][u]);
                const float4 u1 = *reinterpret_cast<const float4*>(&sm.w2[1][u]);
                const float4 u2 = *reinterpret_cast<const float4*>(&sm.w2[2][u]);
                const float b4[4] = {bb.x, bb.y, bb.z, bb.w};
                const float a0[4] = {u0.x, u0.y, u0.z, u0.w}, a1[4] = {u1.x, u1.y, u1.z, u1.w};
                const float a2[4] = {u2.x, u2.y, u2.z, u2.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float zz = __uint_as_float(zc[q + e]) + b4[e];
                    const float tt = fmaf(a0[e], dz2[0], fmaf(a1[e], dz2[1], a2[e] * dz2[2]));
                    vd[q + e] = zz > 0.f ? tt : 0.f;
                    vh[q + e] = fmaxf(zz, 0.f);
                }
            }
            // column groups of four past the inputs hold zero weights: skipped (uniform branch)
#pragma unroll
            for (int k = 0; k < K; k += 4) {
                if (k >= kd) break;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int u = 8 * grp + q;
                    float w4[4];
                    if constexpr (Smem::kW1f) {
                        const float4 f = *reinterpret_cast<const float4*>(&sm.w1f[u * K + k]);
                        w4[0] = f.x; w4[1] = f.y; w4[2] = f.z; w4[3] = f.w;
                    } else {
                        const int o = tc_offset<2 * KS>(u, k);
                        const uint4 wh = *reinterpret_cast<const uint4*>(sm.w_hi + o);
                        const uint4 wl = *reinterpret_cast<const uint4*>(sm.w_lo + o);
                        w4[0] = __uint_as_float(wh.x) + __uint_as_float(wl.x);
                        w4[1] = __uint_as_float(wh.y) + __uint_as_float(wl.y);
                        w4[2] = __uint_as_float(wh.z) + __uint_as_float(wl.z);
                        w4[3] = __uint_as_float(wh.w) + __uint_as_float(wl.w);
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (k + e >= 3) dl[k + e - 3] = fmaf(vd[q], w4[e], dl[k + e - 3]);
                }
            }
            store_col8_t(sm.g_hi, sm.g_lo, grp, r, vd, lane);
            store_col8_t(sm.g_hi, sm.g_lo, 8 + grp, r, vh, lane);
            if (gq + 1 < HH / 8) {
                tc_ld_wait(zn);
#pragma unroll
                for (int q = 0; q < 8; ++q) zc[q] = zn[q];
            }
        }
        // the transposed [X | dZ2 | 1]^T: the first half writes X's columns, the second dz2,
        // ones (zero past the tile's Gaussians) and zeros; the second half also hands its share
        // of dL/dx to the first through tensor memory
        if (half == 0) {
#pragma unroll
            for (int gq = 0; gq < K / 8; ++gq) {
                float v[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) v[q] = xr[8 * gq + q];
                store_col8_t(sm.r_hi, sm.r_lo, gq, r, v, lane);
            }
        } else {
#pragma unroll
            for (int gq = K / 8; gq < NW / 8; ++gq) {
                float v[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int c = 8 * gq + q;
                    v[q] = c < K + 3 ? dz2[c - K] : (c == kOnes && in) ? 1.f : 0.f;
                }
                store_col8_t(sm.r_hi, sm.r_lo, gq, r, v, lane);
            }
            tc_st32(trow + kDlCol, dl);
        }
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
        __syncthreads();
        asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
        // issued (48 instructions) by a thread of the second half, which has nothing left to do in
        // this tile, not by a thread of the first, which still writes dL/dlatent and then stages
        // the next X
        if (t == kTcRows) {
#pragma unroll
            for (int ks = 0; ks < kTcRows / 8; ++ks) {
                const uint32_t off = uint32_t(ks) * 256u;
                const uint64_t ah = tc_desc(g_hi + off, 128, kSboG), al = tc_desc(g_lo + off, 128, kSboG);
                const uint64_t bh = tc_desc(r_hi + off, 128, kSboG), bl = tc_desc(r_lo + off, 128, kSboG);
                tc_mma_tf32(tmem + uint32_t(HID), ah, bh, idesc_g, done > 0 || ks > 0);
                tc_mma_tf32(tmem + uint32_t(HID), ah, bl, idesc_g, true);
                tc_mma_tf32(tmem + uint32_t(HID), al, bh, idesc_g, true);
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(mbar_g)
                         : "memory");
        }
        g_pending = true;
        if (half == 0) {
            float o[32];
            tc_ld_rows<32>(trow + kDlCol, o);
            if (in) {
#pragma unroll
                for (int k = 0; k < K - 3; ++k)
                    if (k < a.L) dlatents[size_t(k) * a.n + i] = dl[k] + o[k];
            }
        }
    }
    // the accumulated weight gradients, once the last product is done
    bool have = done > 0 && !failed;
    if (g_pending) {
        const bool ok = __syncthreads_and(mbar_wait(mbar_g, phase_g));
        phase_g ^= 1u;
        if (!ok) {
            atomicOr(&g_tc_error, 1u);
            failed = true;
            have = false;
        }
    }
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
    if (have && half == 0) {
        // thread r holds row r of G: r < 64 is hidden unit r of dZ1^T (dW1 row r, db1 from the
        // ones column), r >= 64 hidden unit r - 64 of H^T (dW2 column r - 64 from the dz2 columns)
        float gr[NW];
#pragma unroll
        for (int c = 0; c < NW; c += 16) {
            float tv[16];
            tc_ld_rows<16>(trow + uint32_t(HID + c), tv);
#pragma unroll
            for (int q = 0; q < 16; ++q) gr[c + q] = tv[q];
        }
        if (r < HID) {
#pragma unroll
            for (int k = 0; k < K; ++k) {
                if (k < a.D) {
                    const int src = k < 3 ? a.L + k : k - 3;
                    atomicAdd(dW1 + r * a.D + src, gr[k]);
                }
            }
            atomicAdd(db1 + r, gr[kOnes]);
        } else if (r >= 64 && r < 64 + HID) {
#pragma unroll
            for (int c = 0; c < 3; ++c) atomicAdd(dW2 + c * HID + (r - 64), gr[K + c]);
        }
    }
    // db2: the block's sum of dz2 (the first half's rows)
#pragma unroll
    for (int c = 0; c < 3; ++c) {
        float v = db2_acc[c];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
        if (lane == 0 && warp < 4) sm.db2[warp][c] = v;
    }
    // tensor memory goes back once no product is in flight and no warp reads it
    if (failed) {
        (void)mbar_wait(mbar_z, phase_z);
        (void)mbar_wait(mbar_g, phase_g);
    }
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
    if (t < 3 && done > 0 && !failed) atomicAdd(db2 + t, sm.db2[0][t] + sm.db2[1][t] + sm.db2[2][t] + sm.db2[3][t]);
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

__global__ void k_zero_mlp_grads(float* dW1, int nW1, float* db1, int nb1, float* dW2, int nW2, float* db2) {
    RS_PDL_ENTER();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nW1; i += gridDim.x * blockDim.x) dW1[i] = 0.f;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nb1; i += gridDim.x * blockDim.x) db1[i] = 0.f;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nW2; i += gridDim.x * blockDim.x) dW2[i] = 0.f;
    if (blockIdx.x == 0 && threadIdx.x < 3) db2[threadIdx.x] = 0.f;
}

// L1 loss and its gradient; the block sums of |d| go to *loss with one atomic per block.
__global__ void __launch_bounds__(256) k_l1(size_t count, const float* __restrict__ img,
                                            const float* __restrict__ tgt, float scale,
                                            float* __restrict__ dimg, float* __restrict__ loss) {
    RS_PDL_ENTER();
    __shared__ float s_w[8];
    float acc = 0.f;
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < count; i += size_t(gridDim.x) * blockDim.x) {
        const float d = img[i] - tgt[i];
        dimg[i] = d > 0.f ? scale : (d < 0.f ? -scale : 0.f);
        acc += fabsf(d);
    }
    if (!loss) return;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
    if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float b = 0.f;
        for (int w = 0; w < int(blockDim.x >> 5); ++w) b += s_w[w];
        atomicAdd(loss, b * scale);
    }
}

template <int HID, int KS>
cudaError_t launch_fwd_t(const MlpArgs& a, float* colors, cudaStream_t s) {
    const size_t smem = sizeof(TcFwdSmem<HID, KS>) + 1024;  // + room to align the base to 1 KB
    cudaError_t e = cudaFuncSetAttribute(k_mlp_fwd_tc<HID, KS>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    const int tiles = (a.n + kTcRows - 1) / kTcRows;
    // at most 512 / HID CTAs can hold tensor memory on an SM at once
    const int blocks = std::min(tiles, 152 * std::min(8, 512 / HID));
    pdl_launch(k_mlp_fwd_tc<HID, KS>, blocks, kTcRows, smem, s, a, colors);
    return cudaGetLastError();
}

template <int HID, int KS>
cudaError_t launch_bwd_t(const MlpArgs& a, const float* dcol, float* dlat, const rs_mlp_grads& gr, cudaStream_t s) {
    const size_t smem = sizeof(TcBwdSmem<HID, KS>) + 1024;  // + room to align the base to 1 KB
    static_assert(sizeof(TcBwdSmem<HID, KS>) + 1024 <= 232448, "shared memory per CTA");
    cudaError_t e = cudaFuncSetAttribute(k_mlp_bwd_tc<HID, KS>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    pdl_launch(k_zero_mlp_grads, 8, 256, 0, s, gr.d_dW1, HID * a.D, gr.d_db1, HID, gr.d_dW2, 3 * HID, gr.d_db2);
    if (a.n == 0) return cudaGetLastError();
    const int tiles = (a.n + kTcRows - 1) / kTcRows;
    // one CTA per SM (the shared memory of one), each holding 256 columns of tensor memory
    const int blocks = std::min(tiles, 152);
    pdl_launch(k_mlp_bwd_tc<HID, KS>, blocks, kTcBwdThreads, smem, s, a, dcol, dlat, gr.d_dW1, gr.d_db1, gr.d_dW2,
               gr.d_db2);
    return cudaGetLastError();
}

MlpArgs make_args(const CameraF& cam, int n, const float* means, const float* latents, const rs_mlp& m) {
    return MlpArgs{cam, n, m.latent_dim, m.latent_dim + 3, means, latents, m.d_W1, m.d_b1, m.d_W2, m.d_b2};
}

template <int HID>
cudaError_t fwd_ks(const MlpArgs& a, float* colors, cudaStream_t s) {
    switch ((a.D + 7) / 8) {
        case 1: return launch_fwd_t<HID, 1>(a, colors, s);
        case 2: return launch_fwd_t<HID, 2>(a, colors, s);
        case 3: return launch_fwd_t<HID, 3>(a, colors, s);
        default: return launch_fwd_t<HID, 4>(a, colors, s);
    }
}

template <int HID>
cudaError_t bwd_ks(const MlpArgs& a, const float* dcol, float* dlat, const rs_mlp_grads& gr, cudaStream_t s) {
    switch ((a.D + 7) / 8) {
        case 1: return launch_bwd_t<HID, 1>(a, dcol, dlat, gr, s);
        case 2: return launch_bwd_t<HID, 2>(a, dcol, dlat, gr, s);
        case 3: return launch_bwd_t<HID, 3>(a, dcol, dlat, gr, s);
        default: return launch_bwd_t<HID, 4>(a, dcol, dlat, gr, s);
    }
}

}  // namespace

cudaError_t launch_appearance_fwd(const CameraF& cam, int n, const float* means, const float* latents,
                                  const rs_mlp& m, float* colors, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const MlpArgs a = make_args(cam, n, means, latents, m);
    return m.hidden == 32 ? fwd_ks<32>(a, colors, s) : fwd_ks<64>(a, colors, s);
}

cudaError_t launch_appearance_bwd(const CameraF& cam, int n, const float* means, const float* latents,
                                  const rs_mlp& m, const float* dcolors, float* dlatents,
                                  const rs_mlp_grads& gr, cudaStream_t s) {
    const MlpArgs a = make_args(cam, n, means, latents, m);
    return m.hidden == 32 ? bwd_ks<32>(a, dcolors, dlatents, gr, s) : bwd_ks<64>(a, dcolors, dlatents, gr, s);
}

int take_device_error() {
    unsigned int v = 0u;
    if (cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(v)) != cudaSuccess) return -1;
    if (v == 0u) return 0;
    const unsigned int zero = 0u;
    if (cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(zero)) != cudaSuccess) return -1;
    return 1;
}

cudaError_t launch_l1(size_t count, const float* img, const float* tgt, float scale, float* dimg,
                      float* loss, cudaStream_t s) {
    if (loss) {
        cudaError_t e = cudaMemsetAsync(loss, 0, sizeof(float), s);
        if (e != cudaSuccess) return e;
    }
    if (count == 0) return cudaSuccess;
    const unsigned blocks = unsigned(std::min<size_t>((count + 255) / 256, 152 * 8));
    pdl_launch(k_l1, blocks, 256, 0, s, count, img, tgt, scale, dimg, loss);
    return cudaGetLastError();
}


// ---------------------------------------------------------------- L1 + D-SSIM loss
// 3DGS's photometric loss, which rigel trains with ("L1 + D-SSIM"):
//   L = (1 - lambda) mean|I - T| + lambda (1 - mean SSIM(I, T)),
// SSIM per channel and pixel with an 11x11 Gaussian window (sigma 1.5, the separable weights
// normalised over the window, zeros outside the image), C1 = 0.01^2, C2 = 0.03^2:
//   S = (2 mx my + C1)(2 sxy + C2) / ((mx^2 + my^2 + C1)(sx^2 + sy^2 + C2)),
// with mx = G*I, sx^2 = G*I^2 - mx^2, sxy = G*(I T) - mx my.  Its gradient w.r.t. I is the window's
// adjoint (the same symmetric window) applied to dS/dmx, dS/d(G*I^2), dS/d(G*IT):
//   dS_sum/dI_q = (G*a)_q + 2 I_q (G*b)_q + T_q (G*c)_q,
//   a = S (2my/A1 - 2my/A2 - 2mx/B1 + 2mx/B2), b = -S/B2, c = 2S/A2,
// A1 = 2 mx my + C1, A2 = 2 sxy + C2, B1 = mx^2 + my^2 + C1, B2 = sx^2 + sy^2 + C2.
// Two kernels over 32x32 output tiles, each staging its 42x42 input patch (5-pixel halo, zeros
// outside the image) in shared memory and filtering it separably: the first forms the five
// filtered maps, S, a, b, c and the block's sums of S and |I - T|; the second filters a, b, c
// and writes the gradient.  In both passes a thread computes four neighbouring outputs from one
// run of 14 staged inputs (the horizontal pass along a row, the vertical pass down a column),
// so every staged value is loaded once per four outputs instead of once per output.  The
// blocks' sums land in per-block slots, summed in a fixed order by a third kernel.
namespace {

constexpr int kSsimTile = 32;                   // output tile edge
constexpr int kSsimR = 5;                       // window radius
constexpr int kSsimTaps = 2 * kSsimR + 1;
constexpr int kSsimP = kSsimTile + 2 * kSsimR;  // staged patch rows: 42
constexpr int kSsimLead = 3;                    // extra staged columns left of the window's reach
constexpr int kSsimPS = 48;                     // staged columns (x0 - 3 .. x0 + 44): 16-byte groups
constexpr int kSsimThreads = 256;
constexpr int kSsimOut = 4;                     // outputs per thread and pass
constexpr int kSsimGroups = kSsimTile / kSsimOut;  // column groups of a patch row: 8

struct SsimWindow {
    float w[kSsimTaps];  // normalised 1-D Gaussian, sigma 1.5
};

// Stages the plane's rows y0 .. y0 + 41, columns xs .. xs + 47 (xs = x0 - 3, a multiple of 4;
// zeros outside the H x W image) into dst[kSsimP][kSsimPS] with asynchronous copies (cp.async,
// PTX ISA: bytes past the source size are filled with zeros), all in flight together; the
// caller waits with ssim_stage_wait.  VEC: 16-byte copies of four columns (needs W and the
// plane's address to be multiples of 4 floats and 16 bytes); otherwise 4-byte copies.
template <bool VEC>
__device__ __forceinline__ void ssim_stage(const float* __restrict__ plane, int H, int W, int y0, int xs,
                                           float* dst) {
    const unsigned base = static_cast<unsigned>(__cvta_generic_to_shared(dst));
    if (VEC) {
        constexpr int kG = kSsimPS / 4;  // 12 groups per row
        for (int e = threadIdx.x; e < kSsimP * kG; e += kSsimThreads) {
            const int r = e / kG, x = xs + 4 * (e - r * kG), y = y0 + r;
            // a group starts at a multiple of 4, so it is wholly left of column 0 or not at all
            const int n = (y >= 0 && y < H && x >= 0 && x < W) ? 4 * min(4, W - x) : 0;
            const float* src = n ? plane + size_t(y) * W + x : plane;
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(base + 16u * unsigned(e)), "l"(src),
                         "r"(n) : "memory");
        }
    } else {
        for (int e = threadIdx.x; e < kSsimP * kSsimPS; e += kSsimThreads) {
            const int r = e / kSsimPS, x = xs + (e - r * kSsimPS), y = y0 + r;
            const bool in = y >= 0 && y < H && x >= 0 && x < W;
            const float* src = in ? plane + size_t(y) * W + x : plane;
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(base + 4u * unsigned(e)), "l"(src),
                         "r"(in ? 4 : 0) : "memory");
        }
    }
}

__device__ __forceinline__ void ssim_stage_wait() {
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
}

// The staged values of patch row `row` that outputs 4 g .. 4 g + 3 of the horizontal pass read:
// v[3 + o + k] is tap k of output 4 g + o (five 16-byte loads; v[0..2] and v[17..19] unused).
__device__ __forceinline__ void ssim_row_run(const float* patch, int row, int g, float (&v)[20]) {
    const float4* q = reinterpret_cast<const float4*>(patch + row * kSsimPS + g * kSsimOut);
#pragma unroll
    for (int k = 0; k < 5; ++k) {
        const float4 t = q[k];
        v[4 * k] = t.x;
        v[4 * k + 1] = t.y;
        v[4 * k + 2] = t.z;
        v[4 * k + 3] = t.w;
    }
}

template <bool VEC>
__global__ void __launch_bounds__(kSsimThreads) k_ssim_fwd(SsimWindow win, int H, int W,
                                                           const float* __restrict__ img,
                                                           const float* __restrict__ tgt, size_t N,
                                                           float* __restrict__ abc, float2* __restrict__ partial) {
    RS_PDL_ENTER();
    __shared__ __align__(16) float s_x[kSsimP * kSsimPS], s_y[kSsimP * kSsimPS];
    __shared__ __align__(16) float s_h[5][kSsimP][kSsimTile];  // horizontally filtered x, y, xx, yy, xy
    __shared__ float s_red[2][kSsimThreads / 32];
    const int ch = blockIdx.z;
    const int x0 = blockIdx.x * kSsimTile - kSsimR, y0 = blockIdx.y * kSsimTile - kSsimR;
    const size_t plane = size_t(H) * W;
    ssim_stage<VEC>(img + ch * plane, H, W, y0, x0 - kSsimLead, s_x);
    ssim_stage<VEC>(tgt + ch * plane, H, W, y0, x0 - kSsimLead, s_y);
    ssim_stage_wait();
    // horizontal pass: task t = patch row t / 8, outputs 4 (t % 8) .. + 3 of that row
    for (int t = threadIdx.x; t < kSsimP * kSsimGroups; t += kSsimThreads) {
        const int row = t / kSsimGroups, g = t % kSsimGroups;
        float a[20], b[20];
        ssim_row_run(s_x, row, g, a);
        ssim_row_run(s_y, row, g, b);
        // the products once per staged value (14 of them), not once per tap and output
        constexpr int kRun = kSsimOut + 2 * kSsimR;
        float xx[kRun], yy[kRun], xy[kRun];
#pragma unroll
        for (int i = 0; i < kRun; ++i) {
            const float xa = a[kSsimLead + i], yb = b[kSsimLead + i];
            xx[i] = xa * xa;
            yy[i] = yb * yb;
            xy[i] = xa * yb;
        }
        float h[5][kSsimOut];
#pragma unroll
        for (int o = 0; o < kSsimOut; ++o) h[0][o] = h[1][o] = h[2][o] = h[3][o] = h[4][o] = 0.f;
#pragma unroll
        for (int k = 0; k < kSsimTaps; ++k) {
            const float w = win.w[k];
#pragma unroll
            for (int o = 0; o < kSsimOut; ++o) {
                h[0][o] = fmaf(w, a[kSsimLead + o + k], h[0][o]);
                h[1][o] = fmaf(w, b[kSsimLead + o + k], h[1][o]);
                h[2][o] = fmaf(w, xx[o + k], h[2][o]);
                h[3][o] = fmaf(w, yy[o + k], h[3][o]);
                h[4][o] = fmaf(w, xy[o + k], h[4][o]);
            }
        }
#pragma unroll
        for (int q = 0; q < 5; ++q)
            *reinterpret_cast<float4*>(&s_h[q][row][g * kSsimOut]) = make_float4(h[q][0], h[q][1], h[q][2], h[q][3]);
    }
    __syncthreads();
    // vertical pass: lane = output column, warp w = output rows 4 w .. 4 w + 3
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float v[5][kSsimOut];
#pragma unroll
    for (int q = 0; q < 5; ++q) {
        float col[kSsimOut + 2 * kSsimR];
#pragma unroll
        for (int i = 0; i < kSsimOut + 2 * kSsimR; ++i) col[i] = s_h[q][warp * kSsimOut + i][lane];
#pragma unroll
        for (int o = 0; o < kSsimOut; ++o) {
            float acc = 0.f;
#pragma unroll
            for (int k = 0; k < kSsimTaps; ++k) acc = fmaf(win.w[k], col[o + k], acc);
            v[q][o] = acc;
        }
    }
    constexpr float C1 = 0.01f * 0.01f, C2 = 0.03f * 0.03f;
    const int gx = x0 + kSsimR + lane;
    float ssim = 0.f, l1 = 0.f;
#pragma unroll
    for (int o = 0; o < kSsimOut; ++o) {
        const int ty = warp * kSsimOut + o, gy = y0 + kSsimR + ty;
        if (gy >= H || gx >= W) continue;
        const float mx = v[0][o], my = v[1][o];
        const float sxx = v[2][o] - mx * mx, syy = v[3][o] - my * my, sxy = v[4][o] - mx * my;
        const float A1 = 2.f * mx * my + C1, A2 = 2.f * sxy + C2;
        const float B1 = mx * mx + my * my + C1, B2 = sxx + syy + C2;
        // two reciprocals serve every quotient: 1/A1 = A2 rA, 1/A2 = A1 rA, 1/B1 = B2 rB, 1/B2 = B1 rB
        const float rA = __frcp_rn(A1 * A2), rB = __frcp_rn(B1 * B2);
        const float S = (A1 * A2) * rB;
        ssim += S;
        const int cc = (ty + kSsimR) * kSsimPS + kSsimLead + kSsimR + lane;  // the output's own pixel
        l1 += fabsf(s_x[cc] - s_y[cc]);
        const size_t at = ch * plane + size_t(gy) * W + gx;
        abc[at] = S * (2.f * my * (A2 - A1) * rA + 2.f * mx * (B1 - B2) * rB);
        abc[N + at] = -S * B1 * rB;
        abc[2 * N + at] = 2.f * S * A1 * rA;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ssim += __shfl_xor_sync(kFull, ssim, o);
        l1 += __shfl_xor_sync(kFull, l1, o);
    }
    if (lane == 0) {
        s_red[0][warp] = ssim;
        s_red[1][warp] = l1;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float sa = 0.f, sb = 0.f;
        for (int w = 0; w < kSsimThreads / 32; ++w) {
            sa += s_red[0][w];
            sb += s_red[1][w];
        }
        partial[(size_t(ch) * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x] = make_float2(sa, sb);
    }
}

// dL/dI = scale (1 - lambda) sign(I - T) / N - scale lambda / N (G*a + 2 I G*b + T G*c).
template <bool VEC>
__global__ void __launch_bounds__(kSsimThreads) k_ssim_bwd(SsimWindow win, int H, int W,
                                                           const float* __restrict__ img,
                                                           const float* __restrict__ tgt, size_t N,
                                                           const float* __restrict__ abc, float lambda, float scale,
                                                           float* __restrict__ dimg) {
    RS_PDL_ENTER();
    __shared__ __align__(16) float s_in[3][kSsimP * kSsimPS];
    __shared__ __align__(16) float s_h[3][kSsimP][kSsimTile];
    const int ch = blockIdx.z;
    const int x0 = blockIdx.x * kSsimTile - kSsimR, y0 = blockIdx.y * kSsimTile - kSsimR;
    const size_t plane = size_t(H) * W;
#pragma unroll
    for (int q = 0; q < 3; ++q) ssim_stage<VEC>(abc + q * N + ch * plane, H, W, y0, x0 - kSsimLead, s_in[q]);
    // the thread's own outputs' image and target values, loaded now to arrive during the filtering
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gx = x0 + kSsimR + lane;
    float px[kSsimOut], py[kSsimOut];
#pragma unroll
    for (int o = 0; o < kSsimOut; ++o) {
        const int gy = y0 + kSsimR + warp * kSsimOut + o;
        const bool in = gy < H && gx < W;
        const size_t at = ch * plane + size_t(in ? gy : 0) * W + (in ? gx : 0);
        px[o] = in ? img[at] : 0.f;
        py[o] = in ? tgt[at] : 0.f;
    }
    ssim_stage_wait();
    for (int t = threadIdx.x; t < kSsimP * kSsimGroups; t += kSsimThreads) {
        const int row = t / kSsimGroups, g = t % kSsimGroups;
#pragma unroll
        for (int q = 0; q < 3; ++q) {
            float a[20];
            ssim_row_run(s_in[q], row, g, a);
            float h[kSsimOut] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k = 0; k < kSsimTaps; ++k)
#pragma unroll
                for (int o = 0; o < kSsimOut; ++o) h[o] = fmaf(win.w[k], a[kSsimLead + o + k], h[o]);
            *reinterpret_cast<float4*>(&s_h[q][row][g * kSsimOut]) = make_float4(h[0], h[1], h[2], h[3]);
        }
    }
    __syncthreads();
    float gsum[3][kSsimOut];
#pragma unroll
    for (int q = 0; q < 3; ++q) {
        float col[kSsimOut + 2 * kSsimR];
#pragma unroll
        for (int i = 0; i < kSsimOut + 2 * kSsimR; ++i) col[i] = s_h[q][warp * kSsimOut + i][lane];
#pragma unroll
        for (int o = 0; o < kSsimOut; ++o) {
            float acc = 0.f;
#pragma unroll
            for (int k = 0; k < kSsimTaps; ++k) acc = fmaf(win.w[k], col[o + k], acc);
            gsum[q][o] = acc;
        }
    }
    const float inv = scale / float(N);
#pragma unroll
    for (int o = 0; o < kSsimOut; ++o) {
        const int gy = y0 + kSsimR + warp * kSsimOut + o;
        if (gy >= H || gx >= W) continue;
        const size_t at = ch * plane + size_t(gy) * W + gx;
        const float x = px[o], y = py[o];
        const float d = x - y;
        const float sgn = d > 0.f ? 1.f : (d < 0.f ? -1.f : 0.f);
        const float dS = fmaf(2.f * x, gsum[1][o], fmaf(y, gsum[2][o], gsum[0][o]));
        dimg[at] = inv * ((1.f - lambda) * sgn - lambda * dS);
    }
}

// loss = scale ((1 - lambda) sum|I - T| + lambda (N - sum S)) / N from the blocks' sums, added in
// a fixed order.
__global__ void __launch_bounds__(1024) k_ssim_loss(const float2* __restrict__ partial, uint32_t count, size_t N,
                                                    float lambda, float scale, float* loss) {
    RS_PDL_ENTER();
    __shared__ float s_a[32], s_b[32];
    float a = 0.f, b = 0.f;
    for (uint32_t i = threadIdx.x; i < count; i += blockDim.x) {
        const float2 p = partial[i];
        a += p.x;
        b += p.y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_xor_sync(kFull, a, o);
        b += __shfl_xor_sync(kFull, b, o);
    }
    if ((threadIdx.x & 31) == 0) {
        s_a[threadIdx.x >> 5] = a;
        s_b[threadIdx.x >> 5] = b;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float sa = 0.f, sb = 0.f;
        for (int w = 0; w < int(blockDim.x >> 5); ++w) {
            sa += s_a[w];
            sb += s_b[w];
        }
        *loss = scale * ((1.f - lambda) * sb + lambda * (float(N) - sa)) / float(N);
    }
}

size_t ssim_blocks(int C, int H, int W) {
    return size_t((W + kSsimTile - 1) / kSsimTile) * size_t((H + kSsimTile - 1) / kSsimTile) * size_t(C);
}

}  // namespace

size_t ssim_workspace_bytes(int C, int H, int W) {
    const size_t maps = 3 * size_t(C) * H * W * sizeof(float);
    return ((maps + 255) & ~size_t(255)) + ssim_blocks(C, H, W) * sizeof(float2) + 256;
}

cudaError_t launch_l1_dssim(int C, int H, int W, const float* img, const float* tgt, float lambda, float scale,
                            float* dimg, float* loss, void* ws, cudaStream_t s) {
    SsimWindow win;
    double t[kSsimTaps], sum = 0.0;
    for (int i = 0; i < kSsimTaps; ++i) {
        t[i] = std::exp(-double((i - kSsimR) * (i - kSsimR)) / (2.0 * 1.5 * 1.5));
        sum += t[i];
    }
    for (int i = 0; i < kSsimTaps; ++i) win.w[i] = float(t[i] / sum);
    const size_t N = size_t(C) * H * W;
    float* abc = static_cast<float*>(ws);
    float2* partial = reinterpret_cast<float2*>(static_cast<char*>(ws) + ((3 * N * sizeof(float) + 255) & ~size_t(255)));
    const dim3 grid{unsigned((W + kSsimTile - 1) / kSsimTile), unsigned((H + kSsimTile - 1) / kSsimTile), unsigned(C)};
    // 16-byte staging copies need every row of every plane to start on a 16-byte boundary
    const bool vec = W % 4 == 0 && ((reinterpret_cast<uintptr_t>(img) | reinterpret_cast<uintptr_t>(tgt)) & 15u) == 0;
    if (vec) {
        pdl_launch(k_ssim_fwd<true>, grid, kSsimThreads, 0, s, win, H, W, img, tgt, N, abc, partial);
        pdl_launch(k_ssim_bwd<true>, grid, kSsimThreads, 0, s, win, H, W, img, tgt, N, abc, lambda, scale, dimg);
    } else {
        pdl_launch(k_ssim_fwd<false>, grid, kSsimThreads, 0, s, win, H, W, img, tgt, N, abc, partial);
        pdl_launch(k_ssim_bwd<false>, grid, kSsimThreads, 0, s, win, H, W, img, tgt, N, abc, lambda, scale, dimg);
    }
    if (loss)
        pdl_launch(k_ssim_loss, 1, 1024, 0, s, partial, uint32_t(ssim_blocks(C, H, W)), N, lambda, scale, loss);
    return cudaGetLastError();
}

}  // namespace rs
