// Densification of the training loop: clone, split and prune (rigel README: "GaussianModel:
// activations, densify/prune", the training log's per-step clone / split / prune counts, and the
// rule that densification and pruning leave every parameter and its Adam moments the same
// length).  The pages name the three operations but not their criteria; the ones used are those
// of 3D Gaussian Splatting's adaptive density control:
//   - a Gaussian whose mean view-space gradient norm (accumulated by rs_densify_stats) reaches
//     the threshold is cloned when its largest scale is at most `dense_scale`, else split into
//     two children placed at mean + R(q) (s * z) (z standard normal, given) with scales s / 1.6;
//   - every resulting Gaussian whose opacity is below `min_opacity`, or whose largest scale
//     exceeds `max_scale` (if positive), is removed (a clone or split child inherits the test of
//     the values it carries).
// Output order: surviving originals in index order, then the clones in the order of their
// sources, then the first children of the split Gaussians in index order, then their second
// children.  New Gaussians start with zero Adam moments.
//
// rs_densify_plan classifies every Gaussian (one pass over accum, count, log-scales and opacity
// logits), scans the three counts (survivors, clones, splits) over 256-Gaussian blocks and reads
// the totals back: the caller needs the output size to allocate.  rs_densify_apply then moves
// every parameter group in one launch: a block recomputes its Gaussians' ranks from the actions
// with warp ballots, adds its block offsets and writes each output row with the lanes' ranks.
#include <cmath>

#include "rs_internal.cuh"

namespace {

enum Action : uint8_t { kRemove = 0, kKeep = 1, kClone = 2, kSplit = 3 };

constexpr int kBlock = 256;    // Gaussians per classification / apply block
constexpr int kWarps = kBlock / 32;
constexpr float kLn1_6 = 0.47000362924573558f;  // ln 1.6: split children's scales are s / 1.6

struct Rule {
    float grad_threshold;
    float ln_dense;      // ln(dense_scale)
    float logit_min;     // logit(min_opacity): opacity < min_opacity <=> logit < logit_min
    float ln_max;        // ln(max_scale), +inf when the size test is off
};

// Workspace: actions [n] u8 (padded to 256 B), per block {survivors, clones, splits} u32 x 3,
// per block offsets u32 x 3, totals u32 x 4.
struct Plan {
    size_t off_action, off_count, off_offset, off_total, bytes;
    uint32_t blocks;
};
Plan plan_of(int32_t n) {
    Plan p{};
    p.blocks = uint32_t((int64_t(n) + kBlock - 1) / kBlock);
    p.off_action = 0;
    p.off_count = (size_t(n) + 255) & ~size_t(255);
    p.off_offset = p.off_count + ((size_t(p.blocks) * 12 + 255) & ~size_t(255));
    p.off_total = p.off_offset + ((size_t(p.blocks) * 12 + 255) & ~size_t(255));
    p.bytes = p.off_total + 256;
    return p;
}

__global__ void __launch_bounds__(kBlock) k_densify_classify(int n, const float* __restrict__ accum,
                                                              const float* __restrict__ count,
                                                              const float* __restrict__ log_scales,
                                                              const float* __restrict__ logits, Rule rule,
                                                              uint8_t* __restrict__ action, uint32_t* __restrict__ counts) {
    RS_PDL_ENTER();
    __shared__ uint32_t s_n[3][kWarps];
    const int i = blockIdx.x * kBlock + threadIdx.x;
    uint8_t a = kRemove;
    if (i < n) {
        const size_t N = size_t(n);
        const float ls = fmaxf(fmaxf(log_scales[i], log_scales[N + i]), log_scales[2 * N + i]);
        const float c = count[i];
        const bool grow = c > 0.f && accum[i] >= rule.grad_threshold * c;
        const bool dense = ls <= rule.ln_dense;
        const bool faint = logits[i] < rule.logit_min;
        if (grow && !dense) {
            // the children carry s / 1.6 and the parent's opacity
            a = (faint || ls - kLn1_6 > rule.ln_max) ? kRemove : kSplit;
        } else {
            a = (faint || ls > rule.ln_max) ? kRemove : grow ? kClone : kKeep;
        }
        action[i] = a;
    }
    const unsigned lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t b_surv = __ballot_sync(0xffffffffu, a == kKeep || a == kClone);
    const uint32_t b_clone = __ballot_sync(0xffffffffu, a == kClone);
    const uint32_t b_split = __ballot_sync(0xffffffffu, a == kSplit);
    if (lane == 0) {
        s_n[0][warp] = __popc(b_surv);
        s_n[1][warp] = __popc(b_clone);
        s_n[2][warp] = __popc(b_split);
    }
    __syncthreads();
    if (threadIdx.x < 3 * 32) {
        const int k = threadIdx.x >> 5;
        uint32_t v = lane < unsigned(kWarps) ? s_n[k][lane] : 0u;
        v = __reduce_add_sync(0xffffffffu, v);
        if (lane == 0) counts[3 * size_t(blockIdx.x) + k] = v;
    }
}

// Exclusive scan of the per-block counts (one block of 1024 threads, any number of blocks),
// and the totals {survivors, clones, splits, n_out}.
__global__ void __launch_bounds__(1024) k_densify_scan(uint32_t blocks, const uint32_t* __restrict__ counts,
                                                       uint32_t* __restrict__ offsets, uint32_t* __restrict__ totals) {
    RS_PDL_ENTER();
    __shared__ uint32_t s_w[3][32];
    __shared__ uint32_t s_carry[3];
    if (threadIdx.x < 3) s_carry[threadIdx.x] = 0;
    __syncthreads();
    const unsigned lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (uint32_t base = 0; base < blocks; base += 1024) {
        const uint32_t b = base + threadIdx.x;
        uint32_t v[3];
#pragma unroll
        for (int k = 0; k < 3; ++k) v[k] = b < blocks ? counts[3 * size_t(b) + k] : 0u;
        uint32_t incl[3];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            uint32_t x = v[k];
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, x, d);
                if (lane >= unsigned(d)) x += y;
            }
            incl[k] = x;
            if (lane == 31) s_w[k][warp] = x;
        }
        __syncthreads();
        if (warp == 0) {
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                uint32_t x = s_w[k][lane];
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, x, d);
                    if (lane >= unsigned(d)) x += y;
                }
                s_w[k][lane] = x;  // inclusive over warps
            }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const uint32_t before = s_carry[k] + (warp ? s_w[k][warp - 1] : 0u) + incl[k] - v[k];
            if (b < blocks) offsets[3 * size_t(b) + k] = before;
        }
        __syncthreads();
        if (threadIdx.x < 3) s_carry[threadIdx.x] += s_w[threadIdx.x][31];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        totals[0] = s_carry[0];
        totals[1] = s_carry[1];
        totals[2] = s_carry[2];
        totals[3] = s_carry[0] + s_carry[1] + 2u * s_carry[2];
    }
}

struct GroupTable {
    rs_densify_group g[RS_DENSIFY_MAX_GROUPS];
    int n_groups;
};

// R(q) (s * z) for the unit quaternion of q = (w, x, y, z) and s = exp(log-scales).
__device__ __forceinline__ float3 split_offset(const float* quats, const float* log_scales, const float* noise,
                                               size_t N, size_t i, int child) {
    float w = quats[i], x = quats[N + i], y = quats[2 * N + i], z = quats[3 * N + i];
    const float inv = rsqrtf(w * w + x * x + y * y + z * z);
    w *= inv; x *= inv; y *= inv; z *= inv;
    const float* zc = noise + size_t(child) * 3 * N;
    const float a = expf(log_scales[i]) * zc[i];
    const float b = expf(log_scales[N + i]) * zc[N + i];
    const float c = expf(log_scales[2 * N + i]) * zc[2 * N + i];
    // rows of the rotation matrix of a unit quaternion (w, x, y, z)
    float3 o;
    o.x = (1.f - 2.f * (y * y + z * z)) * a + 2.f * (x * y - w * z) * b + 2.f * (x * z + w * y) * c;
    o.y = 2.f * (x * y + w * z) * a + (1.f - 2.f * (x * x + z * z)) * b + 2.f * (y * z - w * x) * c;
    o.z = 2.f * (x * z - w * y) * a + 2.f * (y * z + w * x) * b + (1.f - 2.f * (x * x + y * y)) * c;
    return o;
}

__global__ void __launch_bounds__(kBlock) k_densify_apply(int n, const uint8_t* __restrict__ action,
                                                           const uint32_t* __restrict__ offsets,
                                                           const uint32_t* __restrict__ totals,
                                                           const float* __restrict__ quats,
                                                           const float* __restrict__ log_scales,
                                                           const float* __restrict__ noise, GroupTable T,
                                                           uint32_t n_out) {
    RS_PDL_ENTER();
    __shared__ uint32_t s_w[3][kWarps];
    const int i = blockIdx.x * kBlock + threadIdx.x;
    const uint8_t a = i < n ? action[i] : kRemove;
    const unsigned lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned below = (1u << lane) - 1u;
    const uint32_t b_surv = __ballot_sync(0xffffffffu, a == kKeep || a == kClone);
    const uint32_t b_clone = __ballot_sync(0xffffffffu, a == kClone);
    const uint32_t b_split = __ballot_sync(0xffffffffu, a == kSplit);
    if (lane == 0) {
        s_w[0][warp] = __popc(b_surv);
        s_w[1][warp] = __popc(b_clone);
        s_w[2][warp] = __popc(b_split);
    }
    __syncthreads();
    if (threadIdx.x < 3 * 32) {  // exclusive scan of the warps' counts, per stream
        const int k = threadIdx.x >> 5;
        const uint32_t v = lane < unsigned(kWarps) ? s_w[k][lane] : 0u;
        uint32_t x = v;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, d);
            if (lane >= unsigned(d)) x += y;
        }
        __syncwarp();
        if (lane < unsigned(kWarps)) s_w[k][lane] = x - v;
    }
    __syncthreads();
    if (i >= n || a == kRemove) return;
    const uint32_t* off = offsets + 3 * size_t(blockIdx.x);
    const uint32_t n_surv = totals[0], n_clone = totals[1], n_split = totals[2];
    const size_t N = size_t(n), NO = size_t(n_out);
    // output positions: the original or first child, and the clone or second child
    uint32_t dst0, dst1 = 0;
    int outs;
    if (a == kSplit) {
        const uint32_t r = off[2] + s_w[2][warp] + __popc(b_split & below);
        dst0 = n_surv + n_clone + r;
        dst1 = n_surv + n_clone + n_split + r;
        outs = 2;
    } else {
        dst0 = off[0] + s_w[0][warp] + __popc(b_surv & below);
        if (a == kClone) dst1 = n_surv + off[1] + s_w[1][warp] + __popc(b_clone & below);
        outs = a == kClone ? 2 : 1;
    }
    float3 d0{0.f, 0.f, 0.f}, d1{0.f, 0.f, 0.f};
    if (a == kSplit) {
        d0 = split_offset(quats, log_scales, noise, N, size_t(i), 0);
        d1 = split_offset(quats, log_scales, noise, N, size_t(i), 1);
    }
    for (int gi = 0; gi < T.n_groups; ++gi) {
        const rs_densify_group& G = T.g[gi];
        const float* __restrict__ gp = G.d_param;
        const float* __restrict__ gm = G.d_m;
        const float* __restrict__ gv = G.d_v;
        // four rows' loads in flight before their stores (the outputs never alias the inputs)
        for (int r0 = 0; r0 < G.rows; r0 += 4) {
            float p[4], m[4], v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int r = r0 + q;
                const bool ok = r < G.rows;
                p[q] = ok ? gp[size_t(r) * N + i] : 0.f;
                m[q] = ok && gm ? gm[size_t(r) * N + i] : 0.f;
                v[q] = ok && gv ? gv[size_t(r) * N + i] : 0.f;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int r = r0 + q;
                if (r >= G.rows) break;
                for (int o = 0; o < outs; ++o) {
                    const uint32_t d = o == 0 ? dst0 : dst1;
                    if (d >= n_out) continue;  // an n_out below the plan's count: nothing past it
                    const size_t at = size_t(r) * NO + d;
                    float val = p[q];
                    bool fresh = o == 1;  // a clone or a child: new moments
                    if (a == kSplit) {
                        fresh = true;
                        if (G.kind == RS_DENSIFY_MEANS) {
                            const float3 dd = o == 0 ? d0 : d1;
                            val += r == 0 ? dd.x : r == 1 ? dd.y : dd.z;
                        } else if (G.kind == RS_DENSIFY_LOG_SCALES) {
                            val -= kLn1_6;
                        }
                    }
                    G.d_param_out[at] = val;
                    if (G.d_m_out) G.d_m_out[at] = fresh ? 0.f : m[q];
                    if (G.d_v_out) G.d_v_out[at] = fresh ? 0.f : v[q];
                }
            }
        }
    }
}

bool aligned4(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" {

size_t rs_densify_workspace_size(int32_t n) {
    if (n < 0 || n > RS_MAX_GAUSSIANS) return 0;
    return plan_of(n).bytes;
}

int rs_densify_plan(int32_t n, const float* d_accum, const float* d_count, const float* d_log_scales,
                    const float* d_opacity_logits, const rs_densify_rule* rule, void* d_workspace,
                    size_t workspace_bytes, uint8_t* d_action, int32_t* counts, void* stream) {
    if (n < 0 || n > RS_MAX_GAUSSIANS || !rule || !counts) return RS_ERR_INVALID_ARG;
    if (!(rule->dense_scale > 0.f) || !(rule->min_opacity >= 0.f && rule->min_opacity < 1.f) ||
        !(rule->grad_threshold >= 0.f) || !isfinite(rule->grad_threshold))
        return RS_ERR_INVALID_ARG;
    if (!d_workspace || (reinterpret_cast<uintptr_t>(d_workspace) & 255u)) return RS_ERR_INVALID_ARG;
    if (n > 0 && (!aligned4(d_accum) || !aligned4(d_count) || !aligned4(d_log_scales) || !aligned4(d_opacity_logits)))
        return RS_ERR_INVALID_ARG;
    const Plan p = plan_of(n);
    if (workspace_bytes < p.bytes) return RS_ERR_WORKSPACE;
    for (int k = 0; k < 5; ++k) counts[k] = 0;
    if (n == 0) return RS_OK;
    Rule R;
    R.grad_threshold = rule->grad_threshold;
    R.ln_dense = float(std::log(double(rule->dense_scale)));
    const double mo = double(rule->min_opacity);
    R.logit_min = mo > 0.0 ? float(std::log(mo / (1.0 - mo))) : -INFINITY;
    R.ln_max = rule->max_scale > 0.f ? float(std::log(double(rule->max_scale))) : INFINITY;
    uint8_t* ws = static_cast<uint8_t*>(d_workspace);
    uint8_t* action = ws + p.off_action;
    uint32_t* cnt = reinterpret_cast<uint32_t*>(ws + p.off_count);
    uint32_t* offs = reinterpret_cast<uint32_t*>(ws + p.off_offset);
    uint32_t* tot = reinterpret_cast<uint32_t*>(ws + p.off_total);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    rs::pdl_launch(k_densify_classify, p.blocks, kBlock, 0, s, n, d_accum, d_count, d_log_scales, d_opacity_logits,
                   R, action, cnt);
    rs::pdl_launch(k_densify_scan, 1, 1024, 0, s, p.blocks, static_cast<const uint32_t*>(cnt), offs, tot);
    if (cudaGetLastError() != cudaSuccess) return RS_ERR_CUDA;
    if (d_action && cudaMemcpyAsync(d_action, action, size_t(n), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return RS_ERR_CUDA;
    uint32_t h[4];
    if (cudaMemcpyAsync(h, tot, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return RS_ERR_CUDA;
    counts[0] = int32_t(h[3]);                            // Gaussians after the step
    counts[1] = int32_t(h[0]);                            // originals kept (cloned ones included)
    counts[2] = int32_t(h[1]);                            // clones
    counts[3] = int32_t(h[2]);                            // Gaussians split (two children each)
    counts[4] = n - int32_t(h[0]) - int32_t(h[2]);        // removed outright
    if (int64_t(h[3]) > int64_t(RS_MAX_GAUSSIANS)) return RS_ERR_CAPACITY;
    return RS_OK;
}

int rs_densify_apply(int32_t n, const void* d_workspace, size_t workspace_bytes, const float* d_quats,
                     const float* d_log_scales, const float* d_noise, const rs_densify_group* groups,
                     int32_t n_groups, int32_t n_out, void* stream) {
    if (n < 0 || n > RS_MAX_GAUSSIANS || n_out < 0 || n_out > RS_MAX_GAUSSIANS) return RS_ERR_INVALID_ARG;
    if (n_groups < 0 || n_groups > RS_DENSIFY_MAX_GROUPS || (n_groups > 0 && !groups)) return RS_ERR_INVALID_ARG;
    if (!d_workspace || (reinterpret_cast<uintptr_t>(d_workspace) & 255u)) return RS_ERR_INVALID_ARG;
    const Plan p = plan_of(n);
    if (workspace_bytes < p.bytes) return RS_ERR_WORKSPACE;
    if (n == 0) return RS_OK;
    if (!aligned4(d_quats) || !aligned4(d_log_scales) || !aligned4(d_noise)) return RS_ERR_INVALID_ARG;
    GroupTable T{};
    T.n_groups = n_groups;
    for (int k = 0; k < n_groups; ++k) {
        const rs_densify_group& G = groups[k];
        if (G.rows < 1 || !aligned4(G.d_param) || !aligned4(G.d_param_out)) return RS_ERR_INVALID_ARG;
        if ((G.d_m && !aligned4(G.d_m)) || (G.d_v && !aligned4(G.d_v)) || (G.d_m_out && !aligned4(G.d_m_out)) ||
            (G.d_v_out && !aligned4(G.d_v_out)))
            return RS_ERR_INVALID_ARG;
        if (G.kind != RS_DENSIFY_COPY && G.kind != RS_DENSIFY_MEANS && G.kind != RS_DENSIFY_LOG_SCALES)
            return RS_ERR_INVALID_ARG;
        if (G.kind != RS_DENSIFY_COPY && G.rows != 3) return RS_ERR_INVALID_ARG;
        T.g[k] = G;
    }
    const uint8_t* ws = static_cast<const uint8_t*>(d_workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    rs::pdl_launch(k_densify_apply, p.blocks, kBlock, 0, s, n, ws + p.off_action,
                   reinterpret_cast<const uint32_t*>(ws + p.off_offset),
                   reinterpret_cast<const uint32_t*>(ws + p.off_total), d_quats, d_log_scales, d_noise, T,
                   uint32_t(n_out));
    return cudaGetLastError() == cudaSuccess ? RS_OK : RS_ERR_CUDA;
}

}  // extern "C"
