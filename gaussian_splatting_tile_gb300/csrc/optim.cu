// Fused Adam step over the Gaussian parameters and the densification statistics of the training
// loop (rigel README: the optimisation loop and "GaussianModel: activations, densify/prune",
// with per-group learning rates, e.g. the higher-order SH rate a twentieth of the DC rate).
//
// One launch updates every parameter group: a segment table (by value) maps the flat element
// index to its group.  For a group stored as raw values behind an activation (log-scales behind
// exp, opacity logits behind sigmoid) the given gradient is w.r.t. the activated value, so the
// kernel applies the activation's derivative first and writes the activated value of the updated
// parameter, which is what the projection reads next.  Per element: read param, grad, m, v;
// write param, m, v (and the activated value): HBM-bound.
#include "rs_internal.cuh"

namespace rs {
namespace {

// Per group: `quads` runs of four elements moved with 16-byte loads and stores (when every
// pointer of the group is 16-byte aligned), then the remaining elements one at a time.
struct AdamTable {
    rs_adam_segment seg[RS_ADAM_MAX_SEGMENTS];
    size_t qstart[RS_ADAM_MAX_SEGMENTS + 1];  // cumulative quads
    size_t tstart[RS_ADAM_MAX_SEGMENTS + 1];  // cumulative tail elements
    size_t quads[RS_ADAM_MAX_SEGMENTS];
    int n;
    float beta1, beta2, omb1, omb2, eps, rc1, rc2;  // omb = 1 - beta, rc = 1 / (1 - beta^t)
};

__device__ __forceinline__ float adam_one(const AdamTable& T, int act, float lr, float& p, float g, float& m,
                                          float& v) {
    if (act == RS_ACT_EXP) {
        g *= expf(p);                       // d exp(p)/dp = exp(p)
    } else if (act == RS_ACT_SIGMOID) {
        const float a = 1.0f / (1.0f + expf(-p));
        g *= a * (1.0f - a);                // d sigmoid(p)/dp
    }
    // beta m + (1 - beta) g with both products formed: the second moment stays accurate to
    // float32 when it is small next to g^2 (as in the first steps)
    m = fmaf(T.beta1, m, T.omb1 * g);
    v = fmaf(T.beta2, v, T.omb2 * (g * g));
    p -= lr * (m * T.rc1) / (sqrtf(v * T.rc2) + T.eps);
    return act == RS_ACT_EXP ? expf(p) : act == RS_ACT_SIGMOID ? 1.0f / (1.0f + expf(-p)) : p;
}

__global__ void __launch_bounds__(256) k_adam(AdamTable T) {
    RS_PDL_ENTER();
    const size_t stride = size_t(gridDim.x) * blockDim.x;
    const size_t nq = T.qstart[T.n];
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < nq; i += stride) {
        int s = 0;
        while (s + 1 < T.n && i >= T.qstart[s + 1]) ++s;
        const rs_adam_segment& S = T.seg[s];
        const size_t k = i - T.qstart[s];
        float4 p = reinterpret_cast<const float4*>(S.d_param)[k];
        const float4 g = reinterpret_cast<const float4*>(S.d_grad)[k];
        float4 m = reinterpret_cast<const float4*>(S.d_m)[k];
        float4 v = reinterpret_cast<const float4*>(S.d_v)[k];
        float4 a;
        a.x = adam_one(T, S.activation, S.lr, p.x, g.x, m.x, v.x);
        a.y = adam_one(T, S.activation, S.lr, p.y, g.y, m.y, v.y);
        a.z = adam_one(T, S.activation, S.lr, p.z, g.z, m.z, v.z);
        a.w = adam_one(T, S.activation, S.lr, p.w, g.w, m.w, v.w);
        reinterpret_cast<float4*>(S.d_m)[k] = m;
        reinterpret_cast<float4*>(S.d_v)[k] = v;
        reinterpret_cast<float4*>(S.d_param)[k] = p;
        if (S.d_activated) reinterpret_cast<float4*>(S.d_activated)[k] = a;
    }
    const size_t nt = T.tstart[T.n];
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < nt; i += stride) {
        int s = 0;
        while (s + 1 < T.n && i >= T.tstart[s + 1]) ++s;
        const rs_adam_segment& S = T.seg[s];
        const size_t k = 4 * T.quads[s] + (i - T.tstart[s]);
        float p = S.d_param[k], m = S.d_m[k], v = S.d_v[k];
        const float a = adam_one(T, S.activation, S.lr, p, S.d_grad[k], m, v);
        S.d_m[k] = m;
        S.d_v[k] = v;
        S.d_param[k] = p;
        if (S.d_activated) S.d_activated[k] = a;
    }
}

__global__ void __launch_bounds__(256) k_densify_stats(int n, const float* __restrict__ dm2,
                                                       const int* __restrict__ radius,
                                                       float* __restrict__ accum, float* __restrict__ count) {
    RS_PDL_ENTER();
    const int stride = gridDim.x * blockDim.x;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        if (radius[i] > 0) {
            const float gx = dm2[i], gy = dm2[size_t(n) + i];
            accum[i] += sqrtf(gx * gx + gy * gy);
            count[i] += 1.0f;
        }
    }
}

}  // namespace

cudaError_t launch_adam(const rs_adam_segment* segs, int n, double beta1, double beta2, double eps, int step,
                        cudaStream_t s) {
    AdamTable T{};
    T.n = n;
    for (int i = 0; i < n; ++i) {
        const rs_adam_segment& g = segs[i];
        T.seg[i] = g;
        auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
        const bool vec = al16(g.d_param) && al16(g.d_grad) && al16(g.d_m) && al16(g.d_v) &&
                         (g.d_activated == nullptr || al16(g.d_activated));
        T.quads[i] = vec ? g.count / 4 : 0;
        T.qstart[i + 1] = T.qstart[i] + T.quads[i];
        T.tstart[i + 1] = T.tstart[i] + (g.count - 4 * T.quads[i]);
    }
    T.beta1 = float(beta1);
    T.beta2 = float(beta2);
    T.omb1 = float(1.0 - beta1);
    T.omb2 = float(1.0 - beta2);
    T.eps = float(eps);
    T.rc1 = float(1.0 / (1.0 - std::pow(beta1, double(step))));
    T.rc2 = float(1.0 / (1.0 - std::pow(beta2, double(step))));
    const size_t total = std::max(T.qstart[n], T.tstart[n]);
    if (total == 0) return cudaSuccess;
    const unsigned blocks = unsigned(std::min<size_t>((total + 255) / 256, 152 * 16));
    pdl_launch(k_adam, blocks, 256, 0, s, T);
    return cudaGetLastError();
}

cudaError_t launch_densify_stats(int n, const float* dm2, const int* radius, float* accum, float* count,
                                 cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const unsigned blocks = unsigned(std::min((n + 255) / 256, 152 * 8));
    pdl_launch(k_densify_stats, blocks, 256, 0, s, n, dm2, radius, accum, count);
    return cudaGetLastError();
}

}  // namespace rs
