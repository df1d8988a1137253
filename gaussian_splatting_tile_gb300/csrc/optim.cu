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

struct AdamTable {
    rs_adam_segment seg[RS_ADAM_MAX_SEGMENTS];
    size_t start[RS_ADAM_MAX_SEGMENTS + 1];
    int n;
    float beta1, beta2, omb1, omb2, eps, rc1, rc2;  // omb = 1 - beta, rc = 1 / (1 - beta^t)
};

__global__ void __launch_bounds__(256) k_adam(AdamTable T) {
    const size_t total = T.start[T.n];
    const size_t stride = size_t(gridDim.x) * blockDim.x;
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        int s = 0;
        while (s + 1 < T.n && i >= T.start[s + 1]) ++s;
        const rs_adam_segment& S = T.seg[s];
        const size_t k = i - T.start[s];
        float p = S.d_param[k];
        float g = S.d_grad[k];
        if (S.activation == RS_ACT_EXP) {
            g *= expf(p);                       // d exp(p)/dp = exp(p)
        } else if (S.activation == RS_ACT_SIGMOID) {
            const float a = 1.0f / (1.0f + expf(-p));
            g *= a * (1.0f - a);                // d sigmoid(p)/dp
        }
        // beta m + (1 - beta) g with both products formed: the second moment stays accurate to
        // float32 when it is small next to g^2 (as in the first steps)
        const float m = fmaf(T.beta1, S.d_m[k], T.omb1 * g);
        const float v = fmaf(T.beta2, S.d_v[k], T.omb2 * (g * g));
        p -= S.lr * (m * T.rc1) / (sqrtf(v * T.rc2) + T.eps);
        S.d_m[k] = m;
        S.d_v[k] = v;
        S.d_param[k] = p;
        if (S.d_activated) {
            S.d_activated[k] = S.activation == RS_ACT_EXP ? expf(p)
                             : S.activation == RS_ACT_SIGMOID ? 1.0f / (1.0f + expf(-p)) : p;
        }
    }
}

__global__ void __launch_bounds__(256) k_densify_stats(int n, const float* __restrict__ dm2,
                                                       const int* __restrict__ radius,
                                                       float* __restrict__ accum, float* __restrict__ count) {
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
    T.start[0] = 0;
    for (int i = 0; i < n; ++i) {
        T.seg[i] = segs[i];
        T.start[i + 1] = T.start[i] + segs[i].count;
    }
    T.beta1 = float(beta1);
    T.beta2 = float(beta2);
    T.omb1 = float(1.0 - beta1);
    T.omb2 = float(1.0 - beta2);
    T.eps = float(eps);
    T.rc1 = float(1.0 / (1.0 - std::pow(beta1, double(step))));
    T.rc2 = float(1.0 / (1.0 - std::pow(beta2, double(step))));
    const size_t total = T.start[n];
    if (total == 0) return cudaSuccess;
    const unsigned blocks = unsigned(std::min<size_t>((total + 255) / 256, 152 * 16));
    k_adam<<<blocks, 256, 0, s>>>(T);
    return cudaGetLastError();
}

cudaError_t launch_densify_stats(int n, const float* dm2, const int* radius, float* accum, float* count,
                                 cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const unsigned blocks = unsigned(std::min((n + 255) / 256, 152 * 8));
    k_densify_stats<<<blocks, 256, 0, s>>>(n, dm2, radius, accum, count);
    return cudaGetLastError();
}

}  // namespace rs
