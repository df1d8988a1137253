// [1] projection and [5] projection backward: one thread per Gaussian.
//
// Loads are planar (one coalesced 4-byte row per component), so a warp reads 128 contiguous
// bytes per row; the kernel is bound by those bytes (about 236 per Gaussian at SH degree 3).
// Forward: rigel README "Projection"; "3D Gaussian Splatting ビューワを作る" 2.1-2.3;
// learn-gs "11 - Tiles" tile_spans.  Backward: rigel README "Backward" and "Deliberate
// differences from the reference implementation".
#include "rs_internal.cuh"

namespace rs {
namespace {

// Real SH normalisations of "3D Gaussian Splatting ビューワを作る" 2.2.3 (after Sloan's
// "Stupid Spherical Harmonics (SH) Tricks", Appendix A2).
constexpr float kY0 = 0.28209479177387814f;   // 1 / (2 sqrt(pi))
constexpr float kY1 = 0.4886025119029199f;    // sqrt(3 / (4 pi))
constexpr float kY2a = 1.0925484305920792f;   // sqrt(15 / pi) / 2
constexpr float kY2b = 0.31539156525252005f;  // sqrt(5 / pi) / 4
constexpr float kY2c = 0.5462742152960396f;   // sqrt(15 / pi) / 4
constexpr float kY3a = 0.5900435899266435f;   // sqrt(35 / (2 pi)) / 4
constexpr float kY3b = 2.890611442640554f;    // sqrt(105 / pi) / 2
constexpr float kY3c = 0.4570457994644658f;   // sqrt(21 / (2 pi)) / 4
constexpr float kY3d = 0.3731763325901154f;   // sqrt(7 / pi) / 4
constexpr float kY3e = 1.445305721320277f;    // sqrt(105 / pi) / 4

template <int DEG>
__device__ __forceinline__ void sh_basis(float x, float y, float z, float* Y) {
    Y[0] = kY0;
    if (DEG >= 1) {
        Y[1] = -kY1 * y;
        Y[2] = kY1 * z;
        Y[3] = -kY1 * x;
    }
    if (DEG >= 2) {
        const float xx = x * x, yy = y * y, zz = z * z;
        Y[4] = kY2a * x * y;
        Y[5] = -kY2a * y * z;
        Y[6] = kY2b * (2.f * zz - xx - yy);
        Y[7] = -kY2a * z * x;
        Y[8] = kY2c * (xx - yy);
        if (DEG >= 3) {
            Y[9] = -kY3a * (3.f * xx - yy) * y;
            Y[10] = kY3b * x * y * z;
            Y[11] = -kY3c * (4.f * zz - xx - yy) * y;
            Y[12] = kY3d * z * (2.f * zz - 3.f * xx - 3.f * yy);
            Y[13] = -kY3c * x * (4.f * zz - xx - yy);
            Y[14] = kY3e * (xx - yy) * z;
            Y[15] = -kY3a * x * (xx - 3.f * yy);
        }
    }
}

// d Y_k / d(x, y, z) of the polynomials above, for the backward.
template <int DEG>
__device__ __forceinline__ void sh_basis_grad(float x, float y, float z, float (*G)[3]) {
    G[0][0] = G[0][1] = G[0][2] = 0.f;
    if (DEG >= 1) {
        G[1][0] = 0.f;   G[1][1] = -kY1; G[1][2] = 0.f;
        G[2][0] = 0.f;   G[2][1] = 0.f;  G[2][2] = kY1;
        G[3][0] = -kY1;  G[3][1] = 0.f;  G[3][2] = 0.f;
    }
    if (DEG >= 2) {
        G[4][0] = kY2a * y;          G[4][1] = kY2a * x;          G[4][2] = 0.f;
        G[5][0] = 0.f;               G[5][1] = -kY2a * z;         G[5][2] = -kY2a * y;
        G[6][0] = -2.f * kY2b * x;   G[6][1] = -2.f * kY2b * y;   G[6][2] = 4.f * kY2b * z;
        G[7][0] = -kY2a * z;         G[7][1] = 0.f;               G[7][2] = -kY2a * x;
        G[8][0] = 2.f * kY2c * x;    G[8][1] = -2.f * kY2c * y;   G[8][2] = 0.f;
        if (DEG >= 3) {
            const float xx = x * x, yy = y * y, zz = z * z;
            G[9][0] = -6.f * kY3a * x * y;
            G[9][1] = -3.f * kY3a * (xx - yy);
            G[9][2] = 0.f;
            G[10][0] = kY3b * y * z;
            G[10][1] = kY3b * x * z;
            G[10][2] = kY3b * x * y;
            G[11][0] = 2.f * kY3c * x * y;
            G[11][1] = -kY3c * (4.f * zz - xx - 3.f * yy);
            G[11][2] = -8.f * kY3c * y * z;
            G[12][0] = -6.f * kY3d * x * z;
            G[12][1] = -6.f * kY3d * y * z;
            G[12][2] = kY3d * (6.f * zz - 3.f * xx - 3.f * yy);
            G[13][0] = -kY3c * (4.f * zz - 3.f * xx - yy);
            G[13][1] = 2.f * kY3c * x * y;
            G[13][2] = -8.f * kY3c * x * z;
            G[14][0] = 2.f * kY3e * x * z;
            G[14][1] = -2.f * kY3e * y * z;
            G[14][2] = kY3e * (xx - yy);
            G[15][0] = -3.f * kY3a * (xx - yy);
            G[15][1] = 6.f * kY3a * x * y;
            G[15][2] = 0.f;
        }
    }
}

// Forward geometry of one Gaussian (everything but colour).
struct Geo {
    float p[3];       // camera-space mean
    float qn;         // |q|
    float qh[4];      // q / |q|
    float Rq[9];      // rotation of qh
    float S3[6];      // 3D covariance xx xy xz yy yz zz
    float T[6];       // J R (2x3)
    float tx, ty;
    bool cx, cy;      // clamp active
    float a, b, c;    // dilated 2D covariance
    float det;
    float A, B, C;    // conic
    float u, v;
    int radius;
    int rect[4];
    bool visible;
};

__device__ __forceinline__ void geometry(const CameraF& cam, const float m[3], const float s[3],
                                         const float q[4], Geo& G) {
    G.visible = false;
    G.radius = 0;
#pragma unroll
    for (int r = 0; r < 3; ++r)
        G.p[r] = fmaf(cam.R[r * 3 + 0], m[0], fmaf(cam.R[r * 3 + 1], m[1], fmaf(cam.R[r * 3 + 2], m[2], cam.t[r])));
    const float x = G.p[0], y = G.p[1], z = G.p[2];
    if (!(z > kZNear)) return;
    const float qn2 = q[0] * q[0] + q[1] * q[1] + q[2] * q[2] + q[3] * q[3];
    G.qn = sqrtf(qn2);
    if (!(G.qn > 0.f) || !isfinite(G.qn)) return;
    const float inv_qn = 1.0f / G.qn;
    const float w = q[0] * inv_qn, qx = q[1] * inv_qn, qy = q[2] * inv_qn, qz = q[3] * inv_qn;
    G.qh[0] = w; G.qh[1] = qx; G.qh[2] = qy; G.qh[3] = qz;
    // Hamilton rotation of (w, x, y, z)
    G.Rq[0] = 1.f - 2.f * (qy * qy + qz * qz);
    G.Rq[1] = 2.f * (qx * qy - w * qz);
    G.Rq[2] = 2.f * (qx * qz + w * qy);
    G.Rq[3] = 2.f * (qx * qy + w * qz);
    G.Rq[4] = 1.f - 2.f * (qx * qx + qz * qz);
    G.Rq[5] = 2.f * (qy * qz - w * qx);
    G.Rq[6] = 2.f * (qx * qz - w * qy);
    G.Rq[7] = 2.f * (qy * qz + w * qx);
    G.Rq[8] = 1.f - 2.f * (qx * qx + qy * qy);
    float M[9];
#pragma unroll
    for (int i = 0; i < 3; ++i)
#pragma unroll
        for (int j = 0; j < 3; ++j) M[i * 3 + j] = G.Rq[i * 3 + j] * s[j];
    // Sigma_3d = M M^T (symmetric: xx xy xz yy yz zz)
    G.S3[0] = M[0] * M[0] + M[1] * M[1] + M[2] * M[2];
    G.S3[1] = M[0] * M[3] + M[1] * M[4] + M[2] * M[5];
    G.S3[2] = M[0] * M[6] + M[1] * M[7] + M[2] * M[8];
    G.S3[3] = M[3] * M[3] + M[4] * M[4] + M[5] * M[5];
    G.S3[4] = M[3] * M[6] + M[4] * M[7] + M[5] * M[8];
    G.S3[5] = M[6] * M[6] + M[7] * M[7] + M[8] * M[8];
    // J at the clamped centre
    const float lim_x = kClampFrac * (0.5f * float(cam.W)) / cam.fx;
    const float lim_y = kClampFrac * (0.5f * float(cam.H)) / cam.fy;
    const float xz = x / z, yz = y / z;
    G.cx = xz < -lim_x || xz > lim_x;
    G.cy = yz < -lim_y || yz > lim_y;
    G.tx = z * fminf(lim_x, fmaxf(-lim_x, xz));
    G.ty = z * fminf(lim_y, fmaxf(-lim_y, yz));
    const float iz = 1.0f / z;
    const float j00 = cam.fx * iz, j02 = -cam.fx * G.tx * iz * iz;
    const float j11 = cam.fy * iz, j12 = -cam.fy * G.ty * iz * iz;
    // T = J R
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        G.T[j] = j00 * cam.R[0 * 3 + j] + j02 * cam.R[2 * 3 + j];
        G.T[3 + j] = j11 * cam.R[1 * 3 + j] + j12 * cam.R[2 * 3 + j];
    }
    // Sigma_2d = T Sigma_3d T^T
    const float* S = G.S3;
    float TS[6];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float* t = &G.T[i * 3];
        TS[i * 3 + 0] = t[0] * S[0] + t[1] * S[1] + t[2] * S[2];
        TS[i * 3 + 1] = t[0] * S[1] + t[1] * S[3] + t[2] * S[4];
        TS[i * 3 + 2] = t[0] * S[2] + t[1] * S[4] + t[2] * S[5];
    }
    G.a = TS[0] * G.T[0] + TS[1] * G.T[1] + TS[2] * G.T[2] + kDilation;
    G.b = TS[0] * G.T[3] + TS[1] * G.T[4] + TS[2] * G.T[5];
    G.c = TS[3] * G.T[3] + TS[4] * G.T[4] + TS[5] * G.T[5] + kDilation;
    G.det = G.a * G.c - G.b * G.b;
    if (!(G.det > 0.f) || !isfinite(G.det)) return;
    const float inv = 1.0f / G.det;
    G.A = G.c * inv;
    G.B = -G.b * inv;
    G.C = G.a * inv;
    G.u = cam.fx * x * iz + cam.cx;
    G.v = cam.fy * y * iz + cam.cy;
    if (!isfinite(G.u) || !isfinite(G.v)) return;
    const float mid = 0.5f * (G.a + G.c);
    const float lam = mid + sqrtf(fmaxf(kLambdaFloor, mid * mid - G.det));
    const int r = int(ceilf(3.0f * sqrtf(lam)));
    const float rf = float(r);
    G.rect[0] = span_bound(G.u, rf, cam.TX, false);
    G.rect[1] = span_bound(G.u, rf, cam.TX, true);
    G.rect[2] = span_bound(G.v, rf, cam.TY, false);
    G.rect[3] = span_bound(G.v, rf, cam.TY, true);
    if (G.rect[1] <= G.rect[0] || G.rect[3] <= G.rect[2]) return;
    G.radius = r;
    G.visible = true;
}

__device__ __forceinline__ void view_dir(const CameraF& cam, const float m[3], float d[3], float& len) {
    // camera centre -R^T t
    const float C0 = -(cam.R[0] * cam.t[0] + cam.R[3] * cam.t[1] + cam.R[6] * cam.t[2]);
    const float C1 = -(cam.R[1] * cam.t[0] + cam.R[4] * cam.t[1] + cam.R[7] * cam.t[2]);
    const float C2 = -(cam.R[2] * cam.t[0] + cam.R[5] * cam.t[1] + cam.R[8] * cam.t[2]);
    d[0] = m[0] - C0; d[1] = m[1] - C1; d[2] = m[2] - C2;
    len = sqrtf(d[0] * d[0] + d[1] * d[1] + d[2] * d[2]);
    const float il = len > 0.f ? 1.0f / len : 0.f;
    d[0] *= il; d[1] *= il; d[2] *= il;
}

template <int DEG>
__global__ void __launch_bounds__(256) k_project(CameraF cam, int n, const float* __restrict__ means,
                                                 const float* __restrict__ scales,
                                                 const float* __restrict__ quats,
                                                 const float* __restrict__ opacity,
                                                 const float* __restrict__ sh,
                                                 const float* __restrict__ colors, float* means2d,
                                                 float* depth, float* conic, float* color,
                                                 int* radius, uint32_t* tiles, Record* rec) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const size_t N = size_t(n);
    const float m[3] = {__ldg(means + i), __ldg(means + N + i), __ldg(means + 2 * N + i)};
    const float s[3] = {__ldg(scales + i), __ldg(scales + N + i), __ldg(scales + 2 * N + i)};
    const float q[4] = {__ldg(quats + i), __ldg(quats + N + i), __ldg(quats + 2 * N + i),
                        __ldg(quats + 3 * N + i)};
    Geo G;
    geometry(cam, m, s, q, G);
    if (!G.visible) {
        means2d[i] = 0.f; means2d[N + i] = 0.f;
        depth[i] = 0.f;
        conic[i] = 0.f; conic[N + i] = 0.f; conic[2 * N + i] = 0.f;
        color[i] = 0.f; color[N + i] = 0.f; color[2 * N + i] = 0.f;
        radius[i] = 0;
        tiles[i] = 0;
        return;
    }
    float rgb[3];
    if (DEG < 0) {
        rgb[0] = __ldg(colors + i); rgb[1] = __ldg(colors + N + i); rgb[2] = __ldg(colors + 2 * N + i);
    } else {
        constexpr int K = (DEG + 1) * (DEG + 1);
        float d[3], len;
        view_dir(cam, m, d, len);
        float Y[16];
        sh_basis<(DEG < 0 ? 0 : DEG)>(d[0], d[1], d[2], Y);
#pragma unroll
        for (int ch = 0; ch < 3; ++ch) {
            float acc = 0.f;
#pragma unroll
            for (int k = 0; k < K; ++k) acc = fmaf(__ldg(sh + size_t(k * 3 + ch) * N + i), Y[k], acc);
            rgb[ch] = acc;
        }
    }
    const float o = __ldg(opacity + i);
    means2d[i] = G.u; means2d[N + i] = G.v;
    depth[i] = G.p[2];
    conic[i] = G.A; conic[N + i] = G.B; conic[2 * N + i] = G.C;
    color[i] = rgb[0]; color[N + i] = rgb[1]; color[2 * N + i] = rgb[2];
    radius[i] = G.radius;
    tiles[i] = uint32_t(G.rect[1] - G.rect[0]) * uint32_t(G.rect[3] - G.rect[2]);
    Record r;
    r.p = make_float4(G.u, G.v, o, G.A);
    r.q = make_float4(-0.5f * kLog2e * G.A, -kLog2e * G.B, -0.5f * kLog2e * G.C, G.B);
    r.c = make_float4(rgb[0], rgb[1], rgb[2], G.C);
    rec[i] = r;
}

template <int DEG>
__global__ void __launch_bounds__(256) k_project_bwd(
    CameraF cam, int n, const float* __restrict__ means, const float* __restrict__ scales,
    const float* __restrict__ quats, const float* __restrict__ sh,
    const int* __restrict__ radius, const float* __restrict__ dm2,
    const float* __restrict__ dcon, const float* __restrict__ dcol, float* dmeans,
    float* dscales, float* dquats, float* dsh) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const size_t N = size_t(n);
    constexpr int K = DEG >= 0 ? (DEG + 1) * (DEG + 1) : 0;
    Geo G;
    G.visible = false;
    float m[3], s[3], q[4];
    const bool live = __ldg(radius + i) > 0;
    if (live) {
        m[0] = __ldg(means + i); m[1] = __ldg(means + N + i); m[2] = __ldg(means + 2 * N + i);
        s[0] = __ldg(scales + i); s[1] = __ldg(scales + N + i); s[2] = __ldg(scales + 2 * N + i);
        q[0] = __ldg(quats + i); q[1] = __ldg(quats + N + i); q[2] = __ldg(quats + 2 * N + i);
        q[3] = __ldg(quats + 3 * N + i);
        geometry(cam, m, s, q, G);
    }
    if (!G.visible) {
        for (int k = 0; k < 3; ++k) { dmeans[k * N + i] = 0.f; dscales[k * N + i] = 0.f; }
        for (int k = 0; k < 4; ++k) dquats[k * N + i] = 0.f;
        if (DEG >= 0)
            for (int k = 0; k < 3 * K; ++k) dsh[size_t(k) * N + i] = 0.f;
        return;
    }
    // conic = Q = Sigma_2d^-1: dL/dSigma_2d = -Q Gq Q, Gq = [[gA, gB/2], [gB/2, gC]]
    const float gA = __ldg(dcon + i), gB = 0.5f * __ldg(dcon + N + i), gC = __ldg(dcon + 2 * N + i);
    const float A = G.A, B = G.B, C = G.C;
    const float qg00 = A * gA + B * gB, qg01 = A * gB + B * gC;
    const float qg10 = B * gA + C * gB, qg11 = B * gB + C * gC;
    const float g00 = -(qg00 * A + qg01 * B);
    const float g01 = -(qg00 * B + qg01 * C);
    const float g11 = -(qg10 * B + qg11 * C);
    // Sigma_2d = T S T^T: dT = 2 G2 T S, dS = T^T G2 T (G2 symmetric [[g00, g01], [g01, g11]])
    const float* S = G.S3;
    float TS[6];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const float* t = &G.T[r * 3];
        TS[r * 3 + 0] = t[0] * S[0] + t[1] * S[1] + t[2] * S[2];
        TS[r * 3 + 1] = t[0] * S[1] + t[1] * S[3] + t[2] * S[4];
        TS[r * 3 + 2] = t[0] * S[2] + t[1] * S[4] + t[2] * S[5];
    }
    float dT[6];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        dT[j] = 2.f * (g00 * TS[j] + g01 * TS[3 + j]);
        dT[3 + j] = 2.f * (g01 * TS[j] + g11 * TS[3 + j]);
    }
    float GT[6];  // G2 T
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        GT[j] = g00 * G.T[j] + g01 * G.T[3 + j];
        GT[3 + j] = g01 * G.T[j] + g11 * G.T[3 + j];
    }
    float dS[9];  // T^T G2 T, full 3x3
#pragma unroll
    for (int a = 0; a < 3; ++a)
#pragma unroll
        for (int b = 0; b < 3; ++b) dS[a * 3 + b] = G.T[a] * GT[b] + G.T[3 + a] * GT[3 + b];
    // T = J R -> dJ = dT R^T; only J00, J02, J11, J12 are variables
    float dJ[6];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int k = 0; k < 3; ++k)
            dJ[r * 3 + k] = dT[r * 3 + 0] * cam.R[k * 3 + 0] + dT[r * 3 + 1] * cam.R[k * 3 + 1] +
                            dT[r * 3 + 2] * cam.R[k * 3 + 2];
    const float x = G.p[0], y = G.p[1], z = G.p[2];
    const float iz = 1.0f / z, iz2 = iz * iz, iz3 = iz2 * iz;
    float dp[3] = {0.f, 0.f, 0.f};
    dp[2] += dJ[0] * (-cam.fx * iz2) + dJ[2] * (2.f * cam.fx * G.tx * iz3) + dJ[4] * (-cam.fy * iz2) +
             dJ[5] * (2.f * cam.fy * G.ty * iz3);
    const float dtx = dJ[2] * (-cam.fx * iz2);
    const float dty = dJ[5] * (-cam.fy * iz2);
    if (G.cx) dp[2] += dtx * (G.tx * iz); else dp[0] += dtx;
    if (G.cy) dp[2] += dty * (G.ty * iz); else dp[1] += dty;
    const float du = __ldg(dm2 + i), dv = __ldg(dm2 + N + i);
    dp[0] += du * cam.fx * iz;
    dp[1] += dv * cam.fy * iz;
    dp[2] -= (du * cam.fx * x + dv * cam.fy * y) * iz2;
    float dm[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) dm[j] = cam.R[j] * dp[0] + cam.R[3 + j] * dp[1] + cam.R[6 + j] * dp[2];
    // Sigma_3d = M M^T, M = Rq diag(s): dM = 2 dS M
    float M[9];
#pragma unroll
    for (int a = 0; a < 3; ++a)
#pragma unroll
        for (int b = 0; b < 3; ++b) M[a * 3 + b] = G.Rq[a * 3 + b] * s[b];
    float ds[3] = {0.f, 0.f, 0.f};
    float dR[9];
#pragma unroll
    for (int a = 0; a < 3; ++a)
#pragma unroll
        for (int b = 0; b < 3; ++b) {
            const float dMab = 2.f * (dS[a * 3 + 0] * M[0 * 3 + b] + dS[a * 3 + 1] * M[1 * 3 + b] +
                                      dS[a * 3 + 2] * M[2 * 3 + b]);
            dR[a * 3 + b] = dMab * s[b];
            ds[b] += dMab * G.Rq[a * 3 + b];
        }
    const float w = G.qh[0], qx = G.qh[1], qy = G.qh[2], qz = G.qh[3];
    float dqh[4];
    dqh[0] = 2.f * (-qz * dR[1] + qy * dR[2] + qz * dR[3] - qx * dR[5] - qy * dR[6] + qx * dR[7]);
    dqh[1] = 2.f * (qy * dR[1] + qz * dR[2] + qy * dR[3] - w * dR[5] + qz * dR[6] + w * dR[7]) -
             4.f * qx * (dR[4] + dR[8]);
    dqh[2] = 2.f * (qx * dR[1] + w * dR[2] + qx * dR[3] + qz * dR[5] - w * dR[6] + qz * dR[7]) -
             4.f * qy * (dR[0] + dR[8]);
    dqh[3] = 2.f * (-w * dR[1] + qx * dR[2] + w * dR[3] + qy * dR[5] + qx * dR[6] + qy * dR[7]) -
             4.f * qz * (dR[0] + dR[4]);
    const float dot = dqh[0] * w + dqh[1] * qx + dqh[2] * qy + dqh[3] * qz;
    const float iqn = 1.0f / G.qn;
#pragma unroll
    for (int k = 0; k < 4; ++k) dquats[k * N + i] = (dqh[k] - G.qh[k] * dot) * iqn;
    if (DEG >= 0) {
        float d[3], len;
        view_dir(cam, m, d, len);
        float Y[16], GY[16][3];
        sh_basis<(DEG < 0 ? 0 : DEG)>(d[0], d[1], d[2], Y);
        sh_basis_grad<(DEG < 0 ? 0 : DEG)>(d[0], d[1], d[2], GY);
        const float dc[3] = {__ldg(dcol + i), __ldg(dcol + N + i), __ldg(dcol + 2 * N + i)};
        float dd[3] = {0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < K; ++k) {
            float e = 0.f;
#pragma unroll
            for (int ch = 0; ch < 3; ++ch) {
                const size_t row = size_t(k * 3 + ch) * N + i;
                dsh[row] = dc[ch] * Y[k];
                e = fmaf(dc[ch], __ldg(sh + row), e);
            }
            if (k > 0) {
                dd[0] = fmaf(e, GY[k][0], dd[0]);
                dd[1] = fmaf(e, GY[k][1], dd[1]);
                dd[2] = fmaf(e, GY[k][2], dd[2]);
            }
        }
        const float ddot = dd[0] * d[0] + dd[1] * d[1] + dd[2] * d[2];
        const float il = 1.0f / len;
#pragma unroll
        for (int e = 0; e < 3; ++e) dm[e] += (dd[e] - d[e] * ddot) * il;
    }
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        dmeans[k * N + i] = dm[k];
        dscales[k * N + i] = ds[k];
    }
}

}  // namespace

cudaError_t launch_project(const CameraF& cam, const rs_gaussians& g, const rs_projected& o,
                           cudaStream_t s) {
    if (g.n == 0) return cudaSuccess;
    const int threads = 256;
    const int blocks = (g.n + threads - 1) / threads;
    Record* rec = reinterpret_cast<Record*>(o.d_records);
#define RS_PROJECT(D)                                                                           \
    k_project<D><<<blocks, threads, 0, s>>>(cam, g.n, g.d_means, g.d_scales, g.d_quats,         \
                                             g.d_opacity, g.d_sh, g.d_colors, o.d_means2d,      \
                                             o.d_depth, o.d_conic, o.d_color, o.d_radius,       \
                                             o.d_tiles_touched, rec)
    switch (g.sh_degree) {
        case -1: RS_PROJECT(-1); break;
        case 0: RS_PROJECT(0); break;
        case 1: RS_PROJECT(1); break;
        case 2: RS_PROJECT(2); break;
        default: RS_PROJECT(3); break;
    }
#undef RS_PROJECT
    return cudaGetLastError();
}

cudaError_t launch_project_bwd(const CameraF& cam, const rs_gaussians& g, const rs_projected& p,
                               const float* dm2, const float* dcon, const float* dcol,
                               float* dmeans, float* dscales, float* dquats, float* dsh,
                               cudaStream_t s) {
    if (g.n == 0) return cudaSuccess;
    const int threads = 256;
    const int blocks = (g.n + threads - 1) / threads;
#define RS_PROJECT_BWD(D)                                                                      \
    k_project_bwd<D><<<blocks, threads, 0, s>>>(cam, g.n, g.d_means, g.d_scales, g.d_quats,    \
                                                 g.d_sh, p.d_radius, dm2, dcon, dcol, dmeans,  \
                                                 dscales, dquats, dsh)
    switch (g.sh_degree) {
        case -1: RS_PROJECT_BWD(-1); break;
        case 0: RS_PROJECT_BWD(0); break;
        case 1: RS_PROJECT_BWD(1); break;
        case 2: RS_PROJECT_BWD(2); break;
        default: RS_PROJECT_BWD(3); break;
    }
#undef RS_PROJECT_BWD
    return cudaGetLastError();
}

}  // namespace rs
