// [1] projection and [5] projection backward.
//
// Loads are planar (one coalesced row per component).  The projection of the radius-square
// binning stages each tile's input rows in shared memory by bulk copies when n is a multiple of 4
// and the rows are 16-byte aligned (k_project_staged), else takes RS_PROJ_VEC Gaussians per thread
// with 8- or 16-byte loads and stores of every row when the rows allow it (k_project_vec), else
// one per thread with 4-byte accesses (k_project); its input is about 236 bytes per Gaussian at SH
// degree 3.
// Forward: rigel README "Projection"; "3D Gaussian Splatting ビューワを作る" 2.1-2.3;
// learn-gs "11 - Tiles" tile_spans.  Backward: rigel README "Backward" and "Deliberate
// differences from the reference implementation".
#include <algorithm>

#include "rs_internal.cuh"

namespace rs {
namespace {

// One thread per Gaussian.  Blocks of 128 threads at 9 per SM (at most 56 registers): 160k
// Gaussians then run in a single wave on the 152 SMs (at 256 threads and 64 registers, 4 blocks
// per SM, 608 resident blocks left 17 of 625 for a second wave).
#ifndef RS_PROJ_THREADS
#define RS_PROJ_THREADS 128
#endif
#ifndef RS_PROJ_MIN_BLOCKS
#define RS_PROJ_MIN_BLOCKS 9
#endif
// 1: the square-test projection stages its input rows in shared memory with bulk copies
// (k_project_staged) when n and the rows allow it.
#ifndef RS_PROJ_STAGED
#define RS_PROJ_STAGED 1
#endif
// Gaussians per thread of the vectorised projection (2: 8-byte accesses, 4: 16-byte accesses).
#ifndef RS_PROJ_VEC
#define RS_PROJ_VEC 2
#endif
constexpr int kProjThreads = RS_PROJ_THREADS;
constexpr int kProjMinBlocks = RS_PROJ_MIN_BLOCKS;

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

// Every product and sum below is an explicitly rounded single-precision operation (no contraction
// left to the compiler), so the two projection kernels give bit-identical colours.
__device__ __forceinline__ float mul_rn(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ float sub_rn(float a, float b) { return __fsub_rn(a, b); }

template <int DEG>
__device__ __forceinline__ void sh_basis(float x, float y, float z, float* Y) {
    Y[0] = kY0;
    if (DEG >= 1) {
        Y[1] = mul_rn(-kY1, y);
        Y[2] = mul_rn(kY1, z);
        Y[3] = mul_rn(-kY1, x);
    }
    if (DEG >= 2) {
        const float xx = mul_rn(x, x), yy = mul_rn(y, y), zz = mul_rn(z, z);
        Y[4] = mul_rn(mul_rn(kY2a, x), y);
        Y[5] = mul_rn(mul_rn(-kY2a, y), z);
        Y[6] = mul_rn(kY2b, sub_rn(sub_rn(2.f * zz, xx), yy));
        Y[7] = mul_rn(mul_rn(-kY2a, z), x);
        Y[8] = mul_rn(kY2c, sub_rn(xx, yy));
        if (DEG >= 3) {
            Y[9] = mul_rn(mul_rn(-kY3a, sub_rn(3.f * xx, yy)), y);
            Y[10] = mul_rn(mul_rn(mul_rn(kY3b, x), y), z);
            Y[11] = mul_rn(mul_rn(-kY3c, sub_rn(sub_rn(4.f * zz, xx), yy)), y);
            Y[12] = mul_rn(mul_rn(kY3d, z), sub_rn(sub_rn(2.f * zz, 3.f * xx), 3.f * yy));
            Y[13] = mul_rn(mul_rn(-kY3c, x), sub_rn(sub_rn(4.f * zz, xx), yy));
            Y[14] = mul_rn(mul_rn(kY3e, sub_rn(xx, yy)), z);
            Y[15] = mul_rn(mul_rn(-kY3a, x), sub_rn(xx, 3.f * yy));
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

// a*b - c*d with one rounding error (Kahan's algorithm with a fused multiply-add).
__device__ __forceinline__ float diff_of_products(float a, float b, float c, float d) {
    const float w = c * d;
    const float e = fmaf(-c, d, w);
    const float f = fmaf(a, b, -w);
    return f + e;
}

// Forward geometry of one Gaussian (everything but colour).
struct Geo {
    float p[3];       // camera-space mean
    float qn;         // |q|
    float qh[4];      // q / |q|
    float Rq[9];      // rotation of qh
    float s2[3];      // squared scales
    float T[6];       // J R (2x3)
    float U[6];       // T Rq (2x3): Sigma_2d = U diag(s^2) U^T + 0.3 I
    float m01, m02, m12;  // 2x2 minors of U: m_jk = U0j U1k - U0k U1j
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
    G.s2[0] = s[0] * s[0];
    G.s2[1] = s[1] * s[1];
    G.s2[2] = s[2] * s[2];
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
    // Sigma_2d = T (Rq S^2 Rq^T) T^T = U S^2 U^T with U = T Rq: the same matrix as
    // J W Sigma_3d W^T J^T, evaluated through the 2x3 factor (fewer products, less cancellation)
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int j = 0; j < 3; ++j)
            G.U[k * 3 + j] = G.T[k * 3 + 0] * G.Rq[0 * 3 + j] + G.T[k * 3 + 1] * G.Rq[1 * 3 + j] +
                             G.T[k * 3 + 2] * G.Rq[2 * 3 + j];
    const float ap = G.s2[0] * G.U[0] * G.U[0] + G.s2[1] * G.U[1] * G.U[1] + G.s2[2] * G.U[2] * G.U[2];
    const float cp = G.s2[0] * G.U[3] * G.U[3] + G.s2[1] * G.U[4] * G.U[4] + G.s2[2] * G.U[5] * G.U[5];
    G.a = ap + kDilation;
    G.b = G.s2[0] * G.U[0] * G.U[3] + G.s2[1] * G.U[1] * G.U[4] + G.s2[2] * G.U[2] * G.U[5];
    G.c = cp + kDilation;
    // det = ac - b^2 without its cancellation: by Cauchy-Binet,
    // det(0.3 I + V V^T) = 0.09 + 0.3 tr(V V^T) + sum_{j<k} (s_j s_k m_jk)^2 with V = U diag(s),
    // a sum of non-negative terms (for a needle seen end-on ac and b^2 agree to many digits)
    G.m01 = diff_of_products(G.U[0], G.U[4], G.U[1], G.U[3]);
    G.m02 = diff_of_products(G.U[0], G.U[5], G.U[2], G.U[3]);
    G.m12 = diff_of_products(G.U[1], G.U[5], G.U[2], G.U[4]);
    const float t01 = s[0] * s[1] * G.m01, t02 = s[0] * s[2] * G.m02, t12 = s[1] * s[2] * G.m12;
    G.det = kDilation * kDilation + kDilation * (ap + cp) + (t01 * t01 + t02 * t02 + t12 * t12);
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

// Unit direction from the camera centre -R^T t to the mean, with explicit operations (as sh_basis).
__device__ __forceinline__ void view_dir(const CameraF& cam, const float m[3], float d[3], float& len) {
    const float C0 = -fmaf(cam.R[6], cam.t[2], fmaf(cam.R[3], cam.t[1], mul_rn(cam.R[0], cam.t[0])));
    const float C1 = -fmaf(cam.R[7], cam.t[2], fmaf(cam.R[4], cam.t[1], mul_rn(cam.R[1], cam.t[0])));
    const float C2 = -fmaf(cam.R[8], cam.t[2], fmaf(cam.R[5], cam.t[1], mul_rn(cam.R[2], cam.t[0])));
    d[0] = sub_rn(m[0], C0); d[1] = sub_rn(m[1], C1); d[2] = sub_rn(m[2], C2);
    len = __fsqrt_rn(fmaf(d[2], d[2], fmaf(d[1], d[1], mul_rn(d[0], d[0]))));
    const float il = len > 0.f ? __fdiv_rn(1.0f, len) : 0.f;
    d[0] = mul_rn(d[0], il); d[1] = mul_rn(d[1], il); d[2] = mul_rn(d[2], il);
}

template <int DEG>
__global__ void __launch_bounds__(kProjThreads, kProjMinBlocks) k_project(CameraF cam, int n, const float* __restrict__ means,
                                                 const float* __restrict__ scales,
                                                 const float* __restrict__ quats,
                                                 const float* __restrict__ opacity,
                                                 const float* __restrict__ sh,
                                                 const float* __restrict__ colors, float* means2d,
                                                 float* depth, float* conic, float* color,
                                                 int* radius, uint32_t* tiles, Record* rec,
                                                 int tile_test, float* ellipse) {
    RS_PDL_ENTER();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const size_t N = size_t(n);
    const float m[3] = {__ldg(means + i), __ldg(means + N + i), __ldg(means + 2 * N + i)};
    const float s[3] = {__ldg(scales + i), __ldg(scales + N + i), __ldg(scales + 2 * N + i)};
    const float q[4] = {__ldg(quats + i), __ldg(quats + N + i), __ldg(quats + 2 * N + i),
                        __ldg(quats + 3 * N + i)};
    const float o = __ldg(opacity + i);
    Geo G;
    geometry(cam, m, s, q, G);
    uint32_t nt = 0;
    float ak = 0.f;
    if (G.visible) {
        nt = uint32_t(G.rect[1] - G.rect[0]) * uint32_t(G.rect[3] - G.rect[2]);
        if (tile_test == RS_TILE_TEST_ELLIPSE) {
            // only the tiles the alpha >= 1/255 ellipse meets; none culls the splat
            ak = alpha_k_of(o);
            nt = 0;
            EllipseTiles e;
            if (ellipse_tiles_init(G.u, G.v, G.A, G.B, G.C, ak, G.rect, cam.TY, e)) {
                for (int ty = e.ylo; ty <= e.yhi; ++ty) {
                    int xlo, xhi;
                    ellipse_row(e, ty, cam.TX, xlo, xhi);
                    if (xhi >= xlo) nt += uint32_t(xhi - xlo + 1);
                }
            }
            if (nt > 0) {
                // the per-splat setup, for the binning's expansion
                float w[kEllWords];
                ellipse_pack(e, w);
#pragma unroll
                for (int q = 0; q < kEllWords; ++q) ellipse[(q + 1) * N + i] = w[q];
            }
        }
    }
    if (!G.visible || nt == 0) {
        means2d[i] = 0.f; means2d[N + i] = 0.f;
        depth[i] = 0.f;
        conic[i] = 0.f; conic[N + i] = 0.f; conic[2 * N + i] = 0.f;
        color[i] = 0.f; color[N + i] = 0.f; color[2 * N + i] = 0.f;
        radius[i] = 0;
        tiles[i] = 0;
        if (tile_test == RS_TILE_TEST_ELLIPSE) ellipse[i] = 0.f;
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
    means2d[i] = G.u; means2d[N + i] = G.v;
    depth[i] = G.p[2];
    conic[i] = G.A; conic[N + i] = G.B; conic[2 * N + i] = G.C;
    color[i] = rgb[0]; color[N + i] = rgb[1]; color[2 * N + i] = rgb[2];
    radius[i] = G.radius;
    tiles[i] = nt;
    if (tile_test == RS_TILE_TEST_ELLIPSE) ellipse[i] = ak;
    // Half-extents of the region where opacity * exp(power) >= 1/255, i.e. d^T Q d <= k with
    // k = 2 ln(255 o): the ellipse's bounding box is sqrt(k a) by sqrt(k c) (a, c the diagonal of
    // Sigma_2d = Q^-1).  Inflated by 0.1% in k and 0.01 px so that float rounding in the
    // rasterisers' alpha can never reach 1/255 outside it; negative when o < 1/255 (the Gaussian
    // can never pass the alpha threshold).
    float ext_x = -1.f, ext_y = -1.f;
    const float o255 = 255.f * o;
    if (o255 > 1.f) {
        const float k = 2.002f * logf(o255);
        ext_x = sqrtf(k * G.a) + 0.01f;
        ext_y = sqrtf(k * G.c) + 0.01f;
    }
    Record r;
    r.p = make_float4(G.u, G.v, o, ext_x);
    r.q = make_float4(-0.5f * kLog2e * G.A, -kLog2e * G.B, -0.5f * kLog2e * G.C, ext_y);
    r.c = make_float4(rgb[0], rgb[1], rgb[2], 1.0f / o);
    rec[i] = r;
}

// The projection of V (2 or 4) consecutive Gaussians per thread with 8- or 16-byte loads and
// stores of every planar row (a warp moves 256 or 512 contiguous bytes per row and instruction):
// the same per-Gaussian arithmetic as k_project (geometry, SH colour, record), for the
// radius-square tile test, when n is a multiple of V and every row is 4V-byte aligned.  The SH rows
// are read once any of the V is visible.
template <int V>
struct VecF;
template <>
struct VecF<2> {
    float v[2];
    __device__ __forceinline__ static VecF load(const float* p) {
        const float2 t = __ldg(reinterpret_cast<const float2*>(p));
        return VecF{{t.x, t.y}};
    }
    __device__ __forceinline__ static void store(float* p, const float (&a)[2]) {
        *reinterpret_cast<float2*>(p) = make_float2(a[0], a[1]);
    }
    __device__ __forceinline__ static void store_i(int* p, const int (&a)[2]) {
        *reinterpret_cast<int2*>(p) = make_int2(a[0], a[1]);
    }
    __device__ __forceinline__ static void store_u(uint32_t* p, const uint32_t (&a)[2]) {
        *reinterpret_cast<uint2*>(p) = make_uint2(a[0], a[1]);
    }
};
template <>
struct VecF<4> {
    float v[4];
    __device__ __forceinline__ static VecF load(const float* p) {
        const float4 t = __ldg(reinterpret_cast<const float4*>(p));
        return VecF{{t.x, t.y, t.z, t.w}};
    }
    __device__ __forceinline__ static void store(float* p, const float (&a)[4]) {
        *reinterpret_cast<float4*>(p) = make_float4(a[0], a[1], a[2], a[3]);
    }
    __device__ __forceinline__ static void store_i(int* p, const int (&a)[4]) {
        *reinterpret_cast<int4*>(p) = make_int4(a[0], a[1], a[2], a[3]);
    }
    __device__ __forceinline__ static void store_u(uint32_t* p, const uint32_t (&a)[4]) {
        *reinterpret_cast<uint4*>(p) = make_uint4(a[0], a[1], a[2], a[3]);
    }
};

template <int DEG, int V>
__global__ void __launch_bounds__(kProjThreads) k_project_vec(CameraF cam, int n, const float* __restrict__ means,
                                                             const float* __restrict__ scales,
                                                             const float* __restrict__ quats,
                                                             const float* __restrict__ opacity,
                                                             const float* __restrict__ sh,
                                                             const float* __restrict__ colors, float* means2d,
                                                             float* depth, float* conic, float* color, int* radius,
                                                             uint32_t* tiles, Record* rec) {
    RS_PDL_ENTER();
    using L = VecF<V>;
    const int i0 = V * (blockIdx.x * blockDim.x + threadIdx.x);
    if (i0 >= n) return;
    const size_t N = size_t(n);
    auto row = [&](const float* base, size_t r) { return L::load(base + r * N + size_t(i0)); };
    const L M0 = row(means, 0), M1 = row(means, 1), M2 = row(means, 2);
    const L S0 = row(scales, 0), S1 = row(scales, 1), S2 = row(scales, 2);
    const L Q0 = row(quats, 0), Q1 = row(quats, 1), Q2 = row(quats, 2), Q3 = row(quats, 3);
    const L O = row(opacity, 0);
    float u[V], v[V], z[V], cA[V], cB[V], cC[V], ex[V], ey[V], dir[V][3];
    int rad[V];
    uint32_t nt[V];
    bool vis[V], any = false;
#pragma unroll
    for (int g = 0; g < V; ++g) {
        const float m[3] = {M0.v[g], M1.v[g], M2.v[g]};
        const float sc[3] = {S0.v[g], S1.v[g], S2.v[g]};
        const float q[4] = {Q0.v[g], Q1.v[g], Q2.v[g], Q3.v[g]};
        Geo G;
        geometry(cam, m, sc, q, G);
        vis[g] = G.visible;
        any |= G.visible;
        u[g] = G.visible ? G.u : 0.f;
        v[g] = G.visible ? G.v : 0.f;
        z[g] = G.visible ? G.p[2] : 0.f;
        cA[g] = G.visible ? G.A : 0.f;
        cB[g] = G.visible ? G.B : 0.f;
        cC[g] = G.visible ? G.C : 0.f;
        rad[g] = G.visible ? G.radius : 0;
        nt[g] = G.visible ? uint32_t(G.rect[1] - G.rect[0]) * uint32_t(G.rect[3] - G.rect[2]) : 0u;
        // the alpha >= 1/255 box (as k_project)
        const float o255 = 255.f * O.v[g];
        ex[g] = -1.f;
        ey[g] = -1.f;
        if (G.visible && o255 > 1.f) {
            const float k = 2.002f * logf(o255);
            ex[g] = sqrtf(k * G.a) + 0.01f;
            ey[g] = sqrtf(k * G.c) + 0.01f;
        }
        float len;
        view_dir(cam, m, dir[g], len);
    }
    float rgb[V][3];
#pragma unroll
    for (int g = 0; g < V; ++g) rgb[g][0] = rgb[g][1] = rgb[g][2] = 0.f;
    if (any) {
        if (DEG < 0) {
#pragma unroll
            for (int ch = 0; ch < 3; ++ch) {
                const L c = row(colors, ch);
#pragma unroll
                for (int g = 0; g < V; ++g) rgb[g][ch] = c.v[g];
            }
        } else {
            constexpr int K = (DEG + 1) * (DEG + 1);
            float Y[V][16];
#pragma unroll
            for (int g = 0; g < V; ++g) sh_basis<(DEG < 0 ? 0 : DEG)>(dir[g][0], dir[g][1], dir[g][2], Y[g]);
#pragma unroll
            for (int k = 0; k < K; ++k) {
#pragma unroll
                for (int ch = 0; ch < 3; ++ch) {
                    const L c = row(sh, size_t(k * 3 + ch));
#pragma unroll
                    for (int g = 0; g < V; ++g) rgb[g][ch] = fmaf(c.v[g], Y[g][k], rgb[g][ch]);
                }
            }
        }
    }
    float c0[V], c1[V], c2[V];
#pragma unroll
    for (int g = 0; g < V; ++g) {
        c0[g] = vis[g] ? rgb[g][0] : 0.f;
        c1[g] = vis[g] ? rgb[g][1] : 0.f;
        c2[g] = vis[g] ? rgb[g][2] : 0.f;
    }
    L::store(means2d + i0, u);
    L::store(means2d + N + i0, v);
    L::store(depth + i0, z);
    L::store(conic + i0, cA);
    L::store(conic + N + i0, cB);
    L::store(conic + 2 * N + i0, cC);
    L::store(color + i0, c0);
    L::store(color + N + i0, c1);
    L::store(color + 2 * N + i0, c2);
    L::store_i(radius + i0, rad);
    L::store_u(tiles + i0, nt);
#pragma unroll
    for (int g = 0; g < V; ++g) {
        if (!vis[g]) continue;
        const float o = O.v[g];
        Record r;
        r.p = make_float4(u[g], v[g], o, ex[g]);
        r.q = make_float4(-0.5f * kLog2e * cA[g], -kLog2e * cB[g], -0.5f * kLog2e * cC[g], ey[g]);
        r.c = make_float4(c0[g], c1[g], c2[g], 1.0f / o);
        rec[i0 + g] = r;
    }
}

// ---------------------------------------------------------------- staged projection
// The projection with every planar input row of a tile of Gaussians copied to shared memory
// by bulk asynchronous copies (PTX cp.async.bulk, completion counted in bytes on an mbarrier),
// one thread per Gaussian: the 11 geometry rows on one barrier, the colour rows (48 SH rows at
// degree 3) on a second, so the geometry starts while the colour rows are still in flight.  A
// persistent grid walks the tiles (with two buffers the next tile's rows are requested before the
// current one is computed), so the input streams in bulk instead of in two dependent round trips
// per thread.  Same arithmetic as k_project, Gaussian by Gaussian.
// Taken when n is a multiple of 4 and every input row is 16-byte aligned (the copies' rule).
// Tiles of 64 Gaussians, one buffer, 14 CTAs per SM (15 KB each at degree 3) measured 12.3 us per
// 160k-Gaussian launch under ncu, against 14.3 (128, two buffers, 3 CTAs), 13.1 (128, one, 7)
// and 14.5 (64, two, 7): the per-Gaussian arithmetic needs the warps more than the copies need a
// second buffer.
#ifndef RS_PROJ_STAGE_THREADS
#define RS_PROJ_STAGE_THREADS 64
#endif
#ifndef RS_PROJ_STAGE_BUFS
#define RS_PROJ_STAGE_BUFS 1
#endif
#ifndef RS_PROJ_STAGE_BLOCKS
#define RS_PROJ_STAGE_BLOCKS 14
#endif
constexpr int kStgThreads = RS_PROJ_STAGE_THREADS;   // Gaussians per tile, one per thread
constexpr int kStgBufs = RS_PROJ_STAGE_BUFS;         // 2: the next tile's rows requested ahead
constexpr int kStgBlocksPerSM = RS_PROJ_STAGE_BLOCKS;
static_assert(kStgBufs == 1 || kStgBufs == 2, "one or two buffers");
constexpr int kStgGeoRows = 11;  // means 3, scales 3, quats 4, opacity 1
constexpr uint32_t kStgWaitLimit = 1u << 22;

template <int DEG>
__host__ __device__ constexpr int stg_rows() {
    return kStgGeoRows + (DEG < 0 ? 3 : 3 * (DEG + 1) * (DEG + 1));
}

__device__ unsigned int g_proj_error;  // set when a bounded wait on a staged copy gave up

__device__ __forceinline__ void stg_mbar_init(uint32_t mbar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mbar) : "memory");
}
__device__ __forceinline__ void stg_expect(uint32_t mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void stg_copy(uint32_t dst, const float* src, uint32_t bytes, uint32_t mbar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(mbar)
                 : "memory");
}
__device__ __forceinline__ bool stg_wait(uint32_t mbar, uint32_t parity) {
    for (uint32_t i = 0; i < kStgWaitLimit; ++i) {
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

template <int DEG>
__global__ void __launch_bounds__(kStgThreads) k_project_staged(CameraF cam, int n, const float* __restrict__ means,
                                                              const float* __restrict__ scales,
                                                              const float* __restrict__ quats,
                                                              const float* __restrict__ opacity,
                                                              const float* __restrict__ sh,
                                                              const float* __restrict__ colors, float* means2d,
                                                              float* depth, float* conic, float* color, int* radius,
                                                              uint32_t* tiles, Record* rec) {
    RS_PDL_ENTER();
    constexpr int R = stg_rows<DEG>();
    constexpr int T = kStgThreads;
    extern __shared__ __align__(128) float s_rows[];  // [kStgBufs buffers][R rows][T Gaussians]
    __shared__ __align__(8) uint64_t s_mbar[2][2];     // [buffer][geometry rows, colour rows]
    const int t = threadIdx.x;
    const size_t N = size_t(n);
    const int n_tiles = (n + T - 1) / T;
    if (t == 0) {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            stg_mbar_init(uint32_t(__cvta_generic_to_shared(&s_mbar[b][0])));
            stg_mbar_init(uint32_t(__cvta_generic_to_shared(&s_mbar[b][1])));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // thread 0: request tile `tile`'s rows into buffer b
    auto issue = [&](int tile, int b) {
        const size_t base = size_t(tile) * T;
        const uint32_t bytes = uint32_t(min(size_t(T), N - base)) * 4u;
        const uint32_t dst = uint32_t(__cvta_generic_to_shared(s_rows + size_t(b) * R * T));
        const uint32_t mg = uint32_t(__cvta_generic_to_shared(&s_mbar[b][0]));
        const uint32_t mc = uint32_t(__cvta_generic_to_shared(&s_mbar[b][1]));
        stg_expect(mg, kStgGeoRows * bytes);
        stg_expect(mc, (R - kStgGeoRows) * bytes);
        auto row = [&](int r) { return dst + uint32_t(r * T * 4); };
#pragma unroll
        for (int r = 0; r < 3; ++r) stg_copy(row(r), means + size_t(r) * N + base, bytes, mg);
#pragma unroll
        for (int r = 0; r < 3; ++r) stg_copy(row(3 + r), scales + size_t(r) * N + base, bytes, mg);
#pragma unroll
        for (int r = 0; r < 4; ++r) stg_copy(row(6 + r), quats + size_t(r) * N + base, bytes, mg);
        stg_copy(row(10), opacity + base, bytes, mg);
        const float* crow = DEG < 0 ? colors : sh;
        for (int r = 0; r < R - kStgGeoRows; ++r) stg_copy(row(kStgGeoRows + r), crow + size_t(r) * N + base, bytes, mc);
    };
    int k = 0;
    if (t == 0 && int(blockIdx.x) < n_tiles) issue(blockIdx.x, 0);
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++k) {
        const int b = kStgBufs == 2 ? (k & 1) : 0;
        const uint32_t par = uint32_t(kStgBufs == 2 ? (k >> 1) : k) & 1u;
        const uint32_t mg = uint32_t(__cvta_generic_to_shared(&s_mbar[b][0]));
        const uint32_t mc = uint32_t(__cvta_generic_to_shared(&s_mbar[b][1]));
        const int next = tile + int(gridDim.x);
        if (kStgBufs == 2 && t == 0 && next < n_tiles) {
            // buffer b ^ 1 was last read in the previous step, which ended with a barrier
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(next, b ^ 1);
        }
        const float* S = s_rows + size_t(b) * R * T;
        const int i = tile * T + t;
        const bool live = i < n;
        bool ok = __syncthreads_and(stg_wait(mg, par));
        if (!ok) {
            // give up: flag it, let this CTA's copies in flight land (bounded), leave
            if (t == 0) {
                atomicOr(&g_proj_error, 1u);
                (void)stg_wait(mc, par);
                if (kStgBufs == 2 && next < n_tiles) {
                    (void)stg_wait(uint32_t(__cvta_generic_to_shared(&s_mbar[b ^ 1][0])), uint32_t((k + 1) >> 1) & 1u);
                    (void)stg_wait(uint32_t(__cvta_generic_to_shared(&s_mbar[b ^ 1][1])), uint32_t((k + 1) >> 1) & 1u);
                }
            }
            return;
        }
        const float m[3] = {S[0 * T + t], S[1 * T + t], S[2 * T + t]};
        const float sc[3] = {S[3 * T + t], S[4 * T + t], S[5 * T + t]};
        const float q[4] = {S[6 * T + t], S[7 * T + t], S[8 * T + t], S[9 * T + t]};
        const float o = S[10 * T + t];
        Geo G;
        geometry(cam, m, sc, q, G);
        const bool vis = live && G.visible;
        float d[3], len;
        view_dir(cam, m, d, len);
        ok = __syncthreads_and(stg_wait(mc, par));
        if (!ok) {
            if (t == 0) {
                atomicOr(&g_proj_error, 1u);
                if (kStgBufs == 2 && next < n_tiles) {
                    (void)stg_wait(uint32_t(__cvta_generic_to_shared(&s_mbar[b ^ 1][0])), uint32_t((k + 1) >> 1) & 1u);
                    (void)stg_wait(uint32_t(__cvta_generic_to_shared(&s_mbar[b ^ 1][1])), uint32_t((k + 1) >> 1) & 1u);
                }
            }
            return;
        }
        float rgb[3] = {0.f, 0.f, 0.f};
        if (vis) {
            if (DEG < 0) {
#pragma unroll
                for (int ch = 0; ch < 3; ++ch) rgb[ch] = S[(kStgGeoRows + ch) * T + t];
            } else {
                constexpr int K = (DEG + 1) * (DEG + 1);
                float Y[16];
                sh_basis<(DEG < 0 ? 0 : DEG)>(d[0], d[1], d[2], Y);
#pragma unroll
                for (int ch = 0; ch < 3; ++ch) {
                    float acc = 0.f;
#pragma unroll
                    for (int kk = 0; kk < K; ++kk) acc = fmaf(S[(kStgGeoRows + kk * 3 + ch) * T + t], Y[kk], acc);
                    rgb[ch] = acc;
                }
            }
        }
        if (live) {
            means2d[i] = vis ? G.u : 0.f;
            means2d[N + i] = vis ? G.v : 0.f;
            depth[i] = vis ? G.p[2] : 0.f;
            conic[i] = vis ? G.A : 0.f;
            conic[N + i] = vis ? G.B : 0.f;
            conic[2 * N + i] = vis ? G.C : 0.f;
            color[i] = rgb[0];
            color[N + i] = rgb[1];
            color[2 * N + i] = rgb[2];
            radius[i] = vis ? G.radius : 0;
            tiles[i] = vis ? uint32_t(G.rect[1] - G.rect[0]) * uint32_t(G.rect[3] - G.rect[2]) : 0u;
        }
        if (vis) {
            // the alpha >= 1/255 box, as k_project
            float ext_x = -1.f, ext_y = -1.f;
            const float o255 = 255.f * o;
            if (o255 > 1.f) {
                const float kk = 2.002f * logf(o255);
                ext_x = sqrtf(kk * G.a) + 0.01f;
                ext_y = sqrtf(kk * G.c) + 0.01f;
            }
            Record r;
            r.p = make_float4(G.u, G.v, o, ext_x);
            r.q = make_float4(-0.5f * kLog2e * G.A, -kLog2e * G.B, -0.5f * kLog2e * G.C, ext_y);
            r.c = make_float4(rgb[0], rgb[1], rgb[2], 1.0f / o);
            rec[i] = r;
        }
        __syncthreads();  // buffer b is read before it is requested again
        if (kStgBufs == 1 && t == 0 && next < n_tiles) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(next, 0);
        }
    }
}

template <int DEG>
__global__ void __launch_bounds__(kProjThreads, kProjMinBlocks) k_project_bwd(
    CameraF cam, int n, const float* __restrict__ means, const float* __restrict__ scales,
    const float* __restrict__ quats, const float* __restrict__ sh,
    const int* __restrict__ radius, const float* __restrict__ dm2,
    const float* __restrict__ dcon, const float* __restrict__ dcol, float* dmeans,
    float* dscales, float* dquats, float* dsh) {
    RS_PDL_ENTER();
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
    // conic = Q = Sigma_2d^-1 with Sigma_2d = U S^2 U^T + 0.3 I, U = T Rq; the conic's gradient
    // Gq = [[gA, gB/2], [gB/2, gC]] gives dL/dSigma_2d = -Q Gq Q.  Everything below goes through
    // W = Q U and Q y = adj(Sigma_2d) y / det with
    //   adj(Sigma_2d) y = 0.3 y + sum_k s_k^2 u_k_perp (u_k_perp . y),  u_perp = (-u1, u0),
    // so the large s_j^2 u_j u_j^T part of a needle-like Gaussian is never subtracted from itself:
    //   Z = W^T Gq W,  ds_j = -2 s_j Z_jj,  dRq = -2 Rq Z S^2  (T^T dU with T = U Rq^T),
    //   dU_j = -2 s_j^2 Q (Gq w_j),  dT = dU Rq^T.
    const float gA = __ldg(dcon + i), gB = 0.5f * __ldg(dcon + N + i), gC = __ldg(dcon + 2 * N + i);
    const float mn[3][3] = {{0.f, G.m01, G.m02}, {-G.m01, 0.f, G.m12}, {-G.m02, -G.m12, 0.f}};
    const float inv_det = 1.0f / G.det;
    float Wx[3], Wy[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        float wx = kDilation * G.U[j], wy = kDilation * G.U[3 + j];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            if (k == j) continue;
            const float mm = G.s2[k] * mn[j][k];  // s_k^2 m_jk = -s_k^2 (u_k_perp . u_j)
            wx = fmaf(mm, G.U[3 + k], wx);
            wy = fmaf(-mm, G.U[k], wy);
        }
        Wx[j] = wx * inv_det;
        Wy[j] = wy * inv_det;
    }
    float dU[6];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const float yx = gA * Wx[j] + gB * Wy[j];  // y = Gq w_j
        const float yy = gB * Wx[j] + gC * Wy[j];
        float ax = kDilation * yx, ay = kDilation * yy;  // adj(Sigma_2d) y
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const float ux = G.U[k], uy = G.U[3 + k];
            const float d = G.s2[k] * fmaf(-uy, yx, ux * yy);  // s_k^2 (u_k_perp . y)
            ax = fmaf(-uy, d, ax);
            ay = fmaf(ux, d, ay);
        }
        dU[j] = -2.f * G.s2[j] * ax * inv_det;
        dU[3 + j] = -2.f * G.s2[j] * ay * inv_det;
    }
    float dT[6];
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int r = 0; r < 3; ++r)
            dT[k * 3 + r] = dU[k * 3 + 0] * G.Rq[r * 3 + 0] + dU[k * 3 + 1] * G.Rq[r * 3 + 1] +
                            dU[k * 3 + 2] * G.Rq[r * 3 + 2];
    float Z[3][3];
#pragma unroll
    for (int j = 0; j < 3; ++j)
#pragma unroll
        for (int k = j; k < 3; ++k) {
            Z[j][k] = gA * Wx[j] * Wx[k] + gB * (Wx[j] * Wy[k] + Wy[j] * Wx[k]) + gC * Wy[j] * Wy[k];
            Z[k][j] = Z[j][k];
        }
    float ds[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) ds[j] = -2.f * s[j] * Z[j][j];
    float dR[9];
#pragma unroll
    for (int r = 0; r < 3; ++r)
#pragma unroll
        for (int j = 0; j < 3; ++j)
            dR[r * 3 + j] = -2.f * G.s2[j] *
                            (G.Rq[r * 3 + 0] * Z[0][j] + G.Rq[r * 3 + 1] * Z[1][j] + G.Rq[r * 3 + 2] * Z[2][j]);
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

int take_projection_error() {
    unsigned int v = 0u;
    if (cudaMemcpyFromSymbol(&v, g_proj_error, sizeof(v)) != cudaSuccess) return -1;
    if (v == 0u) return 0;
    const unsigned int zero = 0u;
    if (cudaMemcpyToSymbol(g_proj_error, &zero, sizeof(zero)) != cudaSuccess) return -1;
    return 1;
}

cudaError_t launch_project(const CameraF& cam, const rs_gaussians& g, const rs_projected& o,
                           cudaStream_t s) {
    if (g.n == 0) return cudaSuccess;
    const int threads = kProjThreads;
    Record* rec = reinterpret_cast<Record*>(o.d_records);
#if RS_PROJ_STAGED
    auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & uintptr_t(15)) == 0; };
    if (o.tile_test == RS_TILE_TEST_SQUARE && g.n % 4 == 0 && al16(g.d_means) && al16(g.d_scales) &&
        al16(g.d_quats) && al16(g.d_opacity) && al16(g.sh_degree >= 0 ? g.d_sh : g.d_colors)) {
        int dev = 0, sms = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        const int n_tiles = (g.n + kStgThreads - 1) / kStgThreads;
        const int blocks = std::min(n_tiles, std::max(1, sms) * kStgBlocksPerSM);
#define RS_PROJECT_STAGED(D)                                                                               \
    {                                                                                                      \
        const size_t smem = size_t(kStgBufs) * stg_rows<D>() * kStgThreads * sizeof(float);               \
        e = cudaFuncSetAttribute(k_project_staged<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)); \
        if (e != cudaSuccess) return e;                                                                    \
        pdl_launch(k_project_staged<D>, blocks, kStgThreads, smem, s, cam, g.n, g.d_means, g.d_scales,     \
                   g.d_quats, g.d_opacity, g.d_sh, g.d_colors, o.d_means2d, o.d_depth, o.d_conic, o.d_color, \
                   o.d_radius, o.d_tiles_touched, rec);                                                    \
    }
        switch (g.sh_degree) {
            case -1: RS_PROJECT_STAGED(-1); break;
            case 0: RS_PROJECT_STAGED(0); break;
            case 1: RS_PROJECT_STAGED(1); break;
            case 2: RS_PROJECT_STAGED(2); break;
            default: RS_PROJECT_STAGED(3); break;
        }
#undef RS_PROJECT_STAGED
        return cudaGetLastError();
    }
#endif
    // RS_PROJ_VEC Gaussians per thread (2 or 4) when the rows allow it, else one
    constexpr int V = RS_PROJ_VEC;
    auto al = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & uintptr_t(4 * V - 1)) == 0; };
    const bool vec = o.tile_test == RS_TILE_TEST_SQUARE && g.n % V == 0 && al(g.d_means) && al(g.d_scales) &&
                     al(g.d_quats) && al(g.d_opacity) && al(g.sh_degree >= 0 ? g.d_sh : g.d_colors) &&
                     al(o.d_means2d) && al(o.d_depth) && al(o.d_conic) && al(o.d_color) && al(o.d_radius) &&
                     al(o.d_tiles_touched);
    if (vec) {
        const int blocks_v = (g.n / V + threads - 1) / threads;
#define RS_PROJECT_VEC(D)                                                                          \
    pdl_launch(k_project_vec<D, V>, blocks_v, threads, 0, s, cam, g.n, g.d_means, g.d_scales, g.d_quats,  \
               g.d_opacity, g.d_sh, g.d_colors, o.d_means2d, o.d_depth, o.d_conic, o.d_color, o.d_radius, \
               o.d_tiles_touched, rec)
        switch (g.sh_degree) {
            case -1: RS_PROJECT_VEC(-1); break;
            case 0: RS_PROJECT_VEC(0); break;
            case 1: RS_PROJECT_VEC(1); break;
            case 2: RS_PROJECT_VEC(2); break;
            default: RS_PROJECT_VEC(3); break;
        }
#undef RS_PROJECT_VEC
        return cudaGetLastError();
    }
    const int blocks = (g.n + threads - 1) / threads;
#define RS_PROJECT(D)                                                                           \
    pdl_launch(k_project<D>, blocks, threads, 0, s, cam, g.n, g.d_means, g.d_scales, g.d_quats,         \
                                             g.d_opacity, g.d_sh, g.d_colors, o.d_means2d,      \
                                             o.d_depth, o.d_conic, o.d_color, o.d_radius,       \
                                             o.d_tiles_touched, rec, o.tile_test, o.d_ellipse)
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
    const int threads = kProjThreads;
    const int blocks = (g.n + threads - 1) / threads;
#define RS_PROJECT_BWD(D)                                                                      \
    pdl_launch(k_project_bwd<D>, blocks, threads, 0, s, cam, g.n, g.d_means, g.d_scales, g.d_quats,    \
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
