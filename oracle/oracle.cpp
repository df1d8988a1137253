// Oracle for tile-based 3D Gaussian Splatting rasterisation -- TEST INFRASTRUCTURE ONLY.
//
// Plain, slow, single-threaded statement of the method, stage by stage, in the order and
// notation of the source pages.  It is loaded only by the test suite, the smoke check and
// the benchmark's CPU-baseline leg; it shares nothing with the CUDA library.
// Built with -O2 -ffp-contract=off (no fast-math, no fused multiply-add contraction) so
// that its float arithmetic is the same on every host.
//
// Sources (cited by page title and section):
//   [rigel]  rigel README: "How it works", "Projection", "Binning", "Rasterization",
//            "Backward", "Deliberate differences from the reference implementation",
//            "Appearance MLP".
//   [viewer] "3D Gaussian Splatting ビューワを作る": 2.1 covariance, 2.2 SH, 2.3 outputs,
//            4.1 Prefix Scan, 4.2 Duplicate, 4.3 Radix Sort, 4.4 Tile Range, 4.5 Tile Render.
//   [tiles]  learn-gs notebook "11 - Tiles: the actual 3DGS design": constants,
//            prep_splats, tile_spans, build_tile_lists, the three CPU claims.
#include "oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <utility>
#include <vector>

namespace {

// Constants of the method, stated on the pages ([tiles] constants cell; [rigel] Projection,
// Rasterization, Backward).  The oracle keeps its own copy; nothing is shared with the GPU.
template <typename Real> struct K {
    static Real tile() { return Real(16); }
    static Real dilation() { return Real(0.3); }       // EWA low-pass, [rigel] Projection
    static Real z_near() { return Real(0.05); }        // [tiles] Z_NEAR
    static Real clamp_frac() { return Real(1.3); }     // [rigel] Projection: 1.3x half-width
    static Real alpha_max() { return Real(0.99); }     // [rigel] Rasterization
    static Real alpha_min() { return Real(1) / Real(255); }  // [tiles] ALPHA_MIN
    static Real t_stop() { return Real(1e-4); }        // [rigel] Rasterization, [tiles] T_STOP
    static Real lambda_floor() { return Real(0.1); }   // [viewer] 2.3.3, [tiles] prep_splats
};
const int TILE = 16;

template <typename Real> struct Cam {
    Real R[9], t[3], fx, fy, cx, cy;
    int W, H;
};

template <typename Real> Cam<Real> cam_as(const orc_camera* c) {
    Cam<Real> o;
    for (int i = 0; i < 9; ++i) o.R[i] = Real(c->R[i]);
    for (int i = 0; i < 3; ++i) o.t[i] = Real(c->t[i]);
    o.fx = Real(c->fx); o.fy = Real(c->fy); o.cx = Real(c->cx); o.cy = Real(c->cy);
    o.W = c->width; o.H = c->height;
    return o;
}

bool near_rel(double x, double thr, double margin) {
    return std::fabs(x - thr) <= margin * std::fabs(thr);
}
bool near_int(double x, double margin) {
    return std::fabs(x - std::nearbyint(x)) <= margin * std::max(1.0, std::fabs(x));
}

// Rotation matrix of the unit quaternion (w, x, y, z), Hamilton convention, row-major.
// [viewer] 2.1.1 (Sigma = R S S^T R^T) with the PLY rot_0..rot_3 = (w, x, y, z) order.
template <typename Real> void quat_to_rotmat(Real w, Real x, Real y, Real z, Real* Rq) {
    Rq[0] = 1 - 2 * (y * y + z * z); Rq[1] = 2 * (x * y - w * z);     Rq[2] = 2 * (x * z + w * y);
    Rq[3] = 2 * (x * y + w * z);     Rq[4] = 1 - 2 * (x * x + z * z); Rq[5] = 2 * (y * z - w * x);
    Rq[6] = 2 * (x * z - w * y);     Rq[7] = 2 * (y * z + w * x);     Rq[8] = 1 - 2 * (x * x + y * y);
}

// Real spherical harmonics of degree <= 3 at direction (x, y, z): [viewer] 2.2.3, the table of
// Y_0..Y_15 (after Sloan, "Stupid Spherical Harmonics (SH) Tricks", Appendix A2).  The
// normalisations are written as the page writes them, as closed forms.
template <typename Real> void sh_basis(Real x, Real y, Real z, Real* Y) {
    const double PI = 3.14159265358979323846;
    const Real c0 = Real(1.0 / (2.0 * std::sqrt(PI)));
    const Real c1 = Real(std::sqrt(3.0 / (4.0 * PI)));
    const Real c2a = Real(0.5 * std::sqrt(15.0 / PI));
    const Real c2b = Real(0.25 * std::sqrt(5.0 / PI));
    const Real c2c = Real(0.25 * std::sqrt(15.0 / PI));
    const Real c3a = Real(0.25 * std::sqrt(35.0 / (2.0 * PI)));
    const Real c3b = Real(0.5 * std::sqrt(105.0 / PI));
    const Real c3c = Real(0.25 * std::sqrt(21.0 / (2.0 * PI)));
    const Real c3d = Real(0.25 * std::sqrt(7.0 / PI));
    const Real c3e = Real(0.25 * std::sqrt(105.0 / PI));
    Y[0] = c0;
    Y[1] = -c1 * y;
    Y[2] = c1 * z;
    Y[3] = -c1 * x;
    Y[4] = c2a * x * y;
    Y[5] = -c2a * y * z;
    Y[6] = c2b * (2 * z * z - x * x - y * y);
    Y[7] = -c2a * z * x;
    Y[8] = c2c * (x * x - y * y);
    Y[9] = -c3a * (3 * x * x - y * y) * y;
    Y[10] = c3b * x * y * z;
    Y[11] = -c3c * (4 * z * z - x * x - y * y) * y;
    Y[12] = c3d * z * (2 * z * z - 3 * x * x - 3 * y * y);
    Y[13] = -c3c * x * (4 * z * z - x * x - y * y);
    Y[14] = c3e * (x * x - y * y) * z;
    Y[15] = -c3a * x * (x * x - 3 * y * y);
}

// Gradient of each basis function with respect to the (unnormalised) components (x, y, z);
// obtained by differentiating the polynomials of sh_basis term by term.
void sh_basis_grad(double x, double y, double z, double G[16][3]) {
    const double PI = 3.14159265358979323846;
    const double c1 = std::sqrt(3.0 / (4.0 * PI));
    const double c2a = 0.5 * std::sqrt(15.0 / PI);
    const double c2b = 0.25 * std::sqrt(5.0 / PI);
    const double c2c = 0.25 * std::sqrt(15.0 / PI);
    const double c3a = 0.25 * std::sqrt(35.0 / (2.0 * PI));
    const double c3b = 0.5 * std::sqrt(105.0 / PI);
    const double c3c = 0.25 * std::sqrt(21.0 / (2.0 * PI));
    const double c3d = 0.25 * std::sqrt(7.0 / PI);
    const double c3e = 0.25 * std::sqrt(105.0 / PI);
    const double g[16][3] = {
        {0, 0, 0},
        {0, -c1, 0},
        {0, 0, c1},
        {-c1, 0, 0},
        {c2a * y, c2a * x, 0},
        {0, -c2a * z, -c2a * y},
        {-2 * c2b * x, -2 * c2b * y, 4 * c2b * z},
        {-c2a * z, 0, -c2a * x},
        {2 * c2c * x, -2 * c2c * y, 0},
        {-6 * c3a * x * y, -c3a * (3 * x * x - 3 * y * y), 0},
        {c3b * y * z, c3b * x * z, c3b * x * y},
        {2 * c3c * x * y, -c3c * (4 * z * z - x * x - 3 * y * y), -8 * c3c * y * z},
        {-6 * c3d * x * z, -6 * c3d * y * z, c3d * (6 * z * z - 3 * x * x - 3 * y * y)},
        {-c3c * (4 * z * z - 3 * x * x - y * y), 2 * c3c * x * y, -8 * c3c * x * z},
        {2 * c3e * x * z, -2 * c3e * y * z, c3e * (x * x - y * y)},
        {-c3a * (3 * x * x - 3 * y * y), 6 * c3a * x * y, 0},
    };
    std::memcpy(G, g, sizeof(g));
}

// Camera centre in world space, C = -R^T t (p_cam = R m + t, [rigel] Deliberate differences).
template <typename Real> void camera_centre(const Cam<Real>& c, Real* C) {
    for (int j = 0; j < 3; ++j)
        C[j] = -(c.R[0 * 3 + j] * c.t[0] + c.R[1 * 3 + j] * c.t[1] + c.R[2 * 3 + j] * c.t[2]);
}

// Tile span of a splat's bounding square: [tiles] tile_spans (floor, +1, clamp to the grid),
// evaluated in the caller's precision.  The clamp is applied before conversion to int.
template <typename Real> int span_lo(Real p, Real r, int n_tiles) {
    Real f = std::floor((p - r) / K<Real>::tile());
    if (!(f > Real(0))) f = Real(0);
    if (f > Real(n_tiles)) f = Real(n_tiles);
    return int(f);
}
template <typename Real> int span_hi(Real p, Real r, int n_tiles) {
    Real f = std::floor((p + r) / K<Real>::tile()) + Real(1);
    if (!(f > Real(0))) f = Real(0);
    if (f > Real(n_tiles)) f = Real(n_tiles);
    return int(f);
}

// Everything the projection computes for one Gaussian.
template <typename Real> struct Proj {
    bool visible;
    Real p[3];          // camera-space mean
    Real Rq[9];         // rotation of the normalised quaternion
    Real qn;            // |q|
    Real qhat[4];
    Real S3[9];         // 3D covariance
    Real J[6];          // EWA Jacobian (clamped)
    bool clamp_x, clamp_y;
    Real tx, ty;
    Real T[6];          // T = J W
    Real a, b, c;       // dilated 2D covariance
    Real det;
    Real conic[3];
    Real u, v;
    Real lambda;
    int radius;
    int rect[4];
    unsigned tiles;
    unsigned char amb;
};

// c1: one Gaussian through [rigel] Projection, with the covariance of [viewer] 2.1.1-2.1.2,
// the conic of [viewer] 2.3.1, the radius of [viewer] 2.3.3 / [tiles] prep_splats and the span
// of [tiles] tile_spans.  Culling: z <= 0.05, degenerate, or no tile covered ([rigel] Projection).
template <typename Real>
Proj<Real> project_one(const Cam<Real>& cam, const Real* m, const Real* s, const Real* q,
                       double margin) {
    Proj<Real> P;
    std::memset(&P, 0, sizeof(P));
    P.visible = false;
    // 1. camera transform
    for (int r = 0; r < 3; ++r)
        P.p[r] = cam.R[r * 3 + 0] * m[0] + cam.R[r * 3 + 1] * m[1] + cam.R[r * 3 + 2] * m[2] + cam.t[r];
    const Real x = P.p[0], y = P.p[1], z = P.p[2];
    if (margin > 0 && near_rel(double(z), 0.05, margin)) P.amb |= ORC_AMB_NEAR;
    if (!(z > K<Real>::z_near())) return P;
    // 2. rotation from the normalised quaternion
    P.qn = std::sqrt(q[0] * q[0] + q[1] * q[1] + q[2] * q[2] + q[3] * q[3]);
    if (!(P.qn > Real(0)) || !std::isfinite(double(P.qn))) return P;
    for (int k = 0; k < 4; ++k) P.qhat[k] = q[k] / P.qn;
    quat_to_rotmat(P.qhat[0], P.qhat[1], P.qhat[2], P.qhat[3], P.Rq);
    // 3. Sigma_3d = (R S)(R S)^T
    Real M[9];
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 3; ++j) M[i * 3 + j] = P.Rq[i * 3 + j] * s[j];
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 3; ++j)
            P.S3[i * 3 + j] = M[i * 3 + 0] * M[j * 3 + 0] + M[i * 3 + 1] * M[j * 3 + 1] + M[i * 3 + 2] * M[j * 3 + 2];
    // 4. x/z and y/z clamped to 1.3x the frustum half-width before J is built
    const Real lim_x = K<Real>::clamp_frac() * (Real(cam.W) / Real(2)) / cam.fx;
    const Real lim_y = K<Real>::clamp_frac() * (Real(cam.H) / Real(2)) / cam.fy;
    const Real xz = x / z, yz = y / z;
    if (margin > 0 && (near_rel(std::fabs(double(xz)), double(lim_x), margin) ||
                       near_rel(std::fabs(double(yz)), double(lim_y), margin)))
        P.amb |= ORC_AMB_CLAMP;
    P.clamp_x = xz < -lim_x || xz > lim_x;
    P.clamp_y = yz < -lim_y || yz > lim_y;
    P.tx = z * std::min(lim_x, std::max(-lim_x, xz));
    P.ty = z * std::min(lim_y, std::max(-lim_y, yz));
    // 5. Jacobian of the pinhole at the (clamped) centre
    P.J[0] = cam.fx / z; P.J[1] = 0; P.J[2] = -cam.fx * P.tx / (z * z);
    P.J[3] = 0; P.J[4] = cam.fy / z; P.J[5] = -cam.fy * P.ty / (z * z);
    // 6. Sigma_2d = J W Sigma W^T J^T + 0.3 I
    for (int i = 0; i < 2; ++i)
        for (int j = 0; j < 3; ++j)
            P.T[i * 3 + j] = P.J[i * 3 + 0] * cam.R[0 * 3 + j] + P.J[i * 3 + 1] * cam.R[1 * 3 + j] + P.J[i * 3 + 2] * cam.R[2 * 3 + j];
    Real S2[4];
    for (int i = 0; i < 2; ++i)
        for (int k = 0; k < 2; ++k) {
            Real acc = 0;
            for (int a = 0; a < 3; ++a)
                for (int b = 0; b < 3; ++b) acc += P.T[i * 3 + a] * P.S3[a * 3 + b] * P.T[k * 3 + b];
            S2[i * 2 + k] = acc;
        }
    P.a = S2[0] + K<Real>::dilation();
    P.b = S2[1];
    P.c = S2[3] + K<Real>::dilation();
    // 7. conic = inverse of the 2x2 ([viewer] 2.3.1)
    P.det = P.a * P.c - P.b * P.b;
    if (margin > 0 && std::fabs(double(P.det)) <= margin * std::fabs(double(P.a * P.c))) P.amb |= ORC_AMB_DET;
    if (!(P.det > Real(0)) || !std::isfinite(double(P.det))) return P;
    const Real inv = Real(1) / P.det;
    P.conic[0] = P.c * inv;
    P.conic[1] = -P.b * inv;
    P.conic[2] = P.a * inv;
    // 8. pixel position of the mean (unclamped)
    P.u = cam.fx * x / z + cam.cx;
    P.v = cam.fy * y / z + cam.cy;
    if (!std::isfinite(double(P.u)) || !std::isfinite(double(P.v))) return P;
    // 9. radius = ceil(3 sqrt(lambda_max)), lambda_max with the 0.1 floor
    const Real mid = Real(0.5) * (P.a + P.c);
    P.lambda = mid + std::sqrt(std::max(K<Real>::lambda_floor(), mid * mid - P.det));
    const Real r3 = Real(3) * std::sqrt(P.lambda);
    if (margin > 0 && near_int(double(r3), margin)) P.amb |= ORC_AMB_RADIUS;
    P.radius = int(std::ceil(r3));
    // 10. tile span; nothing covered -> culled
    const int TX = (cam.W + TILE - 1) / TILE, TY = (cam.H + TILE - 1) / TILE;
    const Real r = Real(P.radius);
    if (margin > 0) {
        const double e[4] = {double((P.u - r) / K<Real>::tile()), double((P.u + r) / K<Real>::tile()),
                             double((P.v - r) / K<Real>::tile()), double((P.v + r) / K<Real>::tile())};
        for (double ei : e)
            if (near_int(ei, margin)) P.amb |= ORC_AMB_SPAN;
    }
    P.rect[0] = span_lo(P.u, r, TX);
    P.rect[1] = span_hi(P.u, r, TX);
    P.rect[2] = span_lo(P.v, r, TY);
    P.rect[3] = span_hi(P.v, r, TY);
    const int sx = std::max(0, P.rect[1] - P.rect[0]);
    const int sy = std::max(0, P.rect[3] - P.rect[2]);
    P.tiles = unsigned(sx) * unsigned(sy);
    if (P.tiles == 0) {
        P.radius = 0;
        return P;
    }
    P.visible = true;
    return P;
}

// c6: colour = sum_k sh[k*3+ch] * Y_k(d), d the unit vector from the camera centre to the
// mean ([viewer] 2.2.3).  No offset and no clamp are applied.
template <typename Real>
void sh_colour(const Cam<Real>& cam, const Real* m, const Real* coef /*[3K]*/, int degree,
               Real* rgb, Real* d_out) {
    Real C[3];
    camera_centre(cam, C);
    Real d[3] = {m[0] - C[0], m[1] - C[1], m[2] - C[2]};
    Real len = std::sqrt(d[0] * d[0] + d[1] * d[1] + d[2] * d[2]);
    if (len > Real(0))
        for (int k = 0; k < 3; ++k) d[k] /= len;
    if (d_out)
        for (int k = 0; k < 3; ++k) d_out[k] = d[k];
    Real Y[16];
    sh_basis(d[0], d[1], d[2], Y);
    const int Kc = (degree + 1) * (degree + 1);
    for (int ch = 0; ch < 3; ++ch) {
        Real acc = 0;
        for (int k = 0; k < Kc; ++k) acc += coef[k * 3 + ch] * Y[k];
        rgb[ch] = acc;
    }
}

template <typename Real>
int project_all(const orc_camera* cam_in, int32_t n, const double* means, const double* scales,
                const double* quats, const double* opacity, const double* sh, int32_t sh_degree,
                const double* colors, double* means2d, double* depth, double* conic,
                double* color, int32_t* radius, int32_t* rect, uint32_t* tiles_touched,
                double margin, uint8_t* ambig) {
    (void)opacity;
    const Cam<Real> cam = cam_as<Real>(cam_in);
    const int Kc = sh_degree >= 0 ? (sh_degree + 1) * (sh_degree + 1) : 0;
    std::vector<Real> coef(size_t(3 * std::max(Kc, 1)));
    for (int32_t i = 0; i < n; ++i) {
        Real m[3], s[3], q[4];
        for (int k = 0; k < 3; ++k) m[k] = Real(means[size_t(k) * n + i]);
        for (int k = 0; k < 3; ++k) s[k] = Real(scales[size_t(k) * n + i]);
        for (int k = 0; k < 4; ++k) q[k] = Real(quats[size_t(k) * n + i]);
        const Proj<Real> P = project_one(cam, m, s, q, margin);
        if (ambig) ambig[i] = P.amb;
        if (!P.visible) {
            means2d[i] = means2d[size_t(n) + i] = 0;
            depth[i] = 0;
            for (int k = 0; k < 3; ++k) conic[size_t(k) * n + i] = color[size_t(k) * n + i] = 0;
            radius[i] = 0;
            for (int k = 0; k < 4; ++k) rect[size_t(k) * n + i] = 0;
            tiles_touched[i] = 0;
            continue;
        }
        means2d[i] = double(P.u);
        means2d[size_t(n) + i] = double(P.v);
        depth[i] = double(P.p[2]);
        for (int k = 0; k < 3; ++k) conic[size_t(k) * n + i] = double(P.conic[k]);
        radius[i] = P.radius;
        for (int k = 0; k < 4; ++k) rect[size_t(k) * n + i] = P.rect[k];
        tiles_touched[i] = P.tiles;
        Real rgb[3];
        if (sh_degree >= 0) {
            for (int k = 0; k < 3 * Kc; ++k) coef[size_t(k)] = Real(sh[size_t(k) * n + i]);
            sh_colour(cam, m, coef.data(), sh_degree, rgb, (Real*)nullptr);
        } else {
            for (int k = 0; k < 3; ++k) rgb[k] = Real(colors[size_t(k) * n + i]);
        }
        for (int k = 0; k < 3; ++k) color[size_t(k) * n + i] = double(rgb[k]);
    }
    return 0;
}


// c3: front-to-back compositing of one pixel ([rigel] Rasterization; [viewer] 4.5.4-4.5.5;
// [tiles] constants): power = -1/2 (A dx^2 + C dy^2) - B dx dy, alpha = min(0.99, o exp(power)),
// skip alpha < 1/255, composite C += c alpha T, T *= 1 - alpha, then stop once T < 1e-4.
// The pixel is sampled at its integer coordinates (px, py).  n counts every list entry the pixel
// examined, skipped ones included, and the entry that made it stop.
template <typename Real>
void composite_pixel(int px, int py, const uint32_t* list, uint32_t start, uint32_t end,
                     int32_t n, const double* means2d, const double* conic,
                     const double* opacity, const double* color, const double* bg,
                     double margin, double* out_rgb, double* out_T, uint32_t* out_n,
                     uint8_t* out_amb, uint32_t* out_blend) {
    Real T = 1;
    Real C[3] = {0, 0, 0};
    uint32_t cnt = 0, blended = 0;
    uint8_t amb = 0;
    for (uint32_t j = start; j < end; ++j) {
        const uint32_t g = list[j];
        ++cnt;
        const Real dx = Real(px) - Real(means2d[g]);
        const Real dy = Real(py) - Real(means2d[size_t(n) + g]);
        const Real A = Real(conic[g]), B = Real(conic[size_t(n) + g]), Cc = Real(conic[2 * size_t(n) + g]);
        const Real power = Real(-0.5) * (A * dx * dx + Cc * dy * dy) - B * dx * dy;
        const Real raw = Real(opacity[g]) * std::exp(power);
        const Real alpha = std::min(K<Real>::alpha_max(), raw);
        if (margin > 0) {
            if (near_rel(double(alpha), 1.0 / 255.0, margin)) amb |= ORC_AMB_ALPHA_MIN;
            if (near_rel(double(raw), 0.99, margin)) amb |= ORC_AMB_ALPHA_MAX;
        }
        if (alpha < K<Real>::alpha_min()) continue;
        ++blended;
        for (int ch = 0; ch < 3; ++ch) C[ch] += Real(color[size_t(ch) * n + g]) * alpha * T;
        T = T * (Real(1) - alpha);
        if (margin > 0 && near_rel(double(T), 1e-4, margin)) amb |= ORC_AMB_T_STOP;
        if (T < K<Real>::t_stop()) break;
    }
    for (int ch = 0; ch < 3; ++ch) out_rgb[ch] = double(C[ch] + T * Real(bg[ch]));
    *out_T = double(T);
    *out_n = cnt;
    *out_amb = amb;
    *out_blend = blended;
}

template <typename Real>
int raster_fwd(const orc_camera* cam, int32_t n, const double* means2d, const double* conic,
               const double* opacity, const double* color, const uint32_t* ranges,
               const uint32_t* list, const double* bg, const uint8_t* tile_mask, double* image,
               double* final_T, uint32_t* n_contrib, double margin, uint8_t* ambig,
               uint32_t* n_blend) {
    const int W = cam->width, H = cam->height;
    const int TX = (W + TILE - 1) / TILE, TY = (H + TILE - 1) / TILE;
    const size_t HW = size_t(W) * size_t(H);
    for (int ty = 0; ty < TY; ++ty)
        for (int tx = 0; tx < TX; ++tx) {
            const int t = ty * TX + tx;
            if (tile_mask && !tile_mask[t]) continue;
            const uint32_t start = ranges[2 * size_t(t)], end = ranges[2 * size_t(t) + 1];
            for (int py = ty * TILE; py < std::min(H, (ty + 1) * TILE); ++py)
                for (int px = tx * TILE; px < std::min(W, (tx + 1) * TILE); ++px) {
                    const size_t pix = size_t(py) * W + px;
                    double rgb[3], Tf;
                    uint32_t cnt, blended;
                    uint8_t amb;
                    composite_pixel<Real>(px, py, list, start, end, n, means2d, conic, opacity,
                                          color, bg, margin, rgb, &Tf, &cnt, &amb, &blended);
                    if (n_blend) n_blend[pix] = blended;
                    for (int ch = 0; ch < 3; ++ch) image[size_t(ch) * HW + pix] = rgb[ch];
                    final_T[pix] = Tf;
                    n_contrib[pix] = cnt;
                    if (ambig) ambig[pix] = amb;
                }
        }
    return 0;
}

// c4: backward of the compositing, from its definition ([rigel] Backward):
//   C = sum_i c_i a_i T_i + T_final bg,  T_i = prod_{k<i} (1 - a_k),
//   dC/dc_j = a_j T_j,
//   dC/da_j = c_j T_j - (sum_{i>j} c_i a_i T_i + T_final bg) / (1 - a_j).
// The pixel's first n_contrib entries are re-evaluated front to back (transmittances as forward
// products, not by division), then the suffix sums run back to front.  Skipped entries
// (alpha < 1/255) carry no gradient; an entry whose o exp(power) exceeds 0.99 was clamped and
// passes no gradient to its opacity, conic or mean ([rigel] Deliberate differences).
struct Reached {
    uint32_t g;
    double alpha, T, G, raw, dx, dy;
};

int raster_bwd(const orc_camera* cam, int32_t n, const double* means2d, const double* conic,
               const double* opacity, const double* color, const uint32_t* ranges,
               const uint32_t* list, const double* bg, const uint32_t* n_contrib,
               const double* dL_dimage, const uint8_t* tile_mask, double* dmeans2d,
               double* dconic, double* dopacity, double* dcolor, double* absum) {
    const int W = cam->width, H = cam->height;
    const int TX = (W + TILE - 1) / TILE, TY = (H + TILE - 1) / TILE;
    const size_t HW = size_t(W) * size_t(H);
    std::vector<Reached> seq;
    for (int ty = 0; ty < TY; ++ty)
        for (int tx = 0; tx < TX; ++tx) {
            const int t = ty * TX + tx;
            if (tile_mask && !tile_mask[t]) continue;
            const uint32_t start = ranges[2 * size_t(t)];
            for (int py = ty * TILE; py < std::min(H, (ty + 1) * TILE); ++py)
                for (int px = tx * TILE; px < std::min(W, (tx + 1) * TILE); ++px) {
                    const size_t pix = size_t(py) * W + px;
                    const uint32_t cnt = n_contrib[pix];
                    seq.clear();
                    double T = 1.0;
                    for (uint32_t j = start; j < start + cnt; ++j) {
                        const uint32_t g = list[j];
                        Reached r;
                        r.g = g;
                        r.dx = double(px) - means2d[g];
                        r.dy = double(py) - means2d[size_t(n) + g];
                        const double A = conic[g], B = conic[size_t(n) + g], Cc = conic[2 * size_t(n) + g];
                        const double power = -0.5 * (A * r.dx * r.dx + Cc * r.dy * r.dy) - B * r.dx * r.dy;
                        r.G = std::exp(power);
                        r.raw = opacity[g] * r.G;
                        r.alpha = std::min(0.99, r.raw);
                        if (r.alpha < 1.0 / 255.0) continue;
                        r.T = T;
                        seq.push_back(r);
                        T *= 1.0 - r.alpha;
                    }
                    const double Tfinal = T;
                    double dLdC[3];
                    for (int ch = 0; ch < 3; ++ch) dLdC[ch] = dL_dimage[size_t(ch) * HW + pix];
                    double S[3] = {Tfinal * bg[0], Tfinal * bg[1], Tfinal * bg[2]};
                    for (size_t k = seq.size(); k-- > 0;) {
                        const Reached& r = seq[k];
                        const uint32_t g = r.g;
                        double dalpha = 0, dalpha_mag = 0;
                        for (int ch = 0; ch < 3; ++ch) {
                            const double c = color[size_t(ch) * n + g];
                            dcolor[size_t(ch) * n + g] += r.alpha * r.T * dLdC[ch];
                            dalpha += dLdC[ch] * (c * r.T - S[ch] / (1.0 - r.alpha));
                            dalpha_mag += std::fabs(dLdC[ch]) * (std::fabs(c * r.T) + std::fabs(S[ch] / (1.0 - r.alpha)));
                            if (absum) absum[(6 + size_t(ch)) * n + g] += std::fabs(r.alpha * r.T * dLdC[ch]);
                        }
                        for (int ch = 0; ch < 3; ++ch) S[ch] += color[size_t(ch) * n + g] * r.alpha * r.T;
                        if (r.raw > 0.99) continue;  // clamped: alpha is the constant 0.99
                        // alpha = o G, G = exp(power)
                        dopacity[g] += r.G * dalpha;
                        const double gp = opacity[g] * r.G * dalpha;  // dL/dpower
                        const double A = conic[g], B = conic[size_t(n) + g], Cc = conic[2 * size_t(n) + g];
                        dconic[g] += -0.5 * r.dx * r.dx * gp;
                        dconic[size_t(n) + g] += -r.dx * r.dy * gp;
                        dconic[2 * size_t(n) + g] += -0.5 * r.dy * r.dy * gp;
                        // dpower/du = -dpower/d(dx) = A dx + B dy
                        dmeans2d[g] += gp * (A * r.dx + B * r.dy);
                        dmeans2d[size_t(n) + g] += gp * (Cc * r.dy + B * r.dx);
                        if (absum) {
                            // magnitudes of what the sums above add (with dL/dalpha's own terms
                            // taken in absolute value): the scale of their rounding error
                            const double gm = opacity[g] * r.G * dalpha_mag;
                            absum[2 * size_t(n) + g] += 0.5 * r.dx * r.dx * gm;
                            absum[3 * size_t(n) + g] += std::fabs(r.dx * r.dy) * gm;
                            absum[4 * size_t(n) + g] += 0.5 * r.dy * r.dy * gm;
                            absum[g] += gm * (std::fabs(A * r.dx) + std::fabs(B * r.dy));
                            absum[size_t(n) + g] += gm * (std::fabs(Cc * r.dy) + std::fabs(B * r.dx));
                            absum[5 * size_t(n) + g] += r.G * dalpha_mag;
                        }
                    }
                }
        }
    return 0;
}

// c2: binning from projected float data.  One entry per (visible Gaussian, covered tile), emitted
// in Gaussian index order, tile rows outer and columns inner ([viewer] 4.2; [tiles]
// build_tile_lists); key = (tile_id << 32) | float_bits(depth) ([rigel] Binning); a stable
// ascending sort by key (equal keys keep index order); per-tile [start, end) ranges with
// (0, 0) for empty tiles ([viewer] 4.4.2).
struct Entry {
    uint64_t key;
    uint32_t value;
};

void entries_of(const orc_camera* cam, int32_t n, const float* means2d, const float* depth,
                const int32_t* radius, std::vector<Entry>* out, uint32_t* tiles_touched) {
    const int W = cam->width, H = cam->height;
    const int TX = (W + TILE - 1) / TILE, TY = (H + TILE - 1) / TILE;
    for (int32_t i = 0; i < n; ++i) {
        uint32_t cnt = 0;
        if (radius[i] > 0) {
            const float u = means2d[i], v = means2d[size_t(n) + i], r = float(radius[i]);
            const int xl = span_lo<float>(u, r, TX), xh = span_hi<float>(u, r, TX);
            const int yl = span_lo<float>(v, r, TY), yh = span_hi<float>(v, r, TY);
            for (int ty = yl; ty < yh; ++ty)
                for (int tx = xl; tx < xh; ++tx) {
                    ++cnt;
                    if (out) {
                        uint32_t bits;
                        std::memcpy(&bits, &depth[i], 4);
                        const uint64_t tile = uint64_t(ty) * uint64_t(TX) + uint64_t(tx);
                        out->push_back(Entry{(tile << 32) | uint64_t(bits), uint32_t(i)});
                    }
                }
        }
        if (tiles_touched) tiles_touched[i] = cnt;
    }
}

// c5: reverse mode through c1 and c6 ([rigel] Backward, second paragraph; [rigel] Deliberate
// differences: the quaternion gradient is projected off the radial direction).
void project_bwd_one(const Cam<double>& cam, const double* m, const double* s, const double* q,
                     const double* coef, int degree, const double* dm2, const double* dcon,
                     const double* dcol, double* dm, double* ds, double* dq, double* dcoef) {
    const Proj<double> P = project_one<double>(cam, m, s, q, 0.0);
    for (int k = 0; k < 3; ++k) dm[k] = ds[k] = 0;
    for (int k = 0; k < 4; ++k) dq[k] = 0;
    if (!P.visible) {
        if (dcoef)
            for (int k = 0; k < 3 * (degree + 1) * (degree + 1); ++k) dcoef[k] = 0;
        return;
    }
    const double a = P.a, b = P.b, c = P.c, det = P.det, d2 = det * det;
    // conic = (c, -b, a) / det
    const double gA = dcon[0], gB = dcon[1], gC = dcon[2];
    const double ga = gA * (-c * c / d2) + gB * (b * c / d2) + gC * (-b * b / d2);
    const double gb = gA * (2 * b * c / d2) + gB * (-1.0 / det - 2 * b * b / d2) + gC * (2 * a * b / d2);
    const double gc = gA * (-b * b / d2) + gB * (a * b / d2) + gC * (-a * a / d2);
    // Sigma_2d = T Sigma_3d T^T; G2 = dL/dSigma_2d as a symmetric matrix
    const double G2[4] = {ga, 0.5 * gb, 0.5 * gb, gc};
    double TS[6];  // T Sigma_3d
    for (int i = 0; i < 2; ++i)
        for (int j = 0; j < 3; ++j)
            TS[i * 3 + j] = P.T[i * 3 + 0] * P.S3[0 * 3 + j] + P.T[i * 3 + 1] * P.S3[1 * 3 + j] + P.T[i * 3 + 2] * P.S3[2 * 3 + j];
    double dT[6];  // 2 G2 T Sigma_3d
    for (int i = 0; i < 2; ++i)
        for (int j = 0; j < 3; ++j) dT[i * 3 + j] = 2 * (G2[i * 2 + 0] * TS[0 * 3 + j] + G2[i * 2 + 1] * TS[1 * 3 + j]);
    double dS3[9];  // T^T G2 T
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 3; ++j) {
            double acc = 0;
            for (int k = 0; k < 2; ++k)
                for (int l = 0; l < 2; ++l) acc += P.T[k * 3 + i] * G2[k * 2 + l] * P.T[l * 3 + j];
            dS3[i * 3 + j] = acc;
        }
    // T = J W  ->  dJ = dT W^T
    double dJ[6];
    for (int i = 0; i < 2; ++i)
        for (int k = 0; k < 3; ++k)
            dJ[i * 3 + k] = dT[i * 3 + 0] * cam.R[k * 3 + 0] + dT[i * 3 + 1] * cam.R[k * 3 + 1] + dT[i * 3 + 2] * cam.R[k * 3 + 2];
    const double x = P.p[0], y = P.p[1], z = P.p[2];
    double dp[3] = {0, 0, 0};
    // J = [[fx/z, 0, -fx tx/z^2], [0, fy/z, -fy ty/z^2]]
    dp[2] += dJ[0] * (-cam.fx / (z * z)) + dJ[2] * (2 * cam.fx * P.tx / (z * z * z)) +
             dJ[4] * (-cam.fy / (z * z)) + dJ[5] * (2 * cam.fy * P.ty / (z * z * z));
    const double dtx = dJ[2] * (-cam.fx / (z * z));
    const double dty = dJ[5] * (-cam.fy / (z * z));
    // tx = z clamp(x/z): the clamped branch sends the gradient to z
    if (P.clamp_x) dp[2] += dtx * (P.tx / z); else dp[0] += dtx;
    if (P.clamp_y) dp[2] += dty * (P.ty / z); else dp[1] += dty;
    // u = fx x / z + cx, v = fy y / z + cy
    dp[0] += dm2[0] * cam.fx / z;
    dp[2] += -dm2[0] * cam.fx * x / (z * z);
    dp[1] += dm2[1] * cam.fy / z;
    dp[2] += -dm2[1] * cam.fy * y / (z * z);
    // p = R m + t
    for (int j = 0; j < 3; ++j) dm[j] = cam.R[0 * 3 + j] * dp[0] + cam.R[1 * 3 + j] * dp[1] + cam.R[2 * 3 + j] * dp[2];
    // Sigma_3d = M M^T, M = Rq diag(s)
    double M[9];
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 3; ++j) M[i * 3 + j] = P.Rq[i * 3 + j] * s[j];
    double dM[9];
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 3; ++j)
            dM[i * 3 + j] = 2 * (dS3[i * 3 + 0] * M[0 * 3 + j] + dS3[i * 3 + 1] * M[1 * 3 + j] + dS3[i * 3 + 2] * M[2 * 3 + j]);
    double dRq[9];
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 3; ++j) dRq[i * 3 + j] = dM[i * 3 + j] * s[j];
    for (int j = 0; j < 3; ++j) ds[j] = dM[0 * 3 + j] * P.Rq[0 * 3 + j] + dM[1 * 3 + j] * P.Rq[1 * 3 + j] + dM[2 * 3 + j] * P.Rq[2 * 3 + j];
    // rotation matrix entries as functions of the unit quaternion (w, x, y, z)
    const double w = P.qhat[0], qx = P.qhat[1], qy = P.qhat[2], qz = P.qhat[3];
    const double dR_dw[9] = {0, -2 * qz, 2 * qy, 2 * qz, 0, -2 * qx, -2 * qy, 2 * qx, 0};
    const double dR_dx[9] = {0, 2 * qy, 2 * qz, 2 * qy, -4 * qx, -2 * w, 2 * qz, 2 * w, -4 * qx};
    const double dR_dy[9] = {-4 * qy, 2 * qx, 2 * w, 2 * qx, 0, 2 * qz, -2 * w, 2 * qz, -4 * qy};
    const double dR_dz[9] = {-4 * qz, -2 * w, 2 * qx, 2 * w, -4 * qz, 2 * qy, 2 * qx, 2 * qy, 0};
    double dqhat[4] = {0, 0, 0, 0};
    for (int k = 0; k < 9; ++k) {
        dqhat[0] += dRq[k] * dR_dw[k];
        dqhat[1] += dRq[k] * dR_dx[k];
        dqhat[2] += dRq[k] * dR_dy[k];
        dqhat[3] += dRq[k] * dR_dz[k];
    }
    // qhat = q / |q|
    const double dot = dqhat[0] * P.qhat[0] + dqhat[1] * P.qhat[1] + dqhat[2] * P.qhat[2] + dqhat[3] * P.qhat[3];
    for (int k = 0; k < 4; ++k) dq[k] = (dqhat[k] - P.qhat[k] * dot) / P.qn;
    // colour from SH: colour_ch = sum_k coef[k*3+ch] Y_k(d), d = (m - C)/|m - C|
    if (degree >= 0 && dcoef) {
        double C[3];
        camera_centre(cam, C);
        const double vv[3] = {m[0] - C[0], m[1] - C[1], m[2] - C[2]};
        const double len = std::sqrt(vv[0] * vv[0] + vv[1] * vv[1] + vv[2] * vv[2]);
        const double d[3] = {vv[0] / len, vv[1] / len, vv[2] / len};
        double Y[16], GY[16][3];
        sh_basis(d[0], d[1], d[2], Y);
        sh_basis_grad(d[0], d[1], d[2], GY);
        const int Kc = (degree + 1) * (degree + 1);
        double dd[3] = {0, 0, 0};
        for (int k = 0; k < Kc; ++k)
            for (int ch = 0; ch < 3; ++ch) {
                dcoef[k * 3 + ch] = dcol[ch] * Y[k];
                for (int e = 0; e < 3; ++e) dd[e] += dcol[ch] * coef[k * 3 + ch] * GY[k][e];
            }
        const double ddot = dd[0] * d[0] + dd[1] * d[1] + dd[2] * d[2];
        for (int e = 0; e < 3; ++e) dm[e] += (dd[e] - d[e] * ddot) / len;
    }
}

// c7: the appearance MLP of [rigel] Appearance MLP: per Gaussian an L-float latent concatenated
// with the unit view direction, one ReLU hidden layer, a 3-wide sigmoid output.  The view
// direction is a constant of the backward.
void view_dir(const Cam<double>& cam, const double* m, double* d) {
    double C[3];
    camera_centre(cam, C);
    double v[3] = {m[0] - C[0], m[1] - C[1], m[2] - C[2]};
    const double len = std::sqrt(v[0] * v[0] + v[1] * v[1] + v[2] * v[2]);
    for (int k = 0; k < 3; ++k) d[k] = len > 0 ? v[k] / len : 0.0;
}

}  // namespace

// c2': the ellipse-tile test of the pages' "next" list ([viewer] 2.3.4, footnote 3, names a
// tighter test than the bounding square; the reading taken here is the exact one), stated from
// its definition in double precision.
// The region where a splat can reach alpha >= 1/255 is the ellipse q(d) = d^T Q d <= k, with Q
// the conic ((A, B), (B, C)), d = pixel - mean and k = 2.002 ln(255 o) as given (0.1% wider than
// the exact 2 ln(255 o)).  A tile of the splat's radius square is kept when its pixel-centre
// square [16 tx, 16 tx + 15] x [16 ty, 16 ty + 15] holds a point of that region, i.e. when the
// minimum of q over the square is at most k.

// Minimum of the positive-definite quadratic q(x, y) = A x^2 + 2 B x y + C y^2 over the
// rectangle [x0, x1] x [y0, y1].  If the rectangle holds the origin (q's minimum) it is 0.
// Otherwise the convex q attains its minimum over the rectangle on the boundary; along an edge
// it is a one-variable parabola, smallest at its vertex or, when the vertex is off the edge, at
// the nearer end.
static double quad_min_rect(double A, double B, double C, double x0, double x1, double y0, double y1) {
    if (x0 <= 0.0 && 0.0 <= x1 && y0 <= 0.0 && 0.0 <= y1) return 0.0;
    auto q = [&](double x, double y) { return A * x * x + 2.0 * B * x * y + C * y * y; };
    double best = HUGE_VAL;
    for (double x : {x0, x1}) {  // vertical edge: C y^2 + 2 B x y + A x^2, vertex y = -B x / C
        const double y = std::min(std::max(-B * x / C, y0), y1);
        best = std::min(best, q(x, y));
    }
    for (double y : {y0, y1}) {  // horizontal edge: vertex x = -B y / A
        const double x = std::min(std::max(-B * y / A, x0), x1);
        best = std::min(best, q(x, y));
    }
    return best;
}

// The decision for tile (tx, ty) and whether it is a knife edge.  The test is exact only up to
// rounding in any implementation, so a decision is flagged as ambiguous -- either outcome
// correct -- when it is not clear at a margin: kept for certain needs the minimum over the
// square at most k (1 - margin); dropped for certain needs the minimum over the square widened
// by `widen` pixels on every side above k (1 + margin).
constexpr uint8_t ELL_KEEP = 1, ELL_AMBIG = 2;
static uint8_t ellipse_tile_decision(double u, double v, double A, double B, double C, double k, int tx, int ty,
                              double widen, double margin) {
    if (!(k > 0.0) || !(A > 0.0) || !(C > 0.0) || !(A * C - B * B > 0.0)) return 0;
    const double x0 = TILE * tx - u, x1 = TILE * tx + (TILE - 1) - u;
    const double y0 = TILE * ty - v, y1 = TILE * ty + (TILE - 1) - v;
    const double m = quad_min_rect(A, B, C, x0, x1, y0, y1);
    const double mw = quad_min_rect(A, B, C, x0 - widen, x1 + widen, y0 - widen, y1 + widen);
    const bool keep = m <= k;
    const bool sure_keep = m <= k * (1.0 - margin);
    const bool sure_drop = mw > k * (1.0 + margin);
    return uint8_t((keep ? ELL_KEEP : 0) | (!sure_keep && !sure_drop ? ELL_AMBIG : 0));
}

extern "C" {

int orc_project(int prec, const orc_camera* cam, int32_t n, const double* means,
                const double* scales, const double* quats, const double* opacity,
                const double* sh, int32_t sh_degree, const double* colors, double* means2d,
                double* depth, double* conic, double* color, int32_t* radius, int32_t* rect,
                uint32_t* tiles_touched, double margin, uint8_t* ambig) {
    if (!cam || n < 0 || sh_degree < -1 || sh_degree > 3) return -1;
    if (sh_degree >= 0 && !sh) return -1;
    if (sh_degree < 0 && !colors) return -1;
    if (prec == 32)
        return project_all<float>(cam, n, means, scales, quats, opacity, sh, sh_degree, colors,
                                  means2d, depth, conic, color, radius, rect, tiles_touched,
                                  margin, ambig);
    if (prec == 64)
        return project_all<double>(cam, n, means, scales, quats, opacity, sh, sh_degree, colors,
                                   means2d, depth, conic, color, radius, rect, tiles_touched,
                                   margin, ambig);
    return -1;
}

void orc_project_intermediates(const orc_camera* cam_in, int32_t n, const double* means,
                               const double* scales, const double* quats, double* cov3d,
                               double* cov2d, double* jac, double* pcam) {
    const Cam<double> cam = cam_as<double>(cam_in);
    for (int32_t i = 0; i < n; ++i) {
        double m[3], s[3], q[4];
        for (int k = 0; k < 3; ++k) m[k] = means[size_t(k) * n + i];
        for (int k = 0; k < 3; ++k) s[k] = scales[size_t(k) * n + i];
        for (int k = 0; k < 4; ++k) q[k] = quats[size_t(k) * n + i];
        const Proj<double> P = project_one<double>(cam, m, s, q, 0.0);
        const int sym[6] = {0, 1, 2, 4, 5, 8};
        for (int k = 0; k < 6; ++k) cov3d[size_t(k) * n + i] = P.S3[sym[k]];
        cov2d[i] = P.a;
        cov2d[size_t(n) + i] = P.b;
        cov2d[2 * size_t(n) + i] = P.c;
        for (int k = 0; k < 6; ++k) jac[size_t(k) * n + i] = P.J[k];
        for (int k = 0; k < 3; ++k) pcam[size_t(k) * n + i] = P.p[k];
    }
}

void orc_sh_basis(const double* dirs, int32_t m, double* Y) {
    for (int32_t i = 0; i < m; ++i) {
        double y[16];
        sh_basis<double>(dirs[i], dirs[size_t(m) + i], dirs[2 * size_t(m) + i], y);
        for (int k = 0; k < 16; ++k) Y[size_t(k) * m + i] = y[k];
    }
}

// [viewer] 4.1.1: exclusive scan, each element the sum of those before it.
uint64_t orc_exclusive_scan_u32(const uint32_t* in, int64_t n, uint64_t* out) {
    uint64_t run = 0;
    for (int64_t i = 0; i < n; ++i) {
        out[i] = run;
        run += in[i];
    }
    return run;
}

// [viewer] 4.4.1-4.4.2: a tile's range starts where the tile id differs from the previous
// entry's and ends after the last entry carrying it; tiles absent from the list keep (0, 0).
void orc_tile_ranges(const uint64_t* keys_sorted, int64_t n_entries, int32_t n_tiles,
                     uint32_t* ranges) {
    for (int32_t t = 0; t < n_tiles; ++t) ranges[2 * size_t(t)] = ranges[2 * size_t(t) + 1] = 0;
    for (int64_t e = 0; e < n_entries; ++e) {
        const uint64_t tile = keys_sorted[e] >> 32;
        if (e == 0 || (keys_sorted[e - 1] >> 32) != tile) ranges[2 * tile] = uint32_t(e);
        if (e == n_entries - 1 || (keys_sorted[e + 1] >> 32) != tile) ranges[2 * tile + 1] = uint32_t(e + 1);
    }
}

int64_t orc_bin_count(const orc_camera* cam, int32_t n, const float* means2d,
                      const int32_t* radius) {
    std::vector<uint32_t> tt(size_t(std::max(n, 1)));
    entries_of(cam, n, means2d, nullptr, radius, nullptr, tt.data());
    std::vector<uint64_t> off(size_t(std::max(n, 1)));
    return int64_t(orc_exclusive_scan_u32(tt.data(), n, off.data()));
}

int64_t orc_bin(const orc_camera* cam, int32_t n, const float* means2d, const float* depth,
                const int32_t* radius, int64_t capacity, uint64_t* keys_sorted,
                uint32_t* point_list, uint32_t* ranges, uint32_t* tiles_touched) {
    std::vector<Entry> ent;
    entries_of(cam, n, means2d, depth, radius, &ent, tiles_touched);
    const int64_t E = int64_t(ent.size());
    if (E > capacity) return -2;
    std::stable_sort(ent.begin(), ent.end(),
                     [](const Entry& a, const Entry& b) { return a.key < b.key; });
    for (int64_t e = 0; e < E; ++e) {
        if (keys_sorted) keys_sorted[e] = ent[size_t(e)].key;
        point_list[e] = ent[size_t(e)].value;
    }
    std::vector<uint64_t> ks(static_cast<size_t>(E));
    for (int64_t e = 0; e < E; ++e) ks[size_t(e)] = ent[size_t(e)].key;
    const int TX = (cam->width + TILE - 1) / TILE, TY = (cam->height + TILE - 1) / TILE;
    orc_tile_ranges(ks.data(), E, TX * TY, ranges);
    return E;
}

int orc_raster_fwd(int prec, const orc_camera* cam, int32_t n, const double* means2d,
                   const double* conic, const double* opacity, const double* color,
                   const uint32_t* ranges, const uint32_t* point_list, const double* bg,
                   const uint8_t* tile_mask, double* image, double* final_T,
                   uint32_t* n_contrib, double margin, uint8_t* ambig, uint32_t* n_blend) {
    if (!cam || n < 0) return -1;
    if (prec == 32)
        return raster_fwd<float>(cam, n, means2d, conic, opacity, color, ranges, point_list, bg,
                                 tile_mask, image, final_T, n_contrib, margin, ambig, n_blend);
    if (prec == 64)
        return raster_fwd<double>(cam, n, means2d, conic, opacity, color, ranges, point_list, bg,
                                  tile_mask, image, final_T, n_contrib, margin, ambig, n_blend);
    return -1;
}

int orc_raster_bwd(const orc_camera* cam, int32_t n, const double* means2d,
                   const double* conic, const double* opacity, const double* color,
                   const uint32_t* ranges, const uint32_t* point_list, const double* bg,
                   const uint32_t* n_contrib, const double* dL_dimage,
                   const uint8_t* tile_mask, double* dmeans2d, double* dconic,
                   double* dopacity, double* dcolor, double* absum) {
    if (!cam || n < 0) return -1;
    return raster_bwd(cam, n, means2d, conic, opacity, color, ranges, point_list, bg, n_contrib,
                      dL_dimage, tile_mask, dmeans2d, dconic, dopacity, dcolor, absum);
}

int orc_project_bwd(const orc_camera* cam_in, int32_t n, const double* means,
                    const double* scales, const double* quats, const double* sh,
                    int32_t sh_degree, const int32_t* radius, const double* dmeans2d,
                    const double* dconic, const double* dcolor, double* dmeans,
                    double* dscales, double* dquats, double* dsh) {
    if (!cam_in || n < 0 || sh_degree < -1 || sh_degree > 3) return -1;
    const Cam<double> cam = cam_as<double>(cam_in);
    const int Kc = sh_degree >= 0 ? (sh_degree + 1) * (sh_degree + 1) : 0;
    std::vector<double> coef(size_t(3 * std::max(Kc, 1))), dcoef(size_t(3 * std::max(Kc, 1)));
    for (int32_t i = 0; i < n; ++i) {
        double m[3], s[3], q[4], dm2[2], dcon[3], dcol[3], dm[3], ds[3], dq[4];
        for (int k = 0; k < 3; ++k) m[k] = means[size_t(k) * n + i];
        for (int k = 0; k < 3; ++k) s[k] = scales[size_t(k) * n + i];
        for (int k = 0; k < 4; ++k) q[k] = quats[size_t(k) * n + i];
        for (int k = 0; k < 2; ++k) dm2[k] = dmeans2d[size_t(k) * n + i];
        for (int k = 0; k < 3; ++k) dcon[k] = dconic[size_t(k) * n + i];
        for (int k = 0; k < 3; ++k) dcol[k] = dcolor[size_t(k) * n + i];
        for (int k = 0; k < 3 * Kc; ++k) coef[size_t(k)] = sh[size_t(k) * n + i];
        const bool culled = radius && radius[i] == 0;
        if (culled) {
            for (int k = 0; k < 3; ++k) dm[k] = ds[k] = 0;
            for (int k = 0; k < 4; ++k) dq[k] = 0;
            for (int k = 0; k < 3 * Kc; ++k) dcoef[size_t(k)] = 0;
        } else {
            project_bwd_one(cam, m, s, q, coef.data(), sh_degree, dm2, dcon, dcol, dm, ds, dq,
                            sh_degree >= 0 ? dcoef.data() : nullptr);
        }
        for (int k = 0; k < 3; ++k) dmeans[size_t(k) * n + i] = dm[k];
        for (int k = 0; k < 3; ++k) dscales[size_t(k) * n + i] = ds[k];
        for (int k = 0; k < 4; ++k) dquats[size_t(k) * n + i] = dq[k];
        if (dsh && sh_degree >= 0)
            for (int k = 0; k < 3 * Kc; ++k) dsh[size_t(k) * n + i] = dcoef[size_t(k)];
    }
    return 0;
}

int orc_appearance_fwd(const orc_camera* cam_in, int32_t n, int32_t L, int32_t H,
                       const double* means, const double* latents, const double* W1,
                       const double* b1, const double* W2, const double* b2, double* colors) {
    if (!cam_in || n < 0 || L < 0 || H <= 0) return -1;
    const Cam<double> cam = cam_as<double>(cam_in);
    const int D = L + 3;
    std::vector<double> x(static_cast<size_t>(D)), h(static_cast<size_t>(H));
    for (int32_t i = 0; i < n; ++i) {
        double m[3] = {means[i], means[size_t(n) + i], means[2 * size_t(n) + i]};
        for (int k = 0; k < L; ++k) x[size_t(k)] = latents[size_t(k) * n + i];
        view_dir(cam, m, &x[size_t(L)]);
        for (int j = 0; j < H; ++j) {
            double acc = b1[j];
            for (int k = 0; k < D; ++k) acc += W1[size_t(j) * D + k] * x[size_t(k)];
            h[size_t(j)] = acc > 0 ? acc : 0.0;
        }
        for (int c = 0; c < 3; ++c) {
            double acc = b2[c];
            for (int j = 0; j < H; ++j) acc += W2[size_t(c) * H + j] * h[size_t(j)];
            colors[size_t(c) * n + i] = 1.0 / (1.0 + std::exp(-acc));
        }
    }
    return 0;
}

int orc_appearance_bwd(const orc_camera* cam_in, int32_t n, int32_t L, int32_t H,
                       const double* means, const double* latents, const double* W1,
                       const double* b1, const double* W2, const double* b2,
                       const double* dcolors, double* dlatents, double* dW1, double* db1,
                       double* dW2, double* db2) {
    if (!cam_in || n < 0 || L < 0 || H <= 0) return -1;
    const Cam<double> cam = cam_as<double>(cam_in);
    const int D = L + 3;
    std::vector<double> x(static_cast<size_t>(D)), z1(static_cast<size_t>(H)), h(static_cast<size_t>(H)), dh(static_cast<size_t>(H));
    for (int j = 0; j < H * D; ++j) dW1[j] = 0;
    for (int j = 0; j < H; ++j) db1[j] = 0;
    for (int j = 0; j < 3 * H; ++j) dW2[j] = 0;
    for (int j = 0; j < 3; ++j) db2[j] = 0;
    for (int32_t i = 0; i < n; ++i) {
        double m[3] = {means[i], means[size_t(n) + i], means[2 * size_t(n) + i]};
        for (int k = 0; k < L; ++k) x[size_t(k)] = latents[size_t(k) * n + i];
        view_dir(cam, m, &x[size_t(L)]);
        for (int j = 0; j < H; ++j) {
            double acc = b1[j];
            for (int k = 0; k < D; ++k) acc += W1[size_t(j) * D + k] * x[size_t(k)];
            z1[size_t(j)] = acc;
            h[size_t(j)] = acc > 0 ? acc : 0.0;
        }
        double dz2[3];
        for (int c = 0; c < 3; ++c) {
            double acc = b2[c];
            for (int j = 0; j < H; ++j) acc += W2[size_t(c) * H + j] * h[size_t(j)];
            const double sg = 1.0 / (1.0 + std::exp(-acc));
            dz2[c] = dcolors[size_t(c) * n + i] * sg * (1.0 - sg);
        }
        for (int j = 0; j < H; ++j) {
            double acc = 0;
            for (int c = 0; c < 3; ++c) {
                dW2[size_t(c) * H + j] += dz2[c] * h[size_t(j)];
                acc += W2[size_t(c) * H + j] * dz2[c];
            }
            dh[size_t(j)] = z1[size_t(j)] > 0 ? acc : 0.0;  // relu'(0) = 0
        }
        for (int c = 0; c < 3; ++c) db2[c] += dz2[c];
        for (int k = 0; k < L; ++k) dlatents[size_t(k) * n + i] = 0;
        for (int j = 0; j < H; ++j) {
            db1[j] += dh[size_t(j)];
            for (int k = 0; k < D; ++k) {
                dW1[size_t(j) * D + k] += dh[size_t(j)] * x[size_t(k)];
                if (k < L) dlatents[size_t(k) * n + i] += W1[size_t(j) * D + k] * dh[size_t(j)];
            }
        }
    }
    return 0;
}


// c8: the L1 term of rigel's training loss (README, training: "L1 + D-SSIM"), the absolute error
// summed and scaled by `scale`, and its gradient, written from the definition: |d| and
// d|d|/dd = sign d, with the subgradient 0 taken at d = 0.
int orc_l1_loss_grad(int64_t count, const double* image, const double* target, double scale,
                     double* grad, double* loss) {
    if (count < 0) return -1;
    double acc = 0.0;
    for (int64_t i = 0; i < count; ++i) {
        const double d = image[i] - target[i];
        grad[i] = d > 0.0 ? scale : (d < 0.0 ? -scale : 0.0);
        acc += d < 0.0 ? -d : d;
    }
    if (loss) *loss = scale * acc;
    return 0;
}


// c9: Adam (Kingma & Ba, "Adam: A Method for Stochastic Optimization", Algorithm 1) with the
// bias corrections written as in the paper, one parameter at a time; the gradient of the raw
// parameter is the given gradient times the activation's derivative (rigel README: parameters
// are stored raw and activated in the model layer).
int orc_adam_step(int64_t count, double* param, const double* grad, double* m, double* v,
                  double* activated, double lr, int32_t activation, double beta1, double beta2,
                  double eps, int32_t step) {
    if (count < 0 || step < 1 || activation < 0 || activation > 2) return -1;
    const double c1 = 1.0 - std::pow(beta1, step), c2 = 1.0 - std::pow(beta2, step);
    for (int64_t i = 0; i < count; ++i) {
        double g = grad[i];
        if (activation == 1) g *= std::exp(param[i]);
        if (activation == 2) {
            const double a = 1.0 / (1.0 + std::exp(-param[i]));
            g *= a * (1.0 - a);
        }
        m[i] = beta1 * m[i] + (1.0 - beta1) * g;
        v[i] = beta2 * v[i] + (1.0 - beta2) * g * g;
        const double mhat = m[i] / c1, vhat = v[i] / c2;
        param[i] -= lr * mhat / (std::sqrt(vhat) + eps);
        if (activated) {
            activated[i] = activation == 1 ? std::exp(param[i])
                         : activation == 2 ? 1.0 / (1.0 + std::exp(-param[i])) : param[i];
        }
    }
    return 0;
}

// c10: the view-space gradient statistics that drive densification (rigel README,
// "densify/prune"): norm of dL/dmeans2d accumulated over the views where the Gaussian is visible.
int orc_densify_stats(int32_t n, const double* dmeans2d, const int32_t* radius, double* accum,
                      double* count) {
    if (n < 0) return -1;
    for (int32_t i = 0; i < n; ++i) {
        if (radius[i] <= 0) continue;
        const double gx = dmeans2d[i], gy = dmeans2d[size_t(n) + i];
        accum[i] += std::sqrt(gx * gx + gy * gy);
        count[i] += 1.0;
    }
    return 0;
}


// c11: L1 + D-SSIM, the photometric loss rigel's training uses ("L1 + D-SSIM"; the pages give no
// formula, so 3DGS's, after Wang et al., "Image quality assessment: from error visibility to
// structural similarity"): local means, variances and covariance under a normalised 11 x 11
// Gaussian window (sigma 1.5; pixels outside the image count as zero), SSIM per pixel, averaged.
// The window is applied directly in 2-D.  The gradient follows the chain rule through the five
// filtered maps: S depends on the pixel values only through mx = G*I, sxx' = G*I^2 and
// sxy' = G*(I T), whose derivatives w.r.t. I_q are G(p - q), 2 I_q G(p - q) and T_q G(p - q).
int orc_l1_dssim(int32_t C, int32_t H, int32_t W, const double* image, const double* target,
                 double lambda, double scale, double* grad, double* loss, double* ssim) {
    if (C < 1 || H < 1 || W < 1) return -1;
    const int R = 5;
    double G[11][11], sum = 0.0;
    for (int i = 0; i < 11; ++i)
        for (int j = 0; j < 11; ++j) {
            G[i][j] = std::exp(-double((i - R) * (i - R) + (j - R) * (j - R)) / (2.0 * 1.5 * 1.5));
            sum += G[i][j];
        }
    for (int i = 0; i < 11; ++i)
        for (int j = 0; j < 11; ++j) G[i][j] /= sum;
    const double C1 = 0.01 * 0.01, C2 = 0.03 * 0.03;
    const size_t plane = size_t(H) * W, N = size_t(C) * plane;
    std::vector<double> a(N), b(N), c(N);
    double sum_s = 0.0, sum_l1 = 0.0;
    for (int ch = 0; ch < C; ++ch) {
        const double* X = image + ch * plane;
        const double* Y = target + ch * plane;
        for (int y = 0; y < H; ++y)
            for (int x = 0; x < W; ++x) {
                double mx = 0, my = 0, xx = 0, yy = 0, xy = 0;
                for (int i = -R; i <= R; ++i)
                    for (int j = -R; j <= R; ++j) {
                        const int yy_ = y + i, xx_ = x + j;
                        if (yy_ < 0 || yy_ >= H || xx_ < 0 || xx_ >= W) continue;
                        const double w = G[i + R][j + R];
                        const double u = X[size_t(yy_) * W + xx_], v = Y[size_t(yy_) * W + xx_];
                        mx += w * u; my += w * v; xx += w * u * u; yy += w * v * v; xy += w * u * v;
                    }
                const double sx = xx - mx * mx, sy = yy - my * my, sxy = xy - mx * my;
                const double A1 = 2 * mx * my + C1, A2 = 2 * sxy + C2;
                const double B1 = mx * mx + my * my + C1, B2 = sx + sy + C2;
                const double S = A1 * A2 / (B1 * B2);
                const size_t o = ch * plane + size_t(y) * W + x;
                if (ssim) ssim[o] = S;
                sum_s += S;
                sum_l1 += std::fabs(X[size_t(y) * W + x] - Y[size_t(y) * W + x]);
                // dS/dmx, dS/d(G*I^2), dS/d(G*I T)
                a[o] = S * (2 * my / A1 - 2 * my / A2 - 2 * mx / B1 + 2 * mx / B2);
                b[o] = -S / B2;
                c[o] = 2 * S / A2;
            }
    }
    for (int ch = 0; ch < C; ++ch)
        for (int y = 0; y < H; ++y)
            for (int x = 0; x < W; ++x) {
                const size_t q = ch * plane + size_t(y) * W + x;
                const double u = image[q], v = target[q];
                double dS = 0;
                for (int i = -R; i <= R; ++i)
                    for (int j = -R; j <= R; ++j) {
                        const int py = y + i, px = x + j;  // pixel p whose window holds q
                        if (py < 0 || py >= H || px < 0 || px >= W) continue;
                        const size_t o = ch * plane + size_t(py) * W + px;
                        dS += G[i + R][j + R] * (a[o] + 2 * u * b[o] + v * c[o]);
                    }
                const double d = u - v;
                const double sgn = d > 0 ? 1.0 : (d < 0 ? -1.0 : 0.0);
                grad[q] = scale * ((1 - lambda) * sgn - lambda * dS) / double(N);
            }
    if (loss) *loss = scale * ((1 - lambda) * sum_l1 + lambda * (double(N) - sum_s)) / double(N);
    return 0;
}


int32_t orc_ellipse_tiles(const orc_camera* cam, float u, float v, float A, float B, float C, float k,
                          int32_t radius, double widen, double margin, int32_t* rect, uint8_t* codes,
                          int64_t max_codes) {
    const int TX = (cam->width + TILE - 1) / TILE, TY = (cam->height + TILE - 1) / TILE;
    const float r = float(radius);
    rect[0] = span_lo<float>(u, r, TX);
    rect[1] = span_hi<float>(u, r, TX);
    rect[2] = span_lo<float>(v, r, TY);
    rect[3] = span_hi<float>(v, r, TY);
    if (radius <= 0) rect[1] = rect[0], rect[3] = rect[2];
    const int64_t cols = rect[1] - rect[0], rows = rect[3] - rect[2];
    if (cols * rows > max_codes) return -1;
    for (int ty = rect[2]; ty < rect[3]; ++ty)
        for (int tx = rect[0]; tx < rect[1]; ++tx)
            codes[(ty - rect[2]) * cols + (tx - rect[0])] =
                ellipse_tile_decision(u, v, A, B, C, k, tx, ty, widen, margin);
    return int32_t(cols * rows);
}

int64_t orc_bin_ellipse(const orc_camera* cam, int32_t n, const float* means2d, const float* depth,
                        const int32_t* radius, const float* conic, const float* alpha_k, double widen,
                        double margin, int64_t capacity, uint64_t* keys_sorted, uint32_t* point_list,
                        uint32_t* ranges, uint32_t* tiles_touched, uint8_t* ambig_gauss,
                        int64_t ambig_capacity, uint32_t* ambig_pairs, int64_t* n_ambig) {
    const int TX = (cam->width + TILE - 1) / TILE, TY = (cam->height + TILE - 1) / TILE;
    std::vector<Entry> ent;
    int64_t na = 0;
    for (int32_t i = 0; i < n; ++i) {
        uint32_t cnt = 0;
        uint8_t amb = 0;
        if (radius[i] > 0) {
            const float u = means2d[i], v = means2d[size_t(n) + i], r = float(radius[i]);
            const int xl = span_lo<float>(u, r, TX), xh = span_hi<float>(u, r, TX);
            const int yl = span_lo<float>(v, r, TY), yh = span_hi<float>(v, r, TY);
            uint32_t bits;
            std::memcpy(&bits, &depth[i], 4);
            for (int ty = yl; ty < yh; ++ty)
                for (int tx = xl; tx < xh; ++tx) {
                    const uint8_t d = ellipse_tile_decision(u, v, conic[i], conic[size_t(n) + i],
                                                            conic[2 * size_t(n) + i], alpha_k[i], tx, ty,
                                                            widen, margin);
                    const uint64_t tile = uint64_t(ty) * uint64_t(TX) + uint64_t(tx);
                    if (d & ELL_AMBIG) {
                        amb = 1;
                        if (na < ambig_capacity) {
                            ambig_pairs[2 * na] = uint32_t(i);
                            ambig_pairs[2 * na + 1] = uint32_t(tile);
                        }
                        ++na;
                    }
                    if (d & ELL_KEEP) {
                        ++cnt;
                        ent.push_back(Entry{(tile << 32) | uint64_t(bits), uint32_t(i)});
                    }
                }
        }
        if (tiles_touched) tiles_touched[i] = cnt;
        if (ambig_gauss) ambig_gauss[i] = amb;
    }
    *n_ambig = na;
    const int64_t E = int64_t(ent.size());
    if (E > capacity || na > ambig_capacity) return -2;
    std::stable_sort(ent.begin(), ent.end(), [](const Entry& a, const Entry& b) { return a.key < b.key; });
    std::vector<uint64_t> ks(static_cast<size_t>(E));
    for (int64_t q = 0; q < E; ++q) {
        if (keys_sorted) keys_sorted[q] = ent[size_t(q)].key;
        point_list[q] = ent[size_t(q)].value;
        ks[size_t(q)] = ent[size_t(q)].key;
    }
    orc_tile_ranges(ks.data(), E, TX * TY, ranges);
    return E;
}

// c12: densification ([rigel] "GaussianModel: activations, densify/prune"; the training log's
// clone / split / prune counts).  The pages name the operations only; the criteria are those of
// 3D Gaussian Splatting's adaptive density control, decided here in double precision.  A
// decision within a relative 1e-5 of its threshold is flagged (either outcome is correct there).
int orc_densify_classify(int32_t n, const double* accum, const double* count, const double* log_scales,
                         const double* logits, double grad_threshold, double dense_scale, double min_opacity,
                         double max_scale, int32_t* action, uint8_t* ambig, int32_t* counts) {
    if (n < 0) return -1;
    const double ln_dense = std::log(dense_scale);
    const double logit_min = min_opacity > 0 ? std::log(min_opacity / (1.0 - min_opacity)) : -HUGE_VAL;
    const double ln_max = max_scale > 0 ? std::log(max_scale) : HUGE_VAL;
    const double ln_split = std::log(1.6);  // split children carry s / 1.6
    auto near = [](double x, double thr) {
        return std::isfinite(thr) && std::fabs(x - thr) <= 1e-5 * std::max(1.0, std::fabs(thr));
    };
    int32_t kept = 0, cloned = 0, split = 0, removed = 0;
    for (int32_t i = 0; i < n; ++i) {
        const size_t N = size_t(n);
        const double ls = std::max(std::max(log_scales[i], log_scales[N + i]), log_scales[2 * N + i]);
        // the mean view-space gradient norm reaches the threshold (no views: no growth)
        const bool grow = count[i] > 0 && accum[i] / count[i] >= grad_threshold;
        const bool dense = ls <= ln_dense;
        const bool faint = logits[i] < logit_min;
        uint8_t amb = 0;
        if (count[i] > 0 && std::fabs(accum[i] - grad_threshold * count[i]) <= 1e-5 * grad_threshold * count[i]) amb = 1;
        if (near(logits[i], logit_min)) amb = 1;
        int32_t a;
        if (grow) amb |= near(ls, ln_dense);
        if (grow && !dense) {
            amb |= near(ls - ln_split, ln_max);
            a = (faint || ls - ln_split > ln_max) ? 0 : 3;
        } else {
            amb |= near(ls, ln_max);
            a = (faint || ls > ln_max) ? 0 : grow ? 2 : 1;
        }
        action[i] = a;
        if (ambig) ambig[i] = amb;
        kept += a == 1 || a == 2;
        cloned += a == 2;
        split += a == 3;
        removed += a == 0;
    }
    counts[0] = kept + cloned + 2 * split;
    counts[1] = kept;
    counts[2] = cloned;
    counts[3] = split;
    counts[4] = removed;
    return 0;
}

// One parameter group [rows][n] after densification with the given actions (0 removed, 1 kept,
// 2 kept and cloned, 3 split), in the stated order: kept originals, clones, first children,
// second children.  kind 1: means (children at mean + R(q) (s * z_c)); kind 2: log-scales
// (children log(s / 1.6)); kind 0: copied.  m and v (may be NULL) follow the kept originals;
// clones and children start at zero.  Returns the number of Gaussians written.
int32_t orc_densify_group(int32_t n, const int32_t* action, int32_t rows, int32_t kind, const double* param,
                          const double* m, const double* v, const double* quats, const double* log_scales,
                          const double* noise, int32_t n_out, double* param_out, double* m_out, double* v_out) {
    const size_t N = size_t(n), NO = size_t(n_out);
    int32_t o = 0;
    auto put = [&](int32_t i, const double* value, bool fresh) {
        for (int r = 0; r < rows; ++r) {
            if (o < n_out) {
                param_out[r * NO + o] = value ? value[r] : param[r * N + i];
                if (m_out) m_out[r * NO + o] = fresh || !m ? 0.0 : m[r * N + i];
                if (v_out) v_out[r * NO + o] = fresh || !v ? 0.0 : v[r * N + i];
            }
        }
        ++o;
    };
    for (int32_t i = 0; i < n; ++i)
        if (action[i] == 1 || action[i] == 2) put(i, nullptr, false);
    for (int32_t i = 0; i < n; ++i)
        if (action[i] == 2) put(i, nullptr, true);
    for (int c = 0; c < 2; ++c)
        for (int32_t i = 0; i < n; ++i) {
            if (action[i] != 3) continue;
            double value[64];
            for (int r = 0; r < rows && r < 64; ++r) value[r] = param[r * N + i];
            if (kind == 1) {
                // a sample of N(mean, Sigma_3d): Sigma_3d = R S S^T R^T, so mean + R (s * z)
                const double qn = std::sqrt(quats[i] * quats[i] + quats[N + i] * quats[N + i] +
                                            quats[2 * N + i] * quats[2 * N + i] + quats[3 * N + i] * quats[3 * N + i]);
                double Rq[9];
                quat_to_rotmat<double>(quats[i] / qn, quats[N + i] / qn, quats[2 * N + i] / qn, quats[3 * N + i] / qn, Rq);
                double sz[3];
                for (int k = 0; k < 3; ++k) sz[k] = std::exp(log_scales[k * N + i]) * noise[(size_t(c) * 3 + k) * N + i];
                for (int r = 0; r < 3; ++r) value[r] += Rq[r * 3 + 0] * sz[0] + Rq[r * 3 + 1] * sz[1] + Rq[r * 3 + 2] * sz[2];
            } else if (kind == 2) {
                for (int r = 0; r < 3; ++r) value[r] -= std::log(1.6);
            }
            put(i, value, true);
        }
    return o;
}

double orc_quad_min_rect(double A, double B, double C, double x0, double x1, double y0, double y1) {
    return quad_min_rect(A, B, C, x0, x1, y0, y1);
}

}  // extern "C"
