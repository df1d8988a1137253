/*
 * Oracle for tile-based 3D Gaussian Splatting rasterisation -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU statement of what the GPU path computes, written from
 * the method's description on the source pages (rigel README; "3D Gaussian Splatting
 * ビューワを作る"; learn-gs notebook "11 - Tiles: the actual 3DGS design").  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it.  It shares no
 * source, header, constant or helper with the CUDA library, and never calls it.
 *
 * Conventions (all arrays planar, one row per component, row stride n):
 *   means [3][n], scales [3][n] (linear, already activated), quats [4][n] as (w,x,y,z), any norm,
 *   opacity [n] (already activated), sh [3K][n] with row k*3+ch, K = (degree+1)^2,
 *   colors [3][n] when sh_degree < 0.  Camera: p_cam = R * m + t, R row-major; pinhole fx,fy,cx,cy.
 * Inputs are passed as double; the 32-bit variants round every input to float first and
 * carry out every step in float, so that integer decisions (cull, radius, tile span,
 * contributor counts) are taken in the precision of the GPU kernels.
 *
 * Parity status: every function here is pinned by the CPU test suite (closed forms, worked
 * examples printed on the pages, invariants, brute force, library routines, finite
 * differences).  None is "parity unpinned".
 */
#ifndef GS_ORACLE_H
#define GS_ORACLE_H
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif

typedef struct orc_camera {
    double R[9];
    double t[3];
    double fx, fy, cx, cy;
    int32_t width, height;
} orc_camera;

/* Projection flags (per Gaussian) for decisions that sit within `margin` of their threshold. */
enum {
    ORC_AMB_NEAR = 1,     /* camera-space z close to the near plane            */
    ORC_AMB_DET = 2,      /* determinant of the dilated 2D covariance near 0    */
    ORC_AMB_RADIUS = 4,   /* 3*sqrt(lambda_max) close to an integer              */
    ORC_AMB_SPAN = 8,     /* (u +- r)/16 or (v +- r)/16 close to an integer      */
    ORC_AMB_CLAMP = 16    /* |x/z| or |y/z| close to the 1.3x frustum limit      */
};
/* Rasterisation flags (per pixel). */
enum {
    ORC_AMB_ALPHA_MIN = 1, /* some alpha within margin of the 1/255 skip threshold */
    ORC_AMB_T_STOP = 2,    /* transmittance within margin of the 1e-4 stop test    */
    ORC_AMB_ALPHA_MAX = 4  /* opacity*G within margin of the 0.99 clamp            */
};

/* c1 + c6: projection and colour.  prec = 32 or 64.  Culled Gaussians get radius 0,
 * tiles_touched 0 and zeros everywhere else.  rect = [x_lo, x_hi, y_lo, y_hi][n] in tiles.
 * ambig may be NULL.  Returns 0, or -1 on a bad argument. */
int orc_project(int prec, const orc_camera* cam, int32_t n, const double* means,
                const double* scales, const double* quats, const double* opacity,
                const double* sh, int32_t sh_degree, const double* colors,
                double* means2d, double* depth, double* conic, double* color,
                int32_t* radius, int32_t* rect, uint32_t* tiles_touched,
                double margin, uint8_t* ambig);

/* Intermediates of the projection in double, for the pins: cov3d [6][n] (xx,xy,xz,yy,yz,zz),
 * cov2d [3][n] (a,b,c after the +0.3 dilation), jac [6][n] (J row-major 2x3, clamped),
 * pcam [3][n]. */
void orc_project_intermediates(const orc_camera* cam, int32_t n, const double* means,
                               const double* scales, const double* quats, double* cov3d,
                               double* cov2d, double* jac, double* pcam);

/* c6: the 16 real SH basis functions at unit directions dirs [3][m] -> Y [16][m]. */
void orc_sh_basis(const double* dirs, int32_t m, double* Y);

/* c2 pieces. */
uint64_t orc_exclusive_scan_u32(const uint32_t* in, int64_t n, uint64_t* out);
void orc_tile_ranges(const uint64_t* keys_sorted, int64_t n_entries, int32_t n_tiles,
                     uint32_t* ranges);
/* Count the (Gaussian, tile) entries from projected float data (decisions in float). */
int64_t orc_bin_count(const orc_camera* cam, int32_t n, const float* means2d,
                      const int32_t* radius);
/* Full binning: entries, stable sort, ranges.  keys_sorted/point_list hold `capacity`
 * entries; returns the entry count, or -2 when it exceeds capacity (nothing written). */
int64_t orc_bin(const orc_camera* cam, int32_t n, const float* means2d, const float* depth,
                const int32_t* radius, int64_t capacity, uint64_t* keys_sorted,
                uint32_t* point_list, uint32_t* ranges, uint32_t* tiles_touched);

/* c3: forward compositing of every pixel in the tiles selected by tile_mask (NULL = all).
 * Pixels of unselected tiles are left untouched.  n_blend (may be NULL) receives, per pixel,
 * how many of the examined entries were composited (not skipped). */
int orc_raster_fwd(int prec, const orc_camera* cam, int32_t n, const double* means2d,
                   const double* conic, const double* opacity, const double* color,
                   const uint32_t* ranges, const uint32_t* point_list, const double* bg,
                   const uint8_t* tile_mask, double* image, double* final_T,
                   uint32_t* n_contrib, double margin, uint8_t* ambig, uint32_t* n_blend);

/* c4: backward of the compositing, in double.  Walk length per pixel is n_contrib (as given).
 * Gradients are accumulated into zero-initialised outputs by this call.  absum (may be NULL;
 * zero-initialised, [9][n]: rows dmeans2d 0-1, dconic 2-4, dopacity 5, dcolor 6-8) receives for
 * every output the sum of the magnitudes of the terms it adds up, with dL/dalpha's own terms in
 * absolute value: the scale of the rounding error of any float computation of these sums. */
int orc_raster_bwd(const orc_camera* cam, int32_t n, const double* means2d,
                   const double* conic, const double* opacity, const double* color,
                   const uint32_t* ranges, const uint32_t* point_list, const double* bg,
                   const uint32_t* n_contrib, const double* dL_dimage,
                   const uint8_t* tile_mask, double* dmeans2d, double* dconic,
                   double* dopacity, double* dcolor, double* absum);

/* c5: backward of the projection and colour, in double.  Culled Gaussians (radius 0) get zero
 * gradients.  dsh may be NULL when sh_degree < 0 (then dcolor is the colours' gradient). */
int orc_project_bwd(const orc_camera* cam, int32_t n, const double* means,
                    const double* scales, const double* quats, const double* sh,
                    int32_t sh_degree, const int32_t* radius, const double* dmeans2d,
                    const double* dconic, const double* dcolor, double* dmeans,
                    double* dscales, double* dquats, double* dsh);

/* c7: appearance MLP. x = [latent (L) ; unit view dir (3)], h = relu(W1 x + b1) (H wide),
 * rgb = sigmoid(W2 h + b2).  latents [L][n]; W1 [H][L+3] row-major; W2 [3][H]. */
int orc_appearance_fwd(const orc_camera* cam, int32_t n, int32_t L, int32_t H,
                       const double* means, const double* latents, const double* W1,
                       const double* b1, const double* W2, const double* b2, double* colors);
int orc_appearance_bwd(const orc_camera* cam, int32_t n, int32_t L, int32_t H,
                       const double* means, const double* latents, const double* W1,
                       const double* b1, const double* W2, const double* b2,
                       const double* dcolors, double* dlatents, double* dW1, double* db1,
                       double* dW2, double* db2);

/* c8: L1 loss of the training step.  grad[i] = scale * sign(image[i] - target[i]) (sign(0) = 0),
 * *loss = scale * sum_i |image[i] - target[i]|. */
int orc_l1_loss_grad(int64_t count, const double* image, const double* target, double scale,
                     double* grad, double* loss);

/* c9: Adam step over one parameter group (in place), gradient given w.r.t. act(param);
 * activation 0 identity, 1 exp, 2 sigmoid; activated (may be NULL) receives act(param). */
int orc_adam_step(int64_t count, double* param, const double* grad, double* m, double* v,
                  double* activated, double lr, int32_t activation, double beta1, double beta2,
                  double eps, int32_t step);
/* c10: densification statistics: accum[i] += |dmeans2d_i|, count[i] += 1 where radius[i] > 0. */
int orc_densify_stats(int32_t n, const double* dmeans2d, const int32_t* radius, double* accum,
                      double* count);

/* c11: L1 + D-SSIM loss (3DGS's photometric loss), C channels of H x W images:
 * L = (1 - lambda) mean|I - T| + lambda (1 - mean SSIM), 11 x 11 Gaussian window (sigma 1.5,
 * normalised), zeros outside the image, C1 = 0.01^2, C2 = 0.03^2.  grad = scale dL/dI,
 * *loss = scale L; ssim (may be NULL) receives the per-pixel SSIM map. */
int orc_l1_dssim(int32_t C, int32_t H, int32_t W, const double* image, const double* target,
                 double lambda, double scale, double* grad, double* loss, double* ssim);

/* c2': binning with the ellipse-tile test (the pages' "next" step), from its definition in
 * double precision: per visible Gaussian (radius > 0) only the tiles of its radius square whose
 * pixel-centre square [16 tx, 16 tx + 15] x [16 ty, 16 ty + 15] holds a point with
 * d^T conic d <= alpha_k; otherwise as orc_bin.  A decision is a knife edge (either outcome
 * correct) unless the minimum over the square is at most k (1 - margin) or the minimum over the
 * square widened by `widen` px exceeds k (1 + margin); such (Gaussian, tile) pairs go to
 * ambig_pairs [2 * ambig_capacity] as (index, tile id), their count to *n_ambig, and
 * ambig_gauss [n] (may be NULL) marks Gaussians with any.  Returns E, or -2 when E > capacity or
 * the pairs exceed ambig_capacity (the counts are still written). */
int64_t orc_bin_ellipse(const orc_camera* cam, int32_t n, const float* means2d, const float* depth,
                        const int32_t* radius, const float* conic, const float* alpha_k, double widen,
                        double margin, int64_t capacity, uint64_t* keys_sorted, uint32_t* point_list,
                        uint32_t* ranges, uint32_t* tiles_touched, uint8_t* ambig_gauss,
                        int64_t ambig_capacity, uint32_t* ambig_pairs, int64_t* n_ambig);
/* The decisions of one Gaussian over its radius square: rect = {xl, xh, yl, yh} (half-open),
 * codes [(yh - yl) * (xh - xl)] row-major, bit 0 kept, bit 1 knife edge.  Returns the number of
 * codes, or -1 when they exceed max_codes. */
int32_t orc_ellipse_tiles(const orc_camera* cam, float u, float v, float A, float B, float C, float k,
                          int32_t radius, double widen, double margin, int32_t* rect, uint8_t* codes,
                          int64_t max_codes);
/* c12: densification, decisions in double (3DGS's adaptive density control): action [n] (0 removed,
 * 1 kept, 2 kept and cloned, 3 split), ambig [n] (may be NULL) marks decisions within a relative
 * 1e-5 of a threshold, counts [5] = n_out, kept, cloned, split, removed. */
int orc_densify_classify(int32_t n, const double* accum, const double* count, const double* log_scales,
                         const double* logits, double grad_threshold, double dense_scale, double min_opacity,
                         double max_scale, int32_t* action, uint8_t* ambig, int32_t* counts);
/* One parameter group [rows][n] (rows <= 64) after densification with `action`; kind 0 copy,
 * 1 means (split children at mean + R(q) (s * z_c), noise [2][3][n]), 2 log-scales (children
 * log(s / 1.6)).  Returns the number of Gaussians written to the [rows][n_out] outputs. */
int32_t orc_densify_group(int32_t n, const int32_t* action, int32_t rows, int32_t kind, const double* param,
                          const double* m, const double* v, const double* quats, const double* log_scales,
                          const double* noise, int32_t n_out, double* param_out, double* m_out, double* v_out);
/* Minimum of A x^2 + 2 B x y + C y^2 (positive definite) over [x0, x1] x [y0, y1]. */
double orc_quad_min_rect(double A, double B, double C, double x0, double x1, double y0, double y1);

#ifdef __cplusplus
}
#endif
#endif
