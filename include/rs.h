/*
 * rs.h -- C ABI of the GB300 (sm_103a) tile-based 3D Gaussian Splatting rasteriser.
 *
 * Five calls carry the data-parallel path, in the order the rigel README's "How it works"
 * diagram runs them: rs_project [1], rs_bin [2], rs_rasterize_fwd [3] (forward), then
 * rs_rasterize_bwd [4] and rs_project_bwd [5] (backward).
 *
 * Conventions shared by every call
 *  - Ownership: the caller allocates and owns every buffer, device and host, including the
 *    binning workspace.  The library allocates no device memory, keeps no state between calls
 *    and may be called from several host threads on distinct buffers.
 *  - Pointers named d_* are device pointers; everything else is host memory.
 *  - Layout: planar (structure of arrays) float32, one row per component, row stride n:
 *    element (k, i) of a [K][n] array sits at base[k*n + i].  Images are [3][H][W]; per-pixel
 *    buffers are [H][W].  Device arrays need their natural alignment (4 bytes; 8 bytes for
 *    64-bit keys); the packed records need 16 bytes.
 *  - Streams: every call takes `stream` (a cudaStream_t; NULL = the legacy default stream) and
 *    only enqueues work on it, except rs_bin, which reads the entry count back to the host once
 *    (a stream-ordered copy followed by a synchronisation of that stream).
 *  - Outputs are overwritten, never accumulated into; gradient outputs are zeroed by the callee.
 *  - Arguments are validated before anything is enqueued; a failed check returns
 *    RS_ERR_INVALID_ARG and leaves every buffer untouched.
 *  - n = 0 is valid: no Gaussian work is launched; the image is the background, final_T is 1
 *    and n_contrib is 0.
 *  - Limits: 0 <= n <= RS_MAX_GAUSSIANS; 1 <= width, height <= 32768; the number of
 *    (Gaussian, tile) entries is at most RS_MAX_ENTRIES.
 */
#ifndef RS_H
#define RS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define RS_OK 0
#define RS_ERR_INVALID_ARG (-1)     /* null or misaligned pointer, bad size or parameter      */
#define RS_ERR_CAPACITY (-2)        /* more entries than `capacity`; *n_entries holds the count */
#define RS_ERR_WORKSPACE (-3)       /* workspace smaller than rs_bin_workspace_size reports   */
#define RS_ERR_CUDA (-4)            /* a CUDA runtime call or launch failed                   */
#define RS_ERR_DEVICE_TIMEOUT (-5)  /* a bounded wait inside a kernel gave up (outputs invalid) */
#define RS_ERR_DEVICE_CHECK (-6)    /* a kernel found caller data out of range and skipped it  */

#define RS_TILE 16                  /* tile edge in pixels (rigel "Binning")                    */
#define RS_RECORD_BYTES 48          /* packed per-Gaussian record written by rs_project         */
#define RS_MAX_GAUSSIANS 67108864   /* 2^26                                                     */
#define RS_MAX_ENTRIES 1073741823   /* 2^30 - 1: largest `capacity` of rs_bin                   */

/* Pinhole camera: a world point m maps to p = R m + t (R row-major, world to camera), then to
 * pixel (fx p.x/p.z + cx, fy p.y/p.z + cy).  Pixel (x, y) is sampled at integer coordinates.
 * rigel README, "Deliberate differences from the reference implementation" (row-major
 * world-to-camera matrices and explicit pinhole intrinsics). */
typedef struct rs_camera {
    float R[9];
    float t[3];
    float fx, fy, cx, cy;
    int32_t width, height;
} rs_camera;

/* Gaussian parameters, already activated (scales linear, opacity in [0, 1]).
 *   d_means [3][n], d_scales [3][n], d_quats [4][n] as (w, x, y, z) of any non-zero norm,
 *   d_opacity [n];
 *   sh_degree 0..3: d_sh [3K][n] with K = (sh_degree+1)^2, row k*3+ch holds the coefficient of
 *   basis function k for channel ch (the f_dc / f_rest order of "3D Gaussian Splatting
 *   ビューワを作る", 2.2.3);
 *   sh_degree -1: d_colors [3][n] are the colours and d_sh is ignored. */
typedef struct rs_gaussians {
    int32_t n;
    const float* d_means;
    const float* d_scales;
    const float* d_quats;
    const float* d_opacity;
    const float* d_sh;
    int32_t sh_degree;
    const float* d_colors;
} rs_gaussians;

/* Per-Gaussian results of rs_project (all [n] or [C][n]):
 *   d_means2d [2][n] pixel position (u, v); d_depth [n] camera-space z;
 *   d_conic [3][n] (A, B, C) of the inverse 2D covariance [[A, B], [B, C]];
 *   d_color [3][n]; d_radius [n] int32 bounding radius in pixels, 0 = culled;
 *   d_tiles_touched [n] uint32 number of 16x16 tiles of the radius square;
 *   d_records: n * RS_RECORD_BYTES bytes, 16-byte aligned, the rasterisers' packed copy
 *   (opaque: written by rs_project, read by the two rasterisers).
 * A culled Gaussian has radius 0, tiles_touched 0 and zeros in every other field. */
typedef struct rs_projected {
    float* d_means2d;
    float* d_depth;
    float* d_conic;
    float* d_color;
    int32_t* d_radius;
    uint32_t* d_tiles_touched;
    void* d_records;
    /* Which tiles a splat covers (read by rs_project and rs_bin; a zeroed struct means
     * RS_TILE_TEST_SQUARE):
     *  - RS_TILE_TEST_SQUARE: the tiles of its radius square, the pages' binning (rigel README
     *    "Binning"; learn-gs "11 - Tiles", tile_spans).
     *  - RS_TILE_TEST_ELLIPSE: only the tiles of that square whose pixel centres
     *    [16 tx, 16 tx + 15] x [16 ty, 16 ty + 15] meet the ellipse where opacity exp(power)
     *    >= 1/255, i.e.
     *    d^T conic d <= k with k = 2.002 ln(255 opacity) (0.1% wider than exact, plus 0.01 px),
     *    rows outer and columns inner as before.  The pages list this exact ellipse-tile test as
     *    their next step; the skipped tiles hold only alpha < 1/255, so the image, final_T and
     *    the gradients are those of the square test, with fewer entries; n_contrib counts only
     *    the entries each pixel examined.  A splat meeting no tile is culled (radius 0).
     *    rs_project writes d_ellipse [RS_ELLIPSE_WORDS][n]: row 0 is k (0 when culled), rows
     *    1.. the test's per-splat setup that rs_bin reads (contents otherwise unspecified). */
    float* d_ellipse;
    int32_t tile_test;
} rs_projected;

#define RS_TILE_TEST_SQUARE 0
#define RS_TILE_TEST_ELLIPSE 1
#define RS_ELLIPSE_WORDS 12

/* Human-readable text for a return code; never NULL. */
const char* rs_error_string(int code);

/* [1] Projection, rigel README "Projection"; covariance, conic and radius as in "3D Gaussian
 * Splatting ビューワを作る" 2.1-2.3; tile span as tile_spans in the learn-gs notebook
 * "11 - Tiles".  Per Gaussian: p = R m + t, culled unless p.z > 0.05; Sigma_3d = (R(q) S)(R(q) S)^T
 * with q normalised; J at x/z, y/z clamped to 1.3x the half-widths W/(2 fx), H/(2 fy);
 * Sigma_2d = J R Sigma_3d R^T J^T + 0.3 I; culled unless det > 0; conic = Sigma_2d^-1;
 * (u, v) = (fx x/z + cx, fy y/z + cy); radius = ceil(3 sqrt(lambda_max)) with
 * lambda_max = mid + sqrt(max(0.1, mid^2 - det)); span = [floor((u-r)/16), floor((u+r)/16)+1)
 * clamped to the tile grid (same in y); culled when the span is empty.  Colour: degree-K real
 * SH (viewer 2.2.3) at the unit direction from the camera centre -R^T t to the mean, no offset
 * or clamp; or the given colours.  With the square test, n a multiple of 4 and every input row
 * 16-byte aligned, the input rows are staged through shared memory by bulk asynchronous copies
 * with a bounded wait; a CTA whose wait gives up leaves its Gaussians' outputs unwritten and
 * raises the flag rs_device_error reports (the results are the same on every path).
 * Errors: RS_ERR_INVALID_ARG, RS_ERR_CUDA. */
int rs_project(const rs_camera* camera, const rs_gaussians* gaussians, const rs_projected* out,
               void* stream);

/* Workspace bytes rs_bin needs for n Gaussians on this camera with room for `capacity`
 * entries.  Writes *bytes; returns RS_OK or RS_ERR_INVALID_ARG. */
int rs_bin_workspace_size(int32_t n, const rs_camera* camera, size_t capacity, size_t* bytes);

/* [2] Binning, rigel README "Binning": one entry per (visible Gaussian, covered tile) with
 * key = (tile_id << 32) | float_bits(depth), tile_id = ty * ceil(W/16) + tx, sorted stably by key
 * on the device -- equal keys keep Gaussian index order, the order in which the entries are
 * produced (tile rows outer, columns inner) -- and each tile's [start, end) range extracted
 * (viewer 4.4; empty tiles get (0, 0)).  The 64-bit stable sort runs as an LSD radix sort
 * ("3D Gaussian Splatting ビューワを作る" 4.3) of the Gaussians by depth followed by one of the
 * entries, produced in that depth order, by tile id: the same order, in fewer passes.
 * Inputs: `proj` from rs_project (means2d, depth, radius, tiles_touched are read).
 * Outputs: d_point_list [capacity] uint32 Gaussian index per sorted entry; d_tile_ranges
 * [n_tiles][2] uint32 (8-byte aligned); d_keys_sorted [capacity] uint64 (may be NULL);
 * *n_entries (host) = E.  The entry count is read back to the host once, at the end.  If
 * E > capacity the call writes no entry, returns RS_ERR_CAPACITY and sets *n_entries, so the
 * caller can grow the buffers and call again.
 * d_workspace: at least rs_bin_workspace_size bytes, 256-byte aligned, contents undefined on
 * entry and exit.  Errors: RS_ERR_INVALID_ARG (also capacity > RS_MAX_ENTRIES),
 * RS_ERR_WORKSPACE, RS_ERR_CAPACITY, RS_ERR_CUDA, RS_ERR_DEVICE_TIMEOUT (a bounded wait of the
 * sort's look-back gave up; cannot happen while the GPU runs the call's blocks normally). */
int rs_bin(const rs_camera* camera, const rs_projected* proj, int32_t n, void* d_workspace,
           size_t workspace_bytes, size_t capacity, uint64_t* d_keys_sorted,
           uint32_t* d_point_list, uint32_t* d_tile_ranges, size_t* n_entries, void* stream);

/* Binning without waiting for the entry count (the sync-free pipeline: the host keeps
 * enqueueing the rest of the frame while the GPU bins).  Same arguments, work and outputs as
 * rs_bin, except that the entry count is not waited for: the call enqueues, on `stream`, the
 * writing of two uint64 words into h_result -- h_result[0] = E, h_result[1] = nonzero if a
 * bounded wait of the sort's look-back gave up -- and returns.  h_result must be pinned host
 * memory (cudaHostAlloc, cudaMallocHost, or registered with cudaHostRegister); where it is mapped
 * into the device's address space (always under unified addressing) a one-thread kernel writes
 * it, else a device-to-host copy does.  Read h_result only after the stream has reached that
 * point (cudaStreamSynchronize or an event recorded after the call).  When E > capacity no entry
 * is written and every tile range is (0, 0), so later calls on these buffers render the
 * background and stay within bounds; the caller must then grow the buffers and redo the frame.
 * Nothing in the call waits on the host, so it can be captured in a CUDA graph.
 * Errors (returned at once): RS_ERR_INVALID_ARG, RS_ERR_WORKSPACE, RS_ERR_CUDA. */
int rs_bin_async(const rs_camera* camera, const rs_projected* proj, int32_t n, void* d_workspace,
                 size_t workspace_bytes, size_t capacity, uint64_t* d_keys_sorted,
                 uint32_t* d_point_list, uint32_t* d_tile_ranges, uint64_t* h_result, void* stream);

/* Compositing workspace: the forward's per-pixel state at every RS_RASTER_CHUNK-th position of
 * the point list that falls inside a tile's list, and which tile holds each such position (the
 * backward reads both to walk every 256-entry stretch of the point list as a task of its own);
 * per entry, which 8x4-pixel groups of its tile composited it (the backward skips the others);
 * the order in which the forward takes the tiles (longest lists first); and the backward's work
 * counter.
 * Returns the bytes a point list of `capacity` entries needs for this camera's tile grid; 0 for
 * an invalid camera or capacity > RS_MAX_ENTRIES.  Host-only (no GPU work). */
#define RS_RASTER_CHUNK 256
size_t rs_raster_workspace_size(const rs_camera* camera, size_t capacity);

/* [3] Forward compositing, rigel README "Rasterization"; learn-gs "11 - Tiles", "The kernel".
 * One thread block per half of a 16x16 tile (16x8 pixels); each pixel walks its tile's list
 * front to back:
 * power = -1/2 (A dx^2 + C dy^2) - B dx dy with (dx, dy) = (x - u, y - v),
 * alpha = min(0.99, opacity exp(power)); entries with alpha < 1/255 are skipped;
 * C += colour alpha T, T *= 1 - alpha; the pixel stops after the entry that brings T below 1e-4.
 * image = C + T bg.  n_contrib counts every entry the pixel examined (skipped ones and the one
 * that stopped it included).  bg: host float[3].
 * capacity: the length of d_point_list (the capacity given to rs_bin).  d_workspace: at least
 * rs_raster_workspace_size(camera, capacity) bytes of device memory, 16-byte aligned, owned by
 * the caller; the call fills it for rs_rasterize_bwd (no initial contents needed).
 * Outputs: d_image [3][H][W], d_final_T [H][W], d_n_contrib [H][W] uint32.
 * The kernel checks the caller's list: an entry >= n is skipped (examined, never composited) and
 * a tile whose range ends past capacity (or starts after its end) is drawn empty; either raises
 * the flag rs_device_error reports as RS_ERR_DEVICE_CHECK.  Nothing is read outside the buffers.
 * Errors: RS_ERR_INVALID_ARG, RS_ERR_WORKSPACE (workspace too small), RS_ERR_CUDA. */
int rs_rasterize_fwd(const rs_camera* camera, const rs_projected* proj, int32_t n,
                     const uint32_t* d_tile_ranges, const uint32_t* d_point_list, size_t capacity,
                     const float* bg, float* d_image, float* d_final_T, uint32_t* d_n_contrib,
                     void* d_workspace, size_t workspace_bytes, void* stream);

/* [4] Backward of the compositing, rigel README "Backward": each tile's list is walked back to
 * front, undoing the transmittance one step at a time (T_i = T_{i+1} / (1 - a_i)) and carrying
 * the colour behind the current entry; entries past a pixel's n_contrib and skipped entries
 * (alpha < 1/255) give nothing; an entry whose opacity * exp(power) exceeds 0.99 (clamped)
 * passes no gradient to opacity, conic or mean ("Deliberate differences").
 * The walk is split at every RS_RASTER_CHUNK-th position of the point list: a stretch that ends
 * inside a tile's list starts from the state the forward recorded there (T, and the colour
 * behind that position) instead of from final_T, so long lists are walked in parallel.
 * Per-pixel contributions are reduced across each 8x8 pixel square before they reach global
 * memory.
 * Inputs: the forward's tile_ranges, point_list, capacity, final_T, n_contrib and workspace (as
 * rs_rasterize_fwd left them), bg (host float[3]) and d_dL_dimage [3][H][W].  The call hands out
 * its work through a counter of 8 bytes in the workspace, which the forward sets to zero and the
 * call leaves at zero: two rs_rasterize_bwd calls must not use one workspace at the same time.
 * Outputs (zeroed, then accumulated by the call):
 * d_dL_dmeans2d [2][n], d_dL_dconic [3][n], d_dL_dopacity [n], d_dL_dcolor [3][n].
 * The accumulation order is not fixed, so results may differ in the last bits between runs.
 * The same checks as rs_rasterize_fwd: entries >= n and tiles whose range ends past capacity are
 * skipped and raise the flag rs_device_error reports as RS_ERR_DEVICE_CHECK.
 * Errors: RS_ERR_INVALID_ARG, RS_ERR_WORKSPACE, RS_ERR_CUDA. */
int rs_rasterize_bwd(const rs_camera* camera, const rs_projected* proj, int32_t n,
                     const uint32_t* d_tile_ranges, const uint32_t* d_point_list, size_t capacity,
                     const float* bg, const float* d_final_T, const uint32_t* d_n_contrib,
                     void* d_workspace, size_t workspace_bytes,
                     const float* d_dL_dimage, float* d_dL_dmeans2d, float* d_dL_dconic,
                     float* d_dL_dopacity, float* d_dL_dcolor, void* stream);

/* [5] Backward of the projection and colour, rigel README "Backward" (second paragraph): through
 * the 2x2 inverse, Sigma_2d = T Sigma_3d T^T with T = J R, the Jacobian's dependence on p_cam
 * (a clamped x/z or y/z sends its gradient to z), the pinhole, the camera transform and
 * Sigma_3d = M M^T with M = R(q) S, including the normalisation of q (the quaternion gradient
 * has no component along q); and through the SH basis, including the view direction's
 * dependence on the mean.  Culled Gaussians (radius 0) get zero gradients.
 * Inputs: the forward's gaussians and proj (radius is read), and the gradients of means2d,
 * conic and colour.  Outputs (overwritten): d_dL_dmeans [3][n], d_dL_dscales [3][n],
 * d_dL_dquats [4][n], d_dL_dsh [3K][n] (ignored and may be NULL when sh_degree is -1; then
 * d_dL_dcolor already is the colours' gradient).  Errors: RS_ERR_INVALID_ARG, RS_ERR_CUDA. */
int rs_project_bwd(const rs_camera* camera, const rs_gaussians* gaussians,
                   const rs_projected* proj, const float* d_dL_dmeans2d,
                   const float* d_dL_dconic, const float* d_dL_dcolor, float* d_dL_dmeans,
                   float* d_dL_dscales, float* d_dL_dquats, float* d_dL_dsh, void* stream);

/* Appearance MLP and L1 loss of the training-shaped step (rigel README "Appearance MLP"; the
 * L1 term of its training loss).  rs_appearance_fwd produces the colours that rs_project reads
 * when sh_degree is -1; rs_appearance_bwd takes the colours' gradient that rs_rasterize_bwd
 * returns.  The pages give no device interface for these; this one follows the conventions
 * above. */

/* MLP weights, float32 device arrays: W1 [hidden][latent_dim + 3] and W2 [3][hidden], both
 * row-major, b1 [hidden], b2 [3].  Supported sizes: hidden 32 or 64, 1 <= latent_dim <= 29
 * (the page's MLP is sized for up to 29 latent dims and 64 hidden units). */
typedef struct rs_mlp {
    int32_t latent_dim, hidden;
    const float* d_W1;
    const float* d_b1;
    const float* d_W2;
    const float* d_b2;
} rs_mlp;

/* Weight gradients, same shapes as rs_mlp's arrays. */
typedef struct rs_mlp_grads {
    float* d_dW1;
    float* d_db1;
    float* d_dW2;
    float* d_db2;
} rs_mlp_grads;

/* rigel README "Appearance MLP": for every Gaussian i, x = [latent_i ; (m_i - C) / |m_i - C|]
 * with C = -R^T t the camera centre, h = relu(W1 x + b1), colour = sigmoid(W2 h + b2).
 * Inputs: d_means [3][n], d_latents [latent_dim][n].  Output (overwritten): d_colors [3][n].
 * The products run on the tensor cores in TF32 with split operands (three products per
 * operand pair), which keeps float32 accuracy.  Each CTA waits for its tensor-core products
 * with a bounded wait; one that gives up writes NaN colours for its Gaussians and raises the
 * flag rs_device_error reports.  Errors: RS_ERR_INVALID_ARG, RS_ERR_CUDA. */
int rs_appearance_fwd(const rs_camera* camera, int32_t n, const float* d_means,
                      const float* d_latents, const rs_mlp* mlp, float* d_colors, void* stream);

/* Backward of rs_appearance_fwd with the view direction held constant (rigel README "Appearance
 * MLP": no gradient reaches the means through the MLP).  Input d_dL_dcolors [3][n].  Outputs:
 * d_dL_dlatents [latent_dim][n] (overwritten) and the weight gradients summed over the n
 * Gaussians (zeroed, then accumulated by the call; the accumulation order is not fixed).
 * Errors: RS_ERR_INVALID_ARG, RS_ERR_CUDA. */
int rs_appearance_bwd(const rs_camera* camera, int32_t n, const float* d_means,
                      const float* d_latents, const rs_mlp* mlp, const float* d_dL_dcolors,
                      float* d_dL_dlatents, const rs_mlp_grads* grads, void* stream);

/* Reads and clears the device flags: RS_ERR_DEVICE_CHECK if a compositing kernel skipped caller
 * data out of range (see rs_rasterize_fwd), else RS_ERR_DEVICE_TIMEOUT if a kernel's bounded wait
 * gave up (on the tensor cores, or on the projection's staged copies), since the last call; else
 * RS_OK (RS_ERR_CUDA if a flag cannot be read).  Synchronises the device. */
int rs_device_error(void);

/* L1 loss between an image and its target over `count` floats:
 * d_dL_dimage[i] = scale * sign(d_image[i] - d_target[i]) with sign(0) = 0 and, when d_loss is
 * not NULL, *d_loss (one device float, overwritten) = scale * sum_i |d_image[i] - d_target[i]|
 * (accumulation order not fixed).  With scale = 1 / (3 H W V) this is the gradient of the
 * per-view mean absolute error averaged over V views (rigel README, training loss).
 * Errors: RS_ERR_INVALID_ARG, RS_ERR_CUDA. */
int rs_l1_loss_grad(size_t count, const float* d_image, const float* d_target, float scale,
                    float* d_dL_dimage, float* d_loss, void* stream);

/* L1 + D-SSIM loss, the photometric loss rigel trains with (README: "L1 + D-SSIM"; the pages
 * give no formula, so this is 3DGS's): over C channels of H x W images,
 *   L = (1 - lambda) mean |I - T| + lambda (1 - mean SSIM(I, T)),
 * SSIM per channel and pixel with an 11 x 11 Gaussian window (sigma 1.5, separable weights
 * normalised over the window, zeros outside the image), C1 = 0.01^2, C2 = 0.03^2; means over all
 * C H W values.  Writes d_dL_dimage = scale * dL/dI [C][H][W] and, when d_loss is not NULL,
 * *d_loss = scale * L (one device float, summed in a fixed order).  d_workspace: at least
 * rs_l1_dssim_workspace_size bytes, 16-byte aligned, contents undefined on entry and exit.
 * Errors: RS_ERR_INVALID_ARG, RS_ERR_WORKSPACE, RS_ERR_CUDA. */
int rs_l1_dssim_workspace_size(int32_t channels, int32_t height, int32_t width, size_t* bytes);
int rs_l1_dssim_loss_grad(int32_t channels, int32_t height, int32_t width, const float* d_image,
                          const float* d_target, float lambda, float scale, float* d_dL_dimage,
                          float* d_loss, void* d_workspace, size_t workspace_bytes, void* stream);

/* Optimiser step and densification statistics of the training loop (rigel README: the
 * optimisation loop; "GaussianModel: activations, densify/prune"; per-group learning rates --
 * its higher-order SH rate is a twentieth of the DC rate).  The pages give no device interface
 * for these; this one follows the conventions above. */

#define RS_ACT_IDENTITY 0   /* the parameter is used as it is                                */
#define RS_ACT_EXP 1        /* the parameter is a log (e.g. log-scales): used as exp(param)   */
#define RS_ACT_SIGMOID 2    /* the parameter is a logit (opacity): used as sigmoid(param)     */
#define RS_ADAM_MAX_SEGMENTS 16

/* One parameter group: `count` float32 device values updated in place with their Adam moments.
 * d_grad is the gradient w.r.t. the value the renderer uses, act(param); the step applies the
 * activation's derivative itself.  d_activated (may be NULL) receives act(param) after the step,
 * e.g. the scales or opacities rs_project reads. */
typedef struct rs_adam_segment {
    float* d_param;
    const float* d_grad;
    float* d_m;
    float* d_v;
    float* d_activated;
    size_t count;
    float lr;
    int32_t activation;   /* RS_ACT_* */
} rs_adam_segment;

/* Adam (Kingma & Ba) over up to RS_ADAM_MAX_SEGMENTS groups in one launch, step >= 1:
 *   g = dL/dact * act'(param); m = b1 m + (1 - b1) g; v = b2 v + (1 - b2) g^2;
 *   param -= lr * (m / (1 - b1^step)) / (sqrt(v / (1 - b2^step)) + eps).
 * `segs` is a host array; segments must not overlap.  beta1, beta2 and eps are taken in double:
 * 1 - beta is formed before rounding to float32 (0.999 has no float32 value close enough for
 * 1 - 0.999 to keep more than 4 digits).  Errors: RS_ERR_INVALID_ARG, RS_ERR_CUDA. */
int rs_adam_step(const rs_adam_segment* segs, int32_t n_segs, double beta1, double beta2, double eps,
                 int32_t step, void* stream);

/* Densification statistics (rigel README, "densify/prune" driven by the view-space gradient):
 * for every Gaussian with radius > 0 in this view, d_accum[i] += |dL/dmeans2d_i| (Euclidean norm
 * of d_dL_dmeans2d [2][n]) and d_count[i] += 1; others are left unchanged.  Errors:
 * RS_ERR_INVALID_ARG, RS_ERR_CUDA. */
int rs_densify_stats(int32_t n, const float* d_dL_dmeans2d, const int32_t* d_radius, float* d_accum,
                     float* d_count, void* stream);

/* Densification: clone, split and prune (rigel README: "GaussianModel: activations,
 * densify/prune"; its training log reports clone / split / prune counts per densification, and
 * densification and pruning must leave every parameter and its Adam moments the same length).
 * The pages do not state the criteria; these are 3D Gaussian Splatting's adaptive density control.
 * Per Gaussian i, with g_i = accum_i / count_i the mean view-space gradient norm (rs_densify_stats;
 * no growth when count_i = 0) and s_max the largest of exp(log-scales):
 *   - g_i >= grad_threshold and s_max <= dense_scale: cloned (kept, plus an identical copy);
 *   - g_i >= grad_threshold and s_max > dense_scale: split into two children at
 *     mean + R(q) (s * z_c) (R the rotation of the normalised quaternion, s = exp(log-scales),
 *     z_c the caller's standard normal draws) with log-scales log(s / 1.6), the rest copied; the
 *     parent is removed;
 *   - otherwise kept;
 * and then every Gaussian the step would produce whose opacity sigmoid(logit) is below
 * min_opacity, or whose largest scale exceeds max_scale (when max_scale > 0), is removed (split
 * children are tested with their own scales).  The comparisons run on the stored values:
 * max log-scale against ln(dense_scale) and ln(max_scale), the logit against
 * logit(min_opacity), accum against grad_threshold * count, in float32.
 * Output order: the kept originals in index order, then the clones in the order of their sources,
 * then every split Gaussian's first child in index order, then the second children.  Clones and
 * children start with zero Adam moments; kept Gaussians keep theirs. */
#define RS_DENSIFY_COPY 0        /* copied to every output of the Gaussian                       */
#define RS_DENSIFY_MEANS 1       /* [3][n] means: split children are moved by R(q) (s * z_c)      */
#define RS_DENSIFY_LOG_SCALES 2  /* [3][n] log-scales: split children get log(s / 1.6)           */
#define RS_DENSIFY_MAX_GROUPS 8

typedef struct rs_densify_rule {
    float grad_threshold;   /* on accum / count (3DGS: 0.0002)                                  */
    float dense_scale;      /* > 0: clone at most this largest scale, split above it             */
    float min_opacity;      /* in [0, 1): prune below this opacity (3DGS: 0.005)                 */
    float max_scale;        /* prune above this largest scale; <= 0: no size test                */
} rs_densify_rule;

/* One parameter array [rows][n] and its Adam moments (d_m, d_v may be NULL: no moments), moved
 * to [rows][n_out] outputs (d_m_out, d_v_out may be NULL).  kind RS_DENSIFY_MEANS and
 * RS_DENSIFY_LOG_SCALES need rows = 3. */
typedef struct rs_densify_group {
    const float* d_param;
    const float* d_m;
    const float* d_v;
    float* d_param_out;
    float* d_m_out;
    float* d_v_out;
    int32_t rows;
    int32_t kind;           /* RS_DENSIFY_* */
} rs_densify_group;

/* Workspace bytes of rs_densify_plan / rs_densify_apply for n Gaussians (0 if n is invalid). */
size_t rs_densify_workspace_size(int32_t n);

/* Classifies every Gaussian and counts the outputs; reads the counts back to the host (one
 * stream-ordered copy and a synchronisation of `stream`: the caller allocates the outputs with
 * them).  Inputs: d_accum [n], d_count [n] (rs_densify_stats), d_log_scales [3][n],
 * d_opacity_logits [n].  counts (host int32[5]): n_out, originals kept (cloned ones included),
 * clones, Gaussians split, Gaussians removed.  d_action (device uint8 [n], may be NULL) receives
 * each Gaussian's fate: 0 removed, 1 kept, 2 kept and cloned, 3 split.  d_workspace:
 * rs_densify_workspace_size(n) bytes, 256-byte aligned; it keeps the classification for
 * rs_densify_apply.  Errors: RS_ERR_INVALID_ARG, RS_ERR_WORKSPACE, RS_ERR_CAPACITY (n_out above
 * RS_MAX_GAUSSIANS; counts are still written), RS_ERR_CUDA. */
int rs_densify_plan(int32_t n, const float* d_accum, const float* d_count, const float* d_log_scales,
                    const float* d_opacity_logits, const rs_densify_rule* rule, void* d_workspace,
                    size_t workspace_bytes, uint8_t* d_action, int32_t* counts, void* stream);

/* Writes the densified arrays of up to RS_DENSIFY_MAX_GROUPS groups in one launch, from the
 * classification rs_densify_plan left in d_workspace (same n, same inputs).  d_quats [4][n] and
 * d_log_scales [3][n] are the Gaussians' current quaternions and log-scales (the split offsets),
 * d_noise [2][3][n] standard normal draws (child c, component k of Gaussian i at
 * (c * 3 + k) * n + i).  n_out: counts[0] of the plan; outputs are [rows][n_out] and must not
 * overlap the inputs.  Errors: RS_ERR_INVALID_ARG, RS_ERR_WORKSPACE, RS_ERR_CUDA. */
int rs_densify_apply(int32_t n, const void* d_workspace, size_t workspace_bytes, const float* d_quats,
                     const float* d_log_scales, const float* d_noise, const rs_densify_group* groups,
                     int32_t n_groups, int32_t n_out, void* stream);

/* Allocation-free variant of rs_bin.  The source pages have no counterpart: this entry point
 * exists for callers of this library that cannot allocate device memory -- for example a plug-in
 * whose host application owns and budgets all device memory, or a per-frame loop that must not
 * call cudaMalloc because an allocation synchronises the device and has unbounded latency.
 * Arguments, outputs and errors are those of rs_bin, except that there is no workspace: the
 * scratch is a fixed array of RS_BIN_NOALLOC_SCRATCH_BYTES bytes that is part of the library's
 * device image.  A GPU holds that array from the moment the array's module is loaded on it (with
 * the runtime's lazy module loading, at the first rs_bin_noalloc call on that GPU, see Set-up)
 * until the process exits.
 *  - Limit: the call returns RS_ERR_WORKSPACE, before any work, when
 *    rs_bin_workspace_size(n, camera, capacity) exceeds RS_BIN_NOALLOC_SCRATCH_BYTES
 *    (48 MiB: about 3.5 million entries for 160,000 Gaussians at 1920x1080).
 *  - Set-up: the first call on a device, with that device current, looks up the array's device
 *    address (cudaGetSymbolAddress) and keeps it for later calls.  Under the CUDA runtime's lazy
 *    module loading (its default) that lookup is also what loads the array onto the device, so
 *    this first call may allocate device memory and synchronise: make it once, as a warm-up,
 *    outside any region where allocation is not allowed and before any stream capture.  If the
 *    lookup fails the call returns RS_ERR_CUDA and the next call tries again.
 *  - On RS_ERR_CUDA the call waits for `stream` before returning, so no work of the call still
 *    uses the array when it returns.
 *  - Sharing: all calls use the same array and it keeps the last call's contents; nothing in it
 *    needs to start at zero.  Calls whose work overlaps on the GPU (other streams, other host
 *    threads on the same device) race on the array: serialise them.
 * The call itself allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine. */
#define RS_BIN_NOALLOC_SCRATCH_BYTES (48u << 20)
int rs_bin_noalloc(const rs_camera* camera, const rs_projected* proj, int32_t n, size_t capacity,
                   uint64_t* d_keys_sorted, uint32_t* d_point_list, uint32_t* d_tile_ranges,
                   size_t* n_entries, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* RS_H */
