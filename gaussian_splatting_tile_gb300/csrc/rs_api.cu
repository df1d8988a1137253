// The C ABI of include/rs.h: argument validation, then the kernel launchers.  No device memory
// is allocated here; rs_bin performs the path's single device-to-host read (the entry count).
#include <stdint.h>

#include "rs_internal.cuh"

namespace {

using rs::CameraF;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool camera_ok(const rs_camera* c) {
    if (!c) return false;
    if (c->width < 1 || c->height < 1 || c->width > 32768 || c->height > 32768) return false;
    if (!(c->fx > 0.f) || !(c->fy > 0.f)) return false;
    const float v[] = {c->fx, c->fy, c->cx, c->cy};
    for (float x : v)
        if (!isfinite(x)) return false;
    for (int i = 0; i < 9; ++i)
        if (!isfinite(c->R[i])) return false;
    for (int i = 0; i < 3; ++i)
        if (!isfinite(c->t[i])) return false;
    return true;
}

bool n_ok(int32_t n) { return n >= 0 && n <= RS_MAX_GAUSSIANS; }

bool dev_f(const void* p) { return p && aligned(p, 4); }

bool gaussians_ok(const rs_gaussians* g) {
    if (!g || !n_ok(g->n)) return false;
    if (g->sh_degree < -1 || g->sh_degree > 3) return false;
    if (g->n == 0) return true;
    if (!dev_f(g->d_means) || !dev_f(g->d_scales) || !dev_f(g->d_quats) || !dev_f(g->d_opacity))
        return false;
    if (g->sh_degree >= 0 ? !dev_f(g->d_sh) : !dev_f(g->d_colors)) return false;
    return true;
}

bool projected_ok(const rs_projected* p, bool need_records) {
    if (!p) return false;
    if (!dev_f(p->d_means2d) || !dev_f(p->d_depth) || !dev_f(p->d_conic) || !dev_f(p->d_color) ||
        !dev_f(p->d_radius) || !dev_f(p->d_tiles_touched))
        return false;
    if (need_records && !(p->d_records && aligned(p->d_records, 16))) return false;
    if (p->tile_test != RS_TILE_TEST_SQUARE && p->tile_test != RS_TILE_TEST_ELLIPSE) return false;
    if (p->tile_test == RS_TILE_TEST_ELLIPSE && !dev_f(p->d_ellipse)) return false;
    return true;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? RS_OK : RS_ERR_CUDA; }

bool mlp_ok(const rs_mlp* m) {
    if (!m) return false;
    if (m->hidden != 32 && m->hidden != 64) return false;
    if (m->latent_dim < 1 || m->latent_dim > 29) return false;
    return dev_f(m->d_W1) && dev_f(m->d_b1) && dev_f(m->d_W2) && dev_f(m->d_b2);
}

}  // namespace

extern "C" {

const char* rs_error_string(int code) {
    switch (code) {
        case RS_OK: return "success";
        case RS_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad size or parameter)";
        case RS_ERR_CAPACITY: return "entry count exceeds capacity; *n_entries holds the required count";
        case RS_ERR_WORKSPACE: return "workspace smaller than rs_bin_workspace_size reports";
        case RS_ERR_CUDA: return "CUDA runtime error";
        case RS_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel gave up; the outputs are not valid";
        case RS_ERR_DEVICE_CHECK:
            return "a kernel found an index in the caller's data out of range and skipped it; the outputs are not valid";
        default: return "unknown error code";
    }
}

int rs_project(const rs_camera* camera, const rs_gaussians* gaussians, const rs_projected* out,
               void* stream) {
    if (!camera_ok(camera) || !gaussians_ok(gaussians)) return RS_ERR_INVALID_ARG;
    if (gaussians->n == 0) return RS_OK;
    if (!projected_ok(out, true)) return RS_ERR_INVALID_ARG;
    const CameraF cam = rs::make_camera(*camera);
    return cuda_rc(rs::launch_project(cam, *gaussians, *out, static_cast<cudaStream_t>(stream)));
}

int rs_bin_workspace_size(int32_t n, const rs_camera* camera, size_t capacity, size_t* bytes) {
    if (!camera_ok(camera) || !n_ok(n) || !bytes || capacity > size_t(RS_MAX_ENTRIES))
        return RS_ERR_INVALID_ARG;
    const CameraF cam = rs::make_camera(*camera);
    *bytes = rs::plan_bin(n, cam, capacity).total_bytes;
    return RS_OK;
}

}  // extern "C"

namespace {

// Validation and launches shared by rs_bin and rs_bin_async; on RS_OK the binning is enqueued
// and *result_dev points at the workspace's {E (uint64), error (uint32), pad} block.
int enqueue_bin(const rs_camera* camera, const rs_projected* proj, int32_t n, void* d_workspace,
                size_t workspace_bytes, size_t capacity, uint64_t* d_keys_sorted,
                uint32_t* d_point_list, uint32_t* d_tile_ranges, cudaStream_t s,
                const uint8_t** result_dev) {
    if (!camera_ok(camera) || !n_ok(n) || capacity > size_t(RS_MAX_ENTRIES)) return RS_ERR_INVALID_ARG;
    if (!d_tile_ranges || !aligned(d_tile_ranges, 8)) return RS_ERR_INVALID_ARG;
    if (!d_workspace || !aligned(d_workspace, 256)) return RS_ERR_INVALID_ARG;
    if (n > 0 && !projected_ok(proj, false)) return RS_ERR_INVALID_ARG;
    if (capacity > 0 && (!d_point_list || !aligned(d_point_list, 4))) return RS_ERR_INVALID_ARG;
    if (d_keys_sorted && !aligned(d_keys_sorted, 8)) return RS_ERR_INVALID_ARG;
    const CameraF cam = rs::make_camera(*camera);
    const rs::BinPlan plan = rs::plan_bin(n, cam, capacity);
    if (workspace_bytes < plan.total_bytes) return RS_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(d_workspace);
    rs_projected empty{};
    const rs_projected& p = proj ? *proj : empty;
    cudaError_t e = rs::launch_bin(plan, cam, p, ws, d_keys_sorted, d_point_list, d_tile_ranges, s);
    if (e != cudaSuccess) return RS_ERR_CUDA;
    *result_dev = ws + plan.off_result;
    return RS_OK;
}

}  // namespace

extern "C" {

int rs_bin(const rs_camera* camera, const rs_projected* proj, int32_t n, void* d_workspace,
           size_t workspace_bytes, size_t capacity, uint64_t* d_keys_sorted,
           uint32_t* d_point_list, uint32_t* d_tile_ranges, size_t* n_entries, void* stream) {
    if (!n_entries) return RS_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint8_t* dev = nullptr;
    const int rc = enqueue_bin(camera, proj, n, d_workspace, workspace_bytes, capacity, d_keys_sorted,
                               d_point_list, d_tile_ranges, s, &dev);
    if (rc != RS_OK) return rc;
    // the path's one device-to-host read: the entry count (and the sort's wait flag)
    struct {
        uint64_t E;
        uint32_t error, pad;
    } result{};
    cudaError_t e = cudaMemcpyAsync(&result, dev, sizeof(result), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return RS_ERR_CUDA;
    *n_entries = size_t(result.E);
    if (result.E > uint64_t(capacity)) return RS_ERR_CAPACITY;
    if (result.error != 0) return RS_ERR_DEVICE_TIMEOUT;
    return RS_OK;
}

int rs_bin_async(const rs_camera* camera, const rs_projected* proj, int32_t n, void* d_workspace,
                 size_t workspace_bytes, size_t capacity, uint64_t* d_keys_sorted,
                 uint32_t* d_point_list, uint32_t* d_tile_ranges, uint64_t* h_result, void* stream) {
    if (!h_result || !aligned(h_result, 8)) return RS_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint8_t* dev = nullptr;
    const int rc = enqueue_bin(camera, proj, n, d_workspace, workspace_bytes, capacity, d_keys_sorted,
                               d_point_list, d_tile_ranges, s, &dev);
    if (rc != RS_OK) return rc;
    // pinned host memory is in the device's address space under unified addressing: a one-thread
    // kernel writes the two words there, so the frame has no copy (a copy would queue behind
    // other transfers on the copy engine); memory that is not mapped gets a copy instead
    void* mapped = nullptr;
    if (cudaHostGetDevicePointer(&mapped, h_result, 0) == cudaSuccess && mapped)
        return cuda_rc(rs::launch_report(dev, static_cast<uint64_t*>(mapped), s));
    (void)cudaGetLastError();  // the failed lookup is not an error of this call
    return cuda_rc(cudaMemcpyAsync(h_result, dev, 2 * sizeof(uint64_t), cudaMemcpyDeviceToHost, s));
}

size_t rs_raster_workspace_size(const rs_camera* camera, size_t capacity) {
    if (!camera_ok(camera) || capacity > size_t(RS_MAX_ENTRIES)) return 0;
    const CameraF cam = rs::make_camera(*camera);
    return rs::raster_workspace_bytes(capacity, size_t(cam.TX) * cam.TY);
}

int rs_rasterize_fwd(const rs_camera* camera, const rs_projected* proj, int32_t n,
                     const uint32_t* d_tile_ranges, const uint32_t* d_point_list, size_t capacity,
                     const float* bg, float* d_image, float* d_final_T, uint32_t* d_n_contrib,
                     void* d_workspace, size_t workspace_bytes, void* stream) {
    if (!camera_ok(camera) || !n_ok(n) || !bg || capacity > size_t(RS_MAX_ENTRIES)) return RS_ERR_INVALID_ARG;
    if (!dev_f(d_image) || !dev_f(d_final_T) || !dev_f(d_n_contrib)) return RS_ERR_INVALID_ARG;
    const CameraF cam = rs::make_camera(*camera);
    const float3 b = make_float3(bg[0], bg[1], bg[2]);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (n == 0) return cuda_rc(rs::launch_fill_background(cam, b, d_image, d_final_T, d_n_contrib, s));
    if (!proj || !proj->d_records || !aligned(proj->d_records, 16)) return RS_ERR_INVALID_ARG;
    if (!d_tile_ranges || !aligned(d_tile_ranges, 8) || !dev_f(d_point_list)) return RS_ERR_INVALID_ARG;
    if (!d_workspace || !aligned(d_workspace, 16)) return RS_ERR_INVALID_ARG;
    if (workspace_bytes < rs::raster_workspace_bytes(capacity, size_t(cam.TX) * cam.TY)) return RS_ERR_WORKSPACE;
    return cuda_rc(rs::launch_raster_fwd(cam, n, static_cast<const rs::Record*>(proj->d_records),
                                         d_tile_ranges, d_point_list, capacity, b, d_image, d_final_T,
                                         d_n_contrib, d_workspace, s));
}

int rs_rasterize_bwd(const rs_camera* camera, const rs_projected* proj, int32_t n,
                     const uint32_t* d_tile_ranges, const uint32_t* d_point_list, size_t capacity,
                     const float* bg, const float* d_final_T, const uint32_t* d_n_contrib,
                     void* d_workspace, size_t workspace_bytes,
                     const float* d_dL_dimage, float* d_dL_dmeans2d, float* d_dL_dconic,
                     float* d_dL_dopacity, float* d_dL_dcolor, void* stream) {
    if (!camera_ok(camera) || !n_ok(n) || !bg || capacity > size_t(RS_MAX_ENTRIES)) return RS_ERR_INVALID_ARG;
    if (n == 0) return RS_OK;
    if (!proj || !proj->d_records || !aligned(proj->d_records, 16)) return RS_ERR_INVALID_ARG;
    if (!d_tile_ranges || !aligned(d_tile_ranges, 8) || !dev_f(d_point_list)) return RS_ERR_INVALID_ARG;
    if (!dev_f(d_final_T) || !dev_f(d_n_contrib) || !dev_f(d_dL_dimage)) return RS_ERR_INVALID_ARG;
    if (!dev_f(d_dL_dmeans2d) || !dev_f(d_dL_dconic) || !dev_f(d_dL_dopacity) || !dev_f(d_dL_dcolor))
        return RS_ERR_INVALID_ARG;
    if (!d_workspace || !aligned(d_workspace, 16)) return RS_ERR_INVALID_ARG;
    const CameraF cam = rs::make_camera(*camera);
    if (workspace_bytes < rs::raster_workspace_bytes(capacity, size_t(cam.TX) * cam.TY)) return RS_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (rs::launch_zero_grads(d_dL_dmeans2d, d_dL_dconic, d_dL_dopacity, d_dL_dcolor, size_t(n), s) !=
        cudaSuccess)
        return RS_ERR_CUDA;
    const float3 b = make_float3(bg[0], bg[1], bg[2]);
    return cuda_rc(rs::launch_raster_bwd(cam, n, static_cast<const rs::Record*>(proj->d_records),
                                         d_tile_ranges, d_point_list, capacity, b, d_final_T,
                                         d_n_contrib, d_workspace, d_dL_dimage, d_dL_dmeans2d, d_dL_dconic,
                                         d_dL_dopacity, d_dL_dcolor, s));
}

int rs_project_bwd(const rs_camera* camera, const rs_gaussians* gaussians,
                   const rs_projected* proj, const float* d_dL_dmeans2d,
                   const float* d_dL_dconic, const float* d_dL_dcolor, float* d_dL_dmeans,
                   float* d_dL_dscales, float* d_dL_dquats, float* d_dL_dsh, void* stream) {
    if (!camera_ok(camera) || !gaussians_ok(gaussians)) return RS_ERR_INVALID_ARG;
    if (gaussians->n == 0) return RS_OK;
    if (!proj || !dev_f(proj->d_radius)) return RS_ERR_INVALID_ARG;
    if (!dev_f(d_dL_dmeans2d) || !dev_f(d_dL_dconic) || !dev_f(d_dL_dcolor)) return RS_ERR_INVALID_ARG;
    if (!dev_f(d_dL_dmeans) || !dev_f(d_dL_dscales) || !dev_f(d_dL_dquats)) return RS_ERR_INVALID_ARG;
    if (gaussians->sh_degree >= 0 && !dev_f(d_dL_dsh)) return RS_ERR_INVALID_ARG;
    const CameraF cam = rs::make_camera(*camera);
    return cuda_rc(rs::launch_project_bwd(cam, *gaussians, *proj, d_dL_dmeans2d, d_dL_dconic,
                                          d_dL_dcolor, d_dL_dmeans, d_dL_dscales, d_dL_dquats,
                                          d_dL_dsh, static_cast<cudaStream_t>(stream)));
}

int rs_appearance_fwd(const rs_camera* camera, int32_t n, const float* d_means,
                      const float* d_latents, const rs_mlp* mlp, float* d_colors, void* stream) {
    if (!camera_ok(camera) || !n_ok(n) || !mlp_ok(mlp)) return RS_ERR_INVALID_ARG;
    if (n == 0) return RS_OK;
    if (!dev_f(d_means) || !dev_f(d_latents) || !dev_f(d_colors)) return RS_ERR_INVALID_ARG;
    const CameraF cam = rs::make_camera(*camera);
    return cuda_rc(rs::launch_appearance_fwd(cam, n, d_means, d_latents, *mlp, d_colors,
                                             static_cast<cudaStream_t>(stream)));
}

int rs_appearance_bwd(const rs_camera* camera, int32_t n, const float* d_means,
                      const float* d_latents, const rs_mlp* mlp, const float* d_dL_dcolors,
                      float* d_dL_dlatents, const rs_mlp_grads* grads, void* stream) {
    if (!camera_ok(camera) || !n_ok(n) || !mlp_ok(mlp) || !grads) return RS_ERR_INVALID_ARG;
    if (!dev_f(grads->d_dW1) || !dev_f(grads->d_db1) || !dev_f(grads->d_dW2) || !dev_f(grads->d_db2))
        return RS_ERR_INVALID_ARG;
    if (n > 0 && (!dev_f(d_means) || !dev_f(d_latents) || !dev_f(d_dL_dcolors) || !dev_f(d_dL_dlatents)))
        return RS_ERR_INVALID_ARG;
    const CameraF cam = rs::make_camera(*camera);
    return cuda_rc(rs::launch_appearance_bwd(cam, n, d_means, d_latents, *mlp, d_dL_dcolors,
                                             d_dL_dlatents, *grads, static_cast<cudaStream_t>(stream)));
}

int rs_l1_loss_grad(size_t count, const float* d_image, const float* d_target, float scale,
                    float* d_dL_dimage, float* d_loss, void* stream) {
    if (!isfinite(scale)) return RS_ERR_INVALID_ARG;
    if (d_loss && !aligned(d_loss, 4)) return RS_ERR_INVALID_ARG;
    if (count > 0 && (!dev_f(d_image) || !dev_f(d_target) || !dev_f(d_dL_dimage))) return RS_ERR_INVALID_ARG;
    return cuda_rc(rs::launch_l1(count, d_image, d_target, scale, d_dL_dimage, d_loss,
                                 static_cast<cudaStream_t>(stream)));
}

int rs_adam_step(const rs_adam_segment* segs, int32_t n_segs, double beta1, double beta2, double eps,
                 int32_t step, void* stream) {
    if (!segs || n_segs < 0 || n_segs > RS_ADAM_MAX_SEGMENTS || step < 1) return RS_ERR_INVALID_ARG;
    if (!(beta1 >= 0.0 && beta1 < 1.0) || !(beta2 >= 0.0 && beta2 < 1.0) || !(eps > 0.0) || !isfinite(eps))
        return RS_ERR_INVALID_ARG;
    for (int i = 0; i < n_segs; ++i) {
        const rs_adam_segment& g = segs[i];
        if (g.activation < RS_ACT_IDENTITY || g.activation > RS_ACT_SIGMOID || !isfinite(g.lr)) return RS_ERR_INVALID_ARG;
        if (g.count == 0) continue;
        if (!dev_f(g.d_param) || !dev_f(g.d_grad) || !dev_f(g.d_m) || !dev_f(g.d_v)) return RS_ERR_INVALID_ARG;
        if (g.d_activated && !aligned(g.d_activated, 4)) return RS_ERR_INVALID_ARG;
    }
    return cuda_rc(rs::launch_adam(segs, n_segs, beta1, beta2, eps, step, static_cast<cudaStream_t>(stream)));
}

int rs_densify_stats(int32_t n, const float* d_dL_dmeans2d, const int32_t* d_radius, float* d_accum,
                     float* d_count, void* stream) {
    if (!n_ok(n)) return RS_ERR_INVALID_ARG;
    if (n > 0 && (!dev_f(d_dL_dmeans2d) || !dev_f(d_radius) || !dev_f(d_accum) || !dev_f(d_count)))
        return RS_ERR_INVALID_ARG;
    return cuda_rc(rs::launch_densify_stats(n, d_dL_dmeans2d, d_radius, d_accum, d_count,
                                            static_cast<cudaStream_t>(stream)));
}

int rs_device_error(void) {
    const int a = rs::take_device_error(), b = rs::take_projection_error(), c = rs::take_raster_check();
    if (a < 0 || b < 0 || c < 0) return RS_ERR_CUDA;
    return c > 0 ? RS_ERR_DEVICE_CHECK : a > 0 || b > 0 ? RS_ERR_DEVICE_TIMEOUT : RS_OK;
}

int rs_l1_dssim_workspace_size(int32_t channels, int32_t height, int32_t width, size_t* bytes) {
    if (channels < 1 || height < 1 || width < 1 || height > 32768 || width > 32768 || channels > 64 || !bytes)
        return RS_ERR_INVALID_ARG;
    *bytes = rs::ssim_workspace_bytes(channels, height, width);
    return RS_OK;
}

int rs_l1_dssim_loss_grad(int32_t channels, int32_t height, int32_t width, const float* d_image,
                          const float* d_target, float lambda, float scale, float* d_dL_dimage,
                          float* d_loss, void* d_workspace, size_t workspace_bytes, void* stream) {
    size_t need = 0;
    if (rs_l1_dssim_workspace_size(channels, height, width, &need) != RS_OK) return RS_ERR_INVALID_ARG;
    if (!(lambda >= 0.f && lambda <= 1.f) || !isfinite(scale)) return RS_ERR_INVALID_ARG;
    if (!dev_f(d_image) || !dev_f(d_target) || !dev_f(d_dL_dimage)) return RS_ERR_INVALID_ARG;
    if (d_loss && !aligned(d_loss, 4)) return RS_ERR_INVALID_ARG;
    if (!d_workspace || !aligned(d_workspace, 16)) return RS_ERR_INVALID_ARG;
    if (workspace_bytes < need) return RS_ERR_WORKSPACE;
    return cuda_rc(rs::launch_l1_dssim(channels, height, width, d_image, d_target, lambda, scale, d_dL_dimage,
                                       d_loss, d_workspace, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
