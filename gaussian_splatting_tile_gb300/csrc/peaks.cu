// Throughput microbenchmarks behind the roofline's compute denominators (include/rs_peaks.h):
// the rate at which this GPU, at its current clock, issues the three instructions the
// compositing kernels are bound by -- single-precision fused multiply-adds, the multi-function
// unit's base-2 exponential, and fire-and-forget float atomics to scattered global addresses.
// Each kernel runs long independent chains, so the measured rate is the pipe's, not a latency.
#include "rs_internal.cuh"
#include "rs_peaks.h"

namespace {

constexpr int kThreads = 256;
constexpr int kChains = 8;    // independent dependency chains per thread
constexpr int kUnroll = 32;   // chain steps per loop trip

// kChains x kUnroll FMAs per trip; the result reaches memory only if it is impossible, so the
// compiler keeps every FMA but nothing is written.
__global__ void __launch_bounds__(kThreads) k_peak_ffma(int iters, float* sink) {
    float a[kChains];
    const float m = 1.0f - 1e-7f * float(threadIdx.x & 7), c = 1e-7f;
#pragma unroll
    for (int j = 0; j < kChains; ++j) a[j] = float(threadIdx.x + j);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
#pragma unroll
            for (int j = 0; j < kChains; ++j) a[j] = fmaf(a[j], m, c);
        }
    }
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kChains; ++j) s += a[j];
    if (s == -1.2345f) sink[blockIdx.x * kThreads + threadIdx.x] = s;
}

// x <- 2^(-x): bounded (the iteration settles near 0.64), one ex2 per step and chain.
__global__ void __launch_bounds__(kThreads) k_peak_ex2(int iters, float* sink) {
    float a[kChains];
#pragma unroll
    for (int j = 0; j < kChains; ++j) a[j] = 0.01f * float((threadIdx.x + j) & 63);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
#pragma unroll
            for (int j = 0; j < kChains; ++j) a[j] = rs::ex2_approx(-a[j]);
        }
    }
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kChains; ++j) s += a[j];
    if (s == -1.2345f) sink[blockIdx.x * kThreads + threadIdx.x] = s;
}

// Each lane adds to its own scattered word of a buffer of n words, `iters` times: the lanes of
// a warp hit 32 different 128-byte lines (as the compositing backward's per-Gaussian sums do).
__global__ void __launch_bounds__(kThreads) k_peak_red(int iters, float* target, uint32_t n) {
    const uint32_t tid = blockIdx.x * kThreads + threadIdx.x;
    uint32_t idx = (tid * 2654435761u) % n;
    const uint32_t step = 40503u * 33u;
    for (int i = 0; i < iters; ++i) {
        atomicAdd(target + idx, 1.0f);  // result unused: a red.global.add.f32
        idx += step;
        if (idx >= n) idx -= n * (idx / n);
    }
}

}  // namespace

extern "C" {

int rs_peak_ffma(int32_t blocks, int32_t iters, float* d_sink, double* lane_ops, void* stream) {
    if (blocks < 1 || iters < 1 || !d_sink || !lane_ops) return RS_ERR_INVALID_ARG;
    k_peak_ffma<<<blocks, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(iters, d_sink);
    *lane_ops = double(blocks) * kThreads * double(iters) * kUnroll * kChains;
    return cudaGetLastError() == cudaSuccess ? RS_OK : RS_ERR_CUDA;
}

int rs_peak_ex2(int32_t blocks, int32_t iters, float* d_sink, double* lane_ops, void* stream) {
    if (blocks < 1 || iters < 1 || !d_sink || !lane_ops) return RS_ERR_INVALID_ARG;
    k_peak_ex2<<<blocks, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(iters, d_sink);
    *lane_ops = double(blocks) * kThreads * double(iters) * kUnroll * kChains;
    return cudaGetLastError() == cudaSuccess ? RS_OK : RS_ERR_CUDA;
}

int rs_peak_red(int32_t blocks, int32_t iters, float* d_target, uint32_t n_targets, double* red_ops,
                void* stream) {
    if (blocks < 1 || iters < 1 || !d_target || n_targets < 1 || n_targets > (1u << 30) || !red_ops)
        return RS_ERR_INVALID_ARG;
    k_peak_red<<<blocks, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(iters, d_target, n_targets);
    *red_ops = double(blocks) * kThreads * double(iters);
    return cudaGetLastError() == cudaSuccess ? RS_OK : RS_ERR_CUDA;
}

int rs_device_sm_count(int32_t* sms) {
    if (!sms) return RS_ERR_INVALID_ARG;
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return RS_ERR_CUDA;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return RS_ERR_CUDA;
    *sms = v;
    return RS_OK;
}

}  // extern "C"
