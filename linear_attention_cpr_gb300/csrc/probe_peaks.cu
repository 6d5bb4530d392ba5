// probe_peaks.cu — measures the FP32-pipe peak of this GPU (the roofline denominator
// of the FP32-bound kernels), with scalar FFMA and with paired f32x2 FMA.
//
// extern "C" int cpr_probe_fp32(int paired, int blocks, int threads, int iters,
//                               float* sink, float* ms_out, void* stream)
//   Runs blocks x threads threads, each advancing 16 independent FMA chains (16 scalar
//   lanes, or 16 pairs when paired != 0) for `iters` rounds; returns the kernel time
//   in ms (CUDA events on `stream`).  FLOPs = blocks*threads*iters*16*2*(paired?2:1).
//   sink: device buffer of blocks*threads floats (defeats dead-code elimination).
// extern "C" int cpr_probe_decay_exp(const float* x, float* y, int n, void* stream)
//   The library's decay exponential (numerics.cuh) on n device floats, for its tests.
#include <cuda_runtime.h>

#include "numerics.cuh"

namespace {

__global__ void probe_decay_exp(const float* x, float* y, int n)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) y[i] = cpr::decay_exp(x[i]);
}

__global__ void __launch_bounds__(256) probe_ffma(float* sink, int iters, float a, float b)
{
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = threadIdx.x * 1e-7f + i;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = __fmaf_rn(x[i], a, b);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) s += x[i];
    sink[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void __launch_bounds__(256) probe_ffma2(float* sink, int iters, float a, float b)
{
    float2 x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = make_float2(threadIdx.x * 1e-7f + i, i * 0.5f);
    const float2 a2 = make_float2(a, a), b2 = make_float2(b, b);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = __ffma2_rn(x[i], a2, b2);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) s += x[i].x + x[i].y;
    sink[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

}  // namespace

extern "C" int cpr_probe_fp32(int paired, int blocks, int threads, int iters, float* sink, float* ms_out,
                              void* stream)
{
    if (blocks <= 0 || threads <= 0 || threads > 256 || iters <= 0 || !sink || !ms_out) return -1;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaEvent_t e0, e1;
    if (cudaEventCreate(&e0) != cudaSuccess) return -5;
    if (cudaEventCreate(&e1) != cudaSuccess) {
        cudaEventDestroy(e0);
        return -5;
    }
    cudaEventRecord(e0, s);
    if (paired)
        probe_ffma2<<<blocks, threads, 0, s>>>(sink, iters, 0.999999f, 1e-6f);
    else
        probe_ffma<<<blocks, threads, 0, s>>>(sink, iters, 0.999999f, 1e-6f);
    cudaEventRecord(e1, s);
    cudaError_t err = cudaEventSynchronize(e1);
    float ms = 0.f;
    if (err == cudaSuccess) err = cudaEventElapsedTime(&ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (err != cudaSuccess) return -5;
    *ms_out = ms;
    return 0;
}

// The library's decay exponential applied to n device floats (test hook): y[i] = e^x[i].
extern "C" int cpr_probe_decay_exp(const float* x, float* y, int n, void* stream)
{
    if (!x || !y || n < 0) return -1;
    if (n == 0) return 0;
    probe_decay_exp<<<(n + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, y, n);
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
}
