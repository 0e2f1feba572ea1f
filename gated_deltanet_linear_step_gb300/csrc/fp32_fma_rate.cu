// FP32 FMA throughput of the device, measured: the denominator the ALU-bound decode kernels
// (the tensor-core window kernel's FP32 work, the register tile's token step) are compared with,
// beside the figure derived from the SM count, the 128 FP32 lanes of an SM and the maximum clock.
//
// A standalone program, not part of libgdn.so. Every thread runs kChains independent FMA chains
// (acc = acc * a + b, with a and b runtime arguments so nothing folds), unrolled so the loop
// counter costs a small fraction of the issue slots. Two forms are timed:
//   scalar  fmaf on float, one FMA per lane per instruction;
//   packed  __ffma2_rn on float2, two FMAs per lane per instruction (the form the window kernels'
//           pass A and update use).
// The grid is 4 CTAs of 256 threads per SM (32 warps per SM, 8 per scheduler); 16 independent
// chains per thread cover the FMA latency many times over. Each launch is timed with CUDA events
// after warm-up; the line printed gives the best and median of the timed launches.
//
// Usage: fp32_fma_rate [iterations per launch] [timed launches]
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <vector>

namespace {

constexpr int kThreads = 256;
constexpr int kCtasPerSm = 4;
constexpr int kChains = 16;  // independent accumulators per thread (float or float2)
constexpr int kUnroll = 16;  // FMA rounds per loop iteration

__global__ void __launch_bounds__(kThreads) fma_scalar(float* out, int iters, float a, float b) {
    float acc[kChains];
#pragma unroll
    for (int j = 0; j < kChains; ++j) acc[j] = 1e-3f * (threadIdx.x + j);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
#pragma unroll
            for (int j = 0; j < kChains; ++j) acc[j] = fmaf(acc[j], a, b);
        }
    }
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kChains; ++j) s += acc[j];
    out[blockIdx.x * kThreads + threadIdx.x] = s;
}

__global__ void __launch_bounds__(kThreads) fma_packed(float* out, int iters, float a, float b) {
    float2 acc[kChains];
    const float2 a2 = make_float2(a, a), b2 = make_float2(b, b);
#pragma unroll
    for (int j = 0; j < kChains; ++j) acc[j] = make_float2(1e-3f * (threadIdx.x + j), 2e-3f * (threadIdx.x + j));
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
#pragma unroll
            for (int j = 0; j < kChains; ++j) acc[j] = __ffma2_rn(acc[j], a2, b2);
        }
    }
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kChains; ++j) s += acc[j].x + acc[j].y;
    out[blockIdx.x * kThreads + threadIdx.x] = s;
}

#define CHECK(call)                                                                         \
    do {                                                                                    \
        cudaError_t e_ = (call);                                                            \
        if (e_ != cudaSuccess) {                                                            \
            std::fprintf(stderr, "%s failed: %s\n", #call, cudaGetErrorString(e_));         \
            std::exit(1);                                                                   \
        }                                                                                   \
    } while (0)

struct Timing {
    double best_ms, median_ms;
};

template <typename Kernel>
Timing time_kernel(Kernel k, int grid, float* out, int iters, int timed) {
    cudaEvent_t e0, e1;
    CHECK(cudaEventCreate(&e0));
    CHECK(cudaEventCreate(&e1));
    for (int w = 0; w < 3; ++w) k<<<grid, kThreads>>>(out, iters, 0.999f, 1e-4f);
    CHECK(cudaGetLastError());
    CHECK(cudaDeviceSynchronize());
    std::vector<double> ms;
    for (int r = 0; r < timed; ++r) {
        CHECK(cudaEventRecord(e0));
        k<<<grid, kThreads>>>(out, iters, 0.999f, 1e-4f);
        CHECK(cudaEventRecord(e1));
        CHECK(cudaEventSynchronize(e1));
        float t = 0.f;
        CHECK(cudaEventElapsedTime(&t, e0, e1));
        ms.push_back(t);
    }
    CHECK(cudaEventDestroy(e0));
    CHECK(cudaEventDestroy(e1));
    std::sort(ms.begin(), ms.end());
    return {ms.front(), ms[ms.size() / 2]};
}

}  // namespace

int main(int argc, char** argv) {
    const int iters = argc > 1 ? std::atoi(argv[1]) : 4096;
    const int timed = argc > 2 ? std::atoi(argv[2]) : 20;
    if (iters <= 0 || timed <= 0) {
        std::fprintf(stderr, "usage: fp32_fma_rate [iterations > 0] [timed launches > 0]\n");
        return 2;
    }
    int dev = 0, sms = 0, clock_khz = 0;
    CHECK(cudaGetDevice(&dev));
    CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    CHECK(cudaDeviceGetAttribute(&clock_khz, cudaDevAttrClockRate, dev));
    const int grid = sms * kCtasPerSm;
    float* out = nullptr;
    CHECK(cudaMalloc(&out, sizeof(float) * grid * kThreads));

    // FMAs per launch: threads x iterations x rounds x chains (x 2 lanes for the packed form).
    const double fmas = double(grid) * kThreads * iters * kUnroll * kChains;
    const Timing s = time_kernel(fma_scalar, grid, out, iters, timed);
    const Timing p = time_kernel(fma_packed, grid, out, iters, timed);
    const double derived = double(sms) * 128 * 2 * clock_khz * 1e3 / 1e12;
    auto tflops = [&](double flop, double ms) { return flop / (ms * 1e-3) / 1e12; };
    std::printf(
        "{\"metric\": \"fp32_fma_rate\", \"unit\": \"TFLOP/s\", \"sms\": %d, \"max_sm_mhz\": %d, "
        "\"derived_tflops\": %.2f, \"grid\": %d, \"threads\": %d, \"iterations\": %d, \"timed\": %d, "
        "\"scalar\": {\"best_ms\": %.4f, \"median_ms\": %.4f, \"tflops_best\": %.2f, \"tflops_median\": %.2f}, "
        "\"packed\": {\"best_ms\": %.4f, \"median_ms\": %.4f, \"tflops_best\": %.2f, \"tflops_median\": %.2f}}\n",
        sms, clock_khz / 1000, derived, grid, kThreads, iters, timed,
        s.best_ms, s.median_ms, tflops(2 * fmas, s.best_ms), tflops(2 * fmas, s.median_ms),
        p.best_ms, p.median_ms, tflops(4 * fmas, p.best_ms), tflops(4 * fmas, p.median_ms));
    CHECK(cudaFree(out));
    return 0;
}
