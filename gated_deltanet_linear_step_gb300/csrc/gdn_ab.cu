// gdn_ab.cu - the alpha/beta projections of a GDN layer with their gate
// epilogue, fused (the fused_gdn_ab stage of gdn_layer step 5 on the
// Winery-Strata page src/core/layer.cpp): for every (sequence b, layer l,
// token t) and v head h,
//
//   alpha_raw = x . Wa[l][h],  beta_raw = x . Wb[l][h]      (BF16 weights, fp32 activations, fp32 sums)
//   gate      = softplus(alpha_raw + dt[l][h]) * ssm_a[l][h] (the log of the decay)
//   beta      = sigmoid(beta_raw)
//
// x is read once for both projections. Per layer this is a small GEMM:
// [rows = B*T] x [n_embd] times [n_embd] x [96]. A cluster of kSplit CTAs takes
// 32 rows of one layer, each CTA a contiguous share of n_embd. x and both
// weight blocks stream through double-buffered shared memory (83 KB, dynamic)
// in 128-wide slices by 16-byte asynchronous copies; a share of an odd number
// of 64-wide units ends with one 64-wide slice, and both widths are compiled
// separately. Weight rows are padded by 16 bytes, so a thread reads eight
// weights of an output with one 16-byte load. Each of
// the 128 threads accumulates 4 rows x 6 outputs in fp32 registers, so every
// weight load feeds 32 FMAs. The partial sums then go to the weight buffers,
// which the main loop no longer needs, and meet in a reduce-scatter: rank r of
// the cluster adds the other ranks' sums for row r of each thread's four rows,
// read from their shared memory across the cluster with every load issued
// before any sum uses it, and applies the gate epilogue to that row. No global
// workspace is involved.

#include <cuda_bf16.h>

#include <mutex>
#include <type_traits>

#include "gdn_device.cuh"
#include "gdn_launch.h"

namespace gdn {
namespace {

constexpr int kAbThreads = 128;
constexpr int kRowsPerCta = 32;
constexpr int kOut = 2 * kVHeads;  // 96: alpha heads, then beta heads
constexpr int kKSlice = 128;       // n_embd elements per shared-memory slice
constexpr int kSplit = 4;          // CTAs per cluster, each summing a share of n_embd

using XsBuf = float[2][kRowsPerCta][kKSlice];
using WsBuf = __nv_bfloat16[2][kOut][kKSlice + 8];
constexpr size_t kAbSmem = sizeof(XsBuf) + sizeof(WsBuf);

struct AbParams {
    const float* x;          // [B][L][T][E]
    const uint16_t* wa;      // [L][48][E] bf16 bits
    const uint16_t* wb;      // [L][48][E] bf16 bits
    const float* dt;         // [L][48]
    const float* ssm_a;      // [L][48]
    float* gate;             // [B][L][T][48]
    float* beta;             // [B][L][T][48]
    int B, L, T, E;
};

__global__ void __launch_bounds__(kAbThreads, 1) gdn_ab_gates_kernel(const __grid_constant__ AbParams p) {
    extern __shared__ __align__(16) unsigned char ab_smem[];
    auto& xs = *reinterpret_cast<XsBuf*>(ab_smem);                  // double-buffered x slices
    auto& ws = *reinterpret_cast<WsBuf*>(ab_smem + sizeof(XsBuf));  // weight slices, rows padded by 16 bytes
    // This CTA's partial sums, in the weight buffers once the main loop is done with them.
    float (*part)[24] = reinterpret_cast<float (*)[24]>(&ws[0][0][0]);
    static_assert(sizeof(ws) >= sizeof(float) * kAbThreads * 24, "partial sums fit in the weight buffers");

    const int tid = threadIdx.x;
    const int l = blockIdx.y;
    const int rank = static_cast<int>(cluster_rank());
    const int M = p.B * p.T;                 // rows of this layer
    const int m0 = (blockIdx.x / kSplit) * kRowsPerCta;
    // This rank's share of n_embd, in 64-wide units, taken kKSlice wide at a time: when the share
    // is an odd number of units, its last slice is 64 wide.
    constexpr int kUnit = 64;
    const int n_units = p.E / kUnit;
    const int u_begin = n_units * rank / kSplit, u_end = n_units * (rank + 1) / kSplit;
    const int per = kKSlice / kUnit;
    const int s_begin = 0, s_end = (u_end - u_begin + per - 1) / per;  // slices of this rank
    auto slice_width = [&](int sl) { return min(kKSlice, (u_end - u_begin - sl * per) * kUnit); };
    const int mp = tid >> 4;                 // row quad 0..7 -> rows 4 mp .. 4 mp + 3
    const int n0 = (tid & 15) * 6;           // first of six outputs

    // Global row of layer-local row m (m = b * T + t).
    auto x_row = [&](int m) -> const float* {
        const int b = m / p.T, t = m - (m / p.T) * p.T;
        return p.x + ((static_cast<size_t>(b) * p.L + l) * p.T + t) * p.E;
    };

    float acc[4][6];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 6; ++j) acc[i][j] = 0.f;

    // Slice loads: 16-byte asynchronous copies into buffer `buf`.
    auto load_w = [&](int sl, int buf, auto width_c) {
        constexpr int width = decltype(width_c)::value;
        const int k0 = (u_begin + sl * per) * kUnit;
        for (int i = tid; i < kRowsPerCta * width / 4; i += kAbThreads) {
            const int r = i / (width / 4), c = (i % (width / 4)) * 4;
            const int m = m0 + r < M ? m0 + r : M - 1;  // rows past M read a valid row; their sums are not stored
            cp_async16(smem_addr(&xs[buf][r][c]), x_row(m) + k0 + c);
        }
        for (int i = tid; i < kOut * width / 8; i += kAbThreads) {
            const int n = i / (width / 8), c = (i % (width / 8)) * 8;
            const uint16_t* src = (n < kVHeads ? p.wa + (static_cast<size_t>(l) * kVHeads + n) * p.E
                                               : p.wb + (static_cast<size_t>(l) * kVHeads + n - kVHeads) * p.E) +
                                  k0 + c;
            cp_async16(smem_addr(&ws[buf][n][c]), src);
        }
        cp_async_commit();
    };
    auto load_slice = [&](int sl, int buf) {
        if (slice_width(sl) == kKSlice) load_w(sl, buf, std::integral_constant<int, kKSlice>{});
        else load_w(sl, buf, std::integral_constant<int, kUnit>{});
    };

    if (s_begin < s_end) load_slice(s_begin, 0);
    for (int sl = s_begin; sl < s_end; ++sl) {
        const int buf = (sl - s_begin) & 1;
        if (sl + 1 < s_end) {
            load_slice(sl + 1, buf ^ 1);
            cp_async_wait_one();  // this slice has landed; the next may still be in flight
        } else {
            cp_async_wait_all();
        }
        __syncthreads();
        auto compute = [&](auto width_c) {
            constexpr int width = decltype(width_c)::value;
#pragma unroll 2
            for (int k = 0; k < width; k += 8) {
                float xv[4][8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4 a = *reinterpret_cast<const float4*>(&xs[buf][4 * mp + i][k]);
                    const float4 b = *reinterpret_cast<const float4*>(&xs[buf][4 * mp + i][k + 4]);
                    xv[i][0] = a.x; xv[i][1] = a.y; xv[i][2] = a.z; xv[i][3] = a.w;
                    xv[i][4] = b.x; xv[i][5] = b.y; xv[i][6] = b.z; xv[i][7] = b.w;
                }
#pragma unroll
                for (int j = 0; j < 6; ++j) {
                    const uint4 raw = *reinterpret_cast<const uint4*>(&ws[buf][n0 + j][k]);
                    const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 w = __bfloat1622float2(w2[e]);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            acc[i][j] = fmaf(xv[i][2 * e], w.x, acc[i][j]);
                            acc[i][j] = fmaf(xv[i][2 * e + 1], w.y, acc[i][j]);
                        }
                    }
                }
            }
        };
        if (slice_width(sl) == kKSlice) compute(std::integral_constant<int, kKSlice>{});
        else compute(std::integral_constant<int, kUnit>{});
        __syncthreads();  // the buffer is refilled two slices later
    }

    // Partial sums meet across the cluster.
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 6; ++j) part[tid][6 * i + j] = acc[i][j];
    cluster_sync();
    // Reduce-scatter: rank r finishes row 4 mp + r of each thread's four rows, adding the
    // other ranks' partial sums (two floats per load, all issued before any sum uses them).
    static_assert(kSplit == 4, "one row of a thread's four per rank");
    float2 rv[kSplit - 1][3];
#pragma unroll
    for (int o = 1; o < kSplit; ++o) {
        const uint32_t remote = cluster_map(smem_addr(&part[tid][6 * rank]), (rank + o) % kSplit);
#pragma unroll
        for (int q = 0; q < 3; ++q)
            asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];"
                         : "=f"(rv[o - 1][q].x), "=f"(rv[o - 1][q].y)
                         : "r"(remote + 8 * q));
    }
    float sum[6];
#pragma unroll
    for (int j = 0; j < 6; ++j) sum[j] = part[tid][6 * rank + j];
#pragma unroll
    for (int o = 0; o < kSplit - 1; ++o)
#pragma unroll
        for (int q = 0; q < 3; ++q) {
            sum[2 * q] += rv[o][q].x;
            sum[2 * q + 1] += rv[o][q].y;
        }
    const int m = m0 + 4 * mp + rank;
    if (m < M) {
        const int b = m / p.T, t = m - (m / p.T) * p.T;
        const size_t row = ((static_cast<size_t>(b) * p.L + l) * p.T + t) * kVHeads;
#pragma unroll
        for (int j = 0; j < 6; ++j) {
            const int n = n0 + j;
            if (n < kVHeads) {
                p.gate[row + n] = softplusf_(sum[j] + p.dt[static_cast<size_t>(l) * kVHeads + n]) *
                                  p.ssm_a[static_cast<size_t>(l) * kVHeads + n];
            } else {
                p.beta[row + n - kVHeads] = sigmoidf_(sum[j]);
            }
        }
    }
    cluster_sync();  // no CTA leaves while another may still read its partial sums
}

}  // namespace

cudaError_t launch_ab_gates(const AbArgs& a, cudaStream_t stream) {
    {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        static std::mutex mutex;
        static bool ready[64] = {};
        std::lock_guard<std::mutex> lock(mutex);
        if (!ready[dev]) {
            e = cudaFuncSetAttribute(gdn_ab_gates_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kAbSmem));
            if (e != cudaSuccess) return e;
            ready[dev] = true;
        }
    }
    AbParams p;
    p.x = a.x;
    p.wa = a.w_alpha;
    p.wb = a.w_beta;
    p.dt = a.dt;
    p.ssm_a = a.ssm_a;
    p.gate = a.gate;
    p.beta = a.beta;
    p.B = a.B;
    p.L = a.L;
    p.T = a.T;
    p.E = a.n_embd;
    const int M = a.B * a.T;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(((M + kRowsPerCta - 1) / kRowsPerCta) * kSplit, a.L, 1);
    cfg.blockDim = dim3(kAbThreads, 1, 1);
    cfg.dynamicSmemBytes = kAbSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, gdn_ab_gates_kernel, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace gdn
