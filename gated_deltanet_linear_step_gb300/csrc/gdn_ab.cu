// gdn_ab.cu - the alpha/beta projections of a GDN layer with their gate
// epilogue, fused (the fused_gdn_ab stage of gdn_layer step 5 on the
// Winery-Strata page src/core/layer.cpp), on the 5th-generation tensor cores:
// for every (sequence b, layer l, token t) and v head h,
//
//   alpha_raw = x . Wa[l][h],  beta_raw = x . Wb[l][h]      (BF16 weights, fp32 activations)
//   gate      = softplus(alpha_raw + dt[l][h]) * ssm_a[l][h] (the log of the decay)
//   beta      = sigmoid(beta_raw)
//
// Per layer this is a small GEMM, [B T tokens] x [n_embd] by [n_embd] x [96].
// The 96 weight rows (48 alpha, then 48 beta) are the MMA's M side (M = 128;
// accumulator lanes 96-127 depend only on their own rows and are not stored),
// a block of up to 128 tokens its N side. kind::f16 multiplies BF16 by BF16,
// so x is split as hi + lo, hi = x truncated to BF16 and lo = the remainder
// rounded to BF16 (x to within 2^-16 of its value), and the lo rows follow
// the hi rows on the N side of the same MMA. Sums stay fp32.
//
// A cluster of 4 CTAs takes one (layer, token block), each CTA a quarter of
// n_embd, so even a batch of 64 single-token rows per layer keeps 4 SMs per
// layer busy. Per CTA, per 64-wide slice of its quarter:
//   warp 4 lane 0  - issues the tensor-map loads: the alpha and beta weight
//                    boxes (128-byte swizzle) and the fp32 x rows of the token
//                    block (a 3-D box over [sequence][layer x token][n_embd]);
//   warps 0-3      - convert the x rows into the BF16 hi and lo blocks in the
//                    swizzled K-major layout the MMA reads;
//   warp 5         - holds the tensor memory; lane 0 issues tcgen05.mma.
// The four CTAs' partial sums then meet in a reduce-scatter through
// distributed shared memory: each CTA stores its sums straight into the
// receive area of the rank that finishes the token (rank j mod 4), one cluster
// barrier makes them visible, and each rank adds the four partials of its
// tokens in its own shared memory and applies the gate epilogue. No global
// workspace is used.
// Every wait is bounded; a wait that gives up stops the roles, which still
// take part in the cluster barriers, and the device error word is set.

#include <cstring>
#include <mutex>

#include "gdn_device.cuh"
#include "gdn_launch.h"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int kSplit = 4;                       // CTAs per cluster, each a quarter of n_embd
constexpr int kAbThreads = 192;
constexpr int kBK = 64;                         // n_embd elements per stage
constexpr int kAbRows = kVHeads;                // 48 alpha rows, then 48 beta rows
constexpr int kOut = 2 * kAbRows;               // 96
constexpr uint32_t kWBytes = 128u * 128u;       // the MMA's A block: 128 rows x 64 BF16
constexpr int kMaxStages = 8;
constexpr size_t kStageBudget = 220 * 1024;  // the stages, then the receive area of the reduction
constexpr size_t kBarBytes = 8 * (3 * kMaxStages + 1) + 16 + 2 * kVHeads * 4;  // + the layer's dt and ssm_a
constexpr size_t kAbSmem = kStageBudget + kBarBytes + 1024;  // + alignment slack
// Receive area: [4 source ranks][ceil(n_blk / 4) tokens][96] fp32.
__host__ __device__ constexpr size_t recv_bytes(int n_blk) { return size_t(kSplit) * ((n_blk + 3) / 4) * 2 * kVHeads * 4; }
constexpr uint32_t kTmemCols = 256;

__device__ unsigned int g_ab_error = 0;

struct AbParams {
    CUtensorMap tm_x;      // x as [B][L * T][E] fp32, box {64, Tb, Bb}, no swizzle
    CUtensorMap tm_alpha;  // [L * 48][E] BF16, box {64, 48}, 128-byte swizzle
    CUtensorMap tm_beta;   // [L * 48][E]
    const float* dt;       // [L][48]
    const float* ssm_a;    // [L][48]
    float* gate;           // [B][L][T][48]
    float* beta;           // [B][L][T][48]
    int B, L, T, E;
    int Tb, Bb;            // a token block: Tb tokens of each of Bb sequences
    int n_tt;              // token blocks along T
    int n_blk;             // Bb * Tb rounded up to a multiple of 16: the MMA's N is 2 n_blk
    int n_stages;
};

// A bounded wait that also gives up as soon as another role of the CTA has.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(&g_ab_error, kErrWaitTimeout);
            return false;
        }
    }
}

__global__ void __launch_bounds__(kAbThreads, 1) gdn_ab_gates_kernel(const __grid_constant__ AbParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // the 128-byte swizzle wants 1024-byte alignment
    uint8_t* basep = smem_raw + (base - raw);
    const int n_blk = p.n_blk;
    const uint32_t stage_bytes = kWBytes + 512u * static_cast<uint32_t>(n_blk);  // A, hi, lo, then the fp32 rows
    const int S = p.n_stages;
    const uint32_t bars = base + static_cast<uint32_t>(kStageBudget);
    auto rawf_bar = [&](int s) { return bars + 8u * s; };                     // x rows and weights have landed
    auto conv_bar = [&](int s) { return bars + 8u * (kMaxStages + s); };      // hi and lo written (128 arrivals)
    auto empty_bar = [&](int s) { return bars + 8u * (2 * kMaxStages + s); };  // the MMAs have read the stage
    const uint32_t accf_bar = bars + 8u * (3 * kMaxStages);
    uint8_t* misc = basep + kStageBudget + 8 * (3 * kMaxStages + 1);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
    float* lw = reinterpret_cast<float*>(misc + 16);  // dt[48], then ssm_a[48] of the layer

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int rank = static_cast<int>(cluster_rank());
    const int l = blockIdx.y;
    const int tb = blockIdx.x / kSplit;
    const int t0 = (tb % p.n_tt) * p.Tb, b0 = (tb / p.n_tt) * p.Bb;
    const int rows_box = p.Bb * p.Tb;
    const int n_ks = p.E / kBK;
    const int ks0 = n_ks * rank / kSplit;
    const int steps = n_ks * (rank + 1) / kSplit - ks0;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(rawf_bar(s), 1);
            mbar_init(conv_bar(s), 128);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(accf_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&p.tm_x);
        prefetch_tensormap(&p.tm_alpha);
        prefetch_tensormap(&p.tm_beta);
    }
    if (warp == 5) tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool have_acc = false;  // (warps 0-3) the accumulator holds this CTA's sums
    // Launched with programmatic stream serialization, the next kernel in the stream may start its
    // CTAs (and their set-up above) while this one finishes; every read of global memory below
    // waits until the kernels before this one have completed and their writes are visible.
    griddep_launch_dependents();
    griddep_wait();
    // The layer's dt and ssm_a for the epilogue: loaded now, kept in shared memory after the main loop.
    float lw_val = 0.0f;
    if (tid < 2 * kVHeads)
        lw_val = __ldg((tid < kVHeads ? p.dt : p.ssm_a) + static_cast<size_t>(l) * kVHeads + tid % kVHeads);

    if (warp == 4) {
        if (lane == 0) {
            // ---------------------------------------------------- copies --
            const uint64_t pol = evict_first_policy();
            const uint32_t x_bytes = static_cast<uint32_t>(rows_box) * 256u;
            int issued = 0;
            for (int i = 0; i < steps; ++i) {
                const int s = i % S;
                if (!wait_or_abort(empty_bar(s), ((i / S) & 1) ^ 1u, abort_flag)) break;
                const uint32_t st = base + s * stage_bytes;
                const int k0 = (ks0 + i) * kBK;
                mbar_arrive_expect_tx(rawf_bar(s), 2u * kAbRows * 128u + x_bytes);
                tma_load_2d(st, &p.tm_alpha, k0, l * kAbRows, rawf_bar(s), pol);
                tma_load_2d(st + kAbRows * 128u, &p.tm_beta, k0, l * kAbRows, rawf_bar(s), pol);
                tma_load_3d(st + kWBytes + 256u * n_blk, &p.tm_x, k0, l * p.T + t0, b0, rawf_bar(s), pol);
                ++issued;
            }
            // What is still in flight lands before the CTA leaves.
            for (int j = issued > S ? issued - S : 0; j < issued; ++j)
                if (!mbar_wait_bounded(rawf_bar(j % S), (j / S) & 1)) atomicOr(&g_ab_error, kErrWaitTimeout);
        }
    } else if (warp == 5) {
        if (lane == 0) {
            // ----------------------------------------------- MMA issuer --
            const uint32_t idesc = mma_idesc(2 * n_blk);  // the hi rows, then the lo rows
            for (int i = 0; i < steps; ++i) {
                const int s = i % S;
                if (!wait_or_abort(conv_bar(s), (i / S) & 1, abort_flag)) break;
                tc_fence_after();
                const uint32_t st = base + s * stage_bytes;
                const uint64_t wd = sw128_desc(st);
                const uint64_t xd = sw128_desc(st + kWBytes);
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    // K advances 16 BF16 = 32 bytes inside the swizzled row: +2 in the descriptor's address field.
                    const uint64_t dk = static_cast<uint64_t>(2 * kk);
                    mma_bf16(tmem, wd + dk, xd + dk, idesc, (i | kk) != 0 ? 1u : 0u);
                }
                mma_commit(empty_bar(s));
            }
            // Arrives once every MMA issued above has completed (at once if there were none).
            mma_commit(accf_bar);
            if (!mbar_wait_bounded(accf_bar, 0)) atomicOr(&g_ab_error, kErrWaitTimeout);
        }
    } else {
        // -------------------------------- warps 0-3: x into hi and lo --
        for (int i = 0; i < steps; ++i) {
            const int s = i % S;
            if (!wait_or_abort(rawf_bar(s), (i / S) & 1, abort_flag)) break;
            uint8_t* st = basep + s * stage_bytes;
            const float* xr = reinterpret_cast<const float*>(st + kWBytes + 256u * n_blk);
            for (int it = tid; it < n_blk * 8; it += 128) {
                const int n = it >> 3, c = it & 7;
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
                if (n < rows_box) {
                    a = *reinterpret_cast<const float4*>(xr + n * kBK + 8 * c);
                    b = *reinterpret_cast<const float4*>(xr + n * kBK + 8 * c + 4);
                }
                const uint32_t off = sw128_offset(n, c);
                *reinterpret_cast<uint4*>(st + kWBytes + off) =
                    make_uint4(hi_pair(a.x, a.y), hi_pair(a.z, a.w), hi_pair(b.x, b.y), hi_pair(b.z, b.w));
                *reinterpret_cast<uint4*>(st + kWBytes + 128u * n_blk + off) =
                    make_uint4(lo_pair(a.x, a.y), lo_pair(a.z, a.w), lo_pair(b.x, b.y), lo_pair(b.z, b.w));
            }
            fence_proxy_async_smem();  // the MMA reads the blocks through the async proxy
            mbar_arrive_local(conv_bar(s));
        }
        have_acc = steps > 0 && wait_or_abort(accf_bar, 0, abort_flag);
        tc_fence_after();
    }
    if (tid < 2 * kVHeads) lw[tid] = lw_val;
    __syncthreads();  // every copy and MMA of this CTA is done with the stages

    // ---- push: each sum of this CTA goes straight to the receive area of the rank that finishes its
    //      token (rank j mod 4, slot j / 4), in distributed shared memory; one cluster barrier follows
    const int n_slot = (n_blk + 3) / 4;
    float* recv = reinterpret_cast<float*>(basep + static_cast<size_t>(S) * stage_bytes);
    if (warp < 3) {  // tensor-memory lanes 0-95: the alpha and beta rows
        const int row = 32 * warp + lane;
        const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * warp) << 16);
        const uint32_t mine = smem_addr(recv + rank * n_slot * kOut + row);
        for (int j0 = 0; j0 < n_blk; j0 += 32) {
            uint32_t hi[32], lo[32];
            if (have_acc) {
                tmem_ld32(taddr + static_cast<uint32_t>(j0), hi);
                tmem_ld32(taddr + static_cast<uint32_t>(n_blk + j0), lo);
            }
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int j = j0 + jj;
                if (j < n_blk) {
                    const float val = have_acc ? __uint_as_float(hi[jj]) + __uint_as_float(lo[jj]) : 0.0f;
                    const uint32_t dst = cluster_map(mine + static_cast<uint32_t>((j >> 2) * kOut * 4), j & 3);
                    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dst), "f"(val) : "memory");
                }
            }
        }
    }
    tc_fence_before();
    cluster_sync();  // every rank's sums are in their owners' receive areas

    // ---- rank r finishes the tokens j = r mod 4 (four outputs per item) and applies the gate epilogue
    //      The items run every token's alpha chunks first, then every token's beta chunks, so a warp
    //      takes the softplus or the sigmoid branch, not both.
    constexpr int kChunks = kOut / 4;   // 24 float4 per token
    constexpr int kHalf = kChunks / 2;  // 12 of them alpha, 12 beta
    const int n_mine = (n_blk - rank + kSplit - 1) / kSplit;
    const int n_half = n_mine * kHalf;
    if (!*abort_flag) {
        for (int it = tid; it < 2 * n_half; it += kAbThreads) {
            const bool is_beta = it >= n_half;
            const int k = is_beta ? it - n_half : it;
            const int slot = k / kHalf;
            const int q = k % kHalf + (is_beta ? kHalf : 0);
            const int j = rank + kSplit * slot;
            const int b = b0 + j / p.Tb, t = t0 + j % p.Tb;
            if (j >= rows_box || b >= p.B || t >= p.T) continue;
            float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int o = 0; o < kSplit; ++o) {
                const float4 v = *reinterpret_cast<const float4*>(recv + (o * n_slot + slot) * kOut + 4 * q);
                sum.x += v.x;
                sum.y += v.y;
                sum.z += v.z;
                sum.w += v.w;
            }
            const size_t orow = ((static_cast<size_t>(b) * p.L + l) * p.T + t) * kVHeads;
            const float sv[4] = {sum.x, sum.y, sum.z, sum.w};
            float4 r;
            float* rr = &r.x;
            // chunks 0-11 are gate heads 0-47, chunks 12-23 beta heads 0-47
            if (!is_beta) {
#pragma unroll
                for (int e = 0; e < 4; ++e) rr[e] = softplusf_(sv[e] + lw[4 * q + e]) * lw[kVHeads + 4 * q + e];
                *reinterpret_cast<float4*>(p.gate + orow + 4 * q) = r;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) rr[e] = sigmoidf_(sv[e]);
                *reinterpret_cast<float4*>(p.beta + orow + 4 * q - kAbRows) = r;
            }
        }
    }
    // (no CTA reads another's shared memory after the barrier, so each may leave on its own)
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

std::mutex g_mutex;
bool g_ready[64] = {};

cudaError_t encode_x(CUtensorMap* tm, const float* x, int B, int L, int T, int E, int Tb, int Bb) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(E), static_cast<cuuint64_t>(L) * T,
                                static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(E) * 4, static_cast<cuuint64_t>(L) * T * E * 4};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(Tb), static_cast<cuuint32_t>(Bb)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = tensor_map_encoder()(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(x), dims,
                                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_w(CUtensorMap* tm, const uint16_t* w, int L, int E) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(E), static_cast<cuuint64_t>(L) * kAbRows};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(E) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(kAbRows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = tensor_map_encoder()(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(w), dims,
                                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_ab_gates(const AbArgs& a, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (tensor_map_encoder() == nullptr) return cudaErrorNotSupported;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (!g_ready[dev]) {
            e = cudaFuncSetAttribute(gdn_ab_gates_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kAbSmem));
            if (e != cudaSuccess) return e;
            g_ready[dev] = true;
        }
    }
    AbParams p;
    memset(&p, 0, sizeof(p));
    p.Tb = a.T < 128 ? a.T : 128;
    const int bb = 128 / p.Tb;
    p.Bb = a.B < bb ? a.B : bb;
    p.n_tt = (a.T + p.Tb - 1) / p.Tb;
    p.n_blk = (p.Bb * p.Tb + 15) / 16 * 16;
    const uint32_t stage = kWBytes + 512u * static_cast<uint32_t>(p.n_blk);
    const int fit = static_cast<int>((kStageBudget - recv_bytes(p.n_blk)) / stage);
    p.n_stages = fit < kMaxStages ? fit : kMaxStages;
    e = encode_x(&p.tm_x, a.x, a.B, a.L, a.T, a.n_embd, p.Tb, p.Bb);
    if (e != cudaSuccess) return e;
    e = encode_w(&p.tm_alpha, a.w_alpha, a.L, a.n_embd);
    if (e != cudaSuccess) return e;
    e = encode_w(&p.tm_beta, a.w_beta, a.L, a.n_embd);
    if (e != cudaSuccess) return e;
    p.dt = a.dt;
    p.ssm_a = a.ssm_a;
    p.gate = a.gate;
    p.beta = a.beta;
    p.B = a.B;
    p.L = a.L;
    p.T = a.T;
    p.E = a.n_embd;
    const int n_tb = p.n_tt * ((a.B + p.Bb - 1) / p.Bb);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(n_tb * kSplit), static_cast<unsigned>(a.L), 1);
    cfg.blockDim = dim3(kAbThreads, 1, 1);
    cfg.dynamicSmemBytes = kAbSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, gdn_ab_gates_kernel, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t read_ab_error(uint32_t* out) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_ab_error, sizeof(v));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_ab_error, &zero, sizeof(zero));
    *out = v;
    return e;
}

}  // namespace gdn
