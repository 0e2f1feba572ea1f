// gdn_proj.cu - the mixer's two input projections on the 5th-generation tensor
// cores: qkv = w_qkv x (the 10240 conv channels q|k|v, gdn_layer step 2 on the
// Winery-Strata page src/core/layer.cpp) and z = w_gate x (the 6144-wide output
// gate, the start of gdn_layer step 7), for every (sequence b, layer l, token t).
// The weights are dense BF16 [n_out][n_embd]; x and the outputs are fp32.
//
// Per layer this is a GEMM whose token dimension is small (B T rows) and whose
// weight matrix (16384 x n_embd BF16, 84 MB at n_embd 2560) is read once, so the
// weight stream from HBM bounds it. Weight rows become the MMA's M side (128
// output channels per tile) and tokens its N side; the accumulator lives in
// tensor memory, one lane per output channel and one column per token and half.
//
// Precision. kind::f16 multiplies BF16 by BF16. The weights are BF16 already;
// x is split as x = hi + lo with hi = x truncated to BF16 and lo = the
// remainder rounded to BF16, so every product carries x to within 2^-16 of its
// value. The lo rows follow the hi rows on the MMA's N side: one MMA of
// N = 2 x tokens per K step multiplies the weight slice by both halves (the
// weights are read from shared memory once), and the epilogue adds column j
// and column tokens + j. Sums stay fp32.
//
// With the alpha/beta weights given, every layer gets one more tile: the 48
// alpha rows and the 48 beta rows (two TMA boxes) as the MMA's rows 0-95, with
// the gate epilogue of fused_gdn_ab (gdn_layer step 5): gate = softplus(alpha
// + dt) * ssm_a, the log of the decay, and beta = sigmoid(beta_raw). Rows
// 96-127 of that tile hold whatever the stage held before; each accumulator
// lane depends on its own row only, and those lanes are not stored.
//
// Packed weights. gdn_pack_proj_kernel rearranges the weights once, ahead of
// the calls, into the blocks the MMA reads: per layer 129 tiles (80 of w_qkv,
// 48 of w_gate, then the 48 alpha rows, the 48 beta rows and 32 zero rows),
// per tile n_embd / 64 blocks of [128][64] BF16 (16 KB) in the 128-byte
// swizzled K-major order a tensor-map load with that swizzle would leave in
// shared memory. With packed weights the producer fetches each block with one
// contiguous bulk copy instead of a 128-row tensor-map load whose rows lie
// n_embd x 2 bytes apart in HBM.
//
// Two kernels per call:
// * gdn_x_split_kernel writes hi and lo of every (layer, token block, 64-wide
//   slice of n_embd) as two [N][64] BF16 blocks, already in the 128-byte
//   swizzled K-major layout the MMA reads, into the caller's workspace.
// * gdn_in_proj_kernel, persistent, one CTA per SM, 192 threads:
//     warp 0 lane 0  - producer: per stage, the weight slice [128][64] by TMA
//                      (tensor map, 128-byte swizzle, evict-first) and the
//                      split x blocks by one bulk copy, both on one mbarrier;
//     warp 1         - allocates all 512 tensor-memory columns (two
//                      accumulators of up to 256); lane 0 issues tcgen05.mma
//                      (M 128, N = 2 x token block, K 16) and commits each
//                      stage back to its producer;
//     warps 2-5      - epilogue: tcgen05.ld of the accumulator, 32 tokens at a
//                      time, and coalesced fp32 stores of the outputs.
//   The epilogue of one tile overlaps the next tile's main loop through the
//   two accumulators.
//
// Every wait is bounded; a wait that gives up raises the CTA's abort flag, the
// other roles stop at their next wait, the producer and the MMA issuer wait
// (bounded) for what they have in flight, and the tensor memory is released
// before the CTA exits with the device error word set.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "gdn_device.cuh"
#include "gdn_launch.h"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int kBM = 128;                       // output channels per tile (MMA M)
constexpr int kBK = 64;                        // n_embd elements per stage: one 128-byte BF16 row
constexpr int kMaxTok = 128;                   // tokens per block (MMA N <= 128)
constexpr int kQkvTiles = kConvChannels / kBM;  // 80
constexpr int kGateTiles = kValueDim / kBM;     // 48
constexpr int kChTiles = kQkvTiles + kGateTiles;  // 128; the alpha/beta tile is number 128
constexpr int kPackTiles = kChTiles + 1;           // tiles per layer in the packed weights
constexpr int kAbRows = kVHeads;                   // 48 alpha rows, then 48 beta rows
constexpr int kProjThreads = 192;
constexpr int kMaxStages = 8;
constexpr uint32_t kWBytes = kBM * kBK * 2;    // 16384
constexpr uint32_t kAccCols = 2 * kMaxTok;     // columns per accumulator: hi tokens, then lo tokens
constexpr uint32_t kTmemCols = 2 * kAccCols;
constexpr size_t kStageBudget = 200 * 1024;
constexpr size_t kBarBytes = 256;
constexpr size_t kProjSmem = kStageBudget + kBarBytes + 1024;  // + alignment slack

__device__ unsigned int g_proj_error = 0;

struct ProjParams {
    CUtensorMap tm_qkv;    // [L * 10240][E] BF16, box 64 x 128, 128-byte swizzle
    CUtensorMap tm_gate;   // [L * 6144][E]
    CUtensorMap tm_alpha;  // [L * 48][E], box 64 x 48 (used when n_ct is 129)
    CUtensorMap tm_beta;   // [L * 48][E]
    const float* dt;       // [L][48]
    const float* ssm_a;    // [L][48]
    float* gate;           // [B][L][T][48]
    float* beta;           // [B][L][T][48]
    int n_ct;              // channel tiles per layer: 128, or 129 with the alpha/beta tile
    const uint8_t* wp;     // packed weights [L][129][E / 64][16 KB], or NULL: the tensor maps above
    const uint16_t* xs;   // split x: [L][n_tb][n_ks][2][n_blk][64] BF16, swizzled
    float* qkv;           // [B][L][T][10240]
    float* z;             // [B][L][T][6144]
    int B, L, T, E;
    int n_blk;            // token rows per block in the workspace (multiple of 16, <= 128)
    int n_tb;             // token blocks
    int n_stages;
    long long n_tiles;
};

struct PackParams {
    const uint16_t* w_qkv;    // [L][10240][E]
    const uint16_t* w_gate;   // [L][6144][E]
    const uint16_t* w_alpha;  // [L][48][E], or NULL: zero rows
    const uint16_t* w_beta;   // [L][48][E], or NULL: zero rows
    uint8_t* out;             // [L][129][E / 64][16 KB]
    int L, E;
    long long n_blocks;
};

struct SplitParams {
    const float* x;  // [B][L][T][E]
    uint16_t* xs;
    int B, L, T, E, n_blk, n_tb;
    long long n_items;
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
            atomicOr(&g_proj_error, kErrWaitTimeout);
            return false;
        }
    }
}

// One 16 KB block per iteration: 128 rows x 64 BF16, the 16-byte chunk c of
// row r stored at r * 128 + (c XOR r mod 8) * 16.
__global__ void __launch_bounds__(256) gdn_pack_proj_kernel(const __grid_constant__ PackParams p) {
    const int n_ks = p.E / kBK;
    for (long long blk = blockIdx.x; blk < p.n_blocks; blk += gridDim.x) {
        const int ks = static_cast<int>(blk % n_ks);
        const long long rest = blk / n_ks;
        const int ct = static_cast<int>(rest % kPackTiles);
        const int l = static_cast<int>(rest / kPackTiles);
        uint8_t* dst = p.out + static_cast<size_t>(blk) * kWBytes;
        for (int i = threadIdx.x; i < kBM * 8; i += blockDim.x) {
            const int r = i >> 3, c = i & 7;
            const uint16_t* row = nullptr;
            if (ct < kQkvTiles) {
                row = p.w_qkv + (static_cast<size_t>(l) * kConvChannels + ct * kBM + r) * p.E;
            } else if (ct < kChTiles) {
                row = p.w_gate + (static_cast<size_t>(l) * kValueDim + (ct - kQkvTiles) * kBM + r) * p.E;
            } else if (r < kAbRows) {
                if (p.w_alpha != nullptr) row = p.w_alpha + (static_cast<size_t>(l) * kAbRows + r) * p.E;
            } else if (r < 2 * kAbRows) {
                if (p.w_beta != nullptr) row = p.w_beta + (static_cast<size_t>(l) * kAbRows + r - kAbRows) * p.E;
            }
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (row != nullptr) v = __ldg(reinterpret_cast<const uint4*>(row + ks * kBK + c * 8));
            *reinterpret_cast<uint4*>(dst + r * 128 + ((c ^ (r & 7)) << 4)) = v;
        }
    }
}

__global__ void __launch_bounds__(256) gdn_x_split_kernel(const __grid_constant__ SplitParams p) {
    const int n_ks = p.E / kBK;
    const int M = p.B * p.T;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < p.n_items;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int c = static_cast<int>(i & 7);
        long long r = i >> 3;
        const int n = static_cast<int>(r % p.n_blk);
        r /= p.n_blk;
        const int ks = static_cast<int>(r % n_ks);
        r /= n_ks;
        const int tb = static_cast<int>(r % p.n_tb);
        const int l = static_cast<int>(r / p.n_tb);
        const int m = tb * kMaxTok + n;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
        if (n < kMaxTok && m < M) {
            const int sb = m / p.T, t = m - (m / p.T) * p.T;
            const float* src = p.x + ((static_cast<size_t>(sb) * p.L + l) * p.T + t) * p.E + ks * kBK + c * 8;
            a = __ldg(reinterpret_cast<const float4*>(src));
            b = __ldg(reinterpret_cast<const float4*>(src + 4));
        }
        const uint4 hi = make_uint4(hi_pair(a.x, a.y), hi_pair(a.z, a.w), hi_pair(b.x, b.y), hi_pair(b.z, b.w));
        const uint4 lo = make_uint4(lo_pair(a.x, a.y), lo_pair(a.z, a.w), lo_pair(b.x, b.y), lo_pair(b.z, b.w));
        uint8_t* blk = reinterpret_cast<uint8_t*>(p.xs) +
                       ((static_cast<size_t>(l) * p.n_tb + tb) * n_ks + ks) * (2 * static_cast<size_t>(p.n_blk) * 128);
        const uint32_t off = sw128_offset(n, c);
        *reinterpret_cast<uint4*>(blk + off) = hi;
        *reinterpret_cast<uint4*>(blk + static_cast<size_t>(p.n_blk) * 128 + off) = lo;
    }
}

// --------------------------------------------------------- the projection --
__global__ void __launch_bounds__(kProjThreads, 1) gdn_in_proj_kernel(const __grid_constant__ ProjParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // the 128-byte swizzle wants 1024-byte alignment
    const int n_blk = p.n_blk;
    const uint32_t x_bytes = 2u * static_cast<uint32_t>(n_blk) * 128u;  // hi block, then lo block
    const uint32_t stage_bytes = kWBytes + x_bytes;
    const int n_stages = p.n_stages;
    const uint32_t bars = base + static_cast<uint32_t>(kStageBudget);
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (kMaxStages + s); };
    auto accf_bar = [&](int a) { return bars + 8u * (2 * kMaxStages + a); };
    auto acce_bar = [&](int a) { return bars + 8u * (2 * kMaxStages + 2 + a); };
    uint8_t* misc = smem_raw + (bars - raw) + 8 * (2 * kMaxStages + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_ks = p.E / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < n_stages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(accf_bar(a), 1);
            mbar_init(acce_bar(a), 4 * 32);
        }
        *abort_flag = 0;
        fence_mbar_init();
        if (p.wp == nullptr) prefetch_tensormap(&p.tm_qkv);
        if (p.wp == nullptr) prefetch_tensormap(&p.tm_gate);
        if (p.wp == nullptr && p.n_ct > kChTiles) {
            prefetch_tensormap(&p.tm_alpha);
            prefetch_tensormap(&p.tm_beta);
        }
    }
    if (warp == 1) tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------- producer --
            const uint64_t pol = evict_first_policy();
            uint32_t it = 0;
            for (long long tile = blockIdx.x; tile < p.n_tiles; tile += gridDim.x) {
                const int ct = static_cast<int>(tile % p.n_ct);
                const long long rest = tile / p.n_ct;
                const int tb = static_cast<int>(rest % p.n_tb);
                const int l = static_cast<int>(rest / p.n_tb);
                const bool is_ab = ct == kChTiles;
                const bool is_qkv = ct < kQkvTiles;
                const CUtensorMap* tm = is_qkv ? &p.tm_qkv : &p.tm_gate;
                const int row = is_qkv ? l * kConvChannels + ct * kBM : l * kValueDim + (ct - kQkvTiles) * kBM;
                const uint8_t* xsrc = reinterpret_cast<const uint8_t*>(p.xs) +
                                      (static_cast<size_t>(l) * p.n_tb + tb) * n_ks * static_cast<size_t>(x_bytes);
                bool ok = true;
                for (int ks = 0; ks < n_ks; ++ks) {
                    const int s = static_cast<int>(it % n_stages);
                    const uint32_t ph = (it / n_stages) & 1u;
                    if (!wait_or_abort(empty_bar(s), ph ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = base + s * stage_bytes;
                    if (p.wp != nullptr) {
                        mbar_arrive_expect_tx(full_bar(s), stage_bytes);
                        bulk_load_stream(
                            st, p.wp + ((static_cast<size_t>(l) * kPackTiles + ct) * n_ks + ks) * kWBytes, kWBytes,
                            full_bar(s));
                    } else if (is_ab) {
                        mbar_arrive_expect_tx(full_bar(s), 2u * kAbRows * 128u + x_bytes);
                        tma_load_2d(st, &p.tm_alpha, ks * kBK, l * kAbRows, full_bar(s), pol);
                        tma_load_2d(st + kAbRows * 128u, &p.tm_beta, ks * kBK, l * kAbRows, full_bar(s), pol);
                    } else {
                        mbar_arrive_expect_tx(full_bar(s), stage_bytes);
                        tma_load_2d(st, tm, ks * kBK, row, full_bar(s), pol);
                    }
                    bulk_load(st + kWBytes, xsrc + static_cast<size_t>(ks) * x_bytes, x_bytes, full_bar(s));
                    ++it;
                }
                if (!ok) break;
            }
            // What is still in flight lands before the CTA leaves.
            const uint32_t first = it > static_cast<uint32_t>(n_stages) ? it - n_stages : 0u;
            for (uint32_t j = first; j < it; ++j) {
                if (!mbar_wait_bounded(full_bar(static_cast<int>(j % n_stages)), (j / n_stages) & 1u))
                    atomicOr(&g_proj_error, kErrWaitTimeout);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ----------------------------------------------- MMA issuer --
            const uint32_t idesc = mma_idesc(2 * n_blk);  // the hi rows, then the lo rows
            uint32_t it = 0, local = 0;
            uint32_t last_bar = 0, last_par = 0;
            bool issued = false;
            for (long long tile = blockIdx.x; tile < p.n_tiles; tile += gridDim.x, ++local) {
                const int a = static_cast<int>(local & 1u);
                const uint32_t aph = (local >> 1) & 1u;
                if (!wait_or_abort(acce_bar(a), aph ^ 1u, abort_flag)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + static_cast<uint32_t>(a) * kAccCols;
                bool ok = true;
                for (int ks = 0; ks < n_ks; ++ks) {
                    const int s = static_cast<int>(it % n_stages);
                    const uint32_t ph = (it / n_stages) & 1u;
                    if (!wait_or_abort(full_bar(s), ph, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = base + s * stage_bytes;
                    const uint64_t wd = sw128_desc(st);
                    const uint64_t xd = sw128_desc(st + kWBytes);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        // K advances 16 BF16 = 32 bytes inside the swizzled row: +2 in the descriptor's address field.
                        const uint64_t dk = static_cast<uint64_t>(2 * kk);
                        mma_bf16(d_tmem, wd + dk, xd + dk, idesc, (ks | kk) != 0 ? 1u : 0u);
                    }
                    mma_commit(empty_bar(s));
                    last_bar = empty_bar(s);
                    last_par = ph;
                    issued = true;
                    ++it;
                }
                if (!ok) break;
                mma_commit(accf_bar(a));
                last_bar = accf_bar(a);
                last_par = aph;
            }
            // The last commit covers every MMA issued: they finish before the memory goes away.
            if (issued && !mbar_wait_bounded(last_bar, last_par)) atomicOr(&g_proj_error, kErrWaitTimeout);
        }
    } else {
        // ------------------------------------------------------- epilogue --
        const int q = warp & 3;  // this warp's quarter of the tensor-memory lanes
        const int chan = 32 * q + lane;
        const int M = p.B * p.T;
        uint32_t local = 0;
        for (long long tile = blockIdx.x; tile < p.n_tiles; tile += gridDim.x, ++local) {
            const int a = static_cast<int>(local & 1u);
            const uint32_t aph = (local >> 1) & 1u;
            const int ct = static_cast<int>(tile % p.n_ct);
            const long long rest = tile / p.n_ct;
            const int tb = static_cast<int>(rest % p.n_tb);
            const int l = static_cast<int>(rest / p.n_tb);
            const int m0 = tb * kMaxTok;
            const int P = min(kMaxTok, M - m0);
            // Output of this lane: a qkv or z channel, or in the alpha/beta tile a
            // gate (lanes 0-47) or beta (lanes 48-95) head; lanes 96-127 store nothing.
            float* out;
            int width, ch;
            int kind = 0;  // 0: plain, 1: gate, 2: beta, 3: none
            float dt = 0.f, sa = 0.f;
            if (ct < kQkvTiles) {
                out = p.qkv;
                width = kConvChannels;
                ch = ct * kBM + chan;
            } else if (ct < kChTiles) {
                out = p.z;
                width = kValueDim;
                ch = (ct - kQkvTiles) * kBM + chan;
            } else {
                width = kVHeads;
                if (chan < kAbRows) {
                    kind = 1;
                    out = p.gate;
                    ch = chan;
                    dt = __ldg(p.dt + static_cast<size_t>(l) * kVHeads + ch);
                    sa = __ldg(p.ssm_a + static_cast<size_t>(l) * kVHeads + ch);
                } else {
                    kind = chan < 2 * kAbRows ? 2 : 3;
                    out = p.beta;
                    ch = chan < 2 * kAbRows ? chan - kAbRows : 0;
                }
            }
            if (!wait_or_abort(accf_bar(a), aph, abort_flag)) break;
            tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(a) * kAccCols;
            for (int j0 = 0; j0 < P; j0 += 32) {
                uint32_t hi[32], lo[32];
                tmem_ld32(taddr + static_cast<uint32_t>(j0), hi);
                tmem_ld32(taddr + static_cast<uint32_t>(n_blk + j0), lo);
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = j0 + jj;
                    if (j < P && kind != 3) {
                        const int m = m0 + j;
                        const int sb = m / p.T, t = m - (m / p.T) * p.T;
                        float v = __uint_as_float(hi[jj]) + __uint_as_float(lo[jj]);
                        if (kind == 1) v = softplusf_(v + dt) * sa;
                        else if (kind == 2) v = sigmoidf_(v);
                        out[((static_cast<size_t>(sb) * p.L + l) * p.T + t) * width + ch] = v;
                    }
                }
            }
            tc_fence_before();
            mbar_arrive_local(acce_bar(a));
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------- host --
std::mutex g_mutex;
struct DeviceSetup {
    bool ready = false;
    int sms = 0;
};
DeviceSetup g_setup[64];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t setup(int dev, int* sms) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    if (!g_setup[dev].ready) {
        int n = 0;
        cudaError_t e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(gdn_in_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kProjSmem));
        if (e != cudaSuccess) return e;
        g_setup[dev].sms = n;
        g_setup[dev].ready = true;
    }
    *sms = g_setup[dev].sms;
    return cudaSuccess;
}

cudaError_t encode_weights(CUtensorMap* tm, const uint16_t* w, long long rows, int E, int box_rows) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(E), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(E) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(w), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

ProjGeometry proj_geometry(int B, int T, int E) {
    ProjGeometry g;
    const long long M = static_cast<long long>(B) * T;
    g.n_tb = static_cast<int>((M + kMaxTok - 1) / kMaxTok);
    const long long first = M < kMaxTok ? M : kMaxTok;
    g.n_blk = static_cast<int>((first + 15) / 16 * 16);
    g.n_ks = E / kBK;
    const uint32_t stage = kWBytes + 2u * g.n_blk * 128u;
    const int fit = static_cast<int>(kStageBudget / stage);
    g.n_stages = fit < kMaxStages ? fit : kMaxStages;
    return g;
}

size_t proj_workspace_bytes(int B, int L, int T, int E) {
    const ProjGeometry g = proj_geometry(B, T, E);
    return static_cast<size_t>(L) * g.n_tb * g.n_ks * 2 * static_cast<size_t>(g.n_blk) * 128;
}

cudaError_t launch_in_proj(const ProjArgs& a, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int sms = 0;
    e = setup(dev, &sms);
    if (e != cudaSuccess) return e;
    const ProjGeometry g = proj_geometry(a.B, a.T, a.n_embd);

    SplitParams sp;
    sp.x = a.x;
    sp.xs = static_cast<uint16_t*>(a.workspace);
    sp.B = a.B;
    sp.L = a.L;
    sp.T = a.T;
    sp.E = a.n_embd;
    sp.n_blk = g.n_blk;
    sp.n_tb = g.n_tb;
    sp.n_items = static_cast<long long>(a.L) * g.n_tb * g.n_ks * g.n_blk * 8;
    const long long want = (sp.n_items + 255) / 256;
    const long long cap = static_cast<long long>(sms) * 8;
    gdn_x_split_kernel<<<static_cast<unsigned>(want < cap ? want : cap), 256, 0, stream>>>(sp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    ProjParams p;
    memset(&p, 0, sizeof(p));
    const bool with_ab = a.gate != nullptr;
    if (a.packed != nullptr) {
        p.wp = static_cast<const uint8_t*>(a.packed);
    } else {
        e = encode_weights(&p.tm_qkv, a.w_qkv, static_cast<long long>(a.L) * kConvChannels, a.n_embd, kBM);
        if (e != cudaSuccess) return e;
        e = encode_weights(&p.tm_gate, a.w_gate, static_cast<long long>(a.L) * kValueDim, a.n_embd, kBM);
        if (e != cudaSuccess) return e;
        if (with_ab) {
            e = encode_weights(&p.tm_alpha, a.w_alpha, static_cast<long long>(a.L) * kAbRows, a.n_embd, kAbRows);
            if (e != cudaSuccess) return e;
            e = encode_weights(&p.tm_beta, a.w_beta, static_cast<long long>(a.L) * kAbRows, a.n_embd, kAbRows);
            if (e != cudaSuccess) return e;
        }
    }
    p.n_ct = kChTiles;
    if (with_ab) {
        p.dt = a.dt;
        p.ssm_a = a.ssm_a;
        p.gate = a.gate;
        p.beta = a.beta;
        p.n_ct = kChTiles + 1;
    }
    p.xs = sp.xs;
    p.qkv = a.qkv;
    p.z = a.z;
    p.B = a.B;
    p.L = a.L;
    p.T = a.T;
    p.E = a.n_embd;
    p.n_blk = g.n_blk;
    p.n_tb = g.n_tb;
    p.n_stages = g.n_stages;
    p.n_tiles = static_cast<long long>(a.L) * g.n_tb * p.n_ct;
    const long long grid = p.n_tiles < sms ? p.n_tiles : sms;
    gdn_in_proj_kernel<<<static_cast<unsigned>(grid), kProjThreads, kProjSmem, stream>>>(p);
    return cudaGetLastError();
}

size_t proj_pack_bytes(int L, int E) {
    return static_cast<size_t>(L) * kPackTiles * (E / kBK) * kWBytes;
}

cudaError_t launch_pack_proj(const PackArgs& a, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int sms = 0;
    e = setup(dev, &sms);
    if (e != cudaSuccess) return e;
    PackParams p;
    p.w_qkv = a.w_qkv;
    p.w_gate = a.w_gate;
    p.w_alpha = a.w_alpha;
    p.w_beta = a.w_beta;
    p.out = static_cast<uint8_t*>(a.packed);
    p.L = a.L;
    p.E = a.n_embd;
    p.n_blocks = static_cast<long long>(a.L) * kPackTiles * (a.n_embd / kBK);
    const long long cap = static_cast<long long>(sms) * 16;
    gdn_pack_proj_kernel<<<static_cast<unsigned>(p.n_blocks < cap ? p.n_blocks : cap), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t read_proj_error(uint32_t* out) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_proj_error, sizeof(v));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_proj_error, &zero, sizeof(zero));
    *out = v;
    return e;
}

}  // namespace gdn
