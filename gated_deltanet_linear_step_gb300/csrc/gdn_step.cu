// gdn_step.cu - the fused Gated DeltaNet decode step for GB300 (sm_103a).
//
// One persistent kernel computes, for every (sequence b, layer l, token t), the
// whole recurrent-mixer step listed in the header comment of the Winery-Strata
// page include/strata/core/layer.hpp and composed by gdn_layer (steps 3-7) on
// src/core/layer.cpp: causal conv + SiLU + L2 norm of q and k + q scale +
// beta/decay gates + the gated delta rule on the 128x128 fp32 state + the
// sigmoid-gated RMSNorm.
//
// Work unit. One unit is (b, l, k head g): the 3 v heads 3g..3g+2 that read
// q/k head g, their three 64 KB state tiles, and the 640 conv channels they
// need (q and k of head g, v of the three heads). Because one CTA owns all the
// conv channels of its unit, it reads the old conv history and writes the new
// one with no other CTA touching those channels.
//
// Thread mapping. 384 threads = 3 groups of 128; thread (h, j) owns column j
// of tile h: the 128 fp32 values S[0..127][j] live in its registers for the
// whole unit. Both column reductions of the delta rule (S^T k, S^T q) are then
// sums inside one thread, so a token step needs no cross-thread exchange; the
// rank-1 update touches only the thread's own registers.
//
// Memory pipeline. Each CTA runs on its own SM and walks units u, u + grid,
// ... . A tile reaches shared memory through one 64 KB bulk async copy
// (cp.async.bulk, completion on an mbarrier); as soon as a group has copied
// its tile into registers, the group's leader issues the copy of the same tile
// slot of the CTA's next unit, so the next unit's 192 KB stream in while this
// unit computes. Updated tiles go back with streaming 128-byte-per-warp stores.
//
// Tokens. The conv, norms and gates of up to kChunk tokens are computed in
// parallel into shared-memory records, then the recurrence walks those tokens
// with the tiles held in registers, then y is produced for the chunk. The conv
// history of a chunk is re-read from the previous chunk's qkv rows.
//
// Rounding order. With kv = decay * (S^T k) and o = decay * (S^T q) + d (k.q),
// one read of the pre-update state gives both reductions. This is the
// definition's S *= decay; kv = S^T k; d = (v - kv) beta; S += k d^T;
// o = S^T q rearranged by exact algebra; only the rounding differs.

#include "gdn_launch.h"

#include <cstdio>
#include <mutex>

namespace gdn {
namespace {

constexpr int kS = kHeadDim;
constexpr int kTile = kS * kS;                 // floats per state tile
constexpr uint32_t kTileBytes = kTile * 4;     // 65536
constexpr int kChunk = 8;                      // tokens whose inputs are staged at once
constexpr int kUnitChannels = 2 * kS + kGroup * kS;  // 640 conv channels per unit
constexpr int kWarps = kThreads / 32;          // 12

// Per-token record in shared memory (floats). Channel slot cc of the unit maps
// to record offset cc: q at [0,128), k at [128,256), v at [256,640).
constexpr int kRecQ = 0;
constexpr int kRecK = kS;
constexpr int kRecV = 2 * kS;
constexpr int kRecO = kUnitChannels;           // o of the 3 heads, 384 floats
constexpr int kRecG = kRecO + kGroup * kS;     // beta[3], decay[3], k.q, pad
constexpr int kRecFloats = kRecG + 8;          // 1032 floats = 4128 bytes (16-byte multiple)

constexpr size_t kSmemTiles = size_t(kGroup) * kTileBytes;                 // 196608
constexpr size_t kSmemRecs = size_t(kChunk) * kRecFloats * sizeof(float);  // 33024
constexpr size_t kSmemBars = 64;
constexpr size_t kSmemBytes = kSmemTiles + kSmemRecs + kSmemBars;         // 229696

constexpr float kEps = 1e-6f;
constexpr float kQScale = 0.08838834764831845f;  // 1/sqrt(128)
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per mbarrier wait

constexpr uint32_t kErrWaitTimeout = 1u;

static_assert(kSmemBytes <= 232448, "shared memory budget exceeds 227 KB");
static_assert(kRecFloats % 4 == 0, "records must stay 16-byte aligned");
static_assert(kWarps >= kChunk, "one warp normalises one token's q and k");
static_assert(kChunk >= kDConv - 1, "a chunk's conv history must come from the previous chunk");

__device__ unsigned int g_device_error = 0;

struct Params {
    const float* qkv;
    const float* z;
    const float* alpha;
    const float* beta;
    const float* dt;
    const float* ssm_a;
    const float* conv_w;
    const float* ssm_norm;
    float* conv_state;
    float* state;
    float* y;
    const int32_t* seq_len;
    int B, L, T;
    uint32_t flags;
    long long n_units;
};

// ------------------------------------------------------------ PTX helpers --
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for phase `parity` of the mbarrier, giving up after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// One contiguous global -> shared bulk copy; completion is signalled on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Keeps the compiler from hoisting every shared-memory load of a 128-row loop
// ahead of its FMAs: with the column's 128 state values already in registers,
// hoisted loads would push the thread past its register budget and spill.
__device__ __forceinline__ void compiler_fence() { asm volatile("" ::: "memory"); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float siluf_(float x) { return x / (1.0f + expf(-x)); }
__device__ __forceinline__ float softplusf_(float x) { return fmaxf(x, 0.0f) + log1pf(expf(-fabsf(x))); }

// Global conv channel of unit channel slot cc for k head g.
__device__ __forceinline__ int unit_channel(int cc, int g) {
    return cc < kS ? g * kS + cc : (cc < 2 * kS ? kKOffset + g * kS + (cc - kS) : kVOffset + g * kGroup * kS + (cc - 2 * kS));
}

// Issues the bulk copy of tile `hh` of unit `u` into its shared-memory slot.
__device__ __forceinline__ void issue_tile(const Params& p, long long u, int hh, uint32_t dst, uint32_t bar) {
    const long long bl = u / kKHeads;
    const int g = static_cast<int>(u - bl * kKHeads);
    const float* src = p.state + (static_cast<size_t>(bl) * kVHeads + g * kGroup + hh) * kTile;
    mbar_arrive_expect_tx(bar, kTileBytes);
    bulk_load(dst, src, kTileBytes, bar);
}

// Conv + SiLU of one channel slot for the chunk's tokens [c0, c0 + tc). The
// 3-entry history before c0 (oldest first) comes from conv_state for the first
// chunk and from the previous three qkv rows otherwise (kChunk >= 3), so no
// history has to stay in registers between chunks. After the last chunk the
// rolled window holds the new conv_state.
__device__ __forceinline__ void conv_slot(const Params& p, float* rec, int cc, int g, long long bl, int l, int c0,
                                          int tc, bool last_chunk, bool write_state) {
    const int c = unit_channel(cc, g);
    const float4 w = __ldg(reinterpret_cast<const float4*>(p.conv_w + (static_cast<size_t>(l) * kConvChannels + c) * kDConv));
    float* cs = p.conv_state + (static_cast<size_t>(bl) * kConvChannels + c) * (kDConv - 1);
    const float* xq = p.qkv + (static_cast<size_t>(bl) * p.T + c0) * kConvChannels + c;
    float h0, h1, h2;
    if (c0 == 0) {
        h0 = cs[0];
        h1 = cs[1];
        h2 = cs[2];
    } else {
        h0 = __ldg(xq - 3 * kConvChannels);
        h1 = __ldg(xq - 2 * kConvChannels);
        h2 = __ldg(xq - 1 * kConvChannels);
    }
    float xs[kChunk];
#pragma unroll
    for (int t = 0; t < kChunk; ++t) xs[t] = (t < tc) ? __ldg(xq + static_cast<size_t>(t) * kConvChannels) : 0.0f;
#pragma unroll
    for (int t = 0; t < kChunk; ++t) {
        if (t < tc) {
            float xc = w.x * h0;
            xc = fmaf(w.y, h1, xc);
            xc = fmaf(w.z, h2, xc);
            xc = fmaf(w.w, xs[t], xc);
            h0 = h1;
            h1 = h2;
            h2 = xs[t];
            rec[t * kRecFloats + cc] = siluf_(xc);
        }
    }
    if (last_chunk && write_state) {
        cs[0] = h0;
        cs[1] = h1;
        cs[2] = h2;
    }
}

__global__ void __launch_bounds__(kThreads, 1) gdn_decode_step_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(128) unsigned char smem[];
    float* tiles = reinterpret_cast<float*>(smem);
    float* rec = reinterpret_cast<float*>(smem + kSmemTiles);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kSmemTiles + kSmemRecs);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int hh = tid / kS;  // tile group = v head within the unit
    const int j = tid % kS;   // state column owned by this thread
    const bool group_leader = (j == 0);
    const float* my_tile = tiles + hh * kTile;
    const uint32_t my_tile_s = smem_addr(my_tile);
    const uint32_t my_bar = smem_addr(&bars[hh]);
    const bool write_state = (p.flags & kNoStateWrite) == 0;
    const bool write_y = (p.flags & kNoY) == 0;
    const bool silu_gate = (p.flags & kSiluGate) != 0;

    if (tid == 0) {
        for (int h = 0; h < kGroup; ++h) mbar_init(smem_addr(&bars[h]), 1);
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    __syncthreads();

    long long u = blockIdx.x;
    const long long stride = gridDim.x;
    if (group_leader && u < p.n_units) issue_tile(p, u, hh, my_tile_s, my_bar);
    uint32_t parity = 0;
    bool failed = false;

    for (; u < p.n_units; u += stride) {
        const long long bl = u / kKHeads;
        const int g = static_cast<int>(u - bl * kKHeads);
        const int l = static_cast<int>(bl % p.L);
        const int b = static_cast<int>(bl / p.L);
        int n = p.T;
        if (p.seq_len != nullptr) n = min(max(p.seq_len[b], 0), p.T);

        float s[kS];

        // Chunks of up to kChunk tokens. A sequence with no valid token still
        // runs one empty chunk, so that its tile slot is consumed and refilled.
        int c0 = 0;
        do {
            const int tc = min(kChunk, n - c0);
            const bool last_chunk = (c0 + tc == n) && n > 0;

            // ---- conv + SiLU of the unit's 640 channels; gates of its 3 heads
            conv_slot(p, rec, tid, g, bl, l, c0, tc, last_chunk, write_state);
            if (tid + kThreads < kUnitChannels)
                conv_slot(p, rec, tid + kThreads, g, bl, l, c0, tc, last_chunk, write_state);
            if (tid >= kThreads - kGroup * kChunk) {
                const int idx = tid - (kThreads - kGroup * kChunk);
                const int t = idx / kGroup;
                const int hv = idx - t * kGroup;
                if (t < tc) {
                    const int head = g * kGroup + hv;
                    const size_t row = (static_cast<size_t>(bl) * p.T + c0 + t) * kVHeads + head;
                    const float a = __ldg(p.alpha + row) + __ldg(p.dt + static_cast<size_t>(l) * kVHeads + head);
                    const float gval = softplusf_(a) * __ldg(p.ssm_a + static_cast<size_t>(l) * kVHeads + head);
                    rec[t * kRecFloats + kRecG + hv] = sigmoidf_(__ldg(p.beta + row));
                    rec[t * kRecFloats + kRecG + kGroup + hv] = expf(gval);
                }
            }
            __syncthreads();

            // ---- L2 norm of q and k (one warp per token), q scale, and k.q
            if (warp < tc) {
                float* r = rec + warp * kRecFloats;
                float4 q4 = *reinterpret_cast<float4*>(r + kRecQ + lane * 4);
                float4 k4 = *reinterpret_cast<float4*>(r + kRecK + lane * 4);
                const float sq = warp_sum(q4.x * q4.x + q4.y * q4.y + q4.z * q4.z + q4.w * q4.w);
                const float sk = warp_sum(k4.x * k4.x + k4.y * k4.y + k4.z * k4.z + k4.w * k4.w);
                const float rq = rsqrtf(sq + kEps) * kQScale;
                const float rk = rsqrtf(sk + kEps);
                q4.x *= rq; q4.y *= rq; q4.z *= rq; q4.w *= rq;
                k4.x *= rk; k4.y *= rk; k4.z *= rk; k4.w *= rk;
                *reinterpret_cast<float4*>(r + kRecQ + lane * 4) = q4;
                *reinterpret_cast<float4*>(r + kRecK + lane * 4) = k4;
                const float kq = warp_sum(q4.x * k4.x + q4.y * k4.y + q4.z * k4.z + q4.w * k4.w);
                if (lane == 0) r[kRecG + 2 * kGroup] = kq;
            }
            __syncthreads();

            if (c0 == 0) {
                // This unit's tile: wait for its copy, move it into registers,
                // then hand the slot to the copy of the next unit's tile.
                if (!mbar_wait_bounded(my_bar, parity)) failed = true;
                parity ^= 1u;
#pragma unroll
                for (int i = 0; i < kS; ++i) s[i] = my_tile[i * kS + j];
                named_barrier(1 + hh, kS);
                const long long next = u + stride;
                if (group_leader && next < p.n_units) {
                    fence_proxy_async_smem();
                    issue_tile(p, next, hh, my_tile_s, my_bar);
                }
            }

            // ---- the gated delta rule, token by token, on the column in registers
            for (int t = 0; t < tc; ++t) {
                float* r = rec + t * kRecFloats;
                const float beta_t = r[kRecG + hh];
                const float decay_t = r[kRecG + kGroup + hh];
                const float kq = r[kRecG + 2 * kGroup];
                const float vj = r[kRecV + hh * kS + j];
                float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
                float b0 = 0.f, b1 = 0.f, b2 = 0.f, b3 = 0.f;
#pragma unroll
                for (int i = 0; i < kS; i += 4) {
                    const float4 k4 = *reinterpret_cast<const float4*>(r + kRecK + i);
                    const float4 q4 = *reinterpret_cast<const float4*>(r + kRecQ + i);
                    a0 = fmaf(s[i], k4.x, a0);
                    a1 = fmaf(s[i + 1], k4.y, a1);
                    a2 = fmaf(s[i + 2], k4.z, a2);
                    a3 = fmaf(s[i + 3], k4.w, a3);
                    b0 = fmaf(s[i], q4.x, b0);
                    b1 = fmaf(s[i + 1], q4.y, b1);
                    b2 = fmaf(s[i + 2], q4.z, b2);
                    b3 = fmaf(s[i + 3], q4.w, b3);
                    if ((i & 15) == 12) compiler_fence();
                }
                const float kv = decay_t * ((a0 + a1) + (a2 + a3));
                const float sq = decay_t * ((b0 + b1) + (b2 + b3));
                const float d = beta_t * (vj - kv);
                r[kRecO + hh * kS + j] = fmaf(d, kq, sq);
#pragma unroll
                for (int i = 0; i < kS; i += 4) {
                    const float4 k4 = *reinterpret_cast<const float4*>(r + kRecK + i);
                    s[i] = fmaf(k4.x, d, decay_t * s[i]);
                    s[i + 1] = fmaf(k4.y, d, decay_t * s[i + 1]);
                    s[i + 2] = fmaf(k4.z, d, decay_t * s[i + 2]);
                    s[i + 3] = fmaf(k4.w, d, decay_t * s[i + 3]);
                    if ((i & 15) == 12) compiler_fence();
                }
            }

            if (last_chunk && write_state) {
                float* dst = p.state + (static_cast<size_t>(bl) * kVHeads + g * kGroup + hh) * kTile + j;
#pragma unroll
                for (int i = 0; i < kS; ++i) __stcs(dst + i * kS, s[i]);
            }
            __syncthreads();

            // ---- y = rms_norm(o) * ssm_norm * gate(z), one warp per (token, head)
            if (write_y) {
                for (int pi = warp; pi < tc * kGroup; pi += kWarps) {
                    const int t = pi / kGroup;
                    const int hv = pi - t * kGroup;
                    const int head = g * kGroup + hv;
                    const float4 o4 = *reinterpret_cast<const float4*>(rec + t * kRecFloats + kRecO + hv * kS + lane * 4);
                    const float ss = warp_sum(o4.x * o4.x + o4.y * o4.y + o4.z * o4.z + o4.w * o4.w);
                    const float rr = rsqrtf(ss * (1.0f / kS) + kEps);
                    const size_t off = (static_cast<size_t>(bl) * p.T + c0 + t) * kValueDim + head * kS + lane * 4;
                    const float4 z4 = __ldg(reinterpret_cast<const float4*>(p.z + off));
                    const float4 w4 = __ldg(reinterpret_cast<const float4*>(p.ssm_norm + static_cast<size_t>(l) * kS + lane * 4));
                    float4 y4;
                    if (silu_gate) {
                        y4.x = o4.x * rr * w4.x * siluf_(z4.x);
                        y4.y = o4.y * rr * w4.y * siluf_(z4.y);
                        y4.z = o4.z * rr * w4.z * siluf_(z4.z);
                        y4.w = o4.w * rr * w4.w * siluf_(z4.w);
                    } else {
                        y4.x = o4.x * rr * w4.x * sigmoidf_(z4.x);
                        y4.y = o4.y * rr * w4.y * sigmoidf_(z4.y);
                        y4.z = o4.z * rr * w4.z * sigmoidf_(z4.z);
                        y4.w = o4.w * rr * w4.w * sigmoidf_(z4.w);
                    }
                    *reinterpret_cast<float4*>(p.y + off) = y4;
                }
            }
            c0 += kChunk;
        } while (c0 < n);

        // A wait that gave up anywhere in the CTA stops the whole CTA after this unit.
        if (__syncthreads_or(failed ? 1 : 0)) {
            if (tid == 0) atomicOr(&g_device_error, kErrWaitTimeout);
            // Let the copy already issued for the next unit land before the CTA exits.
            if (u + stride < p.n_units) (void)mbar_wait_bounded(my_bar, parity);
            return;
        }
    }
}

struct DeviceInfo {
    bool ready = false;
    int sms = 0;
};

std::mutex g_mutex;
DeviceInfo g_devices[64];

cudaError_t device_setup(int* sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo& d = g_devices[dev];
    if (!d.ready) {
        e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(gdn_decode_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        d.ready = true;
    }
    *sms = d.sms;
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_decode_step(const StepArgs& a, cudaStream_t stream) {
    int sms = 0;
    cudaError_t e = device_setup(&sms);
    if (e != cudaSuccess) return e;
    Params p;
    p.qkv = a.qkv;
    p.z = a.z;
    p.alpha = a.alpha;
    p.beta = a.beta;
    p.dt = a.dt;
    p.ssm_a = a.ssm_a;
    p.conv_w = a.conv_w;
    p.ssm_norm = a.ssm_norm;
    p.conv_state = a.conv_state;
    p.state = a.state;
    p.y = a.y;
    p.seq_len = a.seq_len;
    p.B = a.B;
    p.L = a.L;
    p.T = a.T;
    p.flags = a.flags;
    p.n_units = static_cast<long long>(a.B) * a.L * kKHeads;
    const long long grid = p.n_units < sms ? p.n_units : sms;
    gdn_decode_step_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t read_device_error(cudaStream_t stream, uint32_t* out) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    unsigned int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    *out = v;
    return e;
}

}  // namespace gdn
