// gdn_step.cu - the fused Gated DeltaNet decode step for GB300 (sm_103a),
// multi-token form (T > 1), plus the dispatch of every call.
//
// One persistent kernel computes, for every (sequence b, layer l, token t), the
// whole recurrent-mixer step listed in the header comment of the Winery-Strata
// page include/strata/core/layer.hpp and composed by gdn_layer (steps 3-7) on
// src/core/layer.cpp: causal conv + SiLU + L2 norm of q and k + q scale +
// beta/decay gates + the gated delta rule on the 128x128 fp32 state + the
// sigmoid-gated RMSNorm. Tokens of a window are applied in order with the
// state held on chip (Verifier::record_window on src/core/verify.cpp).
//
// Work unit. One unit is (b, l, k head g): the 3 v heads 3g..3g+2 that read
// q/k head g, their three 64 KB state tiles, and the 640 conv channels they
// need (q and k of head g, v of the three heads). Because one CTA owns all the
// conv channels of its unit, it reads the old conv history and writes the new
// one with no other CTA touching those channels.
//
// Thread mapping. 384 threads = 3 groups of 128, one group per tile. Within a
// group each thread holds a 32-row x 4-column block of its tile in registers
// for the whole unit (the quad mapping of gdn_device.cuh).
//
// Memory pipeline. Each CTA runs on its own SM and walks units u, u + grid,
// ... . A tile reaches shared memory through one 64 KB bulk async copy
// (cp.async.bulk, completion on an mbarrier, evict-first in L2); as soon as a
// group has copied its tile into registers, the group's leader issues the copy
// of the same tile slot of the CTA's next unit. The next unit's small inputs
// are pulled into L2 one unit ahead. Updated tiles return with 128-bit
// streaming stores.
//
// Tokens. The conv, norms and gates of up to kChunk tokens are computed in
// parallel into shared-memory records, then the recurrence walks those tokens
// with the tiles in registers, then y is produced for the chunk. The conv
// history of a chunk is re-read from the previous chunk's qkv rows.
//
// The single-token call runs gdn_decode_t1.cu instead, with the same
// arithmetic in the same order, so a T-token call equals T one-token calls
// bit for bit.

#include <mutex>

#include "gdn_device.cuh"
#include "gdn_launch.h"

namespace gdn {
namespace {

constexpr int kS = kHeadDim;
constexpr int kTile = kS * kS;                       // floats per state tile
constexpr uint32_t kTileBytes = kTile * 4;           // 65536
constexpr int kChunk = 8;                            // tokens whose inputs are staged at once
constexpr int kUnitChannels = 2 * kS + kGroup * kS;  // 640 conv channels per unit
constexpr int kWarps = kThreads / 32;                // 12

// Per-token record in shared memory (floats). Channel slot cc of the unit maps
// to record offset cc: q at [0,128), k at [128,256), v at [256,640).
constexpr int kRecQ = 0;
constexpr int kRecK = kS;
constexpr int kRecV = 2 * kS;
constexpr int kRecO = kUnitChannels;        // o of the 3 heads, 384 floats
constexpr int kRecG = kRecO + kGroup * kS;  // beta[3], decay[3], pad
constexpr int kRecFloats = kRecG + 8;       // 1032 floats = 4128 bytes (16-byte multiple)

constexpr size_t kSmemTiles = size_t(kGroup) * kTileBytes;                 // 196608
constexpr size_t kSmemRecs = size_t(kChunk) * kRecFloats * sizeof(float);  // 33024
constexpr size_t kSmemBars = 64;
constexpr size_t kSmemBytes = kSmemTiles + kSmemRecs + kSmemBars;         // 229696

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

// Decodes unit u into (b * L + l, k head g).
__device__ __forceinline__ void unit_coords(long long u, long long& bl, int& g) {
    bl = u / kKHeads;
    g = static_cast<int>(u - bl * kKHeads);
}

// Starts L2 prefetches of everything unit u reads besides its state tiles: the
// conv history, conv weights, per-token q/k/v slices, z slices and the alpha
// and beta rows. Issued one unit ahead, these make the next unit's prologue and
// epilogue loads L2 hits instead of DRAM round trips on its critical path.
__device__ __forceinline__ void prefetch_unit_inputs(const Params& p, long long u, int tid) {
    long long bl;
    int g;
    unit_coords(u, bl, g);
    const int l = static_cast<int>(bl % p.L);
    const int b = static_cast<int>(bl / p.L);
    int n = p.T;
    if (p.seq_len != nullptr) n = min(max(__ldg(p.seq_len + b), 0), p.T);
    const int items = 6 + 6 * n;
    for (int it = tid; it < items; it += kThreads) {
        if (it < 6) {
            const int k = it % 3;
            const int c = unit_channel(k == 0 ? 0 : (k == 1 ? kS : 2 * kS), g);
            const int ch = k < 2 ? kS : kGroup * kS;
            if (it < 3)
                prefetch_l2(p.conv_state + (static_cast<size_t>(bl) * kConvChannels + c) * (kDConv - 1),
                            ch * (kDConv - 1) * 4);
            else
                prefetch_l2(p.conv_w + (static_cast<size_t>(l) * kConvChannels + c) * kDConv, ch * kDConv * 4);
        } else {
            const int t = (it - 6) / 6;
            const int k = (it - 6) - 6 * t;
            const size_t row = static_cast<size_t>(bl) * p.T + t;
            if (k < 3) {
                const int c = unit_channel(k == 0 ? 0 : (k == 1 ? kS : 2 * kS), g);
                prefetch_l2(p.qkv + row * kConvChannels + c, (k < 2 ? kS : kGroup * kS) * 4);
            } else if (k == 3) {
                if ((p.flags & kNoY) == 0) prefetch_l2(p.z + row * kValueDim + g * kGroup * kS, kGroup * kS * 4);
            } else {
                prefetch_l2((k == 4 ? p.alpha : p.beta) + row * kVHeads, kVHeads * 4);
            }
        }
    }
}

// Issues the bulk copy of tile `hh` of unit `u` into its shared-memory slot.
__device__ __forceinline__ void issue_tile(const Params& p, long long u, int hh, uint32_t dst, uint32_t bar) {
    long long bl;
    int g;
    unit_coords(u, bl, g);
    const float* src = p.state + (static_cast<size_t>(bl) * kVHeads + g * kGroup + hh) * kTile;
    mbar_arrive_expect_tx(bar, kTileBytes);
    bulk_load_stream(dst, src, kTileBytes, bar);
}

// Conv + SiLU of one channel slot for the chunk's tokens [c0, c0 + tc). The
// 3-entry history before c0 (oldest first) comes from conv_state for the first
// chunk and from the previous three qkv rows otherwise (kChunk >= 3), so no
// history stays in registers between chunks. After the last chunk the rolled
// window is the new conv_state.
__device__ __forceinline__ void conv_slot(const Params& p, float* rec, int cc, int g, long long bl, int l, int c0,
                                          int tc, bool last_chunk, bool write_state) {
    const int c = unit_channel(cc, g);
    const float4 w =
        __ldg(reinterpret_cast<const float4*>(p.conv_w + (static_cast<size_t>(l) * kConvChannels + c) * kDConv));
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
            const float xc = conv4(w, h0, h1, h2, xs[t]);
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
    const Quad qd = quad_of(tid % kS);
    const bool group_leader = (tid % kS) == 0;
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
    if (u < p.n_units) prefetch_unit_inputs(p, u, tid);
    uint32_t parity = 0;
    bool failed = false;

    for (; u < p.n_units; u += stride) {
        if (u + stride < p.n_units) prefetch_unit_inputs(p, u + stride, tid);
        long long bl;
        int g;
        unit_coords(u, bl, g);
        const int l = static_cast<int>(bl % p.L);
        const int b = static_cast<int>(bl / p.L);
        int n = p.T;
        if (p.seq_len != nullptr) n = min(max(p.seq_len[b], 0), p.T);

        float s[128];

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
                    float bt, dc;
                    head_gates(__ldg(p.alpha + row), __ldg(p.beta + row),
                               __ldg(p.dt + static_cast<size_t>(l) * kVHeads + head),
                               __ldg(p.ssm_a + static_cast<size_t>(l) * kVHeads + head), bt, dc);
                    rec[t * kRecFloats + kRecG + hv] = bt;
                    rec[t * kRecFloats + kRecG + kGroup + hv] = dc;
                }
            }
            __syncthreads();

            // ---- L2 norm of q and k (one warp per token) and the q scale
            if (warp < tc) normalize_qk(rec + warp * kRecFloats + kRecQ, rec + warp * kRecFloats + kRecK, lane);
            __syncthreads();

            if (c0 == 0) {
                // This unit's tile: wait for its copy, move it into registers,
                // then hand the slot to the copy of the next unit's tile.
                if (!mbar_wait_bounded(my_bar, parity)) failed = true;
                parity ^= 1u;
                tile_load_quad(s, my_tile, qd);
                named_barrier(1 + hh, kS);
                const long long next = u + stride;
                if (group_leader && next < p.n_units) {
                    fence_proxy_async_smem();
                    issue_tile(p, next, hh, my_tile_s, my_bar);
                }
            }

            // ---- the gated delta rule, token by token, on the tile in registers
            for (int t = 0; t < tc; ++t) {
                float* r = rec + t * kRecFloats;
                const float4 v4 = *reinterpret_cast<const float4*>(r + kRecV + hh * kS + qd.col0);
                const float4 o4 =
                    delta_step_quad(s, r + kRecQ, r + kRecK, qd, v4, r[kRecG + hh], r[kRecG + kGroup + hh]);
                if (qd.rb == 0) *reinterpret_cast<float4*>(r + kRecO + hh * kS + qd.col0) = o4;
            }

            if (last_chunk && write_state)
                tile_store_quad(s, p.state + (static_cast<size_t>(bl) * kVHeads + g * kGroup + hh) * kTile, qd);
            __syncthreads();

            // ---- y = rms_norm(o) * ssm_norm * gate(z), one warp per (token, head)
            if (write_y) {
                for (int pi = warp; pi < tc * kGroup; pi += kWarps) {
                    const int t = pi / kGroup;
                    const int hv = pi - t * kGroup;
                    const int head = g * kGroup + hv;
                    const float4 o4 =
                        *reinterpret_cast<const float4*>(rec + t * kRecFloats + kRecO + hv * kS + lane * 4);
                    const size_t off = (static_cast<size_t>(bl) * p.T + c0 + t) * kValueDim + head * kS + lane * 4;
                    const float4 z4 = __ldg(reinterpret_cast<const float4*>(p.z + off));
                    const float4 w4 =
                        __ldg(reinterpret_cast<const float4*>(p.ssm_norm + static_cast<size_t>(l) * kS + lane * 4));
                    __stcs(reinterpret_cast<float4*>(p.y + off), gated_rms_norm4(o4, z4, w4, silu_gate));
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

std::mutex g_mutex;
int g_sms[64] = {0};

cudaError_t device_setup(int* sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_sms[dev] == 0) {
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(gdn_decode_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        g_sms[dev] = n;
    }
    *sms = g_sms[dev];
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_decode_step(const StepArgs& a, cudaStream_t stream) {
    if (a.T == 1) return launch_decode_t1(a, stream);
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
    if (e != cudaSuccess) return e;
    uint32_t v1 = 0;
    e = read_t1_error(&v1);
    *out = v | v1;
    return e;
}

}  // namespace gdn
