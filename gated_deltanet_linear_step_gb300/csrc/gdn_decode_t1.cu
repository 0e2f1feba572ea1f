// gdn_decode_t1.cu - the single-token decode step (T = 1): the batched-decode
// hot path, where every (sequence, layer) state is read and written once per
// call and the step is bound by HBM bandwidth.
//
// Same arithmetic as the multi-token kernel (the operation
// order of the header comment of Winery-Strata include/strata/core/layer.hpp,
// composed by gdn_layer steps 3-7 on src/core/layer.cpp), organised so that
// nothing on a unit's critical path waits on global memory:
//
// * Unit = (layer l, k head g, sequence b): three 64 KB state tiles plus the
//   640 conv channels of q/k head g and v heads 3g..3g+2. CTA c of the
//   persistent grid (one per SM) owns a contiguous range of units ordered
//   (l, g, b), so consecutive units share their layer weights.
// * Bulk async copies (cp.async.bulk, completion on mbarriers) bring in
//   - each state tile one unit ahead (three 64 KB slots, evict-first in L2),
//   - each unit's small inputs (conv history, q|k|v slice, alpha and beta
//     rows, z slice: 12,160 bytes) two units ahead (two slots),
//   - the layer weights of an (l, g) run (conv taps, dt, ssm_a, ssm_norm).
// * Conv, SiLU, norms and gates then read and write shared memory only.
// * Each tile stays in its shared-memory slot: the group's threads (32x4
//   blocks, the quad mapping of gdn_device.cuh) reduce it, update it in place
//   and accumulate o, then one bulk async store writes it back. The stores
//   drain through the copy engine while the warps go on to y and the next
//   unit; plain per-thread stores of 192 KB per unit would instead clog each
//   SM's memory-instruction path and stall everything behind them. The slot
//   is refilled with the next unit's tile once the store has read it.
// * o overwrites v in the staging slot; y leaves with 128-bit stores.

#include <mutex>

#include "gdn_device.cuh"
#include "gdn_launch.h"

namespace gdn {
namespace {

constexpr int kS = kHeadDim;
constexpr int kTile = kS * kS;
constexpr uint32_t kTileBytes = kTile * 4;
constexpr int kUnitCh = 2 * kS + kGroup * kS;  // 640

// Staging slot (floats): the per-unit inputs.
constexpr int kStCs = 0;                       // conv history [640][3], oldest first
constexpr int kStX = kStCs + kUnitCh * 3;      // qkv slice [640]; becomes q^|k^|v, then q^|k^|o
constexpr int kStAlpha = kStX + kUnitCh;       // alpha row [48] of (b, l)
constexpr int kStBeta = kStAlpha + kVHeads;    // beta row [48]
constexpr int kStZ = kStBeta + kVHeads;        // z slice [384] of the unit's heads
constexpr int kStFloats = kStZ + kGroup * kS;  // 3040 floats = 12160 bytes
// Weight slot (floats): one (l, g) run's weights.
constexpr int kWtConv = 0;                     // conv taps [640][4]
constexpr int kWtDt = kUnitCh * 4;             // dt row [48]
constexpr int kWtA = kWtDt + kVHeads;          // ssm_a row [48]
constexpr int kWtNorm = kWtA + kVHeads;        // ssm_norm [128]
constexpr int kWtFloats = kWtNorm + kS;        // 2784 floats = 11136 bytes

constexpr size_t kOffTiles = 0;
constexpr size_t kOffStage = size_t(kGroup) * kTileBytes;          // 196608
constexpr size_t kOffWt = kOffStage + 2 * size_t(kStFloats) * 4;   // 220928
constexpr size_t kOffBars = kOffWt + size_t(kWtFloats) * 4;        // 232064
constexpr int kBarTile = 0, kBarStage = 3, kBarWt = 5, kNumBars = 6;
constexpr size_t kOffGates = kOffBars + kNumBars * 8;              // beta[3], decay[3], pad
constexpr size_t kSmemBytes = kOffGates + 8 * 4;                   // 232144

static_assert(kSmemBytes <= 232448, "shared memory budget exceeds 227 KB");
static_assert(kOffStage % 16 == 0 && kOffWt % 16 == 0 && (kStFloats * 4) % 16 == 0, "bulk copy alignment");
static_assert((kStX * 4) % 16 == 0 && (kStAlpha * 4) % 16 == 0 && (kStBeta * 4) % 16 == 0 && (kStZ * 4) % 16 == 0,
              "bulk copy alignment");
static_assert((kWtDt * 4) % 16 == 0 && (kWtA * 4) % 16 == 0 && (kWtNorm * 4) % 16 == 0, "bulk copy alignment");

__device__ unsigned int g_t1_error = 0;

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
    int B, L;
    uint32_t flags;
    long long n_units;
};

struct Unit {
    int l, g, b;
    long long bl;  // b * L + l
};

__device__ __forceinline__ Unit unit_of(const Params& p, long long u) {
    Unit x;
    const long long lg = u / p.B;
    x.b = static_cast<int>(u - lg * p.B);
    x.g = static_cast<int>(lg % kKHeads);
    x.l = static_cast<int>(lg / kKHeads);
    x.bl = static_cast<long long>(x.b) * p.L + x.l;
    return x;
}

// The unit after x in (l, g, b) order: b runs fastest, then g, then l.
__device__ __forceinline__ Unit next_unit(const Params& p, Unit x) {
    if (++x.b == p.B) {
        x.b = 0;
        if (++x.g == kKHeads) {
            x.g = 0;
            ++x.l;
        }
    }
    x.bl = static_cast<long long>(x.b) * p.L + x.l;
    return x;
}

__device__ __forceinline__ const float* tile_src(const Params& p, const Unit& x, int hh) {
    return p.state + (static_cast<size_t>(x.bl) * kVHeads + x.g * kGroup + hh) * kTile;
}

// The 9 bulk copies of a unit's small inputs, one per lane 0..8 of the calling
// warp; lane 0 also arms the slot's mbarrier with the total byte count.
__device__ __forceinline__ void issue_stage(const Params& p, const Unit& x, uint32_t dst, uint32_t bar, int lane) {
    const bool with_z = (p.flags & kNoY) == 0;
    if (lane == 0) mbar_arrive_expect_tx(bar, (kStFloats - (with_z ? 0 : kGroup * kS)) * 4);
    const float* cs = p.conv_state + static_cast<size_t>(x.bl) * kConvChannels * (kDConv - 1);
    const float* xr = p.qkv + static_cast<size_t>(x.bl) * kConvChannels;
    switch (lane) {
        case 0: bulk_load(dst + kStCs * 4, cs + x.g * kS * 3, kS * 3 * 4, bar); break;
        case 1: bulk_load(dst + (kStCs + kS * 3) * 4, cs + (kKOffset + x.g * kS) * 3, kS * 3 * 4, bar); break;
        case 2:
            bulk_load(dst + (kStCs + 2 * kS * 3) * 4, cs + (kVOffset + x.g * kGroup * kS) * 3, kGroup * kS * 3 * 4, bar);
            break;
        case 3: bulk_load(dst + kStX * 4, xr + x.g * kS, kS * 4, bar); break;
        case 4: bulk_load(dst + (kStX + kS) * 4, xr + kKOffset + x.g * kS, kS * 4, bar); break;
        case 5: bulk_load(dst + (kStX + 2 * kS) * 4, xr + kVOffset + x.g * kGroup * kS, kGroup * kS * 4, bar); break;
        case 6: bulk_load(dst + kStAlpha * 4, p.alpha + static_cast<size_t>(x.bl) * kVHeads, kVHeads * 4, bar); break;
        case 7: bulk_load(dst + kStBeta * 4, p.beta + static_cast<size_t>(x.bl) * kVHeads, kVHeads * 4, bar); break;
        case 8:
            if (with_z)
                bulk_load(dst + kStZ * 4, p.z + static_cast<size_t>(x.bl) * kValueDim + x.g * kGroup * kS,
                          kGroup * kS * 4, bar);
            break;
        default: break;
    }
}

// The weights of an (l, g) run, issued by one thread.
__device__ __forceinline__ void issue_weights(const Params& p, int l, int g, uint32_t dst, uint32_t bar) {
    const bool with_norm = (p.flags & kNoY) == 0;
    mbar_arrive_expect_tx(bar, (kWtFloats - (with_norm ? 0 : kS)) * 4);
    const float* cw = p.conv_w + static_cast<size_t>(l) * kConvChannels * kDConv;
    bulk_load(dst + kWtConv * 4, cw + g * kS * kDConv, kS * kDConv * 4, bar);
    bulk_load(dst + (kWtConv + kS * kDConv) * 4, cw + (kKOffset + g * kS) * kDConv, kS * kDConv * 4, bar);
    bulk_load(dst + (kWtConv + 2 * kS * kDConv) * 4, cw + (kVOffset + g * kGroup * kS) * kDConv,
              kGroup * kS * kDConv * 4, bar);
    bulk_load(dst + kWtDt * 4, p.dt + static_cast<size_t>(l) * kVHeads, kVHeads * 4, bar);
    bulk_load(dst + kWtA * 4, p.ssm_a + static_cast<size_t>(l) * kVHeads, kVHeads * 4, bar);
    if (with_norm) bulk_load(dst + kWtNorm * 4, p.ssm_norm + static_cast<size_t>(l) * kS, kS * 4, bar);
}

__global__ void __launch_bounds__(kThreads, 1) gdn_decode_t1_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(128) unsigned char smem[];
    float* tiles = reinterpret_cast<float*>(smem + kOffTiles);
    float* stage = reinterpret_cast<float*>(smem + kOffStage);
    float* wt = reinterpret_cast<float*>(smem + kOffWt);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
    float* gates = reinterpret_cast<float*>(smem + kOffGates);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int hh = tid >> 7;  // tile group: v head 3g + hh of the unit
    const Quad q = quad_of(tid & 127);
    const bool group_leader = (tid & 127) == 0;
    const bool write_state = (p.flags & kNoStateWrite) == 0;
    const bool write_y = (p.flags & kNoY) == 0;
    const bool silu_gate = (p.flags & kSiluGate) != 0;
    float* my_tile = tiles + hh * kTile;
    const uint32_t my_tile_s = smem_addr(my_tile);
    const uint32_t my_bar = smem_addr(&bars[kBarTile + hh]);

    const long long u_begin = p.n_units * blockIdx.x / gridDim.x;
    const long long u_end = p.n_units * (blockIdx.x + 1) / gridDim.x;
    if (u_begin >= u_end) return;

    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) mbar_init(smem_addr(&bars[i]), 1);
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    __syncthreads();

    Unit cur = unit_of(p, u_begin);
    int cur_lg = cur.l * kKHeads + cur.g;
    if (tid == 0) issue_weights(p, cur.l, cur.g, smem_addr(wt), smem_addr(&bars[kBarWt]));
    if (warp == 0) {
        issue_stage(p, cur, smem_addr(stage), smem_addr(&bars[kBarStage]), lane);
        if (u_begin + 1 < u_end)
            issue_stage(p, next_unit(p, cur), smem_addr(stage + kStFloats), smem_addr(&bars[kBarStage + 1]), lane);
    }
    if (group_leader) {
        mbar_arrive_expect_tx(my_bar, kTileBytes);
        bulk_load_stream(my_tile_s, tile_src(p, cur, hh), kTileBytes, my_bar);
    }

    uint32_t tile_par = 0, stage_par = 0, wt_par = 0;
    bool wt_pending = true;
    bool failed = false;         // one of this thread's waits gave up
    bool store_pending = false;  // a bulk store of this group's tile has not yet been waited for
    // The phase of a copy whose wait gave up in this thread, or -1: the copy may
    // still land, so it is waited for (bounded) before the CTA leaves.
    int wt_late = -1, stage_late = -1, tile_late = -1;
    bool give_up = (p.flags & kTestGiveUp) != 0;  // the first tile wait gives up (tests this path)

    for (long long u = u_begin; u < u_end; ++u) {
        const int slot = static_cast<int>((u - u_begin) & 1);
        float* S = stage + slot * kStFloats;
        const uint32_t stage_bar = smem_addr(&bars[kBarStage + slot]);
        const Unit x = cur;
        const Unit xn = next_unit(p, cur);
        cur = xn;
        const bool has_next = u + 1 < u_end;
        const int lg = x.l * kKHeads + x.g;
        if (lg != cur_lg) {  // a new (l, g) run: the previous unit has finished with the weights
            cur_lg = lg;
            if (tid == 0) {
                fence_proxy_async_smem();
                issue_weights(p, x.l, x.g, smem_addr(wt), smem_addr(&bars[kBarWt]));
            }
            wt_pending = true;
        }
        if (wt_pending) {
            if (!mbar_wait_bounded(smem_addr(&bars[kBarWt]), wt_par)) {
                failed = true;
                wt_late = static_cast<int>(wt_par);
            }
            wt_par ^= 1u;
            wt_pending = false;
        }
        int n = 1;
        if (p.seq_len != nullptr) n = min(max(__ldg(p.seq_len + x.b), 0), 1);
        if (!mbar_wait_bounded(stage_bar, (stage_par >> slot) & 1u)) {
            failed = true;
            stage_late = static_cast<int>((stage_par >> slot) & 1u);
        }
        stage_par ^= 1u << slot;

        // ---- conv + SiLU (in place over the qkv slice), new conv history, gates.
        // A thread whose wait gave up computes and writes nothing from here on.
        if (n > 0 && !failed) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int cc = tid + k * kThreads;
                if (cc < kUnitCh) {
                    const float h0 = S[kStCs + cc * 3 + 0];
                    const float h1 = S[kStCs + cc * 3 + 1];
                    const float h2 = S[kStCs + cc * 3 + 2];
                    const float xin = S[kStX + cc];
                    const float4 w = *reinterpret_cast<const float4*>(wt + kWtConv + cc * 4);
                    S[kStX + cc] = siluf_(conv4(w, h0, h1, h2, xin));
                    if (write_state) {
                        float* cs = p.conv_state + (static_cast<size_t>(x.bl) * kConvChannels + unit_channel(cc, x.g)) * 3;
                        cs[0] = h1;
                        cs[1] = h2;
                        cs[2] = xin;
                    }
                }
            }
            if (tid >= kThreads - kGroup) {
                const int hv = tid - (kThreads - kGroup);
                const int head = x.g * kGroup + hv;
                float bt, dc;
                head_gates_in((p.flags & kGatesReady) != 0, S[kStAlpha + head], S[kStBeta + head], wt[kWtDt + head],
                              wt[kWtA + head], bt, dc);
                gates[hv] = bt;
                gates[kGroup + hv] = dc;
            }
        }
        __syncthreads();
        // (the norm's shuffles need the whole warp: the decision is the warp's)
        if (n > 0 && warp == 0 && !__any_sync(0xffffffffu, failed)) normalize_qk(S + kStX, S + kStX + kS, lane);
        __syncthreads();

        // ---- this unit's tile
        const bool tile_ok = !give_up && mbar_wait_bounded(my_bar, tile_par);
        give_up = false;
        if (!tile_ok) {
            failed = true;
            tile_late = static_cast<int>(tile_par);
        }
        tile_par ^= 1u;

        // ---- the gated delta rule on the tile in its slot; o replaces v
        if (n > 0 && !__any_sync(0xffffffffu, failed)) {
            float* vo = S + kStX + 2 * kS + hh * kS + q.col0;
            const float4 v4 = *reinterpret_cast<const float4*>(vo);
            const float4 o4 = delta_step_smem(my_tile, S + kStX, S + kStX + kS, q, v4, gates[hh], gates[kGroup + hh]);
            __syncwarp();
            if (q.rb == 0) *reinterpret_cast<float4*>(vo) = o4;
            fence_proxy_async_smem();  // the updated tile is read next by the bulk store
        }
        const bool group_failed = named_barrier_or(1 + hh, kS, failed);
        if (group_leader && n > 0 && write_state && !group_failed) {
            bulk_store(p.state + (static_cast<size_t>(x.bl) * kVHeads + x.g * kGroup + hh) * kTile, my_tile_s,
                       kTileBytes);
            bulk_commit();
            store_pending = true;
        }

        if (__syncthreads_or(failed ? 1 : 0)) {
            // A wait gave up: record it, let every copy still in flight land (each
            // wait bounded), and stop. Each copy is waited for by the thread that
            // issued it, on the phase its own wait gave up on.
            if (tid == 0) {
                atomicOr(&g_t1_error, kErrWaitTimeout);
                if (wt_late >= 0) (void)mbar_wait_bounded(smem_addr(&bars[kBarWt]), static_cast<uint32_t>(wt_late));
                if (stage_late >= 0) (void)mbar_wait_bounded(stage_bar, static_cast<uint32_t>(stage_late));
                if (has_next)
                    (void)mbar_wait_bounded(smem_addr(&bars[kBarStage + (slot ^ 1)]), (stage_par >> (slot ^ 1)) & 1u);
            }
            if (group_leader) {
                if (tile_late >= 0) (void)mbar_wait_bounded(my_bar, static_cast<uint32_t>(tile_late));
                bulk_wait_all();
            }
            return;
        }

        // ---- y = rms_norm(o) * ssm_norm * gate(z), one warp per head
        if (n > 0 && write_y && warp < kGroup) {
            const float4 o4 = *reinterpret_cast<const float4*>(S + kStX + 2 * kS + warp * kS + lane * 4);
            const float4 z4 = *reinterpret_cast<const float4*>(S + kStZ + warp * kS + lane * 4);
            const float4 w4 = *reinterpret_cast<const float4*>(wt + kWtNorm + lane * 4);
            __stcs(reinterpret_cast<float4*>(p.y + static_cast<size_t>(x.bl) * kValueDim + (x.g * kGroup + warp) * kS +
                                             lane * 4),
                   gated_rms_norm4(o4, z4, w4, silu_gate));
        }
        __syncthreads();  // y has read the staging slot before it is refilled

        // The tile slot takes the next unit's tile once the store has read it.
        if (group_leader && has_next) {
            if (store_pending) bulk_wait_read();
            store_pending = false;
            mbar_arrive_expect_tx(my_bar, kTileBytes);
            bulk_load_stream(my_tile_s, tile_src(p, xn, hh), kTileBytes, my_bar);
        }
        // The staging slot is free again: bring in the unit after next.
        if (warp == 0 && u + 2 < u_end) {
            fence_proxy_async_smem();
            issue_stage(p, next_unit(p, xn), smem_addr(S), smem_addr(&bars[kBarStage + slot]), lane);
        }
    }
    if (group_leader) bulk_wait_all();  // the last stores must finish reading shared memory before exit
}

std::mutex g_mutex;
int g_sms[64] = {0};

}  // namespace

cudaError_t launch_decode_t1(const StepArgs& a, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int sms;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (g_sms[dev] == 0) {
            int n = 0;
            e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(gdn_decode_t1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kSmemBytes));
            if (e != cudaSuccess) return e;
            g_sms[dev] = n;
        }
        sms = g_sms[dev];
    }
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
    p.flags = a.flags;
    p.n_units = static_cast<long long>(a.B) * a.L * kKHeads;
    const long long grid = p.n_units < sms ? p.n_units : sms;
    gdn_decode_t1_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t read_t1_error(uint32_t* out) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_t1_error, sizeof(v));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_t1_error, &zero, sizeof(zero));
    *out = v;
    return e;
}

}  // namespace gdn
