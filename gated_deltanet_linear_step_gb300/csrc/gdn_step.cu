// gdn_step.cu - the fused Gated DeltaNet decode step for GB300 (sm_103a),
// register-resident form (windows, and single-token launches too small to fill
// the SMs), plus the dispatch of every call.
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
// q/k head g. A thread-block cluster of 3 CTAs takes a unit; CTA rank h owns
// the 64 KB tile of v head 3g + h, which its 256 threads hold in registers
// (64 values each, the octet mapping of gdn_device.cuh) across all T tokens.
// Two such CTAs fit on an SM, so an SM holds two tiles in registers with room
// to spare and the kernel does not spill.
//
// Conv history. Each CTA convolves its own 128 v channels and, redundantly,
// the 256 q/k channels of head g. All three CTAs read the old q/k history in
// a unit's first chunk; a cluster barrier follows, and only after it does
// rank 0 write the new q/k history (in the unit's last chunk). Each CTA writes
// the history of its own v channels. The barrier also keeps the three CTAs on
// the same unit. In the short-window instance (one chunk per unit) the barrier
// is split: each CTA arrives once it has read the old history and waits only at
// the unit's end, where rank 0 writes the new q/k history, so no CTA stalls on
// the others between its conv and its recurrence.
//
// Tokens. The conv, norms and gates of up to kChunk tokens are computed into
// shared-memory records, the recurrence walks them with the tile in
// registers, then y is produced for the chunk. z arrives in the records, and
// the layer's ssm_norm beside them, by bulk copy while the chunk computes. The conv history of a later chunk is
// re-read from the previous chunk's qkv rows.
//
// Tiles. A unit's tile arrives in the CTA's slot by bulk copy, moves to
// registers, and after the last token returns to the slot and leaves with one
// bulk store; the slot then takes the next unit's tile. The other CTA on the
// SM computes while one waits. Warps 4-7 convolve one channel slot to warps
// 0-3's two, so single threads of warps 4 and 5 issue the copies (z, and the
// tile's store and refill) that would otherwise delay a two-slot warp.
//
// Waits are bounded; a wait that gives up marks the CTA failed, after which it
// computes and writes nothing but still takes part in every cluster barrier,
// waits (bounded) for its own copies, sets the device error word and returns.
//
// A single-token call runs gdn_decode_t1.cu instead unless it is that small
// (the dispatch at the end of this file).

#include <mutex>

#include "gdn_device.cuh"
#include "gdn_launch.h"

namespace gdn {
namespace {

constexpr int kS = kHeadDim;
constexpr int kTile = kS * kS;              // floats per state tile
constexpr uint32_t kTileBytes = kTile * 4;  // 65536
constexpr int kCtaThreads = 256;            // one tile per CTA
constexpr int kWarps = kCtaThreads / 32;    // 8
constexpr int kChunk = 16;                  // tokens whose inputs are staged at once

// Per-token record in shared memory (floats): channel slot cc of the CTA maps
// to offset cc (q at [0,128), k at [128,256), v at [256,384)); the recurrence
// overwrites v with o.
constexpr int kRecQ = 0;
constexpr int kRecK = kS;
constexpr int kRecV = 2 * kS;          // v, then o
constexpr int kRecZ = 3 * kS;          // z of the CTA's head, by bulk copy
constexpr int kRecG = 4 * kS;          // beta, decay, 1 / decay, pad
constexpr int kRecFloats = kRecG + 8;  // 520 floats = 2080 bytes

constexpr size_t kOffRecs = kTileBytes;
constexpr size_t kOffNorm = kOffRecs + size_t(kChunk) * kRecFloats * 4;  // 98816: the layer's ssm_norm
constexpr size_t kOffBars = kOffNorm + kS * 4;                             // 99328
constexpr int kBarTile = 0, kBarZ = 1, kNumBars = 2;
constexpr size_t kSmemBytes = kOffBars + kNumBars * 8;  // 99344
constexpr int kCopyIssuer = 128;  // issues the z and ssm_norm copies (warp 4)
constexpr int kTileIssuer = 160;  // stores and refills the tile slot (warp 5)

static_assert(2 * (kSmemBytes + 1024) <= 233472, "two CTAs must fit in one SM's shared memory");
static_assert((kRecFloats * 4) % 16 == 0 && (kRecZ * 4) % 16 == 0, "records must stay 16-byte aligned");
static_assert(kChunk >= kDConv - 1, "a chunk's conv history must come from the previous chunk");
static_assert(kCtaThreads == 2 * kS, "slot A of a thread is a q/k channel, slot B (first 128 threads) a v channel");

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

// Conv + SiLU of one channel c (record slot cc) for the chunk's tokens
// [c0, c0 + tc). The 3-entry history before c0 (oldest first) is conv_state
// for the first chunk and the previous three qkv rows otherwise; the rolled
// window after the chunk goes to `hist`.
__device__ __forceinline__ void conv_slot(const Params& p, float* rec, int cc, int c, long long bl, int l, int c0,
                                          int tc, float (&hist)[3]) {
    const float4 w =
        __ldg(reinterpret_cast<const float4*>(p.conv_w + (static_cast<size_t>(l) * kConvChannels + c) * kDConv));
    const float* xq = p.qkv + (static_cast<size_t>(bl) * p.T + c0) * kConvChannels + c;
    float h0, h1, h2;
    if (c0 == 0) {
        const float* cs = p.conv_state + (static_cast<size_t>(bl) * kConvChannels + c) * (kDConv - 1);
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
    hist[0] = h0;
    hist[1] = h1;
    hist[2] = h2;
}

// conv_slot for a whole short window (at most kShortWindow tokens) on both slots
// of a thread at once: every load of slot A and slot B is issued before either
// is used, so the two slots cost one round trip to memory instead of two.
constexpr int kShortWindow = 8;

__device__ __forceinline__ void conv_pair_first(const Params& p, float* rec, int tid, int cA, int cB, long long bl,
                                                int l, int tc, float (&histA)[3], float (&histB)[3]) {
    const bool has_b = tid < kS;
    const float4 wA =
        __ldg(reinterpret_cast<const float4*>(p.conv_w + (static_cast<size_t>(l) * kConvChannels + cA) * kDConv));
    float4 wB = make_float4(0.f, 0.f, 0.f, 0.f);
    if (has_b)
        wB = __ldg(reinterpret_cast<const float4*>(p.conv_w + (static_cast<size_t>(l) * kConvChannels + cB) * kDConv));
    const float* csA = p.conv_state + (static_cast<size_t>(bl) * kConvChannels + cA) * (kDConv - 1);
    const float* csB = p.conv_state + (static_cast<size_t>(bl) * kConvChannels + cB) * (kDConv - 1);
    float a0 = csA[0], a1 = csA[1], a2 = csA[2];
    float b0 = 0.f, b1 = 0.f, b2 = 0.f;
    if (has_b) {
        b0 = csB[0];
        b1 = csB[1];
        b2 = csB[2];
    }
    const float* xA = p.qkv + static_cast<size_t>(bl) * p.T * kConvChannels + cA;
    const float* xB = p.qkv + static_cast<size_t>(bl) * p.T * kConvChannels + cB;
    float xa[kShortWindow], xb[kShortWindow];
#pragma unroll
    for (int t = 0; t < kShortWindow; ++t) {
        xa[t] = (t < tc) ? __ldg(xA + static_cast<size_t>(t) * kConvChannels) : 0.0f;
        xb[t] = (has_b && t < tc) ? __ldg(xB + static_cast<size_t>(t) * kConvChannels) : 0.0f;
    }
#pragma unroll
    for (int t = 0; t < kShortWindow; ++t) {
        if (t < tc) {
            rec[t * kRecFloats + tid] = siluf_(conv4(wA, a0, a1, a2, xa[t]));
            a0 = a1;
            a1 = a2;
            a2 = xa[t];
            if (has_b) {
                rec[t * kRecFloats + 2 * kS + tid] = siluf_(conv4(wB, b0, b1, b2, xb[t]));
                b0 = b1;
                b1 = b2;
                b2 = xb[t];
            }
        }
    }
    histA[0] = a0;
    histA[1] = a1;
    histA[2] = a2;
    histB[0] = b0;
    histB[1] = b1;
    histB[2] = b2;
}

__device__ __forceinline__ void store_history(const Params& p, long long bl, int c, const float (&hist)[3]) {
    float* cs = p.conv_state + (static_cast<size_t>(bl) * kConvChannels + c) * (kDConv - 1);
    cs[0] = hist[0];
    cs[1] = hist[1];
    cs[2] = hist[2];
}

// The gated delta rule on the thread's 16x4 block of the tile in registers
// (octet mapping), with two passes: a = S^T k, then the update and o = S_new^T q,
// 16-row partial sums reduced over the warp's 8 row blocks. The decay is
// deferred into a per-tile scale: the tile is S = P s, so S *= decay only
// scales P, and the update is s += k (d / P)^T (three FP32 operations per
// element instead of four). invP tracks 1/P from
// the per-token 1/decay, so no division sits between the two passes. When P
// falls below 2^-64 (decay underflow included) s is rescaled to S and P
// restarts at 1; the branch is uniform over the CTA, which holds one tile.
// Returns o = S_new^T q.
constexpr float kDeferMin = 5.421010862427522e-20f;  // 2^-64

__device__ __forceinline__ float4 delta_step_octet_deferred(float (&s)[64], float& P, float& invP, const float* qv,
                                                            const float* kv, const Octet& q, float4 v4, float beta,
                                                            float decay, float inv_decay) {
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int r = 0; r < 16; r += 4) {
        const float4 k4 = *reinterpret_cast<const float4*>(kv + q.row0 + r);
        const float kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = 4 * (r + e);
            a0 = fmaf(s[i + 0], kk[e], a0);
            a1 = fmaf(s[i + 1], kk[e], a1);
            a2 = fmaf(s[i + 2], kk[e], a2);
            a3 = fmaf(s[i + 3], kk[e], a3);
        }
    }
#pragma unroll
    for (int m = 4; m <= 16; m <<= 1) {
        a0 += __shfl_xor_sync(0xffffffffu, a0, m);
        a1 += __shfl_xor_sync(0xffffffffu, a1, m);
        a2 += __shfl_xor_sync(0xffffffffu, a2, m);
        a3 += __shfl_xor_sync(0xffffffffu, a3, m);
    }
    const float pn = P * decay;  // S_old * decay = pn * s
    float d0 = beta * (v4.x - pn * a0);
    float d1 = beta * (v4.y - pn * a1);
    float d2 = beta * (v4.z - pn * a2);
    float d3 = beta * (v4.w - pn * a3);
    if (pn < kDeferMin) {
#pragma unroll
        for (int i = 0; i < 64; ++i) s[i] *= pn;
        P = 1.0f;
        invP = 1.0f;
    } else {
        P = pn;
        invP *= inv_decay;
        d0 *= invP;
        d1 *= invP;
        d2 *= invP;
        d3 *= invP;
    }
    float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
    for (int r = 0; r < 16; r += 4) {
        const float4 k4 = *reinterpret_cast<const float4*>(kv + q.row0 + r);
        const float4 q4 = *reinterpret_cast<const float4*>(qv + q.row0 + r);
        const float kk[4] = {k4.x, k4.y, k4.z, k4.w};
        const float qq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = 4 * (r + e);
            s[i + 0] = fmaf(kk[e], d0, s[i + 0]);
            s[i + 1] = fmaf(kk[e], d1, s[i + 1]);
            s[i + 2] = fmaf(kk[e], d2, s[i + 2]);
            s[i + 3] = fmaf(kk[e], d3, s[i + 3]);
            o0 = fmaf(s[i + 0], qq[e], o0);
            o1 = fmaf(s[i + 1], qq[e], o1);
            o2 = fmaf(s[i + 2], qq[e], o2);
            o3 = fmaf(s[i + 3], qq[e], o3);
        }
    }
#pragma unroll
    for (int m = 4; m <= 16; m <<= 1) {
        o0 += __shfl_xor_sync(0xffffffffu, o0, m);
        o1 += __shfl_xor_sync(0xffffffffu, o1, m);
        o2 += __shfl_xor_sync(0xffffffffu, o2, m);
        o3 += __shfl_xor_sync(0xffffffffu, o3, m);
    }
    return make_float4(P * o0, P * o1, P * o2, P * o3);
}

// In the short-window instance the per-unit cluster barrier orders one thing:
// the old q/k history loads of ranks 1 and 2 before rank 0's stores of the new
// history (a CTA barrier publishes the records). Each thread's loads have
// returned by the time it arrives (their values feed the conv, which it issues
// before the arrive), so the arrive needs no release fence; a release would
// also stall on the thread's earlier y and history stores.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// kShort: the call's window has at most kShortWindow tokens, so every unit is one
// chunk and the tile never stays in registers from one chunk to the next. That
// leaves room to issue both conv slots' loads at once (conv_pair_first).
template <bool kShort>
__global__ void __launch_bounds__(kCtaThreads, 2) gdn_window_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(128) unsigned char smem[];
    float* tile = reinterpret_cast<float*>(smem);
    float* rec = reinterpret_cast<float*>(smem + kOffRecs);
    float* norm_w = reinterpret_cast<float*>(smem + kOffNorm);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int hh = static_cast<int>(cluster_rank());  // v head 3g + hh of the unit
    const long long cid = cluster_id_x();
    const long long n_clusters = cluster_count_x();
    const Octet oc = octet_of(tid);
    const uint32_t tile_s = smem_addr(tile);
    const uint32_t tile_bar = smem_addr(&bars[kBarTile]);
    const uint32_t z_bar = smem_addr(&bars[kBarZ]);
    const bool write_state = (p.flags & kNoStateWrite) == 0;
    const bool write_y = (p.flags & kNoY) == 0;
    const bool silu_gate = (p.flags & kSiluGate) != 0;

    if (tid == 0) {
        mbar_init(tile_bar, 1);
        mbar_init(z_bar, 1);
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    __syncthreads();  // the barriers are initialized before any thread uses them

    uint32_t tile_par = 0, z_par = 0;
    bool tile_pending = false, z_pending = false;  // copies issued and not yet waited for
    bool failed = false;  // a bounded wait gave up: stop computing, keep taking part in cluster barriers
    bool give_up = (p.flags & kTestGiveUp) != 0;
    if (tid == 0 && cid < p.n_units) {
        const long long bl = cid / kKHeads;
        const int g = static_cast<int>(cid - bl * kKHeads);
        mbar_arrive_expect_tx(tile_bar, kTileBytes);
        bulk_load_stream(tile_s, p.state + (static_cast<size_t>(bl) * kVHeads + g * kGroup + hh) * kTile, kTileBytes,
                         tile_bar);
    }
    tile_pending = cid < p.n_units;
    float s[64];
    float scale = 1.0f;  // the tile in registers is scale * s
    float inv_scale = 1.0f;

    for (long long u = cid; u < p.n_units; u += n_clusters) {
        const long long bl = u / kKHeads;
        const int g = static_cast<int>(u - bl * kKHeads);
        const int l = static_cast<int>(bl % p.L);
        const int b = static_cast<int>(bl / p.L);
        const int vh = g * kGroup + hh;
        const int cA = g * kS + (tid < kS ? tid : kKOffset - kS + tid);  // slot A: q or k channel of head g
        const int cB = kVOffset + vh * kS + tid;                         // slot B: v channel (tid < 128)
        int n = p.T;
        if (p.seq_len != nullptr) n = min(max(__ldg(p.seq_len + b), 0), p.T);

        if (kShort) {
            // The previous unit's tile is dead here; clearing the registers tells the compiler so.
#pragma unroll
            for (int i = 0; i < 64; ++i) s[i] = 0.0f;
        }

        float qk_hist[3] = {0.f, 0.f, 0.f};
        bool qk_store = false;  // short windows: rank 0 writes the q/k history at the unit's end

        int c0 = 0;
        do {
            const int tc = min(kChunk, n - c0);
            const bool last_chunk = (c0 + tc == n) && n > 0;
            const bool work = !failed && tc > 0;

            // ---- z of the chunk's tokens and the layer's ssm_norm by bulk copy, read in the epilogue
            if (work && write_y) {
                if (tid == kCopyIssuer) {
                    mbar_arrive_expect_tx(z_bar, (tc + 1) * kS * 4);
                    bulk_load(smem_addr(norm_w), p.ssm_norm + static_cast<size_t>(l) * kS, kS * 4, z_bar);
                    for (int t = 0; t < tc; ++t)
                        bulk_load(smem_addr(rec + t * kRecFloats + kRecZ),
                                  p.z + (static_cast<size_t>(bl) * p.T + c0 + t) * kValueDim + vh * kS, kS * 4, z_bar);
                }
                z_pending = true;
            }

            // ---- conv + SiLU of the CTA's 384 channels; the gates of its head
            float histA[3], histB[3];
            // Short windows: the gate inputs are loaded with the conv inputs, not after them.
            const int tg = tid - (kCtaThreads - kChunk);
            const bool gate_thread = work && tg >= 0 && tg < tc;
            float g_a = 0.f, g_b = 0.f, g_dt = 0.f, g_sa = 0.f;
            if (kShort && gate_thread) {
                const size_t row = (static_cast<size_t>(bl) * p.T + c0 + tg) * kVHeads + vh;
                g_a = __ldg(p.alpha + row);
                g_b = __ldg(p.beta + row);
                g_dt = __ldg(p.dt + static_cast<size_t>(l) * kVHeads + vh);
                g_sa = __ldg(p.ssm_a + static_cast<size_t>(l) * kVHeads + vh);
            }
            if (work) {
                if (kShort) {
                    conv_pair_first(p, rec, tid, cA, cB, bl, l, tc, histA, histB);
                } else {
                    conv_slot(p, rec, tid, cA, bl, l, c0, tc, histA);
                    if (tid < kS) conv_slot(p, rec, 2 * kS + tid, cB, bl, l, c0, tc, histB);
                }
                if (gate_thread) {
                    if (!kShort) {
                        const size_t row = (static_cast<size_t>(bl) * p.T + c0 + tg) * kVHeads + vh;
                        g_a = __ldg(p.alpha + row);
                        g_b = __ldg(p.beta + row);
                        g_dt = __ldg(p.dt + static_cast<size_t>(l) * kVHeads + vh);
                        g_sa = __ldg(p.ssm_a + static_cast<size_t>(l) * kVHeads + vh);
                    }
                    float bt, dc;
                    head_gates_in((p.flags & kGatesReady) != 0, g_a, g_b, g_dt, g_sa, bt, dc);
                    rec[tg * kRecFloats + kRecG + 0] = bt;
                    rec[tg * kRecFloats + kRecG + 1] = dc;
                    rec[tg * kRecFloats + kRecG + 2] = 1.0f / dc;
                }
            }
            if (kShort) {
                // This CTA has read the unit's old q/k history: it arrives now and waits for the
                // other two only at the unit's end, before rank 0 writes the new history.
                cluster_arrive_relaxed();
                __syncthreads();
                if (last_chunk && write_state && !failed && tid < kS) store_history(p, bl, cB, histB);
                qk_hist[0] = histA[0];
                qk_hist[1] = histA[1];
                qk_hist[2] = histA[2];
                qk_store = last_chunk && write_state && hh == 0;
            } else {
                // All three CTAs have read this unit's old q/k history (first chunk).
                // (Here the barrier also publishes the records, so it keeps its release.)
                if (c0 == 0) cluster_sync();
                else __syncthreads();
                // The new history: q/k by rank 0 only, v by each CTA.
                if (last_chunk && write_state && !failed) {
                    if (hh == 0) store_history(p, bl, cA, histA);
                    if (tid < kS) store_history(p, bl, cB, histB);
                }
            }

            // ---- L2 norm of q and k (one warp per token) and the q scale
            if (work)
                for (int t = warp; t < tc; t += kWarps)
                    normalize_qk(rec + t * kRecFloats + kRecQ, rec + t * kRecFloats + kRecK, lane);
            __syncthreads();

            if (c0 == 0 && !failed) {
                // This unit's tile moves from its slot into registers. (kTestGiveUp: the first
                // wait gives up at once, to exercise this path; the tile then stays pending and
                // is waited for before the CTA leaves.)
                const bool late = give_up || !mbar_wait_bounded(tile_bar, tile_par);
                give_up = false;
                if (__syncthreads_or(late ? 1 : 0)) {
                    failed = true;
                } else {
                    tile_par ^= 1u;
                    tile_pending = false;
                    if (n > 0) tile_load_octet(s, tile, oc);
                    scale = 1.0f;
                    inv_scale = 1.0f;
                }
            }

            // ---- the gated delta rule, token by token; o overwrites v
            if (work && !failed) {
                for (int t = 0; t < tc; ++t) {
                    float* r = rec + t * kRecFloats;
                    float* vo = r + kRecV + oc.col0;
                    const float4 v4 = *reinterpret_cast<const float4*>(vo);
                    const float4 o4 =
                        delta_step_octet_deferred(s, scale, inv_scale, r + kRecQ, r + kRecK, oc, v4, r[kRecG],
                                                  r[kRecG + 1], r[kRecG + 2]);
                    __syncwarp();
                    if (oc.rb == 0) *reinterpret_cast<float4*>(vo) = o4;
                }
            }

            // ---- after the last token the tile returns through its slot
            const bool store_tile = last_chunk && write_state && !failed;
            if (store_tile) {
#pragma unroll
                for (int i = 0; i < 64; ++i) s[i] *= scale;
                tile_save_octet(s, tile, oc);
                fence_proxy_async_smem();
            }
            __syncthreads();
            if (tid == kTileIssuer && store_tile) {
                bulk_store(p.state + (static_cast<size_t>(bl) * kVHeads + vh) * kTile, tile_s, kTileBytes);
                bulk_commit();
            }

            // ---- y = rms_norm(o) * ssm_norm * gate(z), one warp per token
            if (z_pending && !failed) {
                const bool late = !mbar_wait_bounded(z_bar, z_par);
                if (__syncthreads_or(late ? 1 : 0)) {
                    failed = true;
                } else {
                    z_par ^= 1u;
                    z_pending = false;
                    for (int t = warp; t < tc; t += kWarps) {
                        const float* r = rec + t * kRecFloats;
                        const float4 o4 = *reinterpret_cast<const float4*>(r + kRecV + lane * 4);
                        const float4 z4 = *reinterpret_cast<const float4*>(r + kRecZ + lane * 4);
                        const float4 w4 = *reinterpret_cast<const float4*>(norm_w + lane * 4);
                        __stcs(reinterpret_cast<float4*>(p.y + (static_cast<size_t>(bl) * p.T + c0 + t) * kValueDim +
                                                         vh * kS + lane * 4),
                               gated_rms_norm4(o4, z4, w4, silu_gate));
                    }
                }
            }
            c0 += kChunk;
            __syncthreads();  // the records are rewritten by the next chunk
        } while (c0 < n);
        if (kShort) {
            cluster_wait_acquire();
            if (qk_store && !failed) store_history(p, bl, cA, qk_hist);
        }

        // The slot takes the next unit's tile once the store has read it.
        const long long next = u + n_clusters;
        if (next < p.n_units && !failed) {
            if (tid == kTileIssuer) {
                const long long nbl = next / kKHeads;
                const int ng = static_cast<int>(next - nbl * kKHeads);
                bulk_wait_read();
                mbar_arrive_expect_tx(tile_bar, kTileBytes);
                bulk_load_stream(tile_s, p.state + (static_cast<size_t>(nbl) * kVHeads + ng * kGroup + hh) * kTile,
                                 kTileBytes, tile_bar);
            }
            tile_pending = true;
        }
    }

    if (tid == kTileIssuer) {
        // Copies still in flight land before the CTA leaves (bounded), and so do the stores.
        if (tile_pending) (void)mbar_wait_bounded(tile_bar, tile_par);
        if (z_pending) (void)mbar_wait_bounded(z_bar, z_par);
        bulk_wait_read();  // the last store has read the slot (its writes land on their own)
        if (failed) atomicOr(&g_device_error, kErrWaitTimeout);
    }
    // No cluster barrier before leaving: no CTA touches another's shared memory, and the three CTAs
    // of a cluster take the same cluster barriers in the loop, so none is left waiting on one that
    // has gone.
}

std::mutex g_mutex;
struct DeviceSetup {
    bool ready = false;
    int clusters = 0;
    int sms = 0;
};
DeviceSetup g_setup[64];

cudaLaunchConfig_t window_config(unsigned grid, cudaStream_t stream, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kCtaThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kGroup;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

cudaError_t device_setup(int* clusters, int* sms_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceSetup& d = g_setup[dev];
    if (!d.ready) {
        e = cudaFuncSetAttribute(gdn_window_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(gdn_window_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        cudaLaunchAttribute attr[1];
        cudaLaunchConfig_t cfg = window_config(static_cast<unsigned>(kGroup * sms), nullptr, attr);
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, gdn_window_kernel<false>, &cfg);
        if (e != cudaSuccess || n <= 0) {
            (void)cudaGetLastError();
            n = (2 * sms) / kGroup;  // two CTAs per SM
        }
        d.clusters = n;
        d.sms = sms;
        d.ready = true;
    }
    *clusters = d.clusters;
    *sms_out = d.sms;
    return cudaSuccess;
}

}  // namespace

// One token runs the single-token kernel (gdn_decode_t1.cu: one CTA per SM, a
// unit's three tiles on one SM, units taken in rounds of one per SM) or, for
// launches of up to 6 units per SM, gdn_window_kernel (3-CTA clusters, one CTA
// per tile, two CTAs per SM: rounds of one unit per cluster, C units a round, C
// the clusters the occupancy query lets run at once, 97 on 152 SMs) when its
// rounds cost no more (single_token_on_clusters). Measured per round at these
// sizes: about 10.7 us for the single-token kernel, 7.1 us for the clusters, so
// the clusters take a launch when 2 ceil(u / C) <= 3 ceil(u / S);
// 1 x 1 x 1 (16 units): 0.0054 against 0.0108 ms back to back; B x 1 x 1 with B =
// 4, 10, 24, 48: 0.0078 / 0.0137 / 0.0254 / 0.0617 against 0.0113 / 0.0206 /
// 0.0308 / 0.0664 ms; B = 7, 8 (one round against two) and 64 or more they lose.
// Windows of up to GDN_CHUNK_MAX_T tokens run the kernel with the tiles resident
// in shared memory (gdn_chunk.cu, chunks of 8 tokens), unless all their units fit
// one round of 3-CTA clusters (units <= C, window_on_clusters): such a
// launch runs gdn_window_kernel, one v head per CTA (1 x 1 x 8: 0.0090 against
// 0.0150 ms back to back; 4 x 1 x 8: 0.0133 against 0.0155; 4 x 1 x 16: 0.0212
// against 0.0275; at 8 x 1 x 8, two rounds, 0.0210 against 0.0163). Windows of
// GDN_TC_MIN_T tokens or more run the tensor-core chunk kernel
// (gdn_window_tc.cu); any others gdn_window_kernel. The defaults are the
// measured crossovers (16 sequences x 36 layers): the chunked kernel is the
// fastest up to 23 tokens, the tensor-core kernel from there on, so no larger
// window falls to gdn_window_kernel unless a build sets other thresholds (as
// timing comparisons do).
#ifndef GDN_CHUNK_MAX_T
#define GDN_CHUNK_MAX_T 23
#endif
#ifndef GDN_TC_MIN_T
#define GDN_TC_MIN_T 24
#endif

// Whether a single-token launch of `units` units runs on the 3-CTA clusters, `clusters` of which
// run at once (see above).
static bool single_token_on_clusters(long long units, int sms, int clusters) {
    if (units > 6LL * sms || clusters <= 0) return false;
    const long long c = clusters;
    return 2 * ((units + c - 1) / c) <= 3 * ((units + sms - 1) / sms);
}

// Whether a window of at most GDN_CHUNK_MAX_T tokens over `units` units runs on the 3-CTA clusters:
// all its units in one round of them.
static bool window_on_clusters(long long units, int clusters) { return units <= clusters; }

// The kernel a launch of `units` units and T tokens runs, by the rules above.
static DecodeKernel choose_kernel(long long units, int T, int sms, int clusters) {
    if (T == 1)
        return single_token_on_clusters(units, sms, clusters) ? DecodeKernel::kClusters : DecodeKernel::kSingleToken;
    if (T <= GDN_CHUNK_MAX_T)
        return window_on_clusters(units, clusters) ? DecodeKernel::kClusters : DecodeKernel::kChunked;
    if (T >= GDN_TC_MIN_T) return DecodeKernel::kTensorCore;
    return DecodeKernel::kClusters;
}

cudaError_t decode_kernel_for(int B, int L, int T, DecodeKernel* out) {
    int clusters = 0, sms = 0;
    const cudaError_t e = device_setup(&clusters, &sms);
    if (e != cudaSuccess) return e;
    *out = choose_kernel(static_cast<long long>(B) * L * kKHeads, T, sms, clusters);
    return cudaSuccess;
}

cudaError_t launch_decode_step(const StepArgs& a, cudaStream_t stream) {
    const long long units = static_cast<long long>(a.B) * a.L * kKHeads;
    int clusters = 0, sms = 0;
    cudaError_t e = cudaSuccess;
    if (a.T < GDN_TC_MIN_T) {
        e = device_setup(&clusters, &sms);
        if (e != cudaSuccess) return e;
    }
    switch (choose_kernel(units, a.T, sms, clusters)) {
        case DecodeKernel::kSingleToken: return launch_decode_t1(a, stream);
        case DecodeKernel::kChunked: return launch_decode_chunked(a, stream);
        case DecodeKernel::kTensorCore: return launch_decode_window_tc(a, stream);
        case DecodeKernel::kClusters: break;
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
    p.T = a.T;
    p.flags = a.flags;
    p.n_units = units;
    const long long n_cl = p.n_units < clusters ? p.n_units : clusters;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = window_config(static_cast<unsigned>(n_cl * kGroup), stream, attr);
    e = a.T <= kShortWindow ? cudaLaunchKernelEx(&cfg, gdn_window_kernel<true>, p)
                            : cudaLaunchKernelEx(&cfg, gdn_window_kernel<false>, p);
    if (e != cudaSuccess) return e;
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
    uint32_t v1 = 0, v2 = 0, v3 = 0, v4 = 0;
    e = read_t1_error(&v1);
    if (e != cudaSuccess) return e;
    e = read_chunk_error(&v3);
    if (e != cudaSuccess) return e;
    e = read_ab_error(&v4);
    if (e != cudaSuccess) return e;
    e = read_proj_error(&v2);
    if (e != cudaSuccess) return e;
    uint32_t v5 = 0;
    e = read_window_tc_error(&v5);
    *out = v | v1 | v2 | v3 | v4 | v5;
    return e;
}

}  // namespace gdn
