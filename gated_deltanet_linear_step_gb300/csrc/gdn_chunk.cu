// gdn_chunk.cu - the multi-token decode step (T > 1) with the three state
// tiles of a unit resident in shared memory, in chunks of up to 8 tokens.
//
// What it computes is the step listed in the header comment of the
// Winery-Strata page include/strata/core/layer.hpp and composed by gdn_layer
// (steps 3-7) on src/core/layer.cpp, applied to the tokens of a window in
// order (Verifier::record_window on src/core/verify.cpp): per token, conv +
// SiLU, L2 norm of q and k, q scale, gates, then on each v head's tile
//   S *= a_t;  kv_t = S^T k_t;  d_t = beta_t (v_t - kv_t);  S += k_t d_t^T;  o_t = S^T q_t
// and y_t = rms_norm(o_t) * ssm_norm * sigmoid(z_t).
//
// How. Within a chunk of n tokens the recurrence is column-separable and its
// state dependence is linear, so with S_0 the tile at the chunk's start,
//   A_t = a_0 ... a_t,   G(s, t) = a_{s+1} ... a_t  (G(t, t) = 1),
//   S_t = A_t S_0 + sum_{s<=t} G(s, t) k_s d_s^T
// and therefore, exactly,
//   kv_t = A_t (S_0^T k_t) + sum_{s<t}  G(s, t) (k_s . k_t) d_s
//   o_t  = A_t (S_0^T q_t) + sum_{s<=t} G(s, t) (k_s . q_t) d_s
//   S_n  = A_{n-1} S_0 + sum_s k_s (G(s, n-1) d_s)^T.
// A chunk reads each tile once to form S_0^T k_t and S_0^T q_t for all its
// tokens (pass A), solves the recurrence per column from those, the small Gram
// matrices k_s . k_t and k_s . q_t and the decay products (no division), and
// then reads and writes the tile once more with the rank-n update. The
// arithmetic is the definition's, regrouped; the tile crosses shared memory
// three times per chunk whatever n is, instead of three times per token, so
// the tiles can stay in shared memory like the single-token kernel's
// (gdn_decode_t1.cu), arriving by bulk copies.
//
// Layout and roles. One persistent CTA per SM, 384 threads, owns a contiguous
// range of units (layer l, k head g, sequence b), b fastest. Group h (threads
// 128 h .. 128 h + 127) owns the tile of v head 3 g + h. For tile work, lane
// 8 rb + qd of the group's warp w holds columns [32 w + 4 qd, +4) over rows
// i = 4 r + rb (r = 0..31), so consecutive lanes read consecutive rows and
// the shared-memory loads are free of bank conflicts; after pass A the lane
// solves column 32 w + 4 qd + rb. The same thread convolves that column's v
// channel, so v, o and y of the column never leave its registers; threads
// 0-255 also convolve one q or k channel each. Conv histories stay in
// registers from one chunk to the next.
//
// Overlap. Shared memory holds the three tiles, the chunk's raw qkv rows (with
// the heads' alpha, beta, dt and ssm_a) and the normalised q and k (separate
// from the raw rows), so the next chunk's inputs (or the next unit's first
// ones) are requested, by a v-only warp, after the chunk's preparation (the
// copy engine then has little of the tile refills left ahead of them), and
// arrive while the tiles are worked on. Pass A and
// the update run on the packed two-wide FMA. A unit's last update writes the new
// tile straight to HBM with streaming stores, so the slot is free once the
// group has read it: its leader then requests the next unit's tile, which an
// L2 prefetch issued with the next unit's inputs (about half a unit earlier,
// after this unit's preparation) has brought into L2; a prefetch a whole
// unit ahead measured slower than none, its lines evicted before use. The next
// unit's conv histories and taps are loaded into registers a unit ahead. No CTA
// barrier closes a chunk: a group that has finished its update starts the next
// chunk's conv while the others still store theirs (the gate tables alternate
// between two copies so that the next chunk's do not overwrite the ones still
// applied); the next chunk's first barrier gathers them.
// Waits are bounded; a wait that gives up raises a shared abort flag (the
// other threads' waits then return at once), and the CTA stops at the next
// chunk's first barrier after every copy it issued has landed (bounded), with
// the device error word set.

#include <mutex>

#include <cstring>

#include "gdn_launch.h"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int kS = kHeadDim;
constexpr int kTile = kS * kS;
constexpr uint32_t kTileBytes = kTile * 4;
constexpr int kUnitCh = 2 * kS + kGroup * kS;  // 640 conv channels per unit
constexpr int kC = 8;                           // tokens per chunk
constexpr int kXStride = 20;                    // floats per row of X: 16 used, rows 80 B apart (no bank conflicts)

// Per-chunk scalars (floats). The gate inputs of the unit's three heads come first (tensor-map
// boxes land 128-byte aligned): for alpha and beta of each token, and for the layer's dt and
// ssm_a, the 16-byte-aligned run of 8 floats that starts at float gate_base(g) of the 48-wide row.
constexpr int kMGin = 0;                       // [2 (alpha, beta)][kC][8], then [2 (dt, ssm_a)][8]
constexpr int kMPart = kMGin + 2 * kC * 8 + 2 * 8;  // [8][kC] sums of squares per warp (q: warps 0-3, k: 4-7)
constexpr int kMGram = kMPart + 8 * kC;        // [4][64] Gram partial sums of the four k warps
constexpr int kMCoef = kMGram + 4 * 64;        // [3][64] G(s,t) k_s.k_t at 8s+t (s<t), G(t,s) k_t.q_s at 8s+t (t<=s)
constexpr int kMBeta = kMCoef + kGroup * 64;   // [3][kC]
constexpr int kMCum = kMBeta + kGroup * kC;    // [3][kC] A_t
constexpr int kMGam = kMCum + kGroup * kC;     // [3][kC][kC] G(s, t) at [h][s][t]
constexpr int kMRms = kMGam + kGroup * kC * kC;  // [3][4][kC] sums of o^2 per (head, warp, token)
// The gate tables (beta, A_t, G) of alternate chunks: kMBeta .. kMGam, then a second copy at kMGate2
// with the same layout, so that the gate warp may fill the next chunk's while other groups still
// apply the current one (no CTA barrier between a chunk's update and the next chunk's conv).
constexpr int kMGateSpan = kMRms - kMBeta;
constexpr int kMGate2 = kMRms + kGroup * 4 * kC;
constexpr int kMFloats = kMGate2 + kMGateSpan;

constexpr size_t kOffTiles = 0;
constexpr size_t kOffRaw = size_t(kGroup) * kTileBytes;              // 196608: qkv rows [5 segments][kC][128]
constexpr size_t kOffX = kOffRaw + size_t(kC) * kUnitCh * 4;         // 217088: X [128][kXStride]
constexpr size_t kOffMisc = kOffX + size_t(kS) * kXStride * 4;       // 227328
constexpr size_t kOffBars = kOffMisc + size_t(kMFloats) * 4;         // 232256
constexpr int kBarTile = 0, kBarStage = 3, kNumBars = 4;
constexpr size_t kOffAbort = kOffBars + kNumBars * 8;                // a wait gave up (set once, read by waits)
constexpr size_t kSmemBytes = kOffAbort + 8;                         // 232296

static_assert(kSmemBytes <= 232448, "shared memory budget exceeds 227 KB");
static_assert(kOffBars % 8 == 0 && kOffRaw % 16 == 0 && kOffX % 16 == 0 && (kXStride * 4) % 16 == 0, "alignment");
static_assert(kOffMisc % 128 == 0 && kOffRaw % 128 == 0, "tensor-map boxes land 128-byte aligned");
static_assert(kThreads == 384 && kC == 8, "thread roles assume 384 threads and 8-token chunks");

constexpr int kGateWarp = 11;   // loads alpha and beta and builds the decay tables
constexpr int kIssueWarp = 8;   // requests the chunks' inputs (a v-only warp: idle while q and k are normalised)

__device__ unsigned int g_chunk_error = 0;

struct Params {
    CUtensorMap tm_qkv;    // qkv as [B L T rows][10240] fp32, box {128, 8}
    CUtensorMap tm_alpha;  // alpha as [B L T rows][48], box {8, 8}
    CUtensorMap tm_beta;   // beta, the same
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

__device__ __forceinline__ int valid_len(const Params& p, int b) {
    return p.seq_len == nullptr ? p.T : min(max(__ldg(p.seq_len + b), 0), p.T);
}

// Starts pulling `bytes` (a multiple of 16, 16-byte aligned) from global memory into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* ptr, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr), "r"(bytes) : "memory");
}

// First float of the 16-byte-aligned run that holds the gates of v heads 3g..3g+2 in a
// 48-wide row, and the bytes to copy (16 if the three fit in one 16-byte chunk, else 32;
// the run never passes the row's end).
__device__ __forceinline__ int gate_base(int g) { return (kGroup * g) & ~3; }
__device__ __forceinline__ uint32_t gate_bytes(int g) { return (kGroup * g - gate_base(g)) + kGroup <= 4 ? 16u : 32u; }

// The copies of one chunk's inputs (tokens c0 .. c0 + rows - 1 of unit x), 8 token rows per
// tensor-map box: the q and k segments and the three v heads of qkv (a box of 128 columns each,
// into the segment-major rows [5][8][128]), the heads' alpha and beta (a box of 8 columns each),
// and bulk copies of the layer's dt and ssm_a. Issued by the lanes of the calling warp; lane 0
// arms the mbarrier with the byte count first (zero rows: the phase holds dt and ssm_a). Rows
// past the chunk's tokens are read too (other tokens, or zeros past the tensor) and never used.
__device__ __forceinline__ void issue_chunk(const Params& p, const Unit& x, int c0, int rows, uint32_t raw,
                                            uint32_t gin, uint32_t bar, int lane) {
    const int gb = gate_base(x.g);
    const uint32_t gbytes = gate_bytes(x.g);
    if (lane == 0) mbar_arrive_expect_tx(bar, (rows > 0 ? 5u * kC * kS * 4 + 2u * kC * 8 * 4 : 0u) + 2 * gbytes);
    __syncwarp();
    const int row0 = static_cast<int>(x.bl * p.T + c0);
    const uint64_t pol = evict_first_policy();
    if (rows > 0 && lane < 5) {
        const int col = lane == 0 ? x.g * kS : (lane == 1 ? kKOffset + x.g * kS : kVOffset + (x.g * kGroup + lane - 2) * kS);
        tma_load_2d(raw + lane * kC * kS * 4, &p.tm_qkv, col, row0, bar, pol);
    }
    if (rows > 0 && (lane == 5 || lane == 6))
        tma_load_2d(gin + (lane - 5) * kC * 8 * 4, lane == 5 ? &p.tm_alpha : &p.tm_beta, gb, row0, bar, pol);
    if (lane == 7 || lane == 8) {
        const float* src = (lane == 8 ? p.ssm_a : p.dt) + static_cast<size_t>(x.l) * kVHeads + gb;
        bulk_load(gin + (2 * kC * 8 + (lane - 7) * 8) * 4, src, gbytes, bar);
    }
}

// Waits for phase `parity` of the mbarrier: true once it completes; false at once if another
// thread's wait gave up (the abort flag), or after kWaitLimitNs (the flag is then set).
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            return false;
        }
    }
}

// The three entries of a channel's conv history (plain loads: other units'
// entries of conv_state are written while the kernel runs).
__device__ __forceinline__ void load_hist(const Params& p, long long bl, int ch, float (&h)[3]) {
    const float* cs = p.conv_state + (static_cast<size_t>(bl) * kConvChannels + ch) * (kDConv - 1);
    h[0] = cs[0];
    h[1] = cs[1];
    h[2] = cs[2];
}

// The conv history after a chunk of tc tokens: its last three raw inputs, the older
// ones from the history before it (h on entry). Used alone for a channel whose conv
// output is not needed.
__device__ __forceinline__ void roll_history(const float* rows, int cc, int tc, float (&h)[3]) {
    const float i0 = h[0], i1 = h[1], i2 = h[2];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const int tau = tc - 3 + k;  // token of history entry k; < 0 reaches into the old history
        h[k] = tau >= 0 ? rows[(cc >> 7) * kC * kS + max(tau, 0) * kS + (cc & (kS - 1))]
                        : (tau == -3 ? i0 : (tau == -2 ? i1 : i2));
    }
}

// Conv + SiLU of one channel over the chunk's tc tokens (zero past tc), TP >= tc of
// them evaluated; h holds the history before the chunk and leaves holding the one
// after it. The shifts are unconditional and the result a select, so that the
// unrolled tokens interleave (a shift under t < tc became a branch per token);
// rows past tc are re-reads of row tc - 1, and the history after the chunk is read
// back from the rows.
template <int TP>
__device__ __forceinline__ void conv_tokens(float4 w, const float* rows, int cc, int tc, float (&h)[3],
                                            float (&out)[kC]) {
    float h0 = h[0], h1 = h[1], h2 = h[2];
#pragma unroll
    for (int t = 0; t < kC; ++t) {
        out[t] = 0.0f;
        if (t < TP) {
            const float xt = rows[(cc >> 7) * kC * kS + max(min(t, tc - 1), 0) * kS + (cc & (kS - 1))];
            const float xc = conv4(w, h0, h1, h2, xt);
            h0 = h1;
            h1 = h2;
            h2 = xt;
            const float y = siluf_(xc);
            out[t] = t < tc ? y : 0.0f;
        }
    }
    roll_history(rows, cc, tc, h);
}

// conv_tokens with the even token count at or above tc (the SiLUs past it are not
// evaluated: they bound the conv's time on the special-function units).
__device__ __forceinline__ void conv_chunk(float4 w, const float* rows, int cc, int tc, float (&h)[3],
                                           float (&out)[kC]) {
    if (tc <= 2)
        conv_tokens<2>(w, rows, cc, tc, h, out);
    else if (tc <= 4)
        conv_tokens<4>(w, rows, cc, tc, h, out);
    else if (tc <= 6)
        conv_tokens<6>(w, rows, cc, tc, h, out);
    else
        conv_tokens<8>(w, rows, cc, tc, h, out);
}

// Pass A on one tile: red[n] = sum_i S[i][col] X[i][n] for this lane's column
// col = col0 + rb, n < NT (k^ at n < TP, q^ at TP <= n < 2 TP; NT = TP when
// only S^T k is needed, a call that produces no y). The sums run in pairs of n
// on the packed two-wide FMA (each half rounds as fmaf does), half the issue
// slots of scalar FMAs.
template <int NT>
__device__ __forceinline__ void pass_a(const float* tile, const float* X, int col0, int rb, float (&red)[NT]) {
    static_assert(NT % 2 == 0, "X is read in pairs");
    constexpr int NP = NT / 2;
    const int lane = threadIdx.x & 31;
    float2 acc2[4][NP];
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int m = 0; m < NP; ++m) acc2[c][m] = make_float2(0.0f, 0.0f);
#pragma unroll 4
    for (int r = 0; r < 32; ++r) {
        const int i = 4 * r + rb;
        const float4 s = *reinterpret_cast<const float4*>(tile + i * kS + col0);
        float2 xv[NP];
#pragma unroll
        for (int m = 0; m < NP / 2; ++m) {
            const float4 v = *reinterpret_cast<const float4*>(X + i * kXStride + 4 * m);
            xv[2 * m] = make_float2(v.x, v.y);
            xv[2 * m + 1] = make_float2(v.z, v.w);
        }
        if (NP % 2 != 0)  // NT = 2 or 6 (only S^T k): the last pair
            xv[NP - 1] = *reinterpret_cast<const float2*>(X + i * kXStride + NT - 2);
        const float2 s0 = make_float2(s.x, s.x), s1 = make_float2(s.y, s.y);
        const float2 s2 = make_float2(s.z, s.z), s3 = make_float2(s.w, s.w);
#pragma unroll
        for (int m = 0; m < NP; ++m) {
            acc2[0][m] = __ffma2_rn(s0, xv[m], acc2[0][m]);
            acc2[1][m] = __ffma2_rn(s1, xv[m], acc2[1][m]);
            acc2[2][m] = __ffma2_rn(s2, xv[m], acc2[2][m]);
            acc2[3][m] = __ffma2_rn(s3, xv[m], acc2[3][m]);
        }
    }
    float acc[4][NT];
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int m = 0; m < NP; ++m) {
            acc[c][2 * m] = acc2[c][m].x;
            acc[c][2 * m + 1] = acc2[c][m].y;
        }
    // reduce-scatter over the four row sets (lane bits 3-4): the lane keeps column col0 + rb
    const bool b1 = (lane >> 4) & 1;
    const bool b0 = (lane >> 3) & 1;
    float half[2][NT];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const float send = b1 ? acc[c][n] : acc[c + 2][n];
            const float keep = b1 ? acc[c + 2][n] : acc[c][n];
            half[c][n] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const float send = b0 ? half[0][n] : half[1][n];
        const float keep = b0 ? half[1][n] : half[0][n];
        red[n] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
}

// The recurrence of this lane's column from the chunk's start: d_t and (WQ) o_t
// per token from pass A's u_t = red[t] and w_t = red[TP + t], v_t, the gates
// and the group's coefficients.
template <int TP, bool WQ>
__device__ __forceinline__ void solve_column(const float (&red)[WQ ? 2 * TP : TP], const float* M, int gofs2, int hh, int tc,
                                             const float (&v)[kC], float (&d)[kC], float (&o)[kC]) {
    const float* cum = M + kMCum + gofs2 + hh * kC;
    const float* bet = M + kMBeta + gofs2 + hh * kC;
    const float* coef = M + kMCoef + hh * 64;
#pragma unroll
    for (int t = 0; t < kC; ++t) {
        d[t] = 0.0f;
        o[t] = 0.0f;
        if (t < TP && t < tc) {
            float kv = cum[t] * red[t];
#pragma unroll
            for (int s = 0; s < t; ++s) kv = fmaf(coef[8 * s + t], d[s], kv);
            d[t] = bet[t] * (v[t] - kv);
            if (WQ) {
                float ov = cum[t] * red[(WQ ? TP : 0) + t];
#pragma unroll
                for (int s = 0; s <= t; ++s) ov = fmaf(coef[8 * t + s], d[s], ov);
                o[t] = ov;
            }
        }
    }
}

// Pass A, a barrier of the tile's group (its coefficients are then in place),
// and the column recurrence.
template <int TP, bool WQ>
__device__ __forceinline__ void pass_and_solve(const float* tile, const float* X, const float* M, int gofs2, int hh, int col0,
                                               int rb, int tc, const float (&v)[kC], float (&d)[kC],
                                               float (&o)[kC]) {
    float red[WQ ? 2 * TP : TP];
    pass_a<WQ ? 2 * TP : TP>(tile, X, col0, rb, red);
    named_barrier(1 + hh, kS);
    solve_column<TP, WQ>(red, M, gofs2, hh, tc, v, d, o);
}

// The rank-tc update of the thread's 32 x 4 block: S = A_{tc-1} S_0 + sum_s k_s e_s^T,
// e_s = G(s, tc - 1) d_s gathered from the four lanes that solved the block's columns.
// The new block goes back to the tile in shared memory (dst == kToSmem: more chunks follow),
// straight to the state in HBM with streaming stores (dst == kToHbm: the unit's last chunk),
// or nowhere (kDiscard: a window that writes no state).
constexpr int kToSmem = 0, kToHbm = 1, kDiscard = 2;

template <int TP>
__device__ __forceinline__ void update_tile(float* tile, const float* X, const float* M, int gofs2, int hh, int col0, int rb,
                                            int qd, int tc, const float (&d)[kC], int dst, float* gtile) {
    static_assert(TP % 2 == 0, "k is read in pairs");
    constexpr int NP = TP / 2;
    const float* gam = M + kMGam + gofs2 + hh * kC * kC;  // gam[s * kC + t] = G(s, t)
    float e[TP];
#pragma unroll
    for (int s = 0; s < TP; ++s) e[s] = (s < tc) ? gam[s * kC + (tc - 1)] * d[s] : 0.0f;
    // e of the block's four columns, as pairs of tokens (s, s + 1) for the packed FMA
    float2 E[4][NP];
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int m = 0; m < NP; ++m)
            E[c][m] = make_float2(__shfl_sync(0xffffffffu, e[2 * m], (c << 3) | qd),
                                  __shfl_sync(0xffffffffu, e[2 * m + 1], (c << 3) | qd));
    const float al = M[kMCum + gofs2 + hh * kC + tc - 1];
#pragma unroll 2
    for (int r = 0; r < 32; ++r) {
        const int i = 4 * r + rb;
        float4* sp = reinterpret_cast<float4*>(tile + i * kS + col0);
        float4 s = *sp;
        float2 kk[NP];
#pragma unroll
        for (int m = 0; m < NP; ++m) kk[m] = *reinterpret_cast<const float2*>(X + i * kXStride + 2 * m);
        // sum_s k_s e_s per column: token pairs on the packed FMA, the two halves added last
        float2 a0 = __fmul2_rn(kk[0], E[0][0]), a1 = __fmul2_rn(kk[0], E[1][0]);
        float2 a2 = __fmul2_rn(kk[0], E[2][0]), a3 = __fmul2_rn(kk[0], E[3][0]);
#pragma unroll
        for (int m = 1; m < NP; ++m) {
            a0 = __ffma2_rn(kk[m], E[0][m], a0);
            a1 = __ffma2_rn(kk[m], E[1][m], a1);
            a2 = __ffma2_rn(kk[m], E[2][m], a2);
            a3 = __ffma2_rn(kk[m], E[3][m], a3);
        }
        s.x = fmaf(s.x, al, a0.x + a0.y);
        s.y = fmaf(s.y, al, a1.x + a1.y);
        s.z = fmaf(s.z, al, a2.x + a2.y);
        s.w = fmaf(s.w, al, a3.x + a3.y);
        if (dst == kToSmem)
            *sp = s;
        else if (dst == kToHbm)
            __stcs(reinterpret_cast<float4*>(gtile + i * kS + col0), s);
    }
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

__global__ void __launch_bounds__(kThreads, 1) gdn_chunk_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(128) unsigned char smem[];
    float* tiles = reinterpret_cast<float*>(smem + kOffTiles);
    float* raw = reinterpret_cast<float*>(smem + kOffRaw);
    float* X = reinterpret_cast<float*>(smem + kOffX);
    float* M = reinterpret_cast<float*>(smem + kOffMisc);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int hh = tid >> 7;  // tile group: v head 3 g + hh
    const int gtid = tid & 127;
    const int gw = gtid >> 5;
    const int rb = lane >> 3;
    const int qd = lane & 7;
    const int col0 = 32 * gw + 4 * qd;
    const int scol = col0 + rb;  // the column this lane solves, and whose v channel it convolves
    const bool group_leader = gtid == 0;
    const bool write_state = (p.flags & kNoStateWrite) == 0;
    const bool write_y = (p.flags & kNoY) == 0;
    const bool silu_gate = (p.flags & kSiluGate) != 0;
    const bool gates_ready = (p.flags & kGatesReady) != 0;
    float* my_tile = tiles + hh * kTile;
    const uint32_t my_tile_s = smem_addr(my_tile);
    const uint32_t my_bar = smem_addr(&bars[kBarTile + hh]);
    const uint32_t raw_s = smem_addr(raw);
    const uint32_t gin_s = smem_addr(M + kMGin);
    const uint32_t stage_bar = smem_addr(&bars[kBarStage]);
    const int vslot = 2 * kS + hh * kS + scol;  // unit channel slot of this thread's v channel
    const bool has_qk = tid < 2 * kS;           // threads 0-127: q channel tid; 128-255: k channel tid - 128
    const int gh = lane / kC, gt = lane % kC;   // gate warp: lane -> (head, token)

    const long long u_begin = p.n_units * blockIdx.x / gridDim.x;
    const long long u_end = p.n_units * (blockIdx.x + 1) / gridDim.x;
    if (u_begin >= u_end) return;

    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) mbar_init(smem_addr(&bars[i]), 1);
        *abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    __syncthreads();

    Unit x = unit_of(p, u_begin);
    float hv[3], hq[3] = {0.f, 0.f, 0.f};  // conv histories of this thread's channels
    float4 wv, wq = make_float4(0.f, 0.f, 0.f, 0.f);  // conv taps of this thread's channels
    bool tile_pending = false;  // (leaders) a tile load was issued and has not been waited for
    bool stage_pending = false;  // (issue warp) a chunk's inputs were requested and not waited for
    {
        if (warp == kIssueWarp) {
            issue_chunk(p, x, 0, min(kC, valid_len(p, x.b)), raw_s, gin_s, stage_bar, lane);
            stage_pending = true;
        }
        if (group_leader && valid_len(p, x.b) > 0) {  // a unit with no valid token reads no tile
            mbar_arrive_expect_tx(my_bar, kTileBytes);
            bulk_load_stream(my_tile_s, tile_src(p, x, hh), kTileBytes, my_bar);
            tile_pending = true;
        }
        if (group_leader && u_begin + 1 < u_end) {
            const Unit x1 = next_unit(p, x);
            if (valid_len(p, x1.b) > 0) bulk_prefetch_l2(tile_src(p, x1, hh), kTileBytes);
        }
        const int vch = unit_channel(vslot, x.g);
        load_hist(p, x.bl, vch, hv);
        wv = __ldg(reinterpret_cast<const float4*>(p.conv_w + (static_cast<size_t>(x.l) * kConvChannels + vch) * kDConv));
        if (has_qk) {
            const int qkch = unit_channel(tid, x.g);
            load_hist(p, x.bl, qkch, hq);
            wq = __ldg(reinterpret_cast<const float4*>(
                p.conv_w + (static_cast<size_t>(x.l) * kConvChannels + qkch) * kDConv));
        }
    }

    uint32_t tile_par = 0, stage_par = 0;
    bool break_out = false;  // (uniform) a wait gave up: leave the unit loop
    bool failed = false;
    bool give_up = (p.flags & kTestGiveUp) != 0;  // the first tile wait gives up (tests this path)

    int n_carry = valid_len(p, x.b);  // this unit's token count, read a unit ahead
    uint32_t chunk_no = 0;            // chunks done: their parity picks the gate tables
    for (long long u = u_begin; u < u_end; ++u) {
        const bool has_next = u + 1 < u_end;
        const Unit xn = has_next ? next_unit(p, x) : x;
        const int n = n_carry;
        const int n_next = has_next ? valid_len(p, xn.b) : 0;
        const int vch = unit_channel(vslot, x.g);
        const int qkch = unit_channel(tid, x.g);
        const int gofs = kGroup * x.g - gate_base(x.g);  // head 3g's float in the copied gate runs

        for (int c0 = 0;; c0 += kC) {
            const int tc = max(0, min(kC, n - c0));
            const bool last_chunk = c0 + kC >= n;
            const int gofs2 = (chunk_no++ & 1) ? kMGate2 - kMBeta : 0;  // this chunk's gate tables
            const size_t row0 = static_cast<size_t>(x.bl) * p.T + c0;  // (b, l, token c0) row index

            // ---- early loads: z for y, the norm weight
            float zt[kC];
            float nw = 0.f;
#pragma unroll
            for (int t = 0; t < kC; ++t) {
                zt[t] = 0.f;
                if (write_y && t < tc)
                    zt[t] = __ldcs(p.z + (row0 + t) * kValueDim + (x.g * kGroup + hh) * kS + scol);
            }
            if (write_y && tc > 0) nw = __ldg(p.ssm_norm + static_cast<size_t>(x.l) * kS + scol);

            // ---- this chunk's inputs
            if (wait_or_abort(stage_bar, stage_par, abort_flag)) {
                stage_par ^= 1u;
                stage_pending = false;
            } else {
                failed = true;
            }

            // ---- conv + SiLU of this thread's channels; the gates and decay tables
            const int tcw = failed ? 0 : tc;
            float ov[kC], oq[kC];
#pragma unroll
            for (int t = 0; t < kC; ++t) oq[t] = 0.0f;  // (q threads without y convolve nothing)
            conv_chunk(wv, raw, vslot, tcw, hv, ov);
            if (has_qk && (write_y || tid >= kS)) conv_chunk(wq, raw, tid, tcw, hq, oq);
            else if (has_qk) roll_history(raw, tid, tcw, hq);  // no y: q is not needed, its history still rolls
            if (last_chunk) {
                if (write_state && n > 0 && !failed) {
                    float* cs = p.conv_state + (static_cast<size_t>(x.bl) * kConvChannels + vch) * 3;
                    cs[0] = hv[0];
                    cs[1] = hv[1];
                    cs[2] = hv[2];
                    if (has_qk) {
                        cs = p.conv_state + (static_cast<size_t>(x.bl) * kConvChannels + qkch) * 3;
                        cs[0] = hq[0];
                        cs[1] = hq[1];
                        cs[2] = hq[2];
                    }
                }
            }
            if (has_qk && (write_y || tid >= kS)) {
                // q (warps 0-3) and k (warps 4-7): per-warp sums of squares of the eight tokens, as a
                // reduce-scatter over the warp (lanes 4 t .. 4 t + 3 end with token t's sum)
                float sq[kC];
#pragma unroll
                for (int t = 0; t < kC; ++t) sq[t] = oq[t] * oq[t];
#pragma unroll
                for (int m = 16, c = kC; m >= 4; m >>= 1, c >>= 1) {
                    const bool up = (lane & m) != 0;
#pragma unroll
                    for (int j = 0; j < c / 2; ++j) {
                        const float send = up ? sq[j] : sq[j + c / 2];
                        const float keep = up ? sq[j + c / 2] : sq[j];
                        sq[j] = keep + __shfl_xor_sync(0xffffffffu, send, m);
                    }
                }
                sq[0] += __shfl_xor_sync(0xffffffffu, sq[0], 2);
                sq[0] += __shfl_xor_sync(0xffffffffu, sq[0], 1);
                if ((lane & 3) == 0) M[kMPart + warp * kC + (lane >> 2)] = sq[0];
            }
            if (warp == kGateWarp) {
                // lane (h, t): beta and decay, then A_t and G(s, t) from the head's decays by shuffles
                float bt = 0.f, a = 1.f;
                if (lane < kGroup * kC && gt < tc && !failed) {
                    const float* gin = M + kMGin;
                    head_gates_in(gates_ready, gin[gt * 8 + gofs + gh], gin[(kC + gt) * 8 + gofs + gh],
                                  gin[2 * kC * 8 + gofs + gh], gin[2 * kC * 8 + 8 + gofs + gh], bt, a);
                }
                float cum = 1.f;
                float gam[kC];
#pragma unroll
                for (int r = 0; r < kC; ++r) {
                    const float ar = __shfl_sync(0xffffffffu, a, (gh * kC + r) & 31);
                    if (r <= gt) cum *= ar;
                    gam[r] = ar;
                }
                if (lane < kGroup * kC && gt < tc) {
                    M[kMBeta + gofs2 + gh * kC + gt] = bt;
                    M[kMCum + gofs2 + gh * kC + gt] = cum;
                    float gp = 1.f;  // G(s, t) = a_{s+1} ... a_t, for s = t down to 0
#pragma unroll
                    for (int s = kC - 1; s >= 0; --s) {
                        if (s <= gt) {
                            M[kMGam + gofs2 + (gh * kC + s) * kC + gt] = gp;
                            gp *= gam[s];
                        }
                    }
                }
            }
            // (A) the chunk's inputs have been read; sums of squares and gates are in place. Every group has
            // finished the chunk before (no barrier follows a chunk): a wait of it that gave up stops the CTA.
            if (__syncthreads_or(failed ? 1 : 0)) break_out = true;
            if (break_out) break;

            // ---- q^ and k^ (normalised; q scaled) into X; the k warps keep k^ for the Gram matrices
            const int tp = (tc + 1) & ~1;
            if (has_qk && tc > 0 && (write_y || tid >= kS)) {
                const bool is_q = tid < kS;
                const int i = tid & (kS - 1);
                const int pw = is_q ? 0 : 4;
                float* xr = X + i * kXStride + (is_q ? tp : 0);
#pragma unroll
                for (int t = 0; t < kC; ++t) {
                    if (t < tc) {
                        const float ss = M[kMPart + (pw + 0) * kC + t] + M[kMPart + (pw + 1) * kC + t] +
                                         M[kMPart + (pw + 2) * kC + t] + M[kMPart + (pw + 3) * kC + t];
                        oq[t] *= rsqrtf(ss + kEps) * (is_q ? kQScale : 1.0f);
                    }
                }
#pragma unroll
                for (int t = 0; t < kC; t += 2)
                    if (t < tp) *reinterpret_cast<float2*>(xr + t) = make_float2(oq[t], oq[t + 1]);
            }
            __syncthreads();  // (B) X is in place

            // ---- Gram matrices: products at 8s+t (k_s.k_t for s<t, k_t.q_s for t<=s), s in [0, 4) by the q
            //      warps 0-3 (k^ from X) and s in [4, 8) by the k warps 4-7 (q^ from X), 32 per warp, each
            //      reduce-scattered over the warp (lane L keeps product 32 hf + L), partial sums per warp
            if (warp < 8 && tc > 0) {
                const int hf = warp >> 2;
                const int i = tid & (kS - 1);
                float kv[kC], qv[kC];
#pragma unroll
                for (int t = 0; t < kC; ++t) {
                    const float xk = (t < tc) ? X[i * kXStride + t] : 0.0f;
                    const float xq = (t < tc && write_y) ? X[i * kXStride + tp + t] : 0.0f;
                    kv[t] = hf ? oq[t] : xk;
                    qv[t] = hf ? xq : (write_y ? oq[t] : 0.0f);
                }
                float pr[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int sl = j >> 3, t = j & 7;  // s = 4 hf + sl
                    const float ks = hf ? kv[4 + sl] : kv[sl];
                    const float qs = hf ? qv[4 + sl] : qv[sl];
                    pr[j] = (4 * hf + sl < t) ? ks * kv[t] : kv[t] * qs;
                }
#pragma unroll
                for (int m = 16, c = 32; m >= 1; m >>= 1, c >>= 1) {
                    const bool up = (lane & m) != 0;
#pragma unroll
                    for (int j = 0; j < c / 2; ++j) {
                        const float send = up ? pr[j] : pr[j + c / 2];
                        const float keep = up ? pr[j + c / 2] : pr[j];
                        pr[j] = keep + __shfl_xor_sync(0xffffffffu, send, m);
                    }
                }
                M[kMGram + (warp & 3) * 64 + 32 * hf + lane] = pr[0];
            }
            __syncthreads();  // (C) the Gram partials are in place


            // ---- this group's coefficients; this unit's tile (first chunk)
            if (gtid < 64 && tc > 0) {
                const int s = gtid >> 3, t = gtid & 7;
                const float tot = M[kMGram + gtid] + M[kMGram + 64 + gtid] + M[kMGram + 128 + gtid] +
                                  M[kMGram + 192 + gtid];
                const bool in = s < tc && t < tc;
                const float gm = (s < t) ? M[kMGam + gofs2 + (hh * kC + s) * kC + t]
                                         : M[kMGam + gofs2 + (hh * kC + t) * kC + s];
                M[kMCoef + hh * 64 + gtid] = in ? gm * tot : 0.0f;
            }
            // ---- the staging area (free since barrier A) takes the next chunk's inputs, or the next unit's
            //      first ones: requested after the preparation, when the copy engine has little of the
            //      tile refills left ahead of them (requested at barrier A they took a warp 1.4 us to issue)
            if (warp == kIssueWarp && !failed) {
                if (!last_chunk) {
                    fence_proxy_async_smem();
                    issue_chunk(p, x, c0 + kC, min(kC, n - c0 - kC), raw_s, gin_s, stage_bar, lane);
                    stage_pending = true;
                } else if (has_next) {
                    fence_proxy_async_smem();
                    issue_chunk(p, xn, 0, min(kC, n_next), raw_s, gin_s, stage_bar, lane);
                    stage_pending = true;
                    if (n_next > 0 && lane >= 16 && lane < 16 + kGroup)  // the next unit's tiles into L2
                        bulk_prefetch_l2(tile_src(p, xn, lane - 16), kTileBytes);
                }
            }

            if (c0 == 0 && n > 0 && !failed) {
                if (!give_up && wait_or_abort(my_bar, tile_par, abort_flag)) {
                    tile_par ^= 1u;
                    tile_pending = false;
                } else {
                    failed = true;
                    *abort_flag = 1;  // the other groups' next waits return at once
                }
                give_up = false;
            }
            // ---- pass A, then (after the group's coefficients are in place) the column recurrence
            const bool warp_ok = !__any_sync(0xffffffffu, failed);
            float d[kC], o[kC];
#pragma unroll
            for (int t = 0; t < kC; ++t) d[t] = o[t] = 0.0f;
            if (tc > 0 && warp_ok) {
                if (write_y) {
                    if (tc <= 2)
                        pass_and_solve<2, true>(my_tile, X, M, gofs2, hh, col0, rb, tc, ov, d, o);
                    else if (tc <= 4)
                        pass_and_solve<4, true>(my_tile, X, M, gofs2, hh, col0, rb, tc, ov, d, o);
                    else if (tc <= 6)
                        pass_and_solve<6, true>(my_tile, X, M, gofs2, hh, col0, rb, tc, ov, d, o);
                    else
                        pass_and_solve<8, true>(my_tile, X, M, gofs2, hh, col0, rb, tc, ov, d, o);
                } else {  // no y: only S^T k is needed
                    if (tc <= 2)
                        pass_and_solve<2, false>(my_tile, X, M, gofs2, hh, col0, rb, tc, ov, d, o);
                    else if (tc <= 4)
                        pass_and_solve<4, false>(my_tile, X, M, gofs2, hh, col0, rb, tc, ov, d, o);
                    else if (tc <= 6)
                        pass_and_solve<6, false>(my_tile, X, M, gofs2, hh, col0, rb, tc, ov, d, o);
                    else
                        pass_and_solve<8, false>(my_tile, X, M, gofs2, hh, col0, rb, tc, ov, d, o);
                }
            } else {
                named_barrier(1 + hh, kS);
            }

            // ---- y = rms_norm(o) * ssm_norm * gate(z) from the registers: sums of o^2 per token over the
            //      group (reduce-scatter over the warp, then the four warps through shared memory)
            if (write_y && tc > 0) {
                float sq[kC];
#pragma unroll
                for (int t = 0; t < kC; ++t) sq[t] = o[t] * o[t];
#pragma unroll
                for (int m = 16, c = kC; m >= 4; m >>= 1, c >>= 1) {
                    const bool up = (lane & m) != 0;
#pragma unroll
                    for (int j = 0; j < c / 2; ++j) {
                        const float send = up ? sq[j] : sq[j + c / 2];
                        const float keep = up ? sq[j + c / 2] : sq[j];
                        sq[j] = keep + __shfl_xor_sync(0xffffffffu, send, m);
                    }
                }
                sq[0] += __shfl_xor_sync(0xffffffffu, sq[0], 2);
                sq[0] += __shfl_xor_sync(0xffffffffu, sq[0], 1);
                if ((lane & 3) == 0) M[kMRms + (hh * 4 + gw) * kC + (lane >> 2)] = sq[0];
            }
            named_barrier(1 + hh, kS);
            if (write_y && tc > 0 && warp_ok) {
#pragma unroll
                for (int t = 0; t < kC; ++t) {
                    if (t < tc) {
                        const float ss = M[kMRms + (hh * 4 + 0) * kC + t] + M[kMRms + (hh * 4 + 1) * kC + t] +
                                         M[kMRms + (hh * 4 + 2) * kC + t] + M[kMRms + (hh * 4 + 3) * kC + t];
                        const float rr = rsqrtf(ss * (1.0f / kS) + kEps);
                        const float gz = silu_gate ? siluf_(zt[t]) : sigmoidf_(zt[t]);
                        __stcs(p.y + (row0 + t) * kValueDim + (x.g * kGroup + hh) * kS + scol, o[t] * rr * nw * gz);
                    }
                }
            }

            // ---- (last chunk) the next unit's conv histories and taps, one unit ahead
            if (last_chunk && has_next) {
                const int nv = unit_channel(vslot, xn.g);
                load_hist(p, xn.bl, nv, hv);
                wv = __ldg(reinterpret_cast<const float4*>(
                    p.conv_w + (static_cast<size_t>(xn.l) * kConvChannels + nv) * kDConv));
                if (has_qk) {
                    const int nq = unit_channel(tid, xn.g);
                    load_hist(p, xn.bl, nq, hq);
                    wq = __ldg(reinterpret_cast<const float4*>(
                        p.conv_w + (static_cast<size_t>(xn.l) * kConvChannels + nq) * kDConv));
                }
            }

            // ---- the rank-tc update of the tile; after the unit's last chunk the slot takes the
            //      next unit's tile (from L2) as soon as the group has read it
            const int dst = !last_chunk ? kToSmem : (write_state ? kToHbm : kDiscard);
            if (tc > 0 && warp_ok && dst != kDiscard) {
                float* gtile = p.state + (static_cast<size_t>(x.bl) * kVHeads + x.g * kGroup + hh) * kTile;
                if (tc <= 2)
                    update_tile<2>(my_tile, X, M, gofs2, hh, col0, rb, qd, tc, d, dst, gtile);
                else if (tc <= 4)
                    update_tile<4>(my_tile, X, M, gofs2, hh, col0, rb, qd, tc, d, dst, gtile);
                else if (tc <= 6)
                    update_tile<6>(my_tile, X, M, gofs2, hh, col0, rb, qd, tc, d, dst, gtile);
                else
                    update_tile<8>(my_tile, X, M, gofs2, hh, col0, rb, qd, tc, d, dst, gtile);
            }
            fence_proxy_async_smem();  // the slot's reads come before the refill's writes
            const bool group_failed = named_barrier_or(1 + hh, kS, failed);
            if (group_leader && last_chunk && has_next && !group_failed) {
                if (n_next > 0) {
                    mbar_arrive_expect_tx(my_bar, kTileBytes);
                    bulk_load_stream(my_tile_s, tile_src(p, xn, hh), kTileBytes, my_bar);
                    tile_pending = true;
                }
            }

            if (last_chunk) break;
        }
        if (break_out) break;
        x = xn;
        n_carry = n_next;
    }
    if (__syncthreads_or(failed ? 1 : 0)) {
        // A wait gave up: record it, let every copy still in flight land (bounded), stop.
        if (tid == 0) atomicOr(&g_chunk_error, kErrWaitTimeout);
        if (warp == kIssueWarp && lane == 0 && stage_pending) (void)mbar_wait_bounded(stage_bar, stage_par);
        if (group_leader && tile_pending) (void)mbar_wait_bounded(my_bar, tile_par);
    }
}

std::mutex g_mutex;
int g_sms[64] = {0};

// A [rows][cols] fp32 tensor map with boxes of box_cols columns x kC rows, no swizzle.
cudaError_t encode_rows(CUtensorMap* tm, const float* base, int cols, cuuint64_t rows, int box_cols) {
    if (tensor_map_encoder() == nullptr) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), rows};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(kC)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = tensor_map_encoder()(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims,
                                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode_chunked(const StepArgs& a, cudaStream_t stream) {
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
            e = cudaFuncSetAttribute(gdn_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kSmemBytes));
            if (e != cudaSuccess) return e;
            g_sms[dev] = n;
        }
        sms = g_sms[dev];
    }
    Params p;
    memset(&p, 0, sizeof(p));
    const cuuint64_t rows = static_cast<cuuint64_t>(a.B) * a.L * a.T;
    e = encode_rows(&p.tm_qkv, a.qkv, kConvChannels, rows, kS);
    if (e != cudaSuccess) return e;
    e = encode_rows(&p.tm_alpha, a.alpha, kVHeads, rows, 8);
    if (e != cudaSuccess) return e;
    e = encode_rows(&p.tm_beta, a.beta, kVHeads, rows, 8);
    if (e != cudaSuccess) return e;
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
    gdn_chunk_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t read_chunk_error(uint32_t* out) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_chunk_error, sizeof(v));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_chunk_error, &zero, sizeof(zero));
    *out = v;
    return e;
}

}  // namespace gdn
