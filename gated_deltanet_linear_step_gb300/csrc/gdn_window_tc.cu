// gdn_window_tc.cu - the decode step over long windows (24 tokens or more in the
// library's dispatch; the kernel itself takes any length of 2 or more): chunks
// of up to 64 tokens whose contractions run on the tensor cores (tcgen05.mma
// from shared memory into tensor memory), with the conv, the gates, the
// inversion of the solve matrix and the epilogues on the CUDA cores.
//
// Regrouping (exact up to rounding; the method's step is the per-token gated
// delta rule of the Winery-Strata header include/strata/core/layer.hpp, its
// operation-order list, composed over the window by Verifier::record_window on
// src/core/verify.cpp). For one v head, a chunk of n tokens and the state S0
// before it (rows follow k, columns follow v), with decays a_t, betas b_t,
// A_t = a_0 ... a_t and G(s,t) = a_{s+1} ... a_t (G(t,t) = 1):
//
//   the state the token-t update sees, a_t S_{t-1}, is A_t S0 + sum_{s<t} G(s,t) k_s d_s^T, so
//   d_t = b_t (v_t - A_t S0^T k_t) - sum_{s<t} b_t G(s,t) (k_t . k_s) d_s   (a unit lower-triangular system)
//   o_t = A_t S0^T q_t + sum_{s<=t} G(s,t) (q_t . k_s) d_s
//   S_n = A_{n-1} S0 + sum_s k_s (G(s,n-1) d_s)^T
//
// Products on the tensor cores, each as three BF16 MMAs (hi*hi + hi*lo + lo*hi
// of the operands' round-to-nearest hi + lo halves, fp32 accumulation; the
// dropped lo*lo term and the halves' residue are at most about 2^-16 of each
// product, and far less on average):
//   Gram    [K;Q] [K;Q]^T         128x128x128 (k.k, q.k, and the squared norms on the diagonal)
//   state   S0^T [K;Q]^T          128x128x128 (S0^T k_t and S0^T q_t, one TMEM lane per v column)
//   solve   R^T X^T               128x64x64   (d = X r, X the inverse of the solve matrix)
//   output  D^T P^T               128x64x64   (P[t][s] = G(s,t) (q_t . k_s), s <= t)
//   update  E^T K, onto A_{n-1} S0^T held in tensor memory   128x128x64 (K read MN-major)
// q and k enter the MMAs un-normalised; their L2 norms come from the Gram
// diagonal and scale the products' results instead. The solve matrix is
// inverted by 16x16 blocks: diagonal blocks by forward substitution, the blocks
// below by block products, distance by distance.
//
// Work: one CTA (512 threads, 16 warps) per k head of a (sequence, layer), its
// three v heads one after another; one CTA per SM (about 226 KB of shared memory
// and all 512 tensor-memory columns), persistent over the units. For a single
// chunk, the q/k preparation and the Gram matrix serve all three v heads.
// Longer windows run the chunks of one v head in turn with its state in tensor
// memory (fp32) between chunks, redoing the q/k preparation per v head, so
// nothing intermediate is written to global memory (the window may be a verify
// pass that must not write the state).
//
// Rows reach shared memory by bulk copies (the q|k rows of a chunk, a v head's
// v rows, the state tile, the z rows), each signalled on its own mbarrier, so a
// phase waits for one round trip instead of one per token. The next unit's
// inputs are prefetched into L2 during the last v head.
//
// Waits are bounded; a wait that gives up marks the CTA failed, after which it
// writes nothing more, waits (bounded) for the MMAs and copies it issued, frees
// its tensor memory, sets the device error word and returns.

#include <cstring>
#include <mutex>

#include "gdn_launch.h"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int kS = kHeadDim;                // 128
constexpr int kTile = kS * kS;
constexpr int kC = 64;                      // tokens per chunk
constexpr int kTcThreads = 512;
constexpr int kLStride = kC + 4;            // fp32 row stride of the solve matrix (bank spread)

// Shared memory (bytes from a 1024-aligned base). Operand blocks are K-major,
// 128-byte swizzled: rows of 64 BF16, 8-row groups 1024 bytes apart.
constexpr uint32_t kBlk128 = 128 * 128;     // one 64-wide K block of 128 rows
constexpr uint32_t kOffKQ = 0;              // [K;Q] rows (k tokens 0-63, q tokens 64-127) x 128 dims: hi, lo
constexpr uint32_t kOffS = kOffKQ + 4 * kBlk128;    // S0^T: 128 columns x 128 dims: hi, lo
// Before S0^T the region stages the chunk's raw q rows ([64][128] fp32) and k rows
// (the same, 32 KB further), copied 8 tokens per tensor-map box. After the state MMA:
constexpr uint32_t kOffR = kOffS;                   //   R^T, 128 x 64: hi, lo
constexpr uint32_t kOffXop = kOffS + 3 * kBlk128;   //   X as the BF16 operand, 64 x 64: hi, lo
constexpr uint32_t kOffDT = kOffS;                  // then D^T (128 x 64: hi, lo)
constexpr uint32_t kOffET = kOffS + 2 * kBlk128;    //   and E^T (128 x 64: hi, lo)
constexpr uint32_t kOffO = kOffS;                   // then o, fp32 [64][128], for the y epilogue,
constexpr uint32_t kOffZ = kOffS + 2 * kBlk128;     //   beside the chunk's z rows (fp32 [64][128])
constexpr uint32_t kOffP = kOffS + 4 * kBlk128;     // P: 64 tokens x 64 tokens: hi, lo
constexpr uint32_t kOffL = kOffP + 2 * 64 * 128;    // the solve matrix, negated, fp32 [64][kLStride]
constexpr uint32_t kOffV = kOffL + kC * kLStride * 4;  // v rows of a v head: 3 history + 64 tokens, 512 B each
constexpr uint32_t kOffVHist = kOffV + (kC + 3) * kS * 4;  // its conv history at the window start, [128][3]
constexpr uint32_t kOffHist = kOffVHist + kS * 12;     // q/k conv history before the chunk, 3 KB
constexpr uint32_t kOffTab = kOffHist + 3072;
// gates of the unit's three v heads ([head][64] each), then the q/k norms, ssm_norm, scan totals
constexpr int kTabBeta = 0, kTabDec = 192, kTabA = 384, kTabGl = 576, kTabRk = 768, kTabRq = 832, kTabNorm = 896,
              kTabTot = 1024;
constexpr uint32_t kOffBar = kOffTab + 1032 * 4;
constexpr int kXStride = kC + 4;                    // fp32 row stride of the inverse X (bank spread)
constexpr uint32_t kOffX = kOffBar + 80;            // the inverse X, fp32 [64][kXStride], in a region of its own
constexpr uint32_t kSmemUsed = kOffX + kC * kXStride * 4;
constexpr uint32_t kTcSmem = kSmemUsed + 1024;     // room to align the base

static_assert(kOffS % 1024 == 0 && kOffP % 1024 == 0, "operand blocks are 1024-aligned");
static_assert(kC * kS * 4 <= 2 * kBlk128, "o and z fit where S0^T was");
static_assert(kOffXop + 2 * 64 * 128 <= kOffS + 4 * kBlk128, "R^T and X's operand fit where S0^T was");
static_assert(kOffX % 16 == 0, "X rows are read as float4");
static_assert(kC * 1024 <= 4 * kBlk128 && kTile * 4 <= 4 * kBlk128, "the staged rows and tile fit there too");
static_assert(kOffV % 16 == 0 && kOffVHist % 16 == 0 && kOffHist % 16 == 0, "bulk copy destinations");
static_assert(kTcSmem <= 232448, "one CTA per SM");

// Tensor memory columns (512 allocated).
constexpr uint32_t kTmGram = 0, kTmAb = 128, kTmS = 256, kTmPd = 384, kTmD = 448, kTmCols = 512;

__device__ unsigned int g_wtc_error = 0;

constexpr int kBoxRows = 8;  // token rows per tensor-map box (4 KB of one 128-wide head)

struct TcParams {
    CUtensorMap tm_qkv;  // qkv as [B L T rows][10240] fp32, box {128, 8}
    CUtensorMap tm_z;    // z as [B L T rows][6144], box {128, 8} (unused without y)
    CUtensorMap tm_y;    // y, the same geometry (unused without y)
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

__device__ __forceinline__ float u2f(uint32_t v) { return __uint_as_float(v); }

__device__ __forceinline__ void prefetch_l2(const void* ptr, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr), "r"(bytes) : "memory");
}

__device__ __forceinline__ float4 conv_taps(const TcParams& p, int l, int ch) {
    return __ldg(reinterpret_cast<const float4*>(p.conv_w + (static_cast<size_t>(l) * kConvChannels + ch) * kDConv));
}

// One token of the causal conv + SiLU of a channel: xc from the history (h0
// oldest) and x, then the history shifts. Returns SiLU(xc), or 0 for a token
// past the window (whose x and history are then don't-cares: the history after
// the window is read from the staged rows instead). The shift and the result
// are unconditional moves and a select, so that the unrolled tokens interleave;
// a predicated shift became a branch per token and serialised them.
__device__ __forceinline__ float conv_step(float4 w, float& h0, float& h1, float& h2, float x, bool valid) {
    const float xc = conv4(w, h0, h1, h2, x);
    h0 = h1;
    h1 = h2;
    h2 = x;
    const float s = siluf_(xc);
    return valid ? s : 0.0f;
}

// Raw q/k input of staged channel c (q at [0, 128), k at [128, 256)) at token c0 + t (t in
// [-3, tc)): token t >= 0 is row t of the staged q or k rows; before it, the staged history,
// which at the window start is conv_state ([channel][3]) and otherwise the three qkv rows
// before c0 (q and k halves of 1 KB rows).
__device__ __forceinline__ float qk_raw(const float* Rs, const float* Hs, int c0, int c, int t) {
    return t >= 0 ? Rs[(c >> 7) * kC * kS + t * kS + (c & (kS - 1))]
                  : (c0 == 0 ? Hs[3 * c + 3 + t] : Hs[(t + 3) * 2 * kS + c]);
}

// Raw v input of column col at token c0 + t (t in [-3, tc)) from the staged rows: token t is
// row t + 3; before the window start (c0 == 0, t < 0) it is the staged conv history.
__device__ __forceinline__ float v_raw(const float* Vs, const float* VHs, int c0, int col, int t) {
    return (c0 == 0 && t < 0) ? VHs[3 * col + 3 + t] : Vs[(t + 3) * kS + col];
}

// Valid tokens of sequence b: T, or its seq_len clamped to [0, T].
__device__ __forceinline__ int unit_len(const TcParams& p, int b) {
    return p.seq_len != nullptr ? min(max(__ldg(p.seq_len + b), 0), p.T) : p.T;
}

// Three BF16 products of two hi/lo operand pairs into d (accumulate = 0 only for the first).
__device__ __forceinline__ void mma3(uint32_t d, uint64_t ah, uint64_t al, uint64_t bh, uint64_t bl, uint32_t idesc,
                                     bool first) {
    mma_bf16(d, ah, bh, idesc, first ? 0u : 1u);
    mma_bf16(d, ah, bl, idesc, 1u);
    mma_bf16(d, al, bh, idesc, 1u);
}

__global__ void __launch_bounds__(kTcThreads, 1) gdn_window_tc_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    unsigned char* sm = smem_raw + (base - raw_addr);
    float* tab = reinterpret_cast<float*>(sm + kOffTab);
    float* beta_s = tab + kTabBeta;
    float* dec_s = tab + kTabDec;
    float* A_s = tab + kTabA;
    float* gl_s = tab + kTabGl;
    float* rk_s = tab + kTabRk;
    float* rq_s = tab + kTabRq;
    float* nw_s = tab + kTabNorm;
    float* tot_s = tab + kTabTot;
    float* L_s = reinterpret_cast<float*>(sm + kOffL);
    float* O_s = reinterpret_cast<float*>(sm + kOffO);
    float* Xs = reinterpret_cast<float*>(sm + kOffX);  // fp32 [64][kXStride]; blocks above the diagonal hold temporaries
    const float* Rs = reinterpret_cast<const float*>(sm + kOffS);       // staged q|k rows
    const float* Hs = reinterpret_cast<const float*>(sm + kOffHist);    // staged q/k history
    const float* Vs = reinterpret_cast<const float*>(sm + kOffV);       // staged v rows (token t at row t + 3)
    const float* VHs = reinterpret_cast<const float*>(sm + kOffVHist);  // staged v history (window start)
    const float* Zs = reinterpret_cast<const float*>(sm + kOffZ);       // staged z rows
    const uint32_t bar_gram = base + kOffBar, bar_ab = bar_gram + 8, bar_out = bar_gram + 16, bar_d = bar_gram + 24;
    const uint32_t bar_qk = bar_gram + 32, bar_s = bar_gram + 40, bar_z = bar_gram + 48, bar_v = bar_gram + 56;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffBar + 64);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3;                    // the tensor-memory lanes this warp may access
    const int wg = warp >> 2;                        // which of the four warps of its lane quarter
    const int col = 32 * quarter + lane;             // v column (tensor-memory lane) of this thread
    const uint32_t lane_off = static_cast<uint32_t>(32 * quarter) << 16;
    const bool write_state = (p.flags & kNoStateWrite) == 0;
    const bool write_y = (p.flags & kNoY) == 0;
    const bool silu_gate = (p.flags & kSiluGate) != 0;
    const bool gates_ready = (p.flags & kGatesReady) != 0;

    const uint64_t pol_stream = evict_first_policy();  // rows read once per call
    if (tid == 0) {
        prefetch_tensormap(&p.tm_qkv);
        if (write_y) {
            prefetch_tensormap(&p.tm_z);
            prefetch_tensormap(&p.tm_y);
        }
        mbar_init(bar_gram, 1);
        mbar_init(bar_ab, 1);
        mbar_init(bar_out, 1);
        mbar_init(bar_d, 1);
        mbar_init(bar_qk, 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_z, 1);
        mbar_init(bar_v, 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(smem_addr(tmem_slot), kTmCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    uint32_t ph_gram = 0, ph_ab = 0, ph_out = 0, ph_d = 0, ph_qk = 0, ph_s = 0, ph_z = 0, ph_v = 0;
    uint32_t pend_bar = 0, pend_par = 0;  // (thread 0) the last MMA commit, drained if a wait gives up
    bool pend_mma = false;                // (thread 0) an MMA commit not yet waited for
    bool pend_qk = false, pend_s = false, pend_z = false, pend_v = false;  // copies issued, not yet waited for
    bool qk_ahead = false, s_ahead = false;  // the next unit's first q|k rows / state tile already requested
    bool failed = false;
    bool give_up = (p.flags & kTestGiveUp) != 0;

    // Every thread waits for an MMA group or a copy; false (uniform over the CTA) if any wait gave up.
    auto wait_all = [&](uint32_t bar, uint32_t& ph) -> bool {
        const bool late = give_up || !mbar_wait_bounded(bar, ph);
        give_up = false;
        if (__syncthreads_or(late ? 1 : 0)) return false;
        if (bar == pend_bar) pend_mma = false;
        ph ^= 1u;
        tc_fence_after();
        return true;
    };
    // The chunk's q and k rows (8 tokens per tensor-map box) into the region S0^T later holds, the
    // history before them beside it; by warp 1, after its bulk stores have read that region.
    auto issue_qk = [&](long long xbl, int xg, int xc0, int xtc) {
        if (warp == 1) {
            bulk_wait_read();
            const int nb = (xtc + kBoxRows - 1) / kBoxRows;
            if (lane == 0) mbar_arrive_expect_tx(bar_qk, static_cast<uint32_t>(nb) * 2u * kBoxRows * kS * 4 + 3072u);
            __syncwarp();
            const int row0 = static_cast<int>(xbl * p.T + xc0);
            if (lane < 2 * nb) {
                const int j = lane >> 1, kseg = lane & 1;
                tma_load_2d(base + kOffS + kseg * kC * kS * 4 + j * kBoxRows * kS * 4, &p.tm_qkv,
                            (kseg ? kKOffset : 0) + xg * kS, row0 + kBoxRows * j, bar_qk, pol_stream);
            }
            if (lane == 0) {
                if (xc0 == 0) {
                    const float* cs = p.conv_state + static_cast<size_t>(xbl) * kConvChannels * (kDConv - 1);
                    bulk_load(base + kOffHist, cs + xg * kS * 3, kS * 12, bar_qk);
                    bulk_load(base + kOffHist + 1536, cs + (kKOffset + xg * kS) * 3, kS * 12, bar_qk);
                } else {
                    for (int r = 0; r < 3; ++r) {
                        const float* row = p.qkv + (static_cast<size_t>(xbl) * p.T + xc0 - 3 + r) * kConvChannels;
                        bulk_load(base + kOffHist + r * 1024, row + xg * kS, kS * 4, bar_qk);
                        bulk_load(base + kOffHist + r * 1024 + 512, row + kKOffset + xg * kS, kS * 4, bar_qk);
                    }
                }
            }
        }
        pend_qk = true;
    };
    // A state tile in two 32 KB halves: dims [0, 64) into the P and solve-matrix regions, [64, 128)
    // into the v staging, by thread 32 (no bulk copy reads those regions: the new state leaves from
    // tensor memory by plain stores, the y rows from the region S0^T used).
    auto issue_s = [&](long long xbl, int xvh) {
        if (tid == 32) {
            const float* src = p.state + (static_cast<size_t>(xbl) * kVHeads + xvh) * kTile;
            mbar_arrive_expect_tx(bar_s, kTile * 4);
            bulk_load(base + kOffP, src, kTile * 2, bar_s);
            bulk_load(base + kOffV, src + kTile / 2, kTile * 2, bar_s);
        }
        pend_s = true;
    };

    const uint32_t idesc128 = mma_idesc(128), idesc64 = mma_idesc(64);
    const uint32_t kq_hi = base + kOffKQ, kq_lo = kq_hi + 2 * kBlk128;
    const uint32_t s_hi = base + kOffS, s_lo = s_hi + 2 * kBlk128;
    const uint32_t dt_hi = base + kOffDT, dt_lo = dt_hi + kBlk128;
    const uint32_t et_hi = base + kOffET, et_lo = et_hi + kBlk128;
    const uint32_t p_hi = base + kOffP, p_lo = p_hi + 64 * 128;
    const uint32_t r_hi = base + kOffR, r_lo = r_hi + kBlk128;
    const uint32_t x_hi = base + kOffXop, x_lo = x_hi + 64 * 128;

    for (long long u = blockIdx.x; u < p.n_units && !failed; u += gridDim.x) {
        const long long bl = u / kKHeads;
        const int g = static_cast<int>(u - bl * kKHeads);
        const int l = static_cast<int>(bl % p.L);
        const int b = static_cast<int>(bl / p.L);
        const int n = unit_len(p, b);
        if (n == 0) continue;
        const bool multi = n > kC;
        if (write_y && tid < kS) nw_s[tid] = __ldg(p.ssm_norm + static_cast<size_t>(l) * kS + tid);
        // the first chunk's q|k rows and the first v head's state tile, unless requested a unit ahead
        if (!qk_ahead) issue_qk(bl, g, 0, min(n, kC));
        if (!s_ahead) issue_s(bl, g * kGroup);
        qk_ahead = s_ahead = false;

        // q (threads 0-127) or k (128-255) channel of this thread for the conv history
        const bool prep_k = tid >= kS;
        const int prep_col = tid & (kS - 1);
        const int prep_ch = (prep_k ? kKOffset : 0) + g * kS + prep_col;
        float qk_hist[3] = {0.f, 0.f, 0.f};
        float gpre = 1.0f, gsuf = 1.0f;  // (warps 0-5) decay scans of the q/k preparation

        for (int h = 0; h < kGroup && !failed; ++h) {
            const int vh = g * kGroup + h;
            const float* beta_h = beta_s + 64 * h;  // this v head's gates
            const float* dec_h = dec_s + 64 * h;
            const float* A_h = A_s + 64 * h;
            const float* gl_h = gl_s + 64 * h;
            float v_hist[3] = {0.f, 0.f, 0.f};  // (warps 8-11) the v history after the window
            const int v_ch = kVOffset + vh * kS + col;  // (warps 8-15) the v channel of this thread's column

            for (int c0 = 0; c0 < n && !failed; c0 += kC) {
                const int tc = min(kC, n - c0);
                const bool last = c0 + tc == n;
                const int nh = c0 > 0 ? 3 : 0;  // history rows staged with the chunk's rows

                if (h == 0 || multi) {
                    // ---- q/k: the chunk's rows (requested earlier for a unit's first chunk), then conv,
                    //      SiLU and split into the [K;Q] rows; the gates of the three v heads meanwhile
                    if (c0 > 0 || h > 0) issue_qk(bl, g, c0, tc);
                    // gates of the three v heads for the chunk's tokens (warps 0-5: head warp / 2, tokens
                    // [32 (warp & 1), +32)), with in-warp prefix and suffix products of the decays
                    if (warp < 2 * kGroup) {
                        const int hh = warp >> 1, t = 32 * (warp & 1) + lane;
                        float bt = 0.0f, dc = 1.0f;
                        if (t < tc) {
                            const size_t row = (static_cast<size_t>(bl) * p.T + c0 + t) * kVHeads + g * kGroup + hh;
                            const size_t lh = static_cast<size_t>(l) * kVHeads + g * kGroup + hh;
                            head_gates_in(gates_ready, __ldg(p.alpha + row), __ldg(p.beta + row), __ldg(p.dt + lh),
                                          __ldg(p.ssm_a + lh), bt, dc);
                        }
                        gpre = dc;
                        gsuf = dc;
#pragma unroll
                        for (int d = 1; d < 32; d <<= 1) {
                            const float up = __shfl_up_sync(0xffffffffu, gpre, d);
                            const float dn = __shfl_down_sync(0xffffffffu, gsuf, d);
                            if (lane >= d) gpre *= up;
                            if (lane + d < 32) gsuf *= dn;
                        }
                        if (lane == 31) tot_s[warp] = gpre;
                        beta_s[64 * hh + t] = bt;
                        dec_s[64 * hh + t] = dc;
                    }
                    if (!wait_all(bar_qk, ph_qk)) {
                        failed = true;
                        break;
                    }
                    pend_qk = false;
                    {
                        // two adjacent channels per thread (q: tid & 64 == 0, k otherwise), tokens
                        // [16 (tid >> 7), +16); groups past tc are zero rows
                        const int pc = (tid & 64 ? kS : 0) + 2 * (tid & 63);  // staged channel of the pair
                        const int t0 = 16 * (tid >> 7);
                        const int ch = (pc < kS ? 0 : kKOffset - kS) + g * kS + pc;
                        const float4 w0 = conv_taps(p, l, ch), w1 = conv_taps(p, l, ch + 1);
                        float a0 = qk_raw(Rs, Hs, c0, pc, t0 - 3), a1 = qk_raw(Rs, Hs, c0, pc, t0 - 2),
                              a2 = qk_raw(Rs, Hs, c0, pc, t0 - 1);
                        float b0 = qk_raw(Rs, Hs, c0, pc + 1, t0 - 3), b1 = qk_raw(Rs, Hs, c0, pc + 1, t0 - 2),
                              b2 = qk_raw(Rs, Hs, c0, pc + 1, t0 - 1);
                        const int cpos = pc & (kS - 1);
                        const int kb = cpos >> 6, cc = (cpos & 63) >> 3, e = cpos & 7;
#pragma unroll 1
                        for (int j = 0; j < 2; ++j) {
                            const bool any = t0 + 8 * j < tc;
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const int t = t0 + 8 * j + i;
                                float x0 = 0.0f, x1 = 0.0f;
                                if (any) {
                                    const float2 xv = *reinterpret_cast<const float2*>(
                                        Rs + (pc >> 7) * kC * kS + min(t, tc - 1) * kS + (pc & (kS - 1)));
                                    x0 = conv_step(w0, a0, a1, a2, xv.x, t < tc);
                                    x1 = conv_step(w1, b0, b1, b2, xv.y, t < tc);
                                }
                                uint32_t hi, lo;
                                split_pair_rn(x0, x1, hi, lo);
                                const uint32_t off =
                                    kOffKQ + kb * kBlk128 + sw128_offset(pc < kS ? kC + t : t, cc) + 2 * e;
                                *reinterpret_cast<uint32_t*>(sm + off) = hi;
                                *reinterpret_cast<uint32_t*>(sm + off + 2 * kBlk128) = lo;
                            }
                        }
                        if (last && tid < 2 * kS) {
                            // the history after the window: the last three raw inputs of channel tid
                            const int sc = prep_k ? kS + prep_col : prep_col;
                            qk_hist[0] = qk_raw(Rs, Hs, c0, sc, tc - 3);
                            qk_hist[1] = qk_raw(Rs, Hs, c0, sc, tc - 2);
                            qk_hist[2] = qk_raw(Rs, Hs, c0, sc, tc - 1);
                        }
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    __syncthreads();
                    if (tid == 0) {
                        tc_fence_after();
#pragma unroll
                        for (int kb2 = 0; kb2 < 2; ++kb2)
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const uint64_t ah = sw128_desc(kq_hi + kb2 * kBlk128) + 2 * kk;
                                const uint64_t al = sw128_desc(kq_lo + kb2 * kBlk128) + 2 * kk;
                                mma3(tmem + kTmGram, ah, al, ah, al, idesc128, (kb2 | kk) == 0);
                            }
                        mma_commit(bar_gram);
                        pend_bar = bar_gram;
                        pend_mma = true;
                        pend_par = ph_gram;
                    }
                    if (!wait_all(bar_gram, ph_gram)) {
                        failed = true;
                        break;
                    }
                    // ---- A_t (prefix) and G(t, n-1) (exclusive suffix) across the two token halves
                    if (warp < 2 * kGroup) {
                        const int hh = warp >> 1, half = warp & 1, t = 32 * half + lane;
                        float sx = __shfl_down_sync(0xffffffffu, gsuf, 1);
                        if (lane == 31) sx = 1.0f;
                        A_s[64 * hh + t] = half ? tot_s[2 * hh] * gpre : gpre;
                        gl_s[64 * hh + t] = t < tc ? (half ? sx : sx * tot_s[2 * hh + 1]) : 0.0f;
                    }
                    // ---- L2 norms from the Gram diagonal (row r: k token r, or q token r - 64)
                    if (warp < 4) {
                        uint32_t v[32];
                        tmem_ld32(tmem + kTmGram + lane_off + 32 * warp, v);
                        float dg = 0.0f;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (lane == j) dg = u2f(v[j]);
                        const float r = rsqrtf(dg + kEps);
                        if (warp < 2)
                            rk_s[32 * warp + lane] = r;
                        else
                            rq_s[32 * (warp - 2) + lane] = r * kQScale;
                    }
                }

                // ---- the state: S^T (hi, lo) for the MMA, A_{n-1} S into the update accumulator. At
                //      a window start the tile arrived by bulk copy in two halves (P and solve-matrix
                //      regions, v staging); later chunks continue from tensor memory.
                {
                    // thread (column col, dims [32 wg, 32 wg + 32))
                    float sv[32];
                    if (c0 == 0) {
                        if (!wait_all(bar_s, ph_s)) {
                            failed = true;
                            break;
                        }
                        pend_s = false;
                        const float* half_s = reinterpret_cast<const float*>(sm + (wg >= 2 ? kOffV : kOffP));
#pragma unroll
                        for (int k = 0; k < 32; ++k) sv[k] = half_s[(32 * (wg & 1) + k) * kS + col];
                    } else {
                        uint32_t v[32];
                        tmem_ld32(tmem + kTmS + lane_off + 32 * wg, v);
#pragma unroll
                        for (int k = 0; k < 32; ++k) sv[k] = u2f(v[k]);
                    }
                    // the y stores of the previous v head have read the region S0^T goes to; the tile's
                    // halves are read before the v rows and the solve matrix replace them
                    if (warp == 1) bulk_wait_read();
                    __syncthreads();
                    // ---- v rows of this v head (and, at the window start, its conv history) by bulk copy
                    if (warp == 2) {
                        const int nb = (tc + kBoxRows - 1) / kBoxRows;
                        if (lane == 0)
                            mbar_arrive_expect_tx(bar_v, static_cast<uint32_t>(nb) * kBoxRows * kS * 4 +
                                                             static_cast<uint32_t>(nh) * kS * 4 + (c0 == 0 ? kS * 12 : 0));
                        __syncwarp();
                        const int row0 = static_cast<int>(bl * p.T + c0);
                        if (lane < nb)
                            tma_load_2d(base + kOffV + (3 + kBoxRows * lane) * kS * 4, &p.tm_qkv, kVOffset + vh * kS,
                                        row0 + kBoxRows * lane, bar_v, pol_stream);
                        if (lane >= 29 && nh > 0) {  // the three rows before the chunk, one copy each
                            const int t = lane - 32;
                            bulk_load(base + kOffV + (t + 3) * kS * 4,
                                      p.qkv + (static_cast<size_t>(bl) * p.T + c0 + t) * kConvChannels + kVOffset +
                                          vh * kS,
                                      kS * 4, bar_v);
                        }
                        if (lane == 0 && c0 == 0)
                            bulk_load(base + kOffVHist,
                                      p.conv_state + (static_cast<size_t>(bl) * kConvChannels + kVOffset + vh * kS) * 3,
                                      kS * 12, bar_v);
                    }
                    pend_v = true;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t off = kOffS + (wg >> 1) * kBlk128 + sw128_offset(col, 4 * (wg & 1) + j);
                        store_split8(sm + off, sm + off + 2 * kBlk128, sv + 8 * j);
                    }
                    const float al = A_h[tc - 1];
                    uint32_t v[32];
#pragma unroll
                    for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(al * sv[k]);
                    tmem_st32(tmem + kTmS + lane_off + 32 * wg, v);
                    tmem_st_wait();
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncthreads();
                if (tid == 0) {
                    tc_fence_after();
#pragma unroll
                    for (int kb2 = 0; kb2 < 2; ++kb2)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma3(tmem + kTmAb, sw128_desc(s_hi + kb2 * kBlk128) + 2 * kk,
                                 sw128_desc(s_lo + kb2 * kBlk128) + 2 * kk, sw128_desc(kq_hi + kb2 * kBlk128) + 2 * kk,
                                 sw128_desc(kq_lo + kb2 * kBlk128) + 2 * kk, idesc128, (kb2 | kk) == 0);
                    mma_commit(bar_ab);
                    pend_bar = bar_ab;
                    pend_mma = true;
                    pend_par = ph_ab;
                }
                // ---- the next unit's inputs into L2, a third per v head: its state tile h and a third
                //      of its first chunk's rows (warps 12-13)
                if (c0 == 0) {
                    const long long nu = u + gridDim.x;
                    if (nu < p.n_units) {
                        const long long nbl = nu / kKHeads;
                        const int ng = static_cast<int>(nu - nbl * kKHeads);
                        const int nn = min(unit_len(p, static_cast<int>(nbl / p.L)), kC);
                        if (tid == 384 && nn > 0 && h > 0)
                            prefetch_l2(p.state + (static_cast<size_t>(nbl) * kVHeads + ng * kGroup + h) * kTile,
                                        kTile * 4);
                        const int t = tid - 416 + h * 22;  // tokens [22 h, 22 h + 22)
                        if (tid >= 416 && tid < 416 + 22 && t < nn) {
                            const float* row = p.qkv + (static_cast<size_t>(nbl) * p.T + t) * kConvChannels;
                            prefetch_l2(row + kVOffset + ng * kGroup * kS, kGroup * kS * 4);
                            if (write_y)
                                prefetch_l2(p.z + (static_cast<size_t>(nbl) * p.T + t) * kValueDim + ng * kGroup * kS,
                                            kGroup * kS * 4);
                        }
                    }
                }

                // ---- two warp groups at once. Warps 0-7: the solve matrix and P from the Gram rows, then
                //      the inverse X of I - Lneg by 16x16 blocks and X as the operand of d = X r.
                //      Warps 8-15: the v conv and r_t = b_t (v_t - A_t S0^T k_t) into R^T.
                bool group_late = false;
                if (warp < 8) {
                    {
                        // row t of the Gram (k rows: warps 0-1 and 4-5, q rows: warps 2-3 and 6-7), columns
                        // s in [32 (1 - wg), +32), s from the top so that G(s, t) = a_{s+1} ... a_t builds
                        // up as one running product
                        const int t = (32 * quarter + lane) & (kC - 1);
                        const int half = 1 - wg;
                        const bool is_q = quarter >= 2;
                        const bool valid_t = t < tc;
                        const float rt = valid_t ? (is_q ? rq_s[t] : -beta_h[t] * rk_s[t]) : 0.0f;
                        float pr = 1.0f;
                        if (half == 0)
                            for (int r = 33; r <= t; ++r) pr *= dec_h[r];  // a_33 ... a_t, the factors above s = 31
                        uint32_t raw[32];
                        tmem_ld32(tmem + kTmGram + lane_off + 32 * half, raw);
                        float val[32];
#pragma unroll
                        for (int i = 31; i >= 0; --i) {
                            const int s = 32 * half + i;
                            if (s < t) pr *= dec_h[s + 1];
                            // L: s < t (negated, with beta_t); P: s <= t
                            const float gs = s < t ? pr : ((is_q && s == t) ? 1.0f : 0.0f);
                            val[i] = rt * gs * u2f(raw[i]) * rk_s[s];
                        }
                        if (!is_q) {
                            float* Lr = L_s + t * kLStride + 32 * half;
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                *reinterpret_cast<float4*>(Lr + 4 * j) =
                                    make_float4(val[4 * j], val[4 * j + 1], val[4 * j + 2], val[4 * j + 3]);
                        } else {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const uint32_t off = kOffP + sw128_offset(t, 4 * half + j);
                                store_split8(sm + off, sm + off + 64 * 128, val + 8 * j);
                            }
                        }
                    }
                    // X and its BF16 operand are written where S0^T lo was: the state MMA must have read it
                    // (its commit is waited for here; the rhs warps wait for it too, before R^T)
                    const bool ab_late = !mbar_wait_bounded(bar_ab, ph_ab);
                    group_late = named_barrier_or(1, 256, ab_late);
                    if (!group_late) {
                        tc_fence_after();
                        if (tid < kC) {
                            // diagonal blocks: thread (i, j) solves column j of block i by forward substitution
                            const int i = tid >> 4, j = tid & 15;
                            float x[16];
#pragma unroll
                            for (int r = 0; r < 16; ++r) {
                                const float* Lr = L_s + (16 * i + r) * kLStride + 16 * i;
                                float acc = 0.0f;
#pragma unroll
                                for (int m = 0; m < r; ++m) acc = fmaf(Lr[m], x[m], acc);
                                x[r] = r > j ? acc : (r == j ? 1.0f : 0.0f);
                            }
#pragma unroll
                            for (int r = 0; r < 16; ++r) Xs[(16 * i + r) * kXStride + 16 * i + j] = x[r];
                        }
                        named_barrier(1, 256);
                        {
                            // below the diagonal, by distance: X_ij = X_ii sum_{k=j}^{i-1} Lneg_ik X_kj. Thread
                            // (block j = tid / 64, row r, columns [c4, c4 + 4)) of the distance's blocks: rows of
                            // Lneg and X_ii and four columns of X read as float4, each value used four times
                            const int jb = tid >> 6, r = (tid >> 2) & 15, c4 = 4 * (tid & 3);
#pragma unroll
                            for (int dist = 1; dist < 4; ++dist) {
                                if (jb + dist < 4) {
                                    const int j = jb, i = j + dist;
                                    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                                    for (int k = 0; k < 3; ++k) {
                                        if (j + k < i) {
                                            const int kb = j + k;
                                            const float* Lr = L_s + (16 * i + r) * kLStride + 16 * kb;
#pragma unroll
                                            for (int m = 0; m < 16; m += 4) {
                                                const float4 l4 = *reinterpret_cast<const float4*>(Lr + m);
                                                const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                                                for (int e = 0; e < 4; ++e) {
                                                    const float4 x4 = *reinterpret_cast<const float4*>(
                                                        Xs + (16 * kb + m + e) * kXStride + 16 * j + c4);
                                                    y.x = fmaf(lv[e], x4.x, y.x);
                                                    y.y = fmaf(lv[e], x4.y, y.y);
                                                    y.z = fmaf(lv[e], x4.z, y.z);
                                                    y.w = fmaf(lv[e], x4.w, y.w);
                                                }
                                            }
                                        }
                                    }
                                    // temporary in block (j, i)
                                    *reinterpret_cast<float4*>(Xs + (16 * j + r) * kXStride + 16 * i + c4) = y;
                                }
                                named_barrier(1, 256);
                                if (jb + dist < 4) {
                                    const int j = jb, i = j + dist;
                                    const float* Dr = Xs + (16 * i + r) * kXStride + 16 * i;
                                    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                                    for (int m = 0; m < 16; m += 4) {
                                        const float4 d4 = *reinterpret_cast<const float4*>(Dr + m);
                                        const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
                                        for (int e = 0; e < 4; ++e) {
                                            const float4 t4 = *reinterpret_cast<const float4*>(
                                                Xs + (16 * j + m + e) * kXStride + 16 * i + c4);
                                            x.x = fmaf(dv[e], t4.x, x.x);
                                            x.y = fmaf(dv[e], t4.y, x.y);
                                            x.z = fmaf(dv[e], t4.z, x.z);
                                            x.w = fmaf(dv[e], t4.w, x.w);
                                        }
                                    }
                                    *reinterpret_cast<float4*>(Xs + (16 * i + r) * kXStride + 16 * j + c4) = x;
                                }
                                named_barrier(1, 256);
                            }
                        }
                        {
                            // X as the BF16 operand [t][s]; blocks above the diagonal are zero
                            const int t = tid >> 2;
#pragma unroll
                            for (int h2 = 0; h2 < 2; ++h2) {
                                const int j = 2 * (tid & 3) + h2;  // columns [8 j, 8 j + 8)
                                float xv[8];
                                const bool upper = (j >> 1) > (t >> 4);
#pragma unroll
                                for (int e = 0; e < 8; ++e) xv[e] = upper ? 0.0f : Xs[t * kXStride + 8 * j + e];
                                const uint32_t off = kOffXop + sw128_offset(t, j);
                                store_split8(sm + off, sm + off + 64 * 128, xv);
                            }
                        }
                    }
                } else {
                    // warps 8-15: the state MMA and the v rows, then r; warps 8-11 tokens [0, 32), 12-15 [32, 64)
                    bool late = !mbar_wait_bounded(bar_ab, ph_ab);
                    late = late || !mbar_wait_bounded(bar_v, ph_v);
                    group_late = named_barrier_or(2, 256, late);
                    if (!group_late) {
                        tc_fence_after();
                        if (last && wg == 2) {
                            // the v history after the window: the last three raw inputs (the staging is reused later)
                            v_hist[0] = v_raw(Vs, VHs, c0, col, tc - 3);
                            v_hist[1] = v_raw(Vs, VHs, c0, col, tc - 2);
                            v_hist[2] = v_raw(Vs, VHs, c0, col, tc - 1);
                        }
                        const int j0 = wg == 2 ? 0 : kC / 16;
                        float h0 = v_raw(Vs, VHs, c0, col, 8 * j0 - 3), h1 = v_raw(Vs, VHs, c0, col, 8 * j0 - 2),
                              h2 = v_raw(Vs, VHs, c0, col, 8 * j0 - 1);
                        const float4 w = conv_taps(p, l, v_ch);
#pragma unroll 1
                        for (int j = j0; j < j0 + kC / 16; ++j) {
                            float r8[8];
                            if (8 * j < tc) {
                                uint32_t a8[8];
                                tmem_ld8(tmem + kTmAb + lane_off + 8 * j, a8);
#pragma unroll
                                for (int i = 0; i < 8; ++i) {
                                    const int t = 8 * j + i;
                                    const float v =
                                        conv_step(w, h0, h1, h2, Vs[(min(t, tc - 1) + 3) * kS + col], t < tc);
                                    r8[i] = beta_h[t] * (v - A_h[t] * rk_s[t] * u2f(a8[i]));
                                }
                            } else {
#pragma unroll
                                for (int i = 0; i < 8; ++i) r8[i] = 0.0f;
                            }
                            const uint32_t off = kOffR + sw128_offset(col, j);
                            store_split8(sm + off, sm + off + kBlk128, r8);
                        }
                    }
                }
                fence_proxy_async_smem();
                if (__syncthreads_or(group_late ? 1 : 0)) {
                    failed = true;
                    break;
                }
                // every thread follows the two waits' phases (warps 8-15 took them)
                if (pend_bar == bar_ab) pend_mma = false;
                ph_ab ^= 1u;
                ph_v ^= 1u;
                pend_v = false;
                if (tid == 0) {
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma3(tmem + kTmD, sw128_desc(r_hi) + 2 * kk, sw128_desc(r_lo) + 2 * kk, sw128_desc(x_hi) + 2 * kk,
                             sw128_desc(x_lo) + 2 * kk, idesc64, kk == 0);
                    mma_commit(bar_d);
                    pend_bar = bar_d;
                    pend_mma = true;
                    pend_par = ph_d;
                }
                if (!wait_all(bar_d, ph_d)) {
                    failed = true;
                    break;
                }
                {
                    // ---- d, then the D^T and E^T rows (E: d scaled by G(s, n-1) and the k norm); the four
                    //      warps of a lane quarter take 16 tokens each
                    const int j0 = 2 * wg;
#pragma unroll 1
                    for (int j = j0; j < j0 + 2; ++j) {
                        uint32_t d8[8];
                        tmem_ld8(tmem + kTmD + lane_off + 8 * j, d8);
                        float d[8], ev[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            d[e] = u2f(d8[e]);
                            ev[e] = gl_h[8 * j + e] * rk_s[8 * j + e] * d[e];
                        }
                        const uint32_t off = sw128_offset(col, j);
                        store_split8(sm + kOffDT + off, sm + kOffDT + kBlk128 + off, d);
                        store_split8(sm + kOffET + off, sm + kOffET + kBlk128 + off, ev);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncthreads();
                if (tid == 0) {
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma3(tmem + kTmPd, sw128_desc(dt_hi) + 2 * kk, sw128_desc(dt_lo) + 2 * kk,
                             sw128_desc(p_hi) + 2 * kk, sw128_desc(p_lo) + 2 * kk, idesc64, kk == 0);
                    // K as B, MN-major: tokens 16 kk .. 16 kk + 15 are two 8-row groups of the [K;Q] blocks
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma3(tmem + kTmS, sw128_desc(et_hi) + 2 * kk, sw128_desc(et_lo) + 2 * kk,
                             sw128_mn_desc(kq_hi + kk * 2048, kBlk128), sw128_mn_desc(kq_lo + kk * 2048, kBlk128),
                             idesc128 | kIdescBMnMajor, false);
                    mma_commit(bar_out);
                    pend_bar = bar_out;
                    pend_mma = true;
                    pend_par = ph_out;
                }
                if (!wait_all(bar_out, ph_out)) {
                    failed = true;
                    break;
                }
                // ---- the P, solve-matrix and v regions are free: after a v head's last chunk they take the
                //      next state tile now, which then lands during the y epilogue (the next unit's first
                //      tile after the unit's last v head; its q|k rows follow once y has left)
                if (last) {
                    if (h + 1 < kGroup) {
                        issue_s(bl, vh + 1);
                    } else {
                        const long long nu = u + gridDim.x;
                        if (nu < p.n_units) {
                            const long long nbl = nu / kKHeads;
                            const int ng = static_cast<int>(nu - nbl * kKHeads);
                            if (unit_len(p, static_cast<int>(nbl / p.L)) > 0) {
                                issue_s(nbl, ng * kGroup);
                                s_ahead = true;
                            }
                        }
                    }
                }
                if (write_y) {
                    // z rows of the chunk into the half of the region that E^T held
                    if (warp == 1) {
                        const int nb = (tc + kBoxRows - 1) / kBoxRows;
                        if (lane == 0) mbar_arrive_expect_tx(bar_z, static_cast<uint32_t>(nb) * kBoxRows * kS * 4);
                        __syncwarp();
                        if (lane < nb)
                            tma_load_2d(base + kOffZ + lane * kBoxRows * kS * 4, &p.tm_z, vh * kS,
                                        static_cast<int>(bl * p.T + c0) + kBoxRows * lane, bar_z, pol_stream);
                    }
                    pend_z = true;
                    // ---- o_t = A_t S0^T q_t + (D^T P^T)_t into o[t][col] for the y epilogue (16 tokens per
                    //      warp of a lane quarter)
                    const int j0 = 2 * wg;
#pragma unroll 1
                    for (int j = j0; j < j0 + 2 && 8 * j < tc; ++j) {
                        uint32_t bq[8], pd[8];
                        tmem_ld8(tmem + kTmAb + lane_off + kC + 8 * j, bq);
                        tmem_ld8(tmem + kTmPd + lane_off + 8 * j, pd);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int t = 8 * j + i;
                            O_s[t * kS + col] = A_h[t] * rq_s[t] * u2f(bq[i]) + u2f(pd[i]);
                        }
                    }
                }
                if (last && write_state) {
                    // ---- the new state tile from tensor memory straight to HBM: thread (column col, dims
                    //      [32 wg, +32)); a warp's 32 lanes store 32 adjacent columns of a dim's row
                    uint32_t v[32];
                    tmem_ld32(tmem + kTmS + lane_off + 32 * wg, v);
                    float* dst = p.state + (static_cast<size_t>(bl) * kVHeads + vh) * kTile + 32 * wg * kS + col;
#pragma unroll
                    for (int i = 0; i < 32; ++i) __stcs(dst + i * kS, u2f(v[i]));
                }
                tc_fence_before();
                __syncthreads();
                if (write_y) {
                    if (!wait_all(bar_z, ph_z)) {
                        failed = true;
                        break;
                    }
                    pend_z = false;
                    const float4 w4 = *reinterpret_cast<const float4*>(nw_s + lane * 4);
                    for (int t = warp; t < tc; t += kTcThreads / 32) {
                        float4* o4 = reinterpret_cast<float4*>(O_s + t * kS + lane * 4);
                        const float4 z4 = *reinterpret_cast<const float4*>(Zs + t * kS + lane * 4);
                        *o4 = gated_rms_norm4(*o4, z4, w4, silu_gate);
                    }
                    fence_proxy_async_smem();
                    __syncthreads();
                    if (warp == 1) {
                        // full 8-token boxes by tensor map, the rows of a last partial box one by one
                        const int full = tc / kBoxRows;
                        if (lane < full)
                            tma_store_2d(&p.tm_y, vh * kS, static_cast<int>(bl * p.T + c0) + kBoxRows * lane,
                                         base + kOffO + lane * kBoxRows * kS * 4);
                        const int t = kBoxRows * full + lane;
                        if (lane < tc - kBoxRows * full)
                            bulk_store(p.y + (static_cast<size_t>(bl) * p.T + c0 + t) * kValueDim + vh * kS,
                                       base + kOffO + t * kS * 4, kS * 4);
                        bulk_commit();
                    }
                }
                // ---- after the unit's last v head, the next unit's first q|k rows, into the region the y
                //      rows leave once their stores have read it
                if (last && h + 1 == kGroup) {
                    const long long nu = u + gridDim.x;
                    if (nu < p.n_units) {
                        const long long nbl = nu / kKHeads;
                        const int ng = static_cast<int>(nu - nbl * kKHeads);
                        const int nn = unit_len(p, static_cast<int>(nbl / p.L));
                        if (nn > 0) {
                            issue_qk(nbl, ng, 0, min(nn, kC));
                            qk_ahead = true;
                        }
                    }
                }
                __syncthreads();  // o, z and the operand blocks are rewritten next
            }
            if (!failed && write_state && warp >= 8 && wg == 2) {
                float* cs = p.conv_state + (static_cast<size_t>(bl) * kConvChannels + v_ch) * (kDConv - 1);
                cs[0] = v_hist[0];
                cs[1] = v_hist[1];
                cs[2] = v_hist[2];
            }
        }
        // The q/k history last: every v head's pass has read the old one.
        if (!failed && write_state && tid < 2 * kS) {
            float* cs = p.conv_state + (static_cast<size_t>(bl) * kConvChannels + prep_ch) * (kDConv - 1);
            cs[0] = qk_hist[0];
            cs[1] = qk_hist[1];
            cs[2] = qk_hist[2];
        }
    }

    // MMAs and copies still in flight finish before the tensor memory is freed (bounded).
    if (tid == 0 && failed && pend_mma) (void)mbar_wait_bounded(pend_bar, pend_par);
    if (tid == 32) {
        // (a unit-ahead request that no unit consumed is drained too)
        if (pend_qk) (void)mbar_wait_bounded(bar_qk, ph_qk);
        if (pend_s) (void)mbar_wait_bounded(bar_s, ph_s);
        if (pend_z) (void)mbar_wait_bounded(bar_z, ph_z);
        if (pend_v) (void)mbar_wait_bounded(bar_v, ph_v);
    }
    if (warp == 1) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmCols);
    }
    if (tid == 0 && failed) atomicOr(&g_wtc_error, kErrWaitTimeout);
}

std::mutex g_mutex;
int g_sms[64] = {};

// A [rows][cols] fp32 tensor map with boxes of 128 columns x 8 rows, no swizzle.
cudaError_t encode_rows(CUtensorMap* tm, const float* base, int cols, cuuint64_t rows) {
    if (tensor_map_encoder() == nullptr) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), rows};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kS), static_cast<cuuint32_t>(kBoxRows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = tensor_map_encoder()(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims,
                                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode_window_tc(const StepArgs& a, cudaStream_t stream) {
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
            e = cudaFuncSetAttribute(gdn_window_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kTcSmem));
            if (e != cudaSuccess) return e;
            g_sms[dev] = n;
        }
        sms = g_sms[dev];
    }
    TcParams p;
    memset(&p, 0, sizeof(p));
    const cuuint64_t rows = static_cast<cuuint64_t>(a.B) * a.L * a.T;
    e = encode_rows(&p.tm_qkv, a.qkv, kConvChannels, rows);
    if (e != cudaSuccess) return e;
    if ((a.flags & kNoY) == 0) {
        e = encode_rows(&p.tm_z, a.z, kValueDim, rows);
        if (e != cudaSuccess) return e;
        e = encode_rows(&p.tm_y, a.y, kValueDim, rows);
        if (e != cudaSuccess) return e;
    }
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
    gdn_window_tc_kernel<<<static_cast<unsigned>(grid), kTcThreads, kTcSmem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t read_window_tc_error(uint32_t* out) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_wtc_error, sizeof(v));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_wtc_error, &zero, sizeof(zero));
    *out = v;
    return e;
}

}  // namespace gdn
