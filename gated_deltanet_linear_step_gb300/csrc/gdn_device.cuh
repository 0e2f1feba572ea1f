// gdn_device.cuh - device-side pieces shared by the decode-step kernels:
// inline PTX for mbarriers, bulk async copies and clusters, bounded waits,
// warp reductions, the scalar activations of the GDN step, the gated delta rule
// on a tile in shared memory, and the register mapping of a tile held by a
// 256-thread CTA (its step lives with the multi-token kernel).
#pragma once

#include <cstdint>

#include "gdn_launch.h"

namespace gdn {

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per mbarrier wait
constexpr uint32_t kErrWaitTimeout = 1u;
constexpr float kEps = 1e-6f;                    // RMS epsilon of both norms
constexpr float kQScale = 0.08838834764831845f;  // 1/sqrt(128)

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

// Orders this thread's generic-proxy shared-memory accesses before later
// bulk async (async-proxy) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// An L2 policy that marks lines as first to evict: state tiles are touched once per call.
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// One contiguous global -> shared bulk copy (16-byte aligned addresses, size a
// multiple of 16); completion is signalled on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// bulk_load with the evict-first L2 policy, for data read once per call.
__device__ __forceinline__ void bulk_load_stream(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(evict_first_policy())
        : "memory");
}

// One contiguous shared -> global bulk copy, tracked by this thread's bulk
// async-group (commit with bulk_commit, wait with bulk_wait_read / bulk_wait_all).
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until every committed bulk store of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Waits until every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// One 16-byte global -> shared asynchronous copy by this thread (both addresses
// 16-byte aligned), cached in L2 only.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Closes this thread's current group of cp.async copies.
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Waits until at most one of this thread's committed cp.async groups is still in flight.
__device__ __forceinline__ void cp_async_wait_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Waits until all of this thread's committed cp.async groups have landed.
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void named_barrier(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// named_barrier that also returns whether `v` was true in any of the `threads` threads.
__device__ __forceinline__ bool named_barrier_or(int id, int threads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "r"(id), "r"(threads)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

// sigmoid and SiLU through the __expf and __fdividef intrinsics: relative error
// near 1e-6 over the inputs' range, far inside the 1e-4 parity bar, at about a
// fifth of the instructions of expf and an IEEE division. For x below about -88,
// 1 + e^-x is infinite and both return 0 (signed), their limit. The multi-token
// kernel evaluates one SiLU per conv channel and token, and one sigmoid per y
// element. softplus keeps expf and log1pf: it feeds the decay exponent.
__device__ __forceinline__ float sigmoidf_(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }
__device__ __forceinline__ float siluf_(float x) { return __fdividef(x, 1.0f + __expf(-x)); }
__device__ __forceinline__ float softplusf_(float x) { return fmaxf(x, 0.0f) + log1pf(expf(-fabsf(x))); }

// Global conv channel of the unit's channel slot cc (k head g): q of head g at
// slots [0,128), k at [128,256), v of heads 3g..3g+2 at [256,640).
__device__ __forceinline__ int unit_channel(int cc, int g) {
    return cc < kHeadDim ? g * kHeadDim + cc
                         : (cc < 2 * kHeadDim ? kKOffset + g * kHeadDim + (cc - kHeadDim)
                                              : kVOffset + g * kGroup * kHeadDim + (cc - 2 * kHeadDim));
}

// Conv output of one channel: taps 0-2 on the history (oldest first), tap 3 on x.
__device__ __forceinline__ float conv4(float4 w, float h0, float h1, float h2, float x) {
    float xc = w.x * h0;
    xc = fmaf(w.y, h1, xc);
    xc = fmaf(w.z, h2, xc);
    return fmaf(w.w, x, xc);
}

// beta and decay of one v head from the raw projections and the layer's dt, ssm_a.
__device__ __forceinline__ void head_gates(float alpha_raw, float beta_raw, float dt, float ssm_a, float& beta,
                                           float& decay) {
    beta = sigmoidf_(beta_raw);
    decay = expf(softplusf_(alpha_raw + dt) * ssm_a);
}

// beta and decay of one v head, from raw projections or, with `ready`, from
// a precomputed log decay (in alpha_or_gate) and beta (in beta_in).
__device__ __forceinline__ void head_gates_in(bool ready, float alpha_or_gate, float beta_in, float dt, float ssm_a,
                                              float& beta, float& decay) {
    if (ready) {
        beta = beta_in;
        decay = expf(alpha_or_gate);
    } else {
        head_gates(alpha_or_gate, beta_in, dt, ssm_a, beta, decay);
    }
}

// In place, by one warp: q <- q / sqrt(|q|^2 + eps) / sqrt(128) and
// k <- k / sqrt(|k|^2 + eps), 128 floats each, 16-byte aligned.
__device__ __forceinline__ void normalize_qk(float* qv, float* kv, int lane) {
    float4 q4 = *reinterpret_cast<float4*>(qv + lane * 4);
    float4 k4 = *reinterpret_cast<float4*>(kv + lane * 4);
    const float sq = warp_sum(q4.x * q4.x + q4.y * q4.y + q4.z * q4.z + q4.w * q4.w);
    const float sk = warp_sum(k4.x * k4.x + k4.y * k4.y + k4.z * k4.z + k4.w * k4.w);
    const float rq = rsqrtf(sq + kEps) * kQScale;
    const float rk = rsqrtf(sk + kEps);
    q4.x *= rq;
    q4.y *= rq;
    q4.z *= rq;
    q4.w *= rq;
    k4.x *= rk;
    k4.y *= rk;
    k4.z *= rk;
    k4.w *= rk;
    *reinterpret_cast<float4*>(qv + lane * 4) = q4;
    *reinterpret_cast<float4*>(kv + lane * 4) = k4;
}

// y for one head's 128 values (4 per lane): rms_norm(o) * w * gate(z).
__device__ __forceinline__ float4 gated_rms_norm4(float4 o4, float4 z4, float4 w4, bool silu_gate) {
    const float ss = warp_sum(o4.x * o4.x + o4.y * o4.y + o4.z * o4.z + o4.w * o4.w);
    const float rr = rsqrtf(ss * (1.0f / kHeadDim) + kEps);
    float4 y;
    if (silu_gate) {
        y.x = o4.x * rr * w4.x * siluf_(z4.x);
        y.y = o4.y * rr * w4.y * siluf_(z4.y);
        y.z = o4.z * rr * w4.z * siluf_(z4.z);
        y.w = o4.w * rr * w4.w * siluf_(z4.w);
    } else {
        y.x = o4.x * rr * w4.x * sigmoidf_(z4.x);
        y.y = o4.y * rr * w4.y * sigmoidf_(z4.y);
        y.z = o4.z * rr * w4.z * sigmoidf_(z4.z);
        y.w = o4.w * rr * w4.w * sigmoidf_(z4.w);
    }
    return y;
}

// ------------------------------------------------------------------------
// The "quad" mapping of a 128x128 tile onto a 128-thread group (4 warps):
// lane 8 rb + qd of warp wg handles rows [32 rb, 32 rb + 32) of the four
// columns [32 wg + 4 qd, +4). A warp's 128-bit shared accesses then cover four
// full 128-byte row segments without bank conflicts, and a column reduction
// is 32 in-thread FMAs plus two warp shuffles across rb.
// ------------------------------------------------------------------------
struct Quad {
    int row0;  // first row held
    int col0;  // first of the four columns held
    int rb;    // row block (0..3): lane bits 3-4
};

__device__ __forceinline__ Quad quad_of(int tid_in_group) {
    const int lane = tid_in_group & 31;
    Quad q;
    q.rb = lane >> 3;
    q.row0 = 32 * q.rb;
    q.col0 = 32 * (tid_in_group >> 5) + 4 * (lane & 7);
    return q;
}

// One gated delta-rule step on the thread's 32x4 block of a tile that stays in
// shared memory (row-major 128x128). `qv` and `kv` point at the normalised q
// (already scaled) and k of the tile's k head; v4 holds v of the four columns;
// the four lanes of a row-block group compute the same d and o:
//   pass 1:  a_c = sum_i S[i][c] k[i];  d_c = beta (v_c - decay a_c)         (kv = (decay S)^T k)
//   pass 2:  S[i][c] <- decay S[i][c] + k[i] d_c, written back in place;
//            o_c = sum_i S[i][c] q[i]                                       (S += k d^T; o = S^T q)
__device__ __forceinline__ float4 delta_step_smem(float* tile, const float* qv, const float* kv, const Quad& q,
                                                  float4 v4, float beta, float decay) {
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 8
    for (int r = 0; r < 32; ++r) {
        const float4 sv = *reinterpret_cast<const float4*>(tile + (q.row0 + r) * kHeadDim + q.col0);
        const float k = kv[q.row0 + r];
        a0 = fmaf(sv.x, k, a0);
        a1 = fmaf(sv.y, k, a1);
        a2 = fmaf(sv.z, k, a2);
        a3 = fmaf(sv.w, k, a3);
    }
#pragma unroll
    for (int m = 8; m <= 16; m <<= 1) {
        a0 += __shfl_xor_sync(0xffffffffu, a0, m);
        a1 += __shfl_xor_sync(0xffffffffu, a1, m);
        a2 += __shfl_xor_sync(0xffffffffu, a2, m);
        a3 += __shfl_xor_sync(0xffffffffu, a3, m);
    }
    const float d0 = beta * (v4.x - decay * a0);
    const float d1 = beta * (v4.y - decay * a1);
    const float d2 = beta * (v4.z - decay * a2);
    const float d3 = beta * (v4.w - decay * a3);
    float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll 8
    for (int r = 0; r < 32; ++r) {
        float4* row = reinterpret_cast<float4*>(tile + (q.row0 + r) * kHeadDim + q.col0);
        float4 sv = *row;
        const float k = kv[q.row0 + r];
        const float qq = qv[q.row0 + r];
        sv.x = fmaf(k, d0, decay * sv.x);
        sv.y = fmaf(k, d1, decay * sv.y);
        sv.z = fmaf(k, d2, decay * sv.z);
        sv.w = fmaf(k, d3, decay * sv.w);
        *row = sv;
        o0 = fmaf(sv.x, qq, o0);
        o1 = fmaf(sv.y, qq, o1);
        o2 = fmaf(sv.z, qq, o2);
        o3 = fmaf(sv.w, qq, o3);
    }
#pragma unroll
    for (int m = 8; m <= 16; m <<= 1) {
        o0 += __shfl_xor_sync(0xffffffffu, o0, m);
        o1 += __shfl_xor_sync(0xffffffffu, o1, m);
        o2 += __shfl_xor_sync(0xffffffffu, o2, m);
        o3 += __shfl_xor_sync(0xffffffffu, o3, m);
    }
    return make_float4(o0, o1, o2, o3);
}

}  // namespace gdn

namespace gdn {

// ------------------------------------------------------------------------
// Thread-block-cluster helpers (the multi-token kernel runs a 3-CTA cluster
// per unit).
// ------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// All threads of all CTAs of the cluster.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The address of `local` (a shared-memory address of this CTA) in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

// ------------------------------------------------------------------------
// The state tile in registers, 64 values per thread ("octet" mapping) for a
// 256-thread CTA that owns one 128x128 tile. Lane 4 rb + qd of warp w holds
// rows [16 rb, 16 rb + 16) of the four columns [16 w + 4 qd, +4):
// s[4 r + c] = S[16 rb + r][16 w + 4 qd + c]. A column reduction is 16
// in-thread FMAs plus three shuffles across rb.
// ------------------------------------------------------------------------
struct Octet {
    int row0;  // first row held
    int col0;  // first of the four columns held
    int rb;    // row block (0..7): lane bits 2-4
};

__device__ __forceinline__ Octet octet_of(int tid) {
    const int lane = tid & 31;
    Octet q;
    q.rb = lane >> 2;
    q.row0 = 16 * q.rb;
    q.col0 = 16 * (tid >> 5) + 4 * (lane & 3);
    return q;
}

__device__ __forceinline__ void tile_load_octet(float (&s)[64], const float* tile, const Octet& q) {
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const float4 v = *reinterpret_cast<const float4*>(tile + (q.row0 + r) * kHeadDim + q.col0);
        s[4 * r + 0] = v.x;
        s[4 * r + 1] = v.y;
        s[4 * r + 2] = v.z;
        s[4 * r + 3] = v.w;
    }
}

__device__ __forceinline__ void tile_save_octet(const float (&s)[64], float* tile, const Octet& q) {
#pragma unroll
    for (int r = 0; r < 16; ++r)
        *reinterpret_cast<float4*>(tile + (q.row0 + r) * kHeadDim + q.col0) =
            make_float4(s[4 * r + 0], s[4 * r + 1], s[4 * r + 2], s[4 * r + 3]);
}

}  // namespace gdn
