// gdn_tc.cuh - inline PTX for the 5th-generation tensor cores and the tensor
// memory accelerator, shared by the kernels that run tcgen05.mma: tensor-map
// loads, tensor-memory allocation and loads, shared-memory matrix descriptors
// of the 128-byte swizzled K-major layout, the BF16 MMA of kind::f16 with
// M = 128, and the split of fp32 values into BF16 hi + lo halves.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstdint>

#include "gdn_device.cuh"

namespace gdn {

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* tm, int x, int y, int z, uint32_t bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_local(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y, uint32_t bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* tm) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzled
// layout (8-row groups of 128-byte rows, 1024 bytes apart), tcgen05 format.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
    d |= static_cast<uint64_t>(1) << 16;                          // leading offset (unused when swizzled)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;                  // stride between 8-row groups
    d |= static_cast<uint64_t>(1) << 46;                          // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                          // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16: BF16 A and B, both K-major, fp32 D, M 128.
__host__ __device__ constexpr uint32_t mma_idesc(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(128 >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives on `bar` once every tcgen05.mma this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 consecutive accumulator columns of this warp's 32 lanes, one lane per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Byte offset of 16-byte chunk c of row n in a 128-byte swizzled K-major block.
__host__ __device__ __forceinline__ uint32_t sw128_offset(int n, int c) {
    return static_cast<uint32_t>((n >> 3) * 1024 + (n & 7) * 128 + ((c ^ (n & 7)) << 4));
}

// ------------------------------------------------------------- split of x --
// Upper halves of two floats (their BF16 truncations), a in the low 16 bits.
__device__ __forceinline__ uint32_t hi_pair(float a, float b) {
    return __byte_perm(__float_as_uint(a), __float_as_uint(b), 0x7632);
}

// What the truncation left of two floats (exact in fp32), rounded to BF16.
__device__ __forceinline__ uint32_t lo_pair(float a, float b) {
    const float ra = a - __uint_as_float(__float_as_uint(a) & 0xFFFF0000u);
    const float rb = b - __uint_as_float(__float_as_uint(b) & 0xFFFF0000u);
    const __nv_bfloat162 v = __floats2bfloat162_rn(ra, rb);
    return *reinterpret_cast<const uint32_t*>(&v);
}


}  // namespace gdn

namespace gdn {

// The driver's cuTensorMapEncodeTiled, looked up once (NULL if unavailable).
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

}  // namespace gdn

namespace gdn {

// Stores 32 consecutive accumulator columns of this warp's 32 lanes, one lane per thread.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]),
        "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]),
        "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

// Waits until this thread's tensor-memory stores have completed.
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// BF16 hi (truncation) and lo (the rest, rounded) halves of one float, as raw 16-bit patterns.
__device__ __forceinline__ void split_bf16(float x, uint16_t& hi, uint16_t& lo) {
    const uint32_t u = __float_as_uint(x);
    hi = static_cast<uint16_t>(u >> 16);
    lo = __bfloat16_as_ushort(__float2bfloat16_rn(x - __uint_as_float(u & 0xFFFF0000u)));
}

}  // namespace gdn

namespace gdn {

// BF16 hi (rounded to nearest) and lo (the rest, rounded) halves of two floats,
// a in the low 16 bits of each word. hi + lo leaves a relative residue of at most
// 2^-16, against 2^-15 when hi is a truncation.
__device__ __forceinline__ void split_pair_rn(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const uint32_t hu = *reinterpret_cast<const uint32_t*>(&h);
    const __nv_bfloat162 r =
        __floats2bfloat162_rn(a - __uint_as_float(hu << 16), b - __uint_as_float(hu & 0xFFFF0000u));
    hi = hu;
    lo = *reinterpret_cast<const uint32_t*>(&r);
}

// Eight floats as two 16-byte rows of BF16 pairs (hi and lo), stored at hi_dst and lo_dst.
__device__ __forceinline__ void store_split8(unsigned char* hi_dst, unsigned char* lo_dst, const float* x) {
    uint4 h, l;
    split_pair_rn(x[0], x[1], h.x, l.x);
    split_pair_rn(x[2], x[3], h.y, l.y);
    split_pair_rn(x[4], x[5], h.z, l.z);
    split_pair_rn(x[6], x[7], h.w, l.w);
    *reinterpret_cast<uint4*>(hi_dst) = h;
    *reinterpret_cast<uint4*>(lo_dst) = l;
}

// One float as BF16 hi (rounded to nearest) and lo halves, raw 16-bit patterns.
__device__ __forceinline__ void split_rn(float x, uint16_t& hi, uint16_t& lo) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    hi = __bfloat16_as_ushort(h);
    lo = __bfloat16_as_ushort(__float2bfloat16_rn(x - __bfloat162float(h)));
}

}  // namespace gdn

namespace gdn {

// Shared-memory matrix descriptor: MN-major operand in the 128-byte swizzled
// layout, atoms of 8 K-rows x 64 MN-contiguous BF16 (1024 bytes); `mn_stride`
// bytes from one atom to the next along MN, 1024 bytes between 8-row groups
// along K. (A K-major block of 128-byte rows read with its rows as K is this
// layout: its 64-element row halves are the MN atoms.)
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t saddr, uint32_t mn_stride) {
    uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((mn_stride >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Bit 16 of the kind::f16 instruction descriptor: B is MN-major.
constexpr uint32_t kIdescBMnMajor = 1u << 16;

// 8 consecutive accumulator columns of this warp's 32 lanes, one lane per thread.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&v)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr)
                 : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

}  // namespace gdn

namespace gdn {

// Waits until at most one of this thread's committed bulk async-groups is still reading shared memory.
__device__ __forceinline__ void bulk_wait_read_one() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

}  // namespace gdn

namespace gdn {

// A 2-D tensor-map store of one box from shared memory, tracked by this thread's bulk async-group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm, int x, int y, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(tm)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}

}  // namespace gdn

namespace gdn {

// Programmatic dependent launch: lets the next kernel in the stream begin launching (a no-op
// unless it was launched with programmatic stream serialization) ...
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ... and waits until the kernels this one depends on have completed and their memory
// operations are visible (returns at once for an ordinary launch).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace gdn
