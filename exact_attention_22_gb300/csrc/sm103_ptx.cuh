// sm103_ptx.cuh -- thin inline-PTX wrappers for the sm_103a features the
// attention kernel uses: mbarriers, TMA tensor copies, tcgen05 MMA and tensor
// memory (TMEM).  Every wrapper is a single PTX instruction (or a fixed short
// sequence) written by hand; nothing here comes from a library.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace fa103 {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Non-blocking test of three barrier phases at once (bit i set: phase i
// complete); the three tests are in flight together.
__device__ __forceinline__ uint32_t mbar_test3(uint64_t* b0, uint32_t p0, uint64_t* b1, uint32_t p1, uint64_t* b2,
                                               uint32_t p2) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred q0, q1, q2;\n\t.reg .b32 r0, r1, r2;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q0, [%1], %2;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q1, [%3], %4;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q2, [%5], %6;\n\t"
        "selp.b32 r0, 1, 0, q0;\n\t"
        "selp.b32 r1, 2, 0, q1;\n\t"
        "selp.b32 r2, 4, 0, q2;\n\t"
        "or.b32 r0, r0, r1;\n\t"
        "or.b32 %0, r0, r2;\n\t}"
        : "=r"(r)
        : "r"(smem_u32(b0)), "r"(p0), "r"(smem_u32(b1)), "r"(p1), "r"(smem_u32(b2)), "r"(p2)
        : "memory");
    return r;
}
// Wait for the phase of `bar` with the given parity to complete, giving up
// after `timeout_ns` nanoseconds of wall time.  Returns false on time-out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 3-D tiled load global -> shared, completion signalled on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}
// Same, with an L2 eviction-priority policy word.
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* map, uint64_t* bar, int x,
                                                 int y, int z, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "l"(policy)
        : "memory");
}
// 3-D tiled store shared -> global (elements outside the tensor are dropped).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Make generic-proxy writes to shared memory visible to the async proxy (TMA, UMMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------- tcgen05
// TMEM allocation: executed by one whole warp; the base address is written
// to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Commit issued by the lane elect.sync picks from a converged warp (the lowest
// active lane, the same one every time for a full warp): arrive once on `bar`
// when every tcgen05.mma that lane issued before has completed.  The whole
// issuing warp runs the issuer's control flow, which stays warp-uniform.
__device__ __forceinline__ void umma_commit_elect(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------- UMMA groups
// The K-steps of one operation issued as a group under a single elect.sync.
// The shared-memory descriptors' start-address fields (16-byte units in the
// low bits) move by 32-bit adds on their low words, which never carry into the
// high word for shared-memory addresses; the accumulate predicate is the
// caller's for the first step and true after it.  Issuing a group costs the
// issuing warp a handful of instructions per UMMA, and that warp shares its SM
// sub-partition with warps on the critical path of every step.
//
// Step offsets come from a type O: O::a[i] and O::b[i] for step i (a[0] and
// b[0] are 0: the first step uses the bases as given).  For the TMEM-A forms
// O::a[i] is a column offset of the A operand.
template <uint32_t... V>
struct Steps {
    static constexpr uint32_t v[sizeof...(V)] = {V...};
};
template <class A, class B>
struct StepOffsets {
    static constexpr const uint32_t* a = A::v;
    static constexpr const uint32_t* b = B::v;
};

#define FA_UMMA_SS_HEAD                                                     \
    "{\n\t.reg .pred p, e, one;\n\t.reg .b32 al, ah, bl, bh, al2, bl2;\n\t" \
    ".reg .b64 a, b;\n\t"                                                   \
    "mov.b64 {al, ah}, %1;\n\tmov.b64 {bl, bh}, %2;\n\t"                    \
    "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 one, 0, 0;\n\t"                  \
    "elect.sync _|e, 0xffffffff;\n\t"
#define FA_UMMA_SS_FIRST(kind) "@e tcgen05.mma.cta_group::1." kind " [%0], %1, %2, %3, p;\n\t"
#define FA_UMMA_SS_NEXT(kind, ia, ib)                                                          \
    "add.u32 al2, al, %" #ia ";\n\tadd.u32 bl2, bl, %" #ib ";\n\t"                             \
    "mov.b64 a, {al2, ah};\n\tmov.b64 b, {bl2, bh};\n\t"                                       \
    "@e tcgen05.mma.cta_group::1." kind " [%0], a, b, %3, one;\n\t"
#define FA_UMMA_TS_HEAD                                                          \
    "{\n\t.reg .pred p, e, one;\n\t.reg .b32 bl, bh, bl2;\n\t.reg .b64 b;\n\t" \
    "mov.b64 {bl, bh}, %2;\n\t"                                                  \
    "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 one, 0, 0;\n\t"                       \
    "elect.sync _|e, 0xffffffff;\n\t"
#define FA_UMMA_TS_FIRST(kind) "@e tcgen05.mma.cta_group::1." kind " [%0], [%1], %2, %3, p;\n\t"
#define FA_UMMA_TS_NEXT(kind, ia, ib)                                  \
    "add.u32 bl2, bl, %" #ib ";\n\tmov.b64 b, {bl2, bh};\n\t"          \
    "@e tcgen05.mma.cta_group::1." kind " [%0], [%1+%" #ia "], b, %3, one;\n\t"

#define FA_UMMA_OPS4(O) "n"(O::a[1]), "n"(O::b[1]), "n"(O::a[2]), "n"(O::b[2]), "n"(O::a[3]), "n"(O::b[3])
#define FA_UMMA_OPS8(O)                                                                             \
    FA_UMMA_OPS4(O), "n"(O::a[4]), "n"(O::b[4]), "n"(O::a[5]), "n"(O::b[5]), "n"(O::a[6]), "n"(O::b[6]), \
        "n"(O::a[7]), "n"(O::b[7])

// Four / eight steps, both operands in shared memory (kind::f8f6f4 when F8).
template <bool F8, class O>
__device__ __forceinline__ void umma_ss_x4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    if constexpr (F8)
        asm volatile(FA_UMMA_SS_HEAD FA_UMMA_SS_FIRST("kind::f8f6f4") FA_UMMA_SS_NEXT("kind::f8f6f4", 5, 6)
                         FA_UMMA_SS_NEXT("kind::f8f6f4", 7, 8) FA_UMMA_SS_NEXT("kind::f8f6f4", 9, 10) "}" ::"r"(d_tmem),
                     "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), FA_UMMA_OPS4(O)
                     : "memory");
    else
        asm volatile(FA_UMMA_SS_HEAD FA_UMMA_SS_FIRST("kind::f16") FA_UMMA_SS_NEXT("kind::f16", 5, 6)
                         FA_UMMA_SS_NEXT("kind::f16", 7, 8) FA_UMMA_SS_NEXT("kind::f16", 9, 10) "}" ::"r"(d_tmem),
                     "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), FA_UMMA_OPS4(O)
                     : "memory");
}
template <class O>
__device__ __forceinline__ void umma_ss_x8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(FA_UMMA_SS_HEAD FA_UMMA_SS_FIRST("kind::f16") FA_UMMA_SS_NEXT("kind::f16", 5, 6)
                     FA_UMMA_SS_NEXT("kind::f16", 7, 8) FA_UMMA_SS_NEXT("kind::f16", 9, 10)
                         FA_UMMA_SS_NEXT("kind::f16", 11, 12) FA_UMMA_SS_NEXT("kind::f16", 13, 14)
                             FA_UMMA_SS_NEXT("kind::f16", 15, 16) FA_UMMA_SS_NEXT("kind::f16", 17, 18) "}" ::"r"(d_tmem),
                 "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), FA_UMMA_OPS8(O)
                 : "memory");
}
// Four / eight steps, A in tensor memory (its column offsets in O::a).
template <class O>
__device__ __forceinline__ void umma_ts_x4_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(FA_UMMA_TS_HEAD FA_UMMA_TS_FIRST("kind::f8f6f4") FA_UMMA_TS_NEXT("kind::f8f6f4", 5, 6)
                     FA_UMMA_TS_NEXT("kind::f8f6f4", 7, 8) FA_UMMA_TS_NEXT("kind::f8f6f4", 9, 10) "}" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), FA_UMMA_OPS4(O)
                 : "memory");
}
template <class O>
__device__ __forceinline__ void umma_ts_x8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(FA_UMMA_TS_HEAD FA_UMMA_TS_FIRST("kind::f16") FA_UMMA_TS_NEXT("kind::f16", 5, 6)
                     FA_UMMA_TS_NEXT("kind::f16", 7, 8) FA_UMMA_TS_NEXT("kind::f16", 9, 10)
                         FA_UMMA_TS_NEXT("kind::f16", 11, 12) FA_UMMA_TS_NEXT("kind::f16", 13, 14)
                             FA_UMMA_TS_NEXT("kind::f16", 15, 16) FA_UMMA_TS_NEXT("kind::f16", 17, 18) "}" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), FA_UMMA_OPS8(O)
                 : "memory");
}
#undef FA_UMMA_OPS8
#undef FA_UMMA_OPS4
#undef FA_UMMA_TS_NEXT
#undef FA_UMMA_TS_FIRST
#undef FA_UMMA_TS_HEAD
#undef FA_UMMA_SS_NEXT
#undef FA_UMMA_SS_FIRST
#undef FA_UMMA_SS_HEAD

// Common step patterns (descriptor units of 16 bytes; TMEM columns).
// K-major operand over a 128-byte-swizzled head dimension: 32 bytes per step
// (16 16-bit or 32 8-bit elements), the next 128-byte box after four steps.
using StepsK4 = Steps<0, 2, 4, 6>;
template <uint32_t kBox>
using StepsK8 = Steps<0, 2, 4, 6, kBox, kBox + 2, kBox + 4, kBox + 6>;
// MN-major operand: 16 rows (2048 bytes) per step.
using StepsMN8 = Steps<0, 128, 256, 384, 512, 640, 768, 896>;
// 16-bit A operand in TMEM: 16 keys (8 columns of packed pairs) per step.
using StepsCol8 = Steps<0, 8, 16, 24, 32, 40, 48, 56>;
using StepsCol4 = Steps<0, 8, 16, 24>;

// Shared-memory matrix descriptor, 128-byte swizzle.  `lbo` / `sbo` are the
// leading / stride byte offsets of the canonical layout.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;   // descriptor version of the tcgen05 family
    d |= static_cast<uint64_t>(2) << 61;   // swizzle mode: 128 B
    return d;
}

// Instruction descriptor of kind::f16 with fp32 accumulation.
//   bf16: operands are bf16 (else fp16); b_mn_major: B is stored N-contiguous.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, int M, int N, bool b_mn_major) {
    return (1u << 4)                                   // D format: f32
           | ((bf16 ? 1u : 0u) << 7)                   // A format
           | ((bf16 ? 1u : 0u) << 10)                  // B format
           | ((b_mn_major ? 1u : 0u) << 16)            // B major-ness
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// The same with A's major-ness too (a_mn_major: A is stored M-contiguous).
__host__ __device__ constexpr uint32_t idesc_f16_ab(bool bf16, int M, int N, bool a_mn_major, bool b_mn_major) {
    return idesc_f16(bf16, M, N, b_mn_major) | ((a_mn_major ? 1u : 0u) << 15);
}

// 32 lanes x 32 bit, 32 consecutive columns per thread, without the wait.
// The registers are undefined until tmem_ld_wait() names them.
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
// Completes every tcgen05.ld of this thread; naming the registers keeps any
// use of them below the wait.
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}
// Orders the registers of a second load after the same wait (no instruction).
__device__ __forceinline__ void regs_after_wait(uint32_t (&r)[32]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// 16-byte store to shared memory (address in the shared window).
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// 32 lanes x 32 bit, 32 consecutive columns per thread, followed by the wait,
// in one statement so no use of the registers can move above the wait.
__device__ __forceinline__ void tmem_ld32_wait(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
// 16 consecutive columns (32-bit) per thread, followed by the wait.
__device__ __forceinline__ void tmem_ld16_wait(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- math
// Single hardware instructions (no library code): 2^x and packing.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// log2(x) and 1/x for positive normal x, single approximate instructions.
__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// Pack two fp32 values into f16x2 / bf16x2, round to nearest even; `lo` goes
// to the low 16 bits.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Four fp32 values to OCP E4M3 bytes (round to nearest even, saturating to
// +-448), a in the lowest byte.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r)
        : "f"(a), "f"(b), "f"(c), "f"(d));
    return r;
}
// The four E4M3 bytes of w added exactly into two fp32 accumulators
// (bytes 0 and 2 into acc0, bytes 1 and 3 into acc1): each pair of bytes is
// widened to f16x2 (exact) and each half added with one rounding to fp32.
__device__ __forceinline__ void add_e4m3x4(uint32_t w, float& acc0, float& acc1) {
    asm("{\n\t.reg .b16 lo, hi, h0, h1, h2, h3;\n\t.reg .b32 f01, f23;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 f01, lo;\n\t"
        "cvt.rn.f16x2.e4m3x2 f23, hi;\n\t"
        "mov.b32 {h0, h1}, f01;\n\t"
        "mov.b32 {h2, h3}, f23;\n\t"
        "add.rn.f32.f16 %0, h0, %0;\n\t"
        "add.rn.f32.f16 %1, h1, %1;\n\t"
        "add.rn.f32.f16 %0, h2, %0;\n\t"
        "add.rn.f32.f16 %1, h3, %1;\n\t}"
        : "+f"(acc0), "+f"(acc1)
        : "r"(w));
}

// Three-input max.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
// Packed pairs of fp32 in one 64-bit register, and the paired arithmetic on them.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
// acc + (one bf16 half of w, widened exactly), in one mixed-precision add.
__device__ __forceinline__ float add_lo_bf16(uint32_t w, float acc) {
    float r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.bf16 %0, lo, %2;\n\t}"
        : "=f"(r) : "r"(w), "f"(acc));
    return r;
}
__device__ __forceinline__ float add_hi_bf16(uint32_t w, float acc) {
    float r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.bf16 %0, hi, %2;\n\t}"
        : "=f"(r) : "r"(w), "f"(acc));
    return r;
}

}  // namespace fa103
