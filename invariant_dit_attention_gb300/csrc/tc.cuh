// tc.cuh -- sm_103a building blocks written as inline PTX: mbarriers with
// bounded waits, TMA tile loads, tcgen05 tensor-memory allocation, MMA, commit,
// loads and stores, and the shared-memory / instruction descriptors.
//
// Every wait is bounded by a clock budget; when it runs out the wait reports
// failure and the caller records kErrTimeout and unwinds (no trap, no hang).
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace h3 {
namespace tc {

// ~1 s at 2 GHz: far beyond any legitimate wait inside one kernel.
constexpr long long kWaitBudget = 2000000000LL;
// The same bound for the unwinding of an aborted kernel (waits for copies and
// products already issued, which complete on their own).
constexpr long long kDrainBudget = 2000000000LL;

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
// One arrive for the warp, by its lane 0, as a predicated instruction (no branch
// around it); the caller orders the warp's earlier work before it (__syncwarp).
__device__ __forceinline__ void mbar_arrive_lane0(uint32_t bar, int lane) {
    asm volatile("{\n.reg .pred p;\nsetp.eq.s32 p, %1, 0;\n@p mbarrier.arrive.shared::cta.b64 _, [%0];\n}\n"
                 :: "r"(bar), "r"(lane) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
// As mbar_try, but a thread whose phase is not complete yet is suspended by the
// hardware until it completes or about `ns` nanoseconds pass, instead of
// returning at once: waiting warps then issue (almost) no instructions.
__device__ __forceinline__ bool mbar_try_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(bar), "r"(parity), "r"(ns) : "memory");
    return ok != 0;
}
// Non-blocking test of the same condition.  On a phase that has already
// completed this is far cheaper for the issuing thread than try_wait, which
// matters on the MMA thread: the tensor pipe only holds about one instruction
// ahead, so every cycle it spends between MMAs is a cycle the pipe idles.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
// Waits for the phase of the given parity to complete; false on timeout (after
// `budget` clock cycles) or once another thread of the CTA set `abort`.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const volatile int* abort,
                                          long long budget = kWaitBudget) {
    if (mbar_test(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_sleep(bar, parity, 20000u)) return true;
        if (*abort) return false;
        if (clock64() - t0 > budget) return false;
    }
}

// Waits for the phase of the given parity to complete whatever the abort flag
// says: an aborted kernel uses it to wait out the bulk copies and tensor-core
// products it already issued (they complete on their own) before its shared
// and tensor memory are released.  False only past kDrainBudget.
__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity) {
    if (mbar_test(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_sleep(bar, parity, 20000u)) return true;
        if (clock64() - t0 > kDrainBudget) return false;
    }
}

// Waits for every copy a ring's producer issued: the full barriers of slots
// 0 .. slots-1 (8 bytes apart from full0) were armed `armed` times in block
// order, block b in slot b % slots, each arming completed by its copies (or by
// the producer's own arrive).  The last armed phase of each slot is waited on.
__device__ __forceinline__ bool drain_ring(uint32_t full0, int slots, uint32_t armed) {
    bool ok = true;
    for (int s = 0; s < slots && (uint32_t)s < armed; ++s) {
        const uint32_t n = (armed - 1 - (uint32_t)s) / (uint32_t)slots + 1;  // phases armed on slot s
        ok &= mbar_drain(full0 + 8u * s, (n - 1) & 1);
    }
    return ok;
}

// Roles a test can stall once (a bounded wait on a barrier nothing completes)
// to exercise a kernel's unwinding: none, the TMA producer, the MMA issuer, a
// consumer warp (softmax or epilogue).
enum StallRole { kStallNone = 0, kStallProducer = 1, kStallMma = 2, kStallConsumer = 3 };

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 2D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar) : "memory");
}
// 4D tiled TMA load with an L2 cache policy.
__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const CUtensorMap* map, int x, int y, int z, int w,
                                                 uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar), "l"(policy)
        : "memory");
}
// L2 policy: lines of this access are the first to be evicted (streamed data).
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- TMEM

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(dst_smem), "r"(ncols));
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols));
}
__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T   (kind::f16: fp16 or bf16 operands, fp32 accumulate)
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accum) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accum));
}
// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accum) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
        :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accum));
}
// Arrives on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar) : "memory");
}

// 32 lanes x 32 columns of 32-bit, waited, as 16 column pairs (64-bit registers).
__device__ __forceinline__ void tmem_ld32_pairs(uint32_t taddr, uint64_t (&r)[16]) {
    asm volatile(
        "{\n.reg .b32 a<32>;\n"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {a0,a1,a2,a3,a4,a5,a6,a7,a8,a9,a10,a11,a12,a13,a14,a15,a16,a17,a18,a19,a20,a21,a22,a23,a24,a25,a26,a27,a28,a29,a30,a31}, [%16];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        "mov.b64 %0, {a0, a1};\n"
        "mov.b64 %1, {a2, a3};\n"
        "mov.b64 %2, {a4, a5};\n"
        "mov.b64 %3, {a6, a7};\n"
        "mov.b64 %4, {a8, a9};\n"
        "mov.b64 %5, {a10, a11};\n"
        "mov.b64 %6, {a12, a13};\n"
        "mov.b64 %7, {a14, a15};\n"
        "mov.b64 %8, {a16, a17};\n"
        "mov.b64 %9, {a18, a19};\n"
        "mov.b64 %10, {a20, a21};\n"
        "mov.b64 %11, {a22, a23};\n"
        "mov.b64 %12, {a24, a25};\n"
        "mov.b64 %13, {a26, a27};\n"
        "mov.b64 %14, {a28, a29};\n"
        "mov.b64 %15, {a30, a31};\n"
        "}\n"
        : "=l"(r[0]), "=l"(r[1]), "=l"(r[2]), "=l"(r[3]), "=l"(r[4]), "=l"(r[5]), "=l"(r[6]), "=l"(r[7]), "=l"(r[8]), "=l"(r[9]), "=l"(r[10]), "=l"(r[11]), "=l"(r[12]), "=l"(r[13]), "=l"(r[14]), "=l"(r[15])
        : "r"(taddr) : "memory");
}
// 32 lanes x 64 columns of 32-bit in one load, waited, as 32 column pairs.
__device__ __forceinline__ void tmem_ld64_pairs(uint32_t taddr, uint64_t (&r)[32]) {
    asm volatile(
        "{\n.reg .b32 a<64>;\n"
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {a0,a1,a2,a3,a4,a5,a6,a7,a8,a9,a10,a11,a12,a13,a14,a15,a16,a17,a18,a19,a20,a21,a22,a23,a24,a25,a26,a27,a28,a29,a30,a31,a32,a33,a34,a35,a36,a37,a38,a39,a40,a41,a42,a43,a44,a45,a46,a47,a48,a49,a50,a51,a52,a53,a54,a55,a56,a57,a58,a59,a60,a61,a62,a63}, [%32];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        "mov.b64 %0, {a0, a1};\n"
        "mov.b64 %1, {a2, a3};\n"
        "mov.b64 %2, {a4, a5};\n"
        "mov.b64 %3, {a6, a7};\n"
        "mov.b64 %4, {a8, a9};\n"
        "mov.b64 %5, {a10, a11};\n"
        "mov.b64 %6, {a12, a13};\n"
        "mov.b64 %7, {a14, a15};\n"
        "mov.b64 %8, {a16, a17};\n"
        "mov.b64 %9, {a18, a19};\n"
        "mov.b64 %10, {a20, a21};\n"
        "mov.b64 %11, {a22, a23};\n"
        "mov.b64 %12, {a24, a25};\n"
        "mov.b64 %13, {a26, a27};\n"
        "mov.b64 %14, {a28, a29};\n"
        "mov.b64 %15, {a30, a31};\n"
        "mov.b64 %16, {a32, a33};\n"
        "mov.b64 %17, {a34, a35};\n"
        "mov.b64 %18, {a36, a37};\n"
        "mov.b64 %19, {a38, a39};\n"
        "mov.b64 %20, {a40, a41};\n"
        "mov.b64 %21, {a42, a43};\n"
        "mov.b64 %22, {a44, a45};\n"
        "mov.b64 %23, {a46, a47};\n"
        "mov.b64 %24, {a48, a49};\n"
        "mov.b64 %25, {a50, a51};\n"
        "mov.b64 %26, {a52, a53};\n"
        "mov.b64 %27, {a54, a55};\n"
        "mov.b64 %28, {a56, a57};\n"
        "mov.b64 %29, {a58, a59};\n"
        "mov.b64 %30, {a60, a61};\n"
        "mov.b64 %31, {a62, a63};\n"
        "}\n"
        : "=l"(r[0]), "=l"(r[1]), "=l"(r[2]), "=l"(r[3]), "=l"(r[4]), "=l"(r[5]), "=l"(r[6]), "=l"(r[7]), "=l"(r[8]), "=l"(r[9]), "=l"(r[10]), "=l"(r[11]), "=l"(r[12]), "=l"(r[13]), "=l"(r[14]), "=l"(r[15]), "=l"(r[16]), "=l"(r[17]), "=l"(r[18]), "=l"(r[19]), "=l"(r[20]), "=l"(r[21]), "=l"(r[22]), "=l"(r[23]), "=l"(r[24]), "=l"(r[25]), "=l"(r[26]), "=l"(r[27]), "=l"(r[28]), "=l"(r[29]), "=l"(r[30]), "=l"(r[31])
        : "r"(taddr) : "memory");
}
// 32 lanes x 128 columns of 32-bit in one load, waited, as 64 column pairs.
__device__ __forceinline__ void tmem_ld128_pairs(uint32_t taddr, uint64_t (&r)[64]) {
    asm volatile(
        "{\n.reg .b32 a<128>;\n"
        "tcgen05.ld.sync.aligned.32x32b.x128.b32 {a0,a1,a2,a3,a4,a5,a6,a7,a8,a9,a10,a11,a12,a13,a14,a15,a16,a17,a18,a19,a20,a21,a22,a23,a24,a25,a26,a27,a28,a29,a30,a31,a32,a33,a34,a35,a36,a37,a38,a39,a40,a41,a42,a43,a44,a45,a46,a47,a48,a49,a50,a51,a52,a53,a54,a55,a56,a57,a58,a59,a60,a61,a62,a63,a64,a65,a66,a67,a68,a69,a70,a71,a72,a73,a74,a75,a76,a77,a78,a79,a80,a81,a82,a83,a84,a85,a86,a87,a88,a89,a90,a91,a92,a93,a94,a95,a96,a97,a98,a99,a100,a101,a102,a103,a104,a105,a106,a107,a108,a109,a110,a111,a112,a113,a114,a115,a116,a117,a118,a119,a120,a121,a122,a123,a124,a125,a126,a127}, [%64];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        "mov.b64 %0, {a0, a1};\n"
        "mov.b64 %1, {a2, a3};\n"
        "mov.b64 %2, {a4, a5};\n"
        "mov.b64 %3, {a6, a7};\n"
        "mov.b64 %4, {a8, a9};\n"
        "mov.b64 %5, {a10, a11};\n"
        "mov.b64 %6, {a12, a13};\n"
        "mov.b64 %7, {a14, a15};\n"
        "mov.b64 %8, {a16, a17};\n"
        "mov.b64 %9, {a18, a19};\n"
        "mov.b64 %10, {a20, a21};\n"
        "mov.b64 %11, {a22, a23};\n"
        "mov.b64 %12, {a24, a25};\n"
        "mov.b64 %13, {a26, a27};\n"
        "mov.b64 %14, {a28, a29};\n"
        "mov.b64 %15, {a30, a31};\n"
        "mov.b64 %16, {a32, a33};\n"
        "mov.b64 %17, {a34, a35};\n"
        "mov.b64 %18, {a36, a37};\n"
        "mov.b64 %19, {a38, a39};\n"
        "mov.b64 %20, {a40, a41};\n"
        "mov.b64 %21, {a42, a43};\n"
        "mov.b64 %22, {a44, a45};\n"
        "mov.b64 %23, {a46, a47};\n"
        "mov.b64 %24, {a48, a49};\n"
        "mov.b64 %25, {a50, a51};\n"
        "mov.b64 %26, {a52, a53};\n"
        "mov.b64 %27, {a54, a55};\n"
        "mov.b64 %28, {a56, a57};\n"
        "mov.b64 %29, {a58, a59};\n"
        "mov.b64 %30, {a60, a61};\n"
        "mov.b64 %31, {a62, a63};\n"
        "mov.b64 %32, {a64, a65};\n"
        "mov.b64 %33, {a66, a67};\n"
        "mov.b64 %34, {a68, a69};\n"
        "mov.b64 %35, {a70, a71};\n"
        "mov.b64 %36, {a72, a73};\n"
        "mov.b64 %37, {a74, a75};\n"
        "mov.b64 %38, {a76, a77};\n"
        "mov.b64 %39, {a78, a79};\n"
        "mov.b64 %40, {a80, a81};\n"
        "mov.b64 %41, {a82, a83};\n"
        "mov.b64 %42, {a84, a85};\n"
        "mov.b64 %43, {a86, a87};\n"
        "mov.b64 %44, {a88, a89};\n"
        "mov.b64 %45, {a90, a91};\n"
        "mov.b64 %46, {a92, a93};\n"
        "mov.b64 %47, {a94, a95};\n"
        "mov.b64 %48, {a96, a97};\n"
        "mov.b64 %49, {a98, a99};\n"
        "mov.b64 %50, {a100, a101};\n"
        "mov.b64 %51, {a102, a103};\n"
        "mov.b64 %52, {a104, a105};\n"
        "mov.b64 %53, {a106, a107};\n"
        "mov.b64 %54, {a108, a109};\n"
        "mov.b64 %55, {a110, a111};\n"
        "mov.b64 %56, {a112, a113};\n"
        "mov.b64 %57, {a114, a115};\n"
        "mov.b64 %58, {a116, a117};\n"
        "mov.b64 %59, {a118, a119};\n"
        "mov.b64 %60, {a120, a121};\n"
        "mov.b64 %61, {a122, a123};\n"
        "mov.b64 %62, {a124, a125};\n"
        "mov.b64 %63, {a126, a127};\n"
        "}\n"
        : "=l"(r[0]), "=l"(r[1]), "=l"(r[2]), "=l"(r[3]), "=l"(r[4]), "=l"(r[5]), "=l"(r[6]), "=l"(r[7]),
          "=l"(r[8]), "=l"(r[9]), "=l"(r[10]), "=l"(r[11]), "=l"(r[12]), "=l"(r[13]), "=l"(r[14]), "=l"(r[15]),
          "=l"(r[16]), "=l"(r[17]), "=l"(r[18]), "=l"(r[19]), "=l"(r[20]), "=l"(r[21]), "=l"(r[22]), "=l"(r[23]),
          "=l"(r[24]), "=l"(r[25]), "=l"(r[26]), "=l"(r[27]), "=l"(r[28]), "=l"(r[29]), "=l"(r[30]), "=l"(r[31]),
          "=l"(r[32]), "=l"(r[33]), "=l"(r[34]), "=l"(r[35]), "=l"(r[36]), "=l"(r[37]), "=l"(r[38]), "=l"(r[39]),
          "=l"(r[40]), "=l"(r[41]), "=l"(r[42]), "=l"(r[43]), "=l"(r[44]), "=l"(r[45]), "=l"(r[46]), "=l"(r[47]),
          "=l"(r[48]), "=l"(r[49]), "=l"(r[50]), "=l"(r[51]), "=l"(r[52]), "=l"(r[53]), "=l"(r[54]), "=l"(r[55]),
          "=l"(r[56]), "=l"(r[57]), "=l"(r[58]), "=l"(r[59]), "=l"(r[60]), "=l"(r[61]), "=l"(r[62]), "=l"(r[63])
        : "r"(taddr) : "memory");
}
// 32 lanes x 32 columns of 32-bit: thread t of the warp gets lane (base + t), 32 columns.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
           "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
           "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
           "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
           "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// Waits for this thread's TMEM loads; taking the destination registers as operands
// keeps the compiler from reading them before the wait.
__device__ __forceinline__ void tmem_wait_ld_dep(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]),"+r"(r[1]),"+r"(r[2]),"+r"(r[3]),"+r"(r[4]),"+r"(r[5]),"+r"(r[6]),"+r"(r[7]),"+r"(r[8]),"+r"(r[9]),"+r"(r[10]),"+r"(r[11]),"+r"(r[12]),"+r"(r[13]),"+r"(r[14]),"+r"(r[15]),"+r"(r[16]),"+r"(r[17]),"+r"(r[18]),"+r"(r[19]),"+r"(r[20]),"+r"(r[21]),"+r"(r[22]),"+r"(r[23]),"+r"(r[24]),"+r"(r[25]),"+r"(r[26]),"+r"(r[27]),"+r"(r[28]),"+r"(r[29]),"+r"(r[30]),"+r"(r[31]) :: "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ----------------------------------------------------------- descriptors

// Shared-memory matrix descriptor (tcgen05): start address, leading and stride
// byte offsets (16-byte units), fixed version bits 46..48 = 0b001, base offset
// 0 (tiles are 1024-byte aligned), swizzle mode 2 = 128-byte swizzle.
// The same for a 64-byte swizzled operand (atoms of 8 rows x 64 bytes).
__device__ __forceinline__ uint64_t smem_desc_sw64(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 4ull << 61;
    return d;
}
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// Instruction descriptor of kind::f16 with fp32 accumulation.
//   bits 4-5 D format (1 = f32), 7-9 A format and 10-12 B format (0 = f16, 1 = bf16),
//   15 / 16 A / B major (0 = K-major, 1 = MN-major), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, bool b_mn_major, int M, int N) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// The same with A read MN-major as well.
__host__ __device__ constexpr uint32_t idesc_f16_amn(bool bf16, bool b_mn_major, int M, int N) {
    return idesc_f16(bf16, b_mn_major, M, N) | (1u << 15);
}

}  // namespace tc
}  // namespace h3
