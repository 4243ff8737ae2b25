// fwd_tc.cu -- forward attention (K2) on the 5th-generation tensor cores.
//
// Non-causal attention inside each packed sample (the attention node of the
// "ws1_one_h3_block" page of RL-Kernel, PR #539, Bindings table), computed as
// S = q^ k^T (fp16 operands) -> online softmax -> O += P v (bf16 operands),
// FP32 accumulation in tensor memory, one rounding of O at the end.
//
// Persistent kernel, one CTA per SM.  A work item is (sample, head, block of
// 256 query rows anchored at the sample start) = two 128-row subtiles A and B
// that share every K/V tile.  Warp roles (384 threads):
//   warp 0      TMA producer: q^ tiles, then K and V tiles (128 keys each, from
//               the sample start, ascending) through a 4-stage ring;
//   warp 1      tcgen05 issuer: S_X = Q_X K^T into TMEM, then O_X += P_X V with
//               P_X read from TMEM (it overwrites S_X's first 64 columns);
//   warps 4-7   softmax of subtile A, warps 8-11 softmax of subtile B: one
//               thread per query row (TMEM lane), the row max and sum are
//               sequential in that thread, P rounded once to bf16.
// TMEM: S_A cols [0,128), S_B [128,256), O_A [256,384), O_B [384,512).
//
// The running max is only moved when it grows by more than 8 (log2 units);
// P = 2^((s - m) c) <= 2^8 then, and O / l are rescaled exactly when m moves.
// Every row's arithmetic depends only on its sample's data and on tiles
// anchored at the sample start, so a sample gives the same bits alone or
// packed.  Key rows past the sample end are masked by select in S and zeroed in
// shared memory in V (a neighbour's Inf/NaN never reaches the PV product).
#include <cudaTypedefs.h>

#include "common.cuh"
#include "host.cuh"
#include "tc.cuh"

namespace h3 {

namespace fwdt {
constexpr int kThreads = 384;
constexpr int kNST = 4;                      // K/V ring stages
constexpr int kTile = 128 * 128 * 2;         // one 128 x 128 16-bit tile: 32 KB
constexpr int kHalf = 128 * 64 * 2;          // one 64-channel half (the TMA box): 16 KB
constexpr int kOffQ = 0;                     // Q_A, Q_B
constexpr int kOffKV = 2 * kTile;            // ring
constexpr int kOffBar = kOffKV + kNST * kTile;
constexpr int kSmem = kOffBar + 512 + 1024;  // barriers + 1 KB alignment slack
constexpr uint32_t kColS0 = 0, kColO0 = 256;
constexpr float kMaxStale = 8.0f;            // log2 growth of the max tolerated before rescaling
// Column pairs (bit e = columns 2e, 2e + 1 of a 128-key tile) whose 2^x would
// run on the FMA pipe (exp2_poly_pair) instead of the SFU, fixed by the
// column's place in its tile so that every row's arithmetic stays the same
// whatever the packing.  None: measured on the packed 13539-token batch, one
// pair in eight made the kernel 10% slower and one in four 19% (the softmax is
// bound by its instruction stream and latency, not by the SFU).
constexpr uint64_t kPolyPairs = 0x0ull;

// barrier indices (8 bytes each)
enum {
    bQFull = 0, bQEmpty, bKVFull, bKVEmpty = bKVFull + kNST, bSFull = bKVEmpty + kNST, bPFull = bSFull + 2,
    bPVDone = bPFull + 2, bOFree = bPVDone + 2, bTail = bOFree + 2, bDone, bNever, bCount
};
}  // namespace fwdt

struct FwdTcParams {
    Seq seq;
    Plan plan;
    int H;
    float scale_log2;
    __nv_bfloat16* out;
    int out_align32;  // out is 32-byte aligned (else 16: the boundary's promise)
    float* lse;
    int stall;               // tc::StallRole stalled once on the CTA's first item (tests), else 0
    long long stall_budget;  // clock cycles of that stall's bounded wait
};

struct FwdItem {
    int h, seg0, L, row0, nkv;
    bool hasB;
};

__device__ __forceinline__ bool fwd_item(const FwdTcParams& p, int i, FwdItem& it) {
    const int n = p.seq.n;
    const int* cum = p.plan.cum256;
    if (i >= p.H * cum[n]) return false;
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (p.H * cum[mid] <= i) lo = mid; else hi = mid;
    }
    const int nb = cum[lo + 1] - cum[lo];
    const int local = i - p.H * cum[lo];
    const int b = local % nb;
    const int s = p.plan.order[lo];
    it.h = local / nb;
    it.seg0 = p.seq.seg[s];
    it.L = p.seq.seg[s + 1] - it.seg0;
    it.row0 = it.seg0 + 256 * b;
    it.hasB = 256 * b + 128 < it.L;
    it.nkv = (it.L + 127) / 128;
    return true;
}

__global__ void __launch_bounds__(fwdt::kThreads, 1)
fwd_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
              const __grid_constant__ CUtensorMap mv, const FwdTcParams p) {
    using namespace fwdt;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars = sbase + kOffBar;
    auto bar = [&](int i) { return bars + 8u * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * bCount);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + 8 * bCount + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        tc::mbar_init(bar(bQFull), 1);
        tc::mbar_init(bar(bQEmpty), 1);
        for (int i = 0; i < kNST; ++i) {
            tc::mbar_init(bar(bKVFull + i), 1);
            tc::mbar_init(bar(bKVEmpty + i), 1);
        }
        for (int x = 0; x < 2; ++x) {
            tc::mbar_init(bar(bSFull + x), 1);
            tc::mbar_init(bar(bPFull + x), 4);
            tc::mbar_init(bar(bPVDone + x), 1);
            tc::mbar_init(bar(bOFree + x), 4);
        }
        tc::mbar_init(bar(bTail), 1);
        tc::mbar_init(bar(bDone), 1);
        tc::mbar_init(bar(bNever), 1);  // nothing arrives: the target of a test's stall
        *abort_flag = 0;
        tc::fence_mbar_init();
        tc::prefetch_map(&mq);
        tc::prefetch_map(&mk);
        tc::prefetch_map(&mv);
    }
    if (warp == 1) {
        tc::tmem_alloc(smem_u32(tmem_slot), 512);
        tc::tmem_relinquish();
        tc::fence_before_sync();
    }
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    bool failed = false;
    auto fail = [&]() {
        failed = true;
        *abort_flag = 1;
        atomicOr(p.plan.err, kErrTimeout);
    };

    // Register split: the producer/issuer warpgroup gives registers to the two
    // softmax warpgroups (launch: 384 x 168 = 128 x 152 + 256 x 176).
    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 152;");
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 176;");
    }

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        uint32_t kv_it = 0, items = 0, tails = 0;
        // copies issued (lane 0): Q loads, K/V blocks whose full barrier was armed, and
        // a tail block whose own wait gave up with its copy possibly in flight
        uint32_t q_armed = 0, kv_armed = 0;
        bool tail_pending = false;
        for (int k = 0, i = turn_item(0); !failed; i = turn_item(++k)) {
            FwdItem it;
            if (!fwd_item(p, i, it)) break;
            const int x0 = it.h * 128;
            if (lane == 0) {
                if (items > 0 && !tc::mbar_wait(bar(bQEmpty), (items - 1) & 1, abort_flag)) fail();
                if (!failed) {
                    tc::mbar_expect_tx(bar(bQFull), it.hasB ? 2 * kTile : kTile);
                    for (int x = 0; x < (it.hasB ? 2 : 1); ++x)
                        for (int hf = 0; hf < 2; ++hf)
                            tc::tma_load_2d(sbase + kOffQ + x * kTile + hf * kHalf, &mq, x0 + 64 * hf,
                                            it.row0 + 128 * x, bar(bQFull));
                    ++q_armed;
                }
            }
            failed = __shfl_sync(0xffffffffu, failed, 0);
            ++items;
            for (int j = 0; j < it.nkv && !failed; ++j) {
                for (int kv = 0; kv < 2 && !failed; ++kv) {
                    const uint32_t slot = kv_it % kNST, ph = (kv_it / kNST) & 1;
                    const uint32_t dst = sbase + kOffKV + slot * kTile;
                    const int y = it.seg0 + 128 * j;
                    const int valid = it.L - 128 * j;
                    const bool tail = kv == 1 && valid < 128;
                    const CUtensorMap* map = kv == 0 ? &mk : &mv;
                    if (lane == 0) {
                        if (p.stall == tc::kStallProducer && items == 1 && j == 0 && kv == 0 &&
                            !tc::mbar_wait(bar(bNever), 0, abort_flag, p.stall_budget))
                            fail();
                        if (!failed && !tc::mbar_wait(bar(bKVEmpty + slot), ph ^ 1, abort_flag)) fail();
                        if (!failed) {
                            const uint32_t b = tail ? bar(bTail) : bar(bKVFull + slot);
                            tc::mbar_expect_tx(b, kTile);
                            tc::tma_load_2d(dst, map, x0, y, b);
                            tc::tma_load_2d(dst + kHalf, map, x0 + 64, y, b);
                            if (!tail) ++kv_armed;
                            if (tail && !tc::mbar_wait(bar(bTail), tails & 1, abort_flag)) {
                                tail_pending = true;
                                fail();
                            }
                        }
                    }
                    failed = __shfl_sync(0xffffffffu, failed, 0);
                    if (tail && !failed) {
                        ++tails;
                        // zero V rows [valid, 128) of both halves (whole 128-byte rows,
                        // so the swizzle inside a row does not matter)
                        for (int r = valid + (lane >> 3); r < 128; r += 4) {
                            const uint32_t off = (uint32_t)r * 128 + (lane & 7) * 16;
                            asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" :: "r"(dst + off), "r"(0) : "memory");
                            asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" :: "r"(dst + kHalf + off), "r"(0)
                                         : "memory");
                        }
                        tc::fence_proxy_async();
                        __syncwarp();
                        if (lane == 0) {
                            tc::mbar_arrive(bar(bKVFull + slot));
                            ++kv_armed;
                        }
                    }
                    ++kv_it;
                }
            }
        }
        // every copy issued has landed before the CTA's shared memory is released (on
        // an abort, consumers may have left some unread)
        if (lane == 0) {
            bool ok = q_armed == 0 || tc::mbar_drain(bar(bQFull), (q_armed - 1) & 1);
            ok &= tc::drain_ring(bar(bKVFull), kNST, kv_armed);
            if (tail_pending) ok &= tc::mbar_drain(bar(bTail), tails & 1);
            if (!ok) atomicOr(p.plan.err, kErrTimeout);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = tc::idesc_f16(false, false, 128, 128);  // fp16 x fp16, K-major B
            constexpr uint32_t idP = tc::idesc_f16(true, true, 128, 128);    // bf16 x bf16, MN-major B
            uint32_t kv_it = 0, items = 0, cntPV[2] = {0, 0}, itemsX[2] = {0, 0};
            // S_X(j+1) is issued right behind PV_X(j): tcgen05 MMAs of one thread run in
            // order, so PV_X(j) has read P_X(j) before S_X(j+1) overwrites those columns,
            // and S_X(j+1) completing implies PV_X(j) completed (the softmax relies on
            // that before it rescales O_X).
            // descriptors are built once; per MMA only the 16-byte start address moves
            const uint64_t dQ = tc::smem_desc_sw128(sbase + kOffQ, 16, 1024);
            const uint64_t dK = tc::smem_desc_sw128(sbase + kOffKV, 16, 1024);
            const uint64_t dV = tc::smem_desc_sw128(sbase + kOffKV, kHalf, 1024);
            auto issue_s = [&](int x, uint32_t kslot) {
                const uint64_t a0 = dQ + ((uint32_t)(x * kTile) >> 4), b0 = dK + ((kslot * kTile) >> 4);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t koff = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
                    tc::mma_ss(tmem + kColS0 + 128 * x, a0 + koff, b0 + koff, idS, kk > 0);
                }
                tc::mma_commit(bar(bSFull + x));
            };
            for (int k = 0, i = turn_item(0); !failed; i = turn_item(++k)) {
                FwdItem it;
                if (!fwd_item(p, i, it)) break;
                const int nX = it.hasB ? 2 : 1;
                if (!tc::mbar_wait(bar(bQFull), items & 1, abort_flag)) { fail(); break; }
                ++items;
                // ---- S_X(0) = Q_X K_0^T
                uint32_t kslot = kv_it % kNST;
                if (!tc::mbar_wait(bar(bKVFull + kslot), (kv_it / kNST) & 1, abort_flag)) { fail(); break; }
                ++kv_it;
                tc::fence_after_sync();
                for (int x = 0; x < nX; ++x) issue_s(x, kslot);
                tc::mma_commit(bar(bKVEmpty + kslot));
                if (it.nkv == 1) tc::mma_commit(bar(bQEmpty));
                if (p.stall == tc::kStallMma && items == 1 &&
                    !tc::mbar_wait(bar(bNever), 0, abort_flag, p.stall_budget)) {
                    fail();
                    break;
                }
                for (int j = 0; j < it.nkv && !failed; ++j) {
                    const uint32_t vslot = kv_it % kNST;
                    if (!tc::mbar_wait(bar(bKVFull + vslot), (kv_it / kNST) & 1, abort_flag)) { fail(); break; }
                    ++kv_it;
                    const bool more = j + 1 < it.nkv;
                    if (more) {
                        kslot = kv_it % kNST;
                        if (!tc::mbar_wait(bar(bKVFull + kslot), (kv_it / kNST) & 1, abort_flag)) { fail(); break; }
                        ++kv_it;
                    }
                    const uint64_t bv0 = dV + ((vslot * kTile) >> 4);
                    for (int x = 0; x < nX && !failed; ++x) {
                        if (j == 0 && itemsX[x] > 0 &&
                            !tc::mbar_wait(bar(bOFree + x), (itemsX[x] - 1) & 1, abort_flag)) {
                            fail();
                            break;
                        }
                        if (!tc::mbar_wait(bar(bPFull + x), cntPV[x] & 1, abort_flag)) { fail(); break; }
                        tc::fence_after_sync();
                        // ---- O_X += P_X V_j
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            tc::mma_ts(tmem + kColO0 + 128 * x, tmem + kColS0 + 128 * x + 8 * kk,
                                       bv0 + ((kk * 2048) >> 4), idP, (j > 0) || (kk > 0));
                        tc::mma_commit(bar(bPVDone + x));
                        ++cntPV[x];
                        // ---- S_X(j+1) = Q_X K_{j+1}^T
                        if (more) issue_s(x, kslot);
                    }
                    if (failed) break;
                    tc::mma_commit(bar(bKVEmpty + vslot));
                    if (more) {
                        tc::mma_commit(bar(bKVEmpty + kslot));
                        if (j + 2 == it.nkv) tc::mma_commit(bar(bQEmpty));
                    }
                }
                for (int x = 0; x < nX; ++x) ++itemsX[x];
            }
            // every issued MMA has completed before TMEM is released (also on an abort)
            tc::mma_commit(bar(bDone));
            if (!tc::mbar_drain(bar(bDone), 0)) fail();
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------- softmax
        const int x = (warp - 4) >> 2;          // subtile
        const int tx = tid - 128 * (1 + x);     // row in subtile == TMEM lane
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t tS = tmem + lane_base + kColS0 + 128 * x;
        const uint32_t tO = tmem + lane_base + kColO0 + 128 * x;
        const float c = p.scale_log2;
        uint32_t cntS = 0, cntPV = 0;
        for (int k = 0, i = turn_item(0); !failed; i = turn_item(++k)) {
            FwdItem it;
            if (!fwd_item(p, i, it)) break;
            if (x == 1 && !it.hasB) continue;
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < it.nkv; ++j) {
                bool ok = true;
                if (lane == 0) {
                    if (p.stall == tc::kStallConsumer && warp == 4 && cntS == 0)
                        ok = tc::mbar_wait(bar(bNever), 0, abort_flag, p.stall_budget);
                    if (ok) ok = tc::mbar_wait(bar(bSFull + x), cntS & 1, abort_flag);
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) { fail(); break; }
                ++cntS;
                tc::fence_after_sync();
                uint64_t s2[64];  // the row's 128 scores as column pairs, then P
                tc::tmem_ld128_pairs(tS, s2);
                const int valid = it.L - 128 * j;
                if (valid < 128) {  // keys past the sample end: -inf, so P = 0 there
#pragma unroll
                    for (int e = 0; e < 64; ++e) {
                        const float a0 = 2 * e < valid ? pair_lo(s2[e]) : -INFINITY;
                        const float a1 = 2 * e + 1 < valid ? pair_hi(s2[e]) : -INFINITY;
                        s2[e] = f2pack(a0, a1);
                    }
                }
                float mx0 = pair_lo(s2[0]), mx1 = pair_hi(s2[1]), mx2 = pair_lo(s2[2]), mx3 = pair_hi(s2[3]);
                mx0 = fmaxf(mx0, pair_hi(s2[0]));
                mx1 = fmaxf(mx1, pair_lo(s2[1]));
                mx2 = fmaxf(mx2, pair_hi(s2[2]));
                mx3 = fmaxf(mx3, pair_lo(s2[3]));
#pragma unroll
                for (int e = 4; e < 64; e += 4) {
                    mx0 = max3f(mx0, pair_lo(s2[e]), pair_hi(s2[e]));
                    mx1 = max3f(mx1, pair_lo(s2[e + 1]), pair_hi(s2[e + 1]));
                    mx2 = max3f(mx2, pair_lo(s2[e + 2]), pair_hi(s2[e + 2]));
                    mx3 = max3f(mx3, pair_lo(s2[e + 3]), pair_hi(s2[e + 3]));
                }
                const float m_new = fmaxf(fmaxf(m, fmaxf(mx0, mx1)), fmaxf(mx2, mx3));
                const bool need = j == 0 || (m_new - m) * c > kMaxStale;
                float factor = 1.f;
                if (need) {
                    factor = j == 0 ? 0.f : ex2((m - m_new) * c);
                    m = m_new;
                    l *= factor;
                }
                const uint64_t c2 = f2pack(c, c), neg2 = f2pack(-m * c, -m * c);
                uint64_t rs[4] = {0ull, 0ull, 0ull, 0ull};  // pairs of +0.0f
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const uint64_t p2 = ((kPolyPairs >> (16 * q4 + e)) & 1)
                                                ? exp2_poly_pair(s2[16 * q4 + e], c2, neg2)
                                                : exp2_pair(s2[16 * q4 + e], c2, neg2);
                        rs[e & 3] = f2add(rs[e & 3], p2);
                        pk[e] = bf16_pair(p2);
                    }
                    tc::tmem_st16(tS + 16 * q4, pk);
                }
                l += ((pair_lo(rs[0]) + pair_hi(rs[0])) + (pair_lo(rs[1]) + pair_hi(rs[1]))) +
                     ((pair_lo(rs[2]) + pair_hi(rs[2])) + (pair_lo(rs[3]) + pair_hi(rs[3])));
                // O_X was last written by PV_X(j-1), complete before S_X(j) was issued
                if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t r[32];
                        tc::tmem_ld32(tO + 32 * q4, r);
                        tc::tmem_wait_ld_dep(r);
#pragma unroll
                        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * factor);
                        tc::tmem_st32(tO + 32 * q4, r);
                    }
                }
                tc::tmem_wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(bar(bPFull + x));
            }
            if (failed) break;
            // ---- epilogue: O / l -> bf16 rows, lse
            cntPV += it.nkv;
            bool ok = true;
            if (lane == 0) ok = tc::mbar_wait(bar(bPVDone + x), (cntPV - 1) & 1, abort_flag);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) { fail(); break; }
            tc::fence_after_sync();
            const int r_in = 256 * ((it.row0 - it.seg0) / 256) + 128 * x + tx;  // row within the sample
            const int row = it.seg0 + r_in;
            const bool store = r_in < it.L;
            const float inv = 1.0f / l;
            // The row's 128 channels as bf16 pairs, piece k = words 8k .. 8k + 7 (32 bytes).
            uint32_t w[64];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t r[32];
                tc::tmem_ld32(tO + 32 * q4, r);
                tc::tmem_wait_ld_dep(r);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    w[16 * q4 + e] = pack_bf16(__uint_as_float(r[2 * e]) * inv, __uint_as_float(r[2 * e + 1]) * inv);
            }
            // O_X is in registers: the next item's products may overwrite it
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(bar(bOFree + x));
            // Storing the row as is would touch 32 token rows per instruction; lanes first
            // trade pieces (a three-bit transpose of (lane, piece) by xor shuffles within
            // groups of 8), so lane 8g + k holds piece k of rows 8g .. 8g + 7 and store e
            // writes 4 whole 256-byte rows.
            const int m8 = lane & 7;
#pragma unroll
            for (int bit = 1; bit <= 4; bit <<= 1) {
#pragma unroll
                for (int k0 = 0; k0 < 8; ++k0) {
                    if (k0 & bit) continue;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t send = (m8 & bit) ? w[8 * k0 + j] : w[8 * (k0 | bit) + j];
                        const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, bit);
                        if (m8 & bit) w[8 * k0 + j] = recv; else w[8 * (k0 | bit) + j] = recv;
                    }
                }
            }
            const int tx0 = tx - lane;  // the warp's first row of the subtile
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int rr = 256 * ((it.row0 - it.seg0) / 256) + 128 * x + tx0 + (lane & ~7) + e;
                if (rr >= it.L) continue;
                __nv_bfloat16* const d = p.out + ((size_t)(it.seg0 + rr) * p.H + it.h) * kD + 16 * m8;
                if (p.out_align32) {
                    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                                 ::"l"(d), "r"(w[8 * e]), "r"(w[8 * e + 1]), "r"(w[8 * e + 2]), "r"(w[8 * e + 3]),
                                 "r"(w[8 * e + 4]), "r"(w[8 * e + 5]), "r"(w[8 * e + 6]), "r"(w[8 * e + 7]) : "memory");
                } else {
                    *reinterpret_cast<uint4*>(d) = make_uint4(w[8 * e], w[8 * e + 1], w[8 * e + 2], w[8 * e + 3]);
                    *reinterpret_cast<uint4*>(d + 8) = make_uint4(w[8 * e + 4], w[8 * e + 5], w[8 * e + 6], w[8 * e + 7]);
                }
            }
            if (store && p.lse) p.lse[(size_t)it.h * p.seq.S + row] = (m * c + log2f(l)) * 0.69314718055994531f;
        }
    }

    // the producer has waited out its copies and the issuer its products
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ host

namespace {
bool encode_rows(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int H, int S) {
    const cuuint64_t dims[2] = {(cuuint64_t)H * kD, (cuuint64_t)S};
    const cuuint64_t strides[1] = {(cuuint64_t)H * kD * 2};
    const cuuint32_t box[2] = {64, 128};
    const cuuint32_t es[2] = {1, 1};
    return tensor_map_encoder()(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

cudaError_t set_fwd_attributes() {
    return cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, fwdt::kSmem);
}

cudaError_t launch_fwd(const Problem& p, const Workspace& ws, __nv_bfloat16* out, float* lse, cudaStream_t st) {
    CUtensorMap mq, mk, mv;
    if (!encode_rows(&mq, ws.qhat, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p.H, p.seq.S) ||
        !encode_rows(&mk, ws.khat, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p.H, p.seq.S) ||
        !encode_rows(&mv, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.H, p.seq.S))
        return cudaErrorInvalidValue;
    FwdTcParams prm;
    prm.seq = p.seq;
    prm.plan = ws.plan;
    prm.H = p.H;
    prm.scale_log2 = p.scale * 1.4426950408889634f;
    prm.out = out;
    prm.out_align32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
    prm.lse = lse;
    prm.stall = p.stall.kernel == kStallKernelFwd ? p.stall.role : 0;
    prm.stall_budget = p.stall.budget;
    const int sms = device_sms();
    if (sms < 1) return cudaErrorNotSupported;
    fwd_tc_kernel<<<sms, fwdt::kThreads, fwdt::kSmem, st>>>(mq, mk, mv, prm);
    return cudaGetLastError();
}

}  // namespace h3
