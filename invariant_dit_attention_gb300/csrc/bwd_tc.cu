// bwd_tc.cu -- backward of the attention core on the 5th-generation tensor cores.
//
// Gradients of sum(out * dout) (the per-leaf gradient checks of the
// "ws1_one_h3_block" page of RL-Kernel, PR #539, Results and Tests; the
// 128-element norm-weight gradient of its Status section):
//   Delta_i = sum_c dO_ic O_ic                                         (delta_kernel, bwd_rows.cu)
//   P_ij = exp(scale q^_i.k^_j - lse_i),  dP_ij = dO_i . v_j,  dS_ij = P_ij (dP_ij - Delta_i)
//   dV_j = sum_i P_ij dO_i,  dk^_j = scale sum_i dS_ij q^_i              (dkdv_tc_kernel)
//   dq^_i = scale sum_j dS_ij k^_j                        (dq_ds_kernel or dq_tc_kernel)
// They leave scale * dk^ and scale * dq^ as FP32 rows for the row backward
// (RoPE^-1 and the RMSNorm backward, rows_bwd.cuh): run by 8 warps of
// dq_ds_kernel, or by rows_bwd_kernel (bwd_rows.cu) after dq_tc_kernel.
//
// No atomics anywhere: dQ is a second pass, either over the dS blocks that
// dkdv stored (dq_ds_kernel) or recomputing S and P (dq_tc_kernel: 7 tile
// products for the 5 of the algorithm), and every sum runs over tiles anchored
// at the sample start in ascending order, so a sample's gradients are the same
// bits alone or packed.
//
// dkdv and dq_tc are persistent (one CTA per SM): warps 0 and 2 TMA producers
// (one per streamed ring), warp 1 the single-thread tcgen05 issuer, in dkdv warp 3
// the stager of each block's lse / Delta columns in shared memory; then the
// warpgroups that split each 128 x 128 score block by columns (thread = TMEM
// lane = one row of the CTA's 128-row tile) and compute on register pairs: two
// of 64 columns in dkdv (384 threads), four of 32 in dq_tc (640 threads).  Operands: S on fp16 q^/k^, dP on bf16 dO/v, P (bf16) and dS
// (fp16) for the accumulating products.  An item's accumulators are drained to
// HBM as soon as its last MMA completed, so the next item's loads and products
// start right away.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "host.cuh"
#include "rows_bwd.cuh"
#include "tc.cuh"

namespace h3 {

namespace bwdt {
constexpr int kTile = 128 * 128 * 2;   // 32 KB
constexpr int kHalf = 128 * 64 * 2;    // 16 KB
constexpr int kPair = 2 * kTile;       // two tiles (q^ + dO, or k^ + v): 64 KB
constexpr float kLog2e = 1.4426950408889634f;
}  // namespace bwdt

struct BwdTcParams {
    Seq seq;
    Plan plan;
    int H;
    float scale;
    const float* lse;
    const float* delta;
    __nv_bfloat16* dv;  // dkdv kernel only
    int dv_align32;     // dv is 32-byte aligned (else 16: the boundary's promise)
    float* dyhat;       // scale * dk^ (dkdv) or scale * dq^ (dq): FP32 [S, H, 128]
    __half* ds;         // stored dS^T blocks (dkdv writes, dq_ds reads), or null
    long long ds_blocks;
    int stall;               // tc::StallRole stalled once on the CTA's first item (tests), else 0
    long long stall_budget;  // clock cycles of that stall's bounded wait
};

struct BwdItem {
    int h, seg0, L, tile, row0, n_other, tile_global, rank;
};

// First stored block of (sample of plan rank r, head h): the blocks of one head
// of a sample with nq tiles are (key tile j, query tile i) at + j nq + i.
__device__ __forceinline__ long long ds_base(const BwdTcParams& p, const BwdItem& it) {
    return (long long)p.H * p.plan.cumsq[it.rank] + (long long)it.h * it.n_other * it.n_other;
}

// Item i over (rank, head, 128-token tile), samples longest first.
__device__ __forceinline__ bool bwd_item(const BwdTcParams& p, int i, BwdItem& it) {
    const int n = p.seq.n;
    const int* cum = p.plan.cum128;
    if (i >= p.H * cum[n]) return false;
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (p.H * cum[mid] <= i) lo = mid; else hi = mid;
    }
    const int nb = cum[lo + 1] - cum[lo];
    const int local = i - p.H * cum[lo];
    const int s = p.plan.order[lo];
    it.h = local / nb;
    it.tile = local % nb;
    it.seg0 = p.seq.seg[s];
    it.L = p.seq.seg[s + 1] - it.seg0;
    it.row0 = it.seg0 + 128 * it.tile;
    it.n_other = nb;
    it.tile_global = cum[lo] + it.tile;
    it.rank = lo;
    return true;
}

// Zeroes rows [valid, rows) of a 64-channel-half tile (whole 128-byte rows).
__device__ __forceinline__ void zero_rows(uint32_t half, int valid, int rows, int lane) {
    for (int r = valid + (lane >> 3); r < rows; r += 4)
        asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" :: "r"(half + (uint32_t)r * 128 + (lane & 7) * 16),
                     "r"(0) : "memory");
}

// One ring of 128-row streamed tiles and the warp that fills it.
struct RingSpec {
    const CUtensorMap* map;
    uint32_t base;        // shared address of slot 0 (slots kTile apart)
    int slots;
    uint32_t full, empty;  // barrier addresses of slot 0 (8 bytes apart)
    uint32_t tail;        // barrier of a block that runs past the sample end
    bool zero_tail;       // zero the rows past the sample end before publishing
};
// The item's fixed tile pair, loaded by the first ring's warp once the previous
// item's last MMA completed.
struct FixedSpec {
    const CUtensorMap* map0;
    const CUtensorMap* map1;
    uint32_t base, full, acc_done;
};

// Producer warp of one ring (lane 0 issues): for every streamed 128-row block of
// every item of this CTA, waits until its slot is released, loads the block's
// two 64-channel halves with TMA and publishes it.  One warp per ring, so a
// ring never waits behind a slot of the other.  Before returning it waits for
// every copy it issued (an aborted kernel's consumers may have left some
// unread), so no copy lands after the CTA's shared memory is released.
// `never`: a barrier nothing completes, the target of a test's stall (`stall`).
__device__ __forceinline__ void ring_producer(const BwdTcParams& p, const RingSpec& r, const FixedSpec* fx,
                                              volatile int* abort_flag, int lane, uint32_t never, bool stall) {
    constexpr int kTile = 128 * 128 * 2, kHalf = 128 * 64 * 2;
    bool failed = false;
    auto fail = [&]() {
        failed = true;
        *abort_flag = 1;
        atomicOr(p.plan.err, kErrTimeout);
    };
    uint32_t blk = 0, items = 0, tails = 0;
    // copies issued (lane 0): fixed tile pairs, ring blocks whose full barrier was
    // armed, and a tail block whose own wait gave up with its copy possibly in flight
    uint32_t fixed_armed = 0, armed = 0;
    bool tail_pending = false;
    for (int k = 0, i = turn_item(0); !failed; i = turn_item(++k)) {
        BwdItem it;
        if (!bwd_item(p, i, it)) break;
        const int x0 = it.h * 128;
        if (fx && lane == 0) {
            if (items > 0 && !tc::mbar_wait(fx->acc_done, (items - 1) & 1, abort_flag)) fail();
            if (!failed) {
                tc::fence_proxy_async();
                tc::mbar_expect_tx(fx->full, 2 * kTile);
                for (int hf = 0; hf < 2; ++hf) {
                    tc::tma_load_2d(fx->base + hf * kHalf, fx->map0, x0 + 64 * hf, it.row0, fx->full);
                    tc::tma_load_2d(fx->base + kTile + hf * kHalf, fx->map1, x0 + 64 * hf, it.row0, fx->full);
                }
                ++fixed_armed;
            }
        }
        failed = __shfl_sync(0xffffffffu, failed, 0);
        ++items;
        const int nb = (it.L + 127) / 128;
        for (int j = 0; j < nb && !failed; ++j) {
            const uint32_t sl = blk % r.slots, ph = (blk / r.slots) & 1;
            const uint32_t dst = r.base + sl * kTile;
            const int y = it.seg0 + 128 * j, valid = it.L - 128 * j;
            const bool tail = r.zero_tail && valid < 128;
            if (lane == 0) {
                if (stall && items == 1 && j == 0 && !tc::mbar_wait(never, 0, abort_flag, p.stall_budget)) fail();
                if (!failed && !tc::mbar_wait(r.empty + 8 * sl, ph ^ 1, abort_flag)) fail();
                if (!failed) {
                    const uint32_t b = tail ? r.tail : r.full + 8 * sl;
                    tc::mbar_expect_tx(b, kTile);
                    for (int hf = 0; hf < 2; ++hf) tc::tma_load_2d(dst + hf * kHalf, r.map, x0 + 64 * hf, y, b);
                    if (!tail) ++armed;
                    if (tail && !tc::mbar_wait(r.tail, tails & 1, abort_flag)) {
                        tail_pending = true;
                        fail();
                    }
                }
            }
            failed = __shfl_sync(0xffffffffu, failed, 0);
            if (tail && !failed) {
                ++tails;
                for (int hf = 0; hf < 2; ++hf) zero_rows(dst + hf * kHalf, valid, 128, lane);
                tc::fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(r.full + 8 * sl);
                    ++armed;
                }
            }
            ++blk;
        }
    }
    if (lane == 0) {
        bool ok = !fx || fixed_armed == 0 || tc::mbar_drain(fx->full, (fixed_armed - 1) & 1);
        ok &= tc::drain_ring(r.full, r.slots, armed);
        if (tail_pending) ok &= tc::mbar_drain(r.tail, tails & 1);
        if (!ok) atomicOr(p.plan.err, kErrTimeout);
    }
    __syncwarp();
}

// ------------------------------------------------------------------ dK, dV
//
// 128-query blocks (N = 128 MMAs run at the full rate).  TMEM: S^T [0, 128),
// the block buffer B [128, 256), dV [256, 384), dK [384, 512).  Four warpgroups
// split each block's 128 query columns (thread = key row, 32 columns each).
// Per block b a warpgroup
//   loads S^T(b) and computes P (FP32, registers); the S^T buffer is refilled
//     with S^T(b+1) right away;
//   loads dP^T(b) from B, then writes P^T(b) (bf16) over the first 16 of its
//     32 B columns -> dV(b) = P^T(b) dO(b) reads it as the TMEM A operand;
//   computes dS = P (dP - Delta) and writes dS^T(b) (fp16) over the other 16
//     -> dK(b) = dS^T(b) q^(b), TMEM A operand as well;
// and dP^T(b+1) is issued into B right behind dK(b) (in-order MMAs).  So the
// tensor cores never wait on a whole softmax-gradient pass, and the softmax
// warps wait on the tensor cores only for dP^T.  q^ streams through a 3-slot
// ring (a slot is held from S^T(b), one block ahead, to dK(b)), dO through a
// 2-slot ring (dP^T(b) to dV(b)).
namespace kvt {
constexpr int kThreads = 384;                       // warps 0-3: producers, MMA issuer, column stager; 4-11: two warpgroups
constexpr int kQSlots = 3, kOSlots = 2;
constexpr int kOffFixed = 0;                        // k^ + v tiles
constexpr int kOffQ = bwdt::kPair;                  // q^ ring
constexpr int kOffO = kOffQ + kQSlots * bwdt::kTile;  // dO ring
constexpr int kOffBar = kOffO + kOSlots * bwdt::kTile;
// per warpgroup and block parity: the block's 64 query columns as -lse2 then -Delta (FP32)
// (written by warp 3, read by the warpgroup's four softmax warps)
constexpr int kOffCol = kOffBar + 256;
constexpr int kSmem = kOffCol + 4 * 2 * 64 * 4;     // the dynamic shared memory base is 1024-aligned (checked)
enum { bFixedFull = 0, bQFull, bQEmpty = bQFull + kQSlots, bOFull = bQEmpty + kQSlots, bOEmpty = bOFull + kOSlots,
       bSFull = bOEmpty + kOSlots, bPFull, bSUsed, bPtFull, bDsFull, bAccDone, bTailQ, bTailO, bDone, bNever,
       bColReady, bColFree = bColReady + 2, bCount = bColFree + 2 };
static_assert(8 * bCount + 8 <= 256, "barrier area");
static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
constexpr uint32_t cB = 128;
}  // namespace kvt

// TMEM column of the A operand for K-step kk (queries 16kk .. 16kk + 15) of P^T
// (half = 0) or dS^T (half = 1): warpgroup kk / 4 packed its 64 queries at
// B + 64 (kk / 4) + 32 half.
__device__ __forceinline__ uint32_t kv_acol(int kk, int half) { return kvt::cB + 64 * (kk >> 2) + 32 * half + 8 * (kk & 3); }


__global__ void __launch_bounds__(kvt::kThreads, 1)
dkdv_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
               const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
               const BwdTcParams p) {
    using namespace kvt;
    using bwdt::kHalf;
    using bwdt::kLog2e;
    using bwdt::kPair;
    using bwdt::kTile;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {  // the layout below needs a 1024-byte aligned base
        if (threadIdx.x == 0) atomicOr(p.plan.err, kErrTimeout);
        return;
    }
    uint8_t* smem = smem_raw;
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) { return sbase + kOffBar + 8u * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * bCount);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + 8 * bCount + 4);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        tc::mbar_init(bar(bFixedFull), 1);
        for (int i = 0; i < kQSlots; ++i) {
            tc::mbar_init(bar(bQFull + i), 1);
            tc::mbar_init(bar(bQEmpty + i), 1);
        }
        for (int i = 0; i < kOSlots; ++i) {
            tc::mbar_init(bar(bOFull + i), 1);
            tc::mbar_init(bar(bOEmpty + i), 1);
        }
        tc::mbar_init(bar(bSFull), 1);
        tc::mbar_init(bar(bPFull), 1);
        tc::mbar_init(bar(bSUsed), 8);
        tc::mbar_init(bar(bPtFull), 8);
        tc::mbar_init(bar(bDsFull), 8);
        tc::mbar_init(bar(bAccDone), 1);
        tc::mbar_init(bar(bTailQ), 1);
        tc::mbar_init(bar(bTailO), 1);
        tc::mbar_init(bar(bDone), 1);
        tc::mbar_init(bar(bNever), 1);  // nothing arrives: the target of a test's stall
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(bar(bColReady + i), 1);  // warp 3
            tc::mbar_init(bar(bColFree + i), 8);  // the softmax warps
        }
        *abort_flag = 0;
        tc::fence_mbar_init();
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
    // 384 threads x 168 registers, no setmaxnreg split (a 152 / 176 split made the
    // softmax warps spill)

    if (warp == 0 || warp == 2) {
        // ------------------------------------- TMA producers: warp 0 the fixed k^ / v
        // tiles and the q^ ring, warp 2 the dO ring; rows past the sample end are
        // zeroed in both, so no neighbour value reaches the dV and dK products
        const FixedSpec fx = {&mk, &mv, sbase + kOffFixed, bar(bFixedFull), bar(bAccDone)};
        const RingSpec r = warp == 0 ? RingSpec{&mq, sbase + kOffQ, kQSlots, bar(bQFull), bar(bQEmpty), bar(bTailQ), true}
                                     : RingSpec{&mdo, sbase + kOffO, kOSlots, bar(bOFull), bar(bOEmpty), bar(bTailO), true};
        ring_producer(p, r, warp == 0 ? &fx : nullptr, abort_flag, lane, bar(bNever),
                      warp == 0 && p.stall == tc::kStallProducer);
    } else if (warp == 1) {
        // ----------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS16 = tc::idesc_f16(false, false, 128, 128);
            constexpr uint32_t idSbf = tc::idesc_f16(true, false, 128, 128);
            constexpr uint32_t idAbf = tc::idesc_f16(true, true, 128, 128);
            constexpr uint32_t idA16 = tc::idesc_f16(false, true, 128, 128);
            // descriptors are built once; per MMA only the 16-byte start address moves
            const uint64_t dK = tc::smem_desc_sw128(sbase + kOffFixed, 16, 1024);
            const uint64_t dV = dK + (kTile >> 4);
            const uint64_t dQr = tc::smem_desc_sw128(sbase + kOffQ, 16, 1024);
            const uint64_t dOr = tc::smem_desc_sw128(sbase + kOffO, 16, 1024);
            const uint64_t dQrMN = tc::smem_desc_sw128(sbase + kOffQ, kHalf, 1024);
            const uint64_t dOrMN = tc::smem_desc_sw128(sbase + kOffO, kHalf, 1024);
            uint32_t blk = 0, items = 0, cnt = 0;
            // S^T(b) = k^ q^(b)^T into [0, 128)
            auto issue_st = [&](uint32_t b) -> bool {
                const uint32_t qs = b % kQSlots;
                if (!tc::mbar_wait(bar(bQFull + qs), (b / kQSlots) & 1, abort_flag)) return false;
                tc::fence_after_sync();
                const uint64_t bq = dQr + ((qs * kTile) >> 4);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t koff = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
                    tc::mma_ss(tmem + 0, dK + koff, bq + koff, idS16, kk > 0);
                }
                tc::mma_commit(bar(bSFull));
                return true;
            };
            // dP^T(b) = v dO(b)^T into B
            auto issue_dpt = [&](uint32_t b) -> bool {
                const uint32_t os = b % kOSlots;
                if (!tc::mbar_wait(bar(bOFull + os), (b / kOSlots) & 1, abort_flag)) return false;
                tc::fence_after_sync();
                const uint64_t bo = dOr + ((os * kTile) >> 4);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t koff = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
                    tc::mma_ss(tmem + cB, dV + koff, bo + koff, idSbf, kk > 0);
                }
                tc::mma_commit(bar(bPFull));
                return true;
            };
            for (int k = 0, i = turn_item(0); !failed; i = turn_item(++k)) {
                BwdItem it;
                if (!bwd_item(p, i, it)) break;
                if (!tc::mbar_wait(bar(bFixedFull), items & 1, abort_flag)) { fail(); break; }
                ++items;
                const int nq = (it.L + 127) / 128;
                const uint32_t b0 = blk;
                if (!issue_st(b0) || !issue_dpt(b0)) { fail(); break; }
                if (p.stall == tc::kStallMma && items == 1 &&
                    !tc::mbar_wait(bar(bNever), 0, abort_flag, p.stall_budget)) {
                    fail();
                    break;
                }
                for (int qj = 0; qj < nq && !failed; ++qj) {
                    const uint32_t b = b0 + qj;
                    const bool more = qj + 1 < nq;
                    // S^T(b) is in registers: refill the S^T buffer with block b+1
                    if (!tc::mbar_wait(bar(bSUsed), cnt & 1, abort_flag)) { fail(); break; }
                    if (more && !issue_st(b + 1)) { fail(); break; }
                    // dV += P^T(b) dO(b)
                    if (!tc::mbar_wait(bar(bPtFull), cnt & 1, abort_flag)) { fail(); break; }
                    tc::fence_after_sync();
                    const uint64_t bo = dOrMN + (((b % kOSlots) * kTile) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc::mma_ts(tmem + 256, tmem + kv_acol(kk, 0), bo + ((kk * 2048) >> 4), idAbf,
                                   (qj > 0) || (kk > 0));
                    tc::mma_commit(bar(bOEmpty + (b % kOSlots)));
                    // dK += dS^T(b) q^(b)
                    if (!tc::mbar_wait(bar(bDsFull), cnt & 1, abort_flag)) { fail(); break; }
                    tc::fence_after_sync();
                    const uint64_t bq = dQrMN + (((b % kQSlots) * kTile) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc::mma_ts(tmem + 384, tmem + kv_acol(kk, 1), bq + ((kk * 2048) >> 4), idA16,
                                   (qj > 0) || (kk > 0));
                    tc::mma_commit(bar(bQEmpty + (b % kQSlots)));
                    // dP^T(b+1) overwrites P^T(b) and dS^T(b): in-order MMAs, dV and dK read them
                    if (more && !issue_dpt(b + 1)) { fail(); break; }
                    ++cnt;
                }
                if (failed) break;
                blk = b0 + nq;
                tc::mma_commit(bar(bAccDone));
            }
            // every issued MMA has completed before TMEM is released (also on an abort)
            tc::mma_commit(bar(bDone));
            if (!tc::mbar_drain(bar(bDone), 0)) fail();
        }
        __syncwarp();
    } else if (warp == 3) {
        // ------------------------------------- lse / Delta column stager
        // Block n's 128 query columns, -lse in log2 units and -Delta (+0 past the
        // sample end), into buffer n & 1: warpgroup w's 64 columns at 256 w + 128 (n & 1)
        // floats, their Delta 64 floats further.  The values are loaded before waiting for the buffer (the softmax
        // warps' release of block n - 2), so the stager runs up to two blocks ahead
        // and the softmax warps issue no global loads in their block loop.
        float* const colbase = reinterpret_cast<float*>(smem + kOffCol) + lane;
        uint32_t n = 0;
        for (int k = 0, i = turn_item(0); !failed; i = turn_item(++k)) {
            BwdItem it;
            if (!bwd_item(p, i, it)) break;
            const int nq = (it.L + 127) / 128;
            const size_t col0 = (size_t)it.h * p.seq.S + it.seg0;
            for (int qj = 0; qj < nq; ++qj, ++n) {
                float rl[4], rd[4];
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const int c = 128 * qj + 32 * g + lane;
                    rl[g] = c < it.L ? p.lse[col0 + c] : 0.f;
                    rd[g] = c < it.L ? p.delta[col0 + c] : 0.f;
                }
                bool ok = true;
                if (lane == 0 && n >= 2) ok = tc::mbar_wait(bar(bColFree + (n & 1)), ((n - 2) >> 1) & 1, abort_flag);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) { fail(); break; }
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    colbase[256 * (g >> 1) + 128 * (n & 1) + 32 * (g & 1)] = 0.f - rl[g] * kLog2e;
                    colbase[256 * (g >> 1) + 128 * (n & 1) + 32 * (g & 1) + 64] = 0.f - rd[g];
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(bar(bColReady + (n & 1)));
            }
        }
    } else if (warp >= 4) {
        // ------------------------------------- softmax gradient + drain
        const int wg = (warp - 4) >> 2;                 // query half of the score tile
        const int t = tid - 128 * (1 + wg);             // key row == TMEM lane
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t tS = tmem + lane_base + 64 * wg, tB = tmem + lane_base + cB + 64 * wg;
        const float c = p.scale * kLog2e;
        const uint64_t pol = tc::policy_evict_first();  // the stored dS blocks are streamed once
        uint32_t cntS = 0, items = 0;
        for (int k = 0, i = turn_item(0); !failed; i = turn_item(++k)) {
            BwdItem it;
            if (!bwd_item(p, i, it)) break;
            const int nq = (it.L + 127) / 128;
            const bool key_ok = 128 * it.tile + t < it.L;
            // the item's stored dS rows of this thread: chunks 2 wg and 2 wg + 1 of block qj at
            // dsrow + qj * 8192 words and 2048 words further (layout [32-query chunk][key][32 queries])
            const long long blk0 = p.ds ? ds_base(p, it) + (long long)it.tile * nq : 0;
            const int ds_in = (int)max(0LL, min((long long)nq, p.ds_blocks - blk0));
            const size_t dsrow = (size_t)blk0 * (128 * 128 / 2) + ((size_t)(2 * wg) * 128 + t) * 16;  // in 32-bit words
            // lse / Delta of the warpgroup's 64 query columns come staged in shared memory
            // (warp 3, above) and are read as broadcast 16-byte loads
            for (int qj = 0; qj < nq; ++qj) {
                const uint32_t n = cntS;
                const int validq = it.L - 128 * qj - 64 * wg;  // columns of this half inside the sample
                bool ok = true;
                if (lane == 0) {
                    if (p.stall == tc::kStallConsumer && warp == 4 && cntS == 0)
                        ok = tc::mbar_wait(bar(bNever), 0, abort_flag, p.stall_budget);
                    if (ok) ok = tc::mbar_wait(bar(bSFull), cntS & 1, abort_flag);
                    if (ok) ok = tc::mbar_wait(bar(bColReady + (n & 1)), (n >> 1) & 1, abort_flag);
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) { fail(); break; }
                __syncwarp();  // lane 0's acquire of the staged columns covers the warp
                tc::fence_after_sync();
                const float4* const cl = reinterpret_cast<const float4*>(smem + kOffCol) + 64 * wg + 32 * (n & 1);
                const float4* const cd = cl + 16;
                uint64_t p2[32];  // S^T column pairs, then P in FP32
                tc::tmem_ld64_pairs(tS, p2);
                tc::fence_before_sync();
                __syncwarp();
                tc::mbar_arrive_lane0(bar(bSUsed), lane);
                // ---- P = 2^(s c - lse2_col)
                const uint64_t c2 = f2pack(c, c);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float4 v = cl[j];
                    p2[2 * j] = exp2_pair(p2[2 * j], c2, f2pack(v.x, v.y));
                    p2[2 * j + 1] = exp2_pair(p2[2 * j + 1], c2, f2pack(v.z, v.w));
                }
                if (validq < 64) {  // tail block: columns past the sample end are exact zeros
#pragma unroll
                    for (int e = 0; e < 32; ++e) p2[e] = mask_pair(p2[e], 2 * e, validq);
                }
                // ---- dP^T(b) from B, then P^T (bf16) over B's first 32 columns of this half
                if (lane == 0) ok = tc::mbar_wait(bar(bPFull), cntS & 1, abort_flag);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) { fail(); break; }
                ++cntS;
                tc::fence_after_sync();
                // dP^T in two halves: the first (queries 0-31) before P^T is written over it,
                // the second (queries 32-63) before dS^T is
                uint64_t d2[16];
                tc::tmem_ld32_pairs(tB, d2);
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) pk[e] = bf16_pair(p2[16 * h2 + e]);
                    tc::tmem_st16(tB + 16 * h2, pk);
                }
                tc::tmem_wait_st();
                tc::fence_before_sync();
                __syncwarp();
                tc::mbar_arrive_lane0(bar(bPtFull), lane);
                // ---- dS = P (dP - Delta_col), fp16, over B's other 32 columns (zero where P is)
                uint32_t dk[32];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 v = cd[j];
                    dk[2 * j] = ds_f16_pair(p2[2 * j], d2[2 * j], f2pack(v.x, v.y));
                    dk[2 * j + 1] = ds_f16_pair(p2[2 * j + 1], d2[2 * j + 1], f2pack(v.z, v.w));
                }
                tc::tmem_ld32_pairs(tB + 32, d2);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 v = cd[8 + j];
                    dk[16 + 2 * j] = ds_f16_pair(p2[16 + 2 * j], d2[2 * j], f2pack(v.x, v.y));
                    dk[16 + 2 * j + 1] = ds_f16_pair(p2[16 + 2 * j + 1], d2[2 * j + 1], f2pack(v.z, v.w));
                }
                tc::tmem_st32(tB + 32, dk);
                tc::tmem_wait_st();
                tc::fence_before_sync();
                __syncwarp();
                tc::mbar_arrive_lane0(bar(bDsFull), lane);
                tc::mbar_arrive_lane0(bar(bColFree + (n & 1)), lane);  // the warp's reads of the columns are done
                if (p.ds) {  // the block for the dQ kernel (key row t, this half's two 32-query chunks)
                    if (qj < ds_in) {
                        uint32_t* const dst = reinterpret_cast<uint32_t*>(p.ds) + dsrow + (size_t)qj * (128 * 128 / 2);
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            if (key_ok) {
#pragma unroll
                                for (int e = 0; e < 2; ++e)
                                    asm volatile("st.global.L2::cache_hint.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}, %9;"
                                                 ::"l"(dst + 2048 * h2 + 8 * e), "r"(dk[16 * h2 + 8 * e]),
                                                 "r"(dk[16 * h2 + 8 * e + 1]), "r"(dk[16 * h2 + 8 * e + 2]),
                                                 "r"(dk[16 * h2 + 8 * e + 3]), "r"(dk[16 * h2 + 8 * e + 4]),
                                                 "r"(dk[16 * h2 + 8 * e + 5]), "r"(dk[16 * h2 + 8 * e + 6]),
                                                 "r"(dk[16 * h2 + 8 * e + 7]), "l"(pol)
                                                 : "memory");
                            } else {
#pragma unroll
                                for (int e = 0; e < 2; ++e)
                                    asm volatile("st.global.L2::cache_hint.v8.b32 [%0], {%1, %1, %1, %1, %1, %1, %1, %1}, %2;"
                                                 ::"l"(dst + 2048 * h2 + 8 * e), "r"(0u), "l"(pol) : "memory");
                            }
                        }
                    } else if (lane == 0) {
                        atomicOr(p.plan.err, kErrRange);
                    }
                }
            }
            if (failed) break;
            // ---- drain: each warpgroup its 64 channels of dV (bf16 output rows) and of
            // scale * dk^ (FP32 rows for the RoPE^-1 / RMSNorm backward)
            bool ok = true;
            if (lane == 0) ok = tc::mbar_wait(bar(bAccDone), items & 1, abort_flag);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) { fail(); break; }
            ++items;
            tc::fence_after_sync();
            // A thread holds its key row's 64 channels of this half, drained 32 at a time: 64
            // bytes of dV and 128 of scale * dk^ per 32.  Lanes trade 32-byte pieces first
            // (pairs for dV, quads for dk^: one- and two-bit transposes of (lane, piece) by
            // xor shuffles), so that each store instruction writes 16 rows' 64 contiguous
            // bytes of dV, or 8 rows' whole 128-byte lines of dk^.
            const int m = lane & 3;
            const int r0 = 32 * (warp & 3);  // the warp's first row of the tile
#pragma unroll 1
            for (int hq = 0; hq < 2; ++hq) {
                const int ch = 64 * wg + 32 * hq;  // first channel of this 32
                auto row_ptr = [&](int r) {        // row r of the warp's 32, if inside the sample
                    return 128 * it.tile + r0 + r < it.L ? ((size_t)(it.row0 + r0 + r) * p.H + it.h) * kD + ch
                                                         : (size_t)-1;
                };
                {
                    uint32_t r[32];
                    tc::tmem_ld32(tmem + lane_base + 256 + ch, r);
                    tc::tmem_wait_ld_dep(r);
                    uint32_t w[16];  // pieces 0, 1: channels 0-15, 16-31 as bf16 pairs
#pragma unroll
                    for (int e = 0; e < 16; ++e) w[e] = pack_bf16(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
#pragma unroll
                    for (int j = 0; j < 8; ++j) {  // lane 2k + b ends with piece b of rows 2k, 2k + 1
                        const uint32_t send = (m & 1) ? w[j] : w[8 + j];
                        const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 1);
                        if (m & 1) w[j] = recv; else w[8 + j] = recv;
                    }
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const size_t off = row_ptr((lane & ~1) + e);
                        __nv_bfloat16* const d = p.dv + off + 16 * (m & 1);
                        if (off == (size_t)-1) continue;
                        if (p.dv_align32) {
                            asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                                         ::"l"(d), "r"(w[8 * e]), "r"(w[8 * e + 1]), "r"(w[8 * e + 2]), "r"(w[8 * e + 3]),
                                         "r"(w[8 * e + 4]), "r"(w[8 * e + 5]), "r"(w[8 * e + 6]), "r"(w[8 * e + 7])
                                         : "memory");
                        } else {
                            *reinterpret_cast<uint4*>(d) = make_uint4(w[8 * e], w[8 * e + 1], w[8 * e + 2], w[8 * e + 3]);
                            *reinterpret_cast<uint4*>(d + 8) =
                                make_uint4(w[8 * e + 4], w[8 * e + 5], w[8 * e + 6], w[8 * e + 7]);
                        }
                    }
                }
                {
                    uint32_t r[32];  // pieces 0-3: channels 8q .. 8q + 7
                    tc::tmem_ld32(tmem + lane_base + 384 + ch, r);
                    tc::tmem_wait_ld_dep(r);
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * p.scale);
#pragma unroll
                    for (int bit = 1; bit <= 2; bit <<= 1) {  // lane 4k + q ends with piece q of rows 4k .. 4k + 3
#pragma unroll
                        for (int q0 = 0; q0 < 4; ++q0) {
                            if (q0 & bit) continue;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const uint32_t send = (m & bit) ? r[8 * q0 + j] : r[8 * (q0 | bit) + j];
                                const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, bit);
                                if (m & bit) r[8 * q0 + j] = recv; else r[8 * (q0 | bit) + j] = recv;
                            }
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const size_t off = row_ptr((lane & ~3) + e);
                        if (off != (size_t)-1)
                            asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                                         ::"l"(p.dyhat + off + 8 * m), "r"(r[8 * e]), "r"(r[8 * e + 1]), "r"(r[8 * e + 2]),
                                         "r"(r[8 * e + 3]), "r"(r[8 * e + 4]), "r"(r[8 * e + 5]), "r"(r[8 * e + 6]),
                                         "r"(r[8 * e + 7]) : "memory");
                    }
                }
            }
            // the next item's first dV/dK products overwrite the accumulators only after
            // this warpgroup's P^T / dS^T of its first block, which follow in program order
        }
    }

    // the producers have waited out their copies and the issuer its products
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ dQ
//
// 128-key blocks (N = 128 MMAs run at the full rate).  TMEM: S [0, 128),
// dP [128, 256), dQ [256, 384), dS [384, 448).  Four warpgroups split each
// block's 128 key columns (thread = query row, 32 keys each).  The score buffer is refilled
// with block j+1 as soon as both warpgroups have loaded block j; dS (fp16) is
// written to its own TMEM columns and read by the dQ MMAs from there, and is
// rewritten for block j+1 only after dQ(j) completed.  k^ tiles stream through
// a 3-slot ring (held until dQ(j)), v tiles through a 2-slot ring (released
// as soon as dP(j) completed), so the next tiles load while a block is used.
namespace dqt {
constexpr int kThreads = 640;                      // warps 0-3: producer, MMA issuer; 4-19: four warpgroups
constexpr int kOffFixed = 0;                       // q^ + dO tiles
constexpr int kKSlots = 3, kVSlots = 2;
constexpr int kOffK = bwdt::kPair;                 // k^ ring
constexpr int kOffV = kOffK + kKSlots * bwdt::kTile;  // v ring
constexpr int kOffBar = kOffV + kVSlots * bwdt::kTile;
constexpr int kSmem = kOffBar + 256;               // the dynamic shared memory base is 1024-aligned (checked)
enum { bFixedFull = 0, bKFull, bKEmpty = bKFull + kKSlots, bVFull = bKEmpty + kKSlots,
       bVEmpty = bVFull + kVSlots, bSFull = bVEmpty + kVSlots, bSUsed, bPFull, bDsFree, bAccDone, bTail, bDone,
       bNever, bCount };
constexpr uint32_t cDs = 384;
}  // namespace dqt

__global__ void __launch_bounds__(dqt::kThreads, 1)
dq_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
             const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
             const BwdTcParams p) {
    using namespace dqt;
    using bwdt::kHalf;
    using bwdt::kLog2e;
    using bwdt::kPair;
    using bwdt::kTile;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {  // the layout below needs a 1024-byte aligned base
        if (threadIdx.x == 0) atomicOr(p.plan.err, kErrTimeout);
        return;
    }
    uint8_t* smem = smem_raw;
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) { return sbase + kOffBar + 8u * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * bCount);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + 8 * bCount + 4);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        tc::mbar_init(bar(bFixedFull), 1);
        for (int i = 0; i < kKSlots; ++i) {
            tc::mbar_init(bar(bKFull + i), 1);
            tc::mbar_init(bar(bKEmpty + i), 1);
        }
        for (int i = 0; i < kVSlots; ++i) {
            tc::mbar_init(bar(bVFull + i), 1);
            tc::mbar_init(bar(bVEmpty + i), 1);
        }
        tc::mbar_init(bar(bSFull), 1);
        tc::mbar_init(bar(bSUsed), 16);
        tc::mbar_init(bar(bPFull), 16);
        tc::mbar_init(bar(bDsFree), 1);
        tc::mbar_init(bar(bAccDone), 1);
        tc::mbar_init(bar(bTail), 1);
        tc::mbar_init(bar(bDone), 1);
        tc::mbar_init(bar(bNever), 1);  // nothing arrives: the target of a test's stall
        *abort_flag = 0;
        tc::fence_mbar_init();
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
    // 640 threads x 96 registers for every role (no setmaxnreg split)

    if (warp == 0 || warp == 2) {
        // ------------------------------------- TMA producers: warp 0 the fixed q^ / dO
        // tiles and the k^ ring (key rows past the sample end zeroed: dS is 0 there,
        // k^ may not be finite), warp 2 the v ring
        const FixedSpec fx = {&mq, &mdo, sbase + kOffFixed, bar(bFixedFull), bar(bAccDone)};
        const RingSpec r = warp == 0 ? RingSpec{&mk, sbase + kOffK, kKSlots, bar(bKFull), bar(bKEmpty), bar(bTail), true}
                                     : RingSpec{&mv, sbase + kOffV, kVSlots, bar(bVFull), bar(bVEmpty), bar(bTail), false};
        ring_producer(p, r, warp == 0 ? &fx : nullptr, abort_flag, lane, bar(bNever),
                      warp == 0 && p.stall == tc::kStallProducer);
    } else if (warp == 1) {
        // ----------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS16 = tc::idesc_f16(false, false, 128, 128);
            constexpr uint32_t idSbf = tc::idesc_f16(true, false, 128, 128);
            constexpr uint32_t idA16 = tc::idesc_f16(false, true, 128, 128);
            // descriptors are built once; per MMA only the 16-byte start address moves
            const uint64_t dQ = tc::smem_desc_sw128(sbase + kOffFixed, 16, 1024);
            const uint64_t dO = dQ + (kTile >> 4);
            const uint64_t dKr = tc::smem_desc_sw128(sbase + kOffK, 16, 1024);
            const uint64_t dKrMN = tc::smem_desc_sw128(sbase + kOffK, kHalf, 1024);
            const uint64_t dVr = tc::smem_desc_sw128(sbase + kOffV, 16, 1024);
            uint32_t kr = 0, vr = 0, items = 0, cntS = 0;
            // S(j) = q^ k^(j)^T and dP(j) = dO v(j)^T into the score buffer
            auto issue_s = [&]() -> bool {
                const uint32_t ks = kr % kKSlots, vs = vr % kVSlots;
                if (!tc::mbar_wait(bar(bKFull + ks), (kr / kKSlots) & 1, abort_flag)) return false;
                if (!tc::mbar_wait(bar(bVFull + vs), (vr / kVSlots) & 1, abort_flag)) return false;
                tc::fence_after_sync();
                const uint64_t bk = dKr + ((ks * kTile) >> 4), bv = dVr + ((vs * kTile) >> 4);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t koff = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
                    tc::mma_ss(tmem + 0, dQ + koff, bk + koff, idS16, kk > 0);
                }
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t koff = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
                    tc::mma_ss(tmem + 128, dO + koff, bv + koff, idSbf, kk > 0);
                }
                tc::mma_commit(bar(bSFull));
                tc::mma_commit(bar(bVEmpty + vs));  // v(j) is free once dP(j) completed
                ++vr;
                return true;
            };
            for (int k = 0, i = turn_item(0); !failed; i = turn_item(++k)) {
                BwdItem it;
                if (!bwd_item(p, i, it)) break;
                if (!tc::mbar_wait(bar(bFixedFull), items & 1, abort_flag)) { fail(); break; }
                ++items;
                const int nk = (it.L + 127) / 128;
                uint32_t kcur = kr;  // ring index of the k^ tile of block kj
                if (!issue_s()) { fail(); break; }
                ++kr;
                if (p.stall == tc::kStallMma && items == 1 &&
                    !tc::mbar_wait(bar(bNever), 0, abort_flag, p.stall_budget)) {
                    fail();
                    break;
                }
                for (int kj = 0; kj < nk && !failed; ++kj) {
                    // block kj's scores are in registers: refill the buffer with block kj+1
                    if (!tc::mbar_wait(bar(bSUsed), cntS & 1, abort_flag)) { fail(); break; }
                    ++cntS;
                    if (kj + 1 < nk) {
                        if (!issue_s()) { fail(); break; }
                        ++kr;
                    }
                    if (!tc::mbar_wait(bar(bPFull), (cntS - 1) & 1, abort_flag)) { fail(); break; }
                    tc::fence_after_sync();
                    const uint32_t ks = kcur % kKSlots;
                    const uint64_t bk = dKrMN + ((ks * kTile) >> 4);
                    // dQ += dS(j) k^(j): K = the block's 128 keys, dS from TMEM
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc::mma_ts(tmem + 256, tmem + cDs + 8 * kk, bk + ((kk * 2048) >> 4), idA16, (kj > 0) || (kk > 0));
                    tc::mma_commit(bar(bDsFree));
                    tc::mma_commit(bar(bKEmpty + ks));
                    ++kcur;
                }
                if (failed) break;
                tc::mma_commit(bar(bAccDone));
            }
            // every issued MMA has completed before TMEM is released (also on an abort)
            tc::mma_commit(bar(bDone));
            if (!tc::mbar_drain(bar(bDone), 0)) fail();
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------- softmax gradient + drain
        const int wg = (warp - 4) >> 2;                 // key quarter of the score tile
        const int t = tid - 128 * (1 + wg);             // query row of the tile
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t tS = tmem + lane_base + 32 * wg, tDP = tmem + lane_base + 128 + 32 * wg;
        const uint32_t tDs = tmem + lane_base + cDs + 16 * wg;
        const float c = p.scale * kLog2e;
        uint32_t cntS = 0, items = 0, nds = 0;
        for (int k = 0, i = turn_item(0); !failed; i = turn_item(++k)) {
            BwdItem it;
            if (!bwd_item(p, i, it)) break;
            const int nk = (it.L + 127) / 128;
            const bool row_ok = 128 * it.tile + t < it.L;
            const size_t idx = (size_t)it.h * p.seq.S + (row_ok ? it.row0 + t : it.seg0);
            const float lse2 = row_ok ? p.lse[idx] * kLog2e : 0.f;
            const float dlt = row_ok ? p.delta[idx] : 0.f;
            const uint64_t c2 = f2pack(c, c), nl2 = f2pack(-lse2, -lse2), nd2 = f2pack(-dlt, -dlt);
            for (int kj = 0; kj < nk; ++kj) {
                bool ok = true;
                if (lane == 0) {
                    if (p.stall == tc::kStallConsumer && warp == 4 && cntS == 0)
                        ok = tc::mbar_wait(bar(bNever), 0, abort_flag, p.stall_budget);
                    if (ok) ok = tc::mbar_wait(bar(bSFull), cntS & 1, abort_flag);
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) { fail(); break; }
                ++cntS;
                tc::fence_after_sync();
                uint64_t p2[16], d2[16];  // S then P column pairs; dP column pairs
                tc::tmem_ld32_pairs(tS, p2);
                tc::tmem_ld32_pairs(tDP, d2);
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(bar(bSUsed));
                // dS of the previous block must have been read by its dQ MMAs
                if (nds > 0) {
                    bool fr = true;
                    if (lane == 0) fr = tc::mbar_wait(bar(bDsFree), (nds - 1) & 1, abort_flag);
                    fr = __shfl_sync(0xffffffffu, fr, 0);
                    if (!fr) { fail(); break; }
                    tc::fence_after_sync();
                }
                ++nds;
                const int validk = it.L - 128 * kj - 32 * wg;  // keys of this quarter inside the sample
                // P = 2^(s c - lse2); dS = P (dP - Delta), fp16 into TMEM
#pragma unroll
                for (int e = 0; e < 16; ++e) p2[e] = exp2_pair(p2[e], c2, nl2);
                if (validk < 32) {  // tail block: keys past the sample end give exact zeros
#pragma unroll
                    for (int e = 0; e < 16; ++e) p2[e] = mask_pair(p2[e], 2 * e, validk);
                }
                {
                    uint32_t dk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) dk[e] = ds_f16_pair(p2[e], d2[e], nd2);
                    tc::tmem_st16(tDs, dk);
                }
                tc::tmem_wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(bar(bPFull));
            }
            if (failed) break;
            // ---- drain: scale * dq^ as FP32 rows, each warpgroup its 32 channels
            bool ok = true;
            if (lane == 0) ok = tc::mbar_wait(bar(bAccDone), items & 1, abort_flag);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) { fail(); break; }
            ++items;
            tc::fence_after_sync();
            {
                uint32_t r[32];
                tc::tmem_ld32(tmem + lane_base + 256 + 32 * wg, r);
                tc::tmem_wait_ld_dep(r);
                if (row_ok) {
                    float* dst = p.dyhat + ((size_t)(it.row0 + t) * p.H + it.h) * kD + 32 * wg;
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4*>(dst + e) =
                            make_float4(__uint_as_float(r[e]) * p.scale, __uint_as_float(r[e + 1]) * p.scale,
                                        __uint_as_float(r[e + 2]) * p.scale, __uint_as_float(r[e + 3]) * p.scale);
                }
            }
        }
    }

    // the producers have waited out their copies and the issuer its products
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------- dQ from stored dS
//
// When the dK/dV kernel has written every dS^T block (fp16, keys past the
// sample end zero), dq^_i = scale sum_j dS_ij k^_j needs no recomputation of S
// and dP: it is one product per block.  Item = (sample, head, pair of 128-query
// tiles), so each k^ tile is loaded once for two tiles' products.  Warp 0
// loads, per key block j, dS^T(j, i0), dS^T(j, i1) and k^(j) (key rows past the
// sample end zeroed: k^ may not be finite there) into one of two 96 KB stages;
// warp 1 issues dQ0 += dS0 k^ and dQ1 += dS1 k^ (A = a dS^T tile read MN-major
// from its 64-byte swizzled chunks, B = k^ MN-major) into one of two pairs of
// TMEM accumulators; warps 4-7 drain the finished pair as scale * dq^ FP32 rows
// while the next item accumulates.  The sum over j runs in ascending order
// from the sample start.  Bound by HBM: every stored block is read once.
// Warps 8-15 run the row backward (RoPE^-1 + RMSNorm backward, rows_bwd.cuh)
// beside the products: the k tiles first, then the q tiles of this CTA's items
// once the drain has stored their rows, so its row traffic rides on the same
// HBM-bound pass.  Items are dealt round-robin (item i to CTA i mod G): the
// alternating order of the other kernels measured 0.5% slower here.
namespace dqs {
constexpr int kThreads = 512;  // warps 0-1: producer, MMA issuer; 4-7: drain; 8-15: row backward
constexpr int kRingStages = 2;
constexpr int kStage = 3 * bwdt::kTile;  // dS^T of two query tiles + k^: 96 KB
constexpr int kOffBar = kRingStages * kStage;
constexpr int kOffRows = kOffBar + 256;  // the rotary table, then 8 x 128 floats for the row units' sums
constexpr int kSmem = kOffRows + (int)sizeof(RopeTable) + 8 * kD * 4;  // the base is 1024-aligned (checked)
enum { bFull = 0, bEmpty = bFull + kRingStages, bAccFull = bEmpty + kRingStages, bAccEmpty = bAccFull + 2,
       bTail = bAccEmpty + 2, bDone, bNever, bCount };
}  // namespace dqs

struct DqsItem {
    int h, seg0, L, pair, nq, rank;
    bool has1;  // the pair's second query tile exists
};

// Item i over (rank, head, 256-token query pair), samples longest first.
__device__ __forceinline__ bool dqs_item(const BwdTcParams& p, int i, DqsItem& it) {
    const int n = p.seq.n;
    const int* cum = p.plan.cum256;
    if (i >= p.H * cum[n]) return false;
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (p.H * cum[mid] <= i) lo = mid; else hi = mid;
    }
    const int np = cum[lo + 1] - cum[lo];
    const int local = i - p.H * cum[lo];
    const int s = p.plan.order[lo];
    it.h = local / np;
    it.pair = local % np;
    it.seg0 = p.seq.seg[s];
    it.L = p.seq.seg[s + 1] - it.seg0;
    it.nq = (it.L + 127) / 128;
    it.rank = lo;
    it.has1 = 2 * it.pair + 1 < it.nq;
    return true;
}

__global__ void __launch_bounds__(dqs::kThreads, 1)
dq_ds_kernel(const __grid_constant__ CUtensorMap mds, const __grid_constant__ CUtensorMap mk, const BwdTcParams p,
             const __grid_constant__ RopeTable rt, const RowsParams rp) {
    using namespace dqs;
    using bwdt::kHalf;
    using bwdt::kTile;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {  // the layout below needs a 1024-byte aligned base
        if (threadIdx.x == 0) atomicOr(p.plan.err, kErrTimeout);
        return;
    }
    uint8_t* smem = smem_raw;
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) { return sbase + kOffBar + 8u * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * bCount);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + 8 * bCount + 4);
    // the drain warps' count of finished items (4 per item), read by the row warps
    const uint32_t drained = sbase + kOffBar + 8 * bCount + 8;
    volatile int* row_ok = reinterpret_cast<volatile int*>(smem + kOffBar + 8 * bCount + 12);  // [2]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int i = 0; i < kRingStages; ++i) {
            tc::mbar_init(bar(bFull + i), 1);
            tc::mbar_init(bar(bEmpty + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(bar(bAccFull + i), 1);
            tc::mbar_init(bar(bAccEmpty + i), 4);
        }
        tc::mbar_init(bar(bTail), 1);
        tc::mbar_init(bar(bDone), 1);
        tc::mbar_init(bar(bNever), 1);  // nothing arrives: the target of a test's stall
        *abort_flag = 0;
        *reinterpret_cast<volatile uint32_t*>(smem + kOffBar + 8 * bCount + 8) = 0;
        tc::fence_mbar_init();
        tc::prefetch_map(&mds);
        tc::prefetch_map(&mk);
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

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        const uint64_t pol = tc::policy_evict_first();
        uint32_t blk = 0, tails = 0;
        // copies issued (lane 0): stages whose full barrier was armed, and a tail stage
        // whose own wait gave up with its copies possibly in flight
        uint32_t armed = 0;
        bool tail_pending = false, first = true;
        for (int i = blockIdx.x; !failed; i += gridDim.x, first = false) {
            DqsItem it;
            if (!dqs_item(p, i, it)) break;
            const long long base = (long long)p.H * p.plan.cumsq[it.rank] + (long long)it.h * it.nq * it.nq;
            for (int j = 0; j < it.nq && !failed; ++j, ++blk) {
                const uint32_t s = blk % kRingStages, ph = (blk / kRingStages) & 1;
                const uint32_t dst = sbase + s * kStage;
                const int valid = it.L - 128 * j;
                const bool tail = valid < 128;
                if (lane == 0) {
                    if (p.stall == tc::kStallProducer && first && j == 0 &&
                        !tc::mbar_wait(bar(bNever), 0, abort_flag, p.stall_budget))
                        fail();
                    if (!failed && !tc::mbar_wait(bar(bEmpty + s), ph ^ 1, abort_flag)) fail();
                    if (!failed) {
                        const uint32_t b = tail ? bar(bTail) : bar(bFull + s);
                        const int b0 = (int)(base + (long long)j * it.nq + 2 * it.pair);
                        tc::mbar_expect_tx(b, (it.has1 ? 3 : 2) * kTile);
                        for (int hf = 0; hf < 2; ++hf) {
                            // chunks 2 hf, 2 hf + 1 (queries 64 hf .. 64 hf + 63), read once
                            tc::tma_load_4d_hint(dst + hf * kHalf, &mds, 0, 0, 2 * hf, b0, b, pol);
                            if (it.has1) tc::tma_load_4d_hint(dst + kTile + hf * kHalf, &mds, 0, 0, 2 * hf, b0 + 1, b, pol);
                            tc::tma_load_2d(dst + 2 * kTile + hf * kHalf, &mk, it.h * 128 + 64 * hf, it.seg0 + 128 * j, b);
                        }
                        if (!tail) ++armed;
                        if (tail && !tc::mbar_wait(bar(bTail), tails & 1, abort_flag)) {
                            tail_pending = true;
                            fail();
                        }
                    }
                }
                failed = __shfl_sync(0xffffffffu, failed, 0);
                if (tail && !failed) {
                    ++tails;
                    for (int hf = 0; hf < 2; ++hf) zero_rows(dst + 2 * kTile + hf * kHalf, valid, 128, lane);
                    tc::fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) {
                        tc::mbar_arrive(bar(bFull + s));
                        ++armed;
                    }
                }
            }
        }
        // every copy issued has landed before the CTA's shared memory is released
        if (lane == 0) {
            bool ok = tc::drain_ring(bar(bFull), kRingStages, armed);
            if (tail_pending) ok &= tc::mbar_drain(bar(bTail), tails & 1);
            if (!ok) atomicOr(p.plan.err, kErrTimeout);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t id = tc::idesc_f16_amn(false, true, 128, 128);  // fp16, A and B MN-major
            // A: a dS^T tile as [32-query chunk][key][32 queries], 64-byte swizzled: atoms of
            // 8 keys x 32 queries (512 bytes), 8 KB from one chunk to the next
            const uint64_t dA = tc::smem_desc_sw64(sbase, 128 * 64, 512);
            const uint64_t dB = tc::smem_desc_sw128(sbase + 2 * kTile, kHalf, 1024);
            uint32_t blk = 0, items = 0;
            for (int i = blockIdx.x; !failed; i += gridDim.x, ++items) {
                DqsItem it;
                if (!dqs_item(p, i, it)) break;
                const uint32_t b = items & 1;
                // the epilogue has drained this accumulator pair (two items ago)
                if (items >= 2 && !tc::mbar_wait(bar(bAccEmpty + b), ((items >> 1) - 1) & 1, abort_flag)) {
                    fail();
                    break;
                }
                tc::fence_after_sync();
                for (int j = 0; j < it.nq; ++j, ++blk) {
                    const uint32_t s = blk % kRingStages;
                    if (!tc::mbar_wait(bar(bFull + s), (blk / kRingStages) & 1, abort_flag)) { fail(); break; }
                    tc::fence_after_sync();
                    const uint32_t so = (s * kStage) >> 4;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)  // 16 keys per step: 1 KB of A, 2 KB of B
                        tc::mma_ss(tmem + 256 * b, dA + so + ((kk * 1024) >> 4), dB + so + ((kk * 2048) >> 4), id,
                                   (j > 0) || (kk > 0));
                    if (it.has1) {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            tc::mma_ss(tmem + 256 * b + 128, dA + so + ((kTile + kk * 1024) >> 4),
                                       dB + so + ((kk * 2048) >> 4), id, (j > 0) || (kk > 0));
                    }
                    tc::mma_commit(bar(bEmpty + s));
                    if (p.stall == tc::kStallMma && items == 0 && j == 0 &&
                        !tc::mbar_wait(bar(bNever), 0, abort_flag, p.stall_budget)) {
                        fail();
                        break;
                    }
                }
                if (failed) break;
                tc::mma_commit(bar(bAccFull + b));
            }
            // every issued MMA has completed before TMEM is released (also on an abort)
            tc::mma_commit(bar(bDone));
            if (!tc::mbar_drain(bar(bDone), 0)) fail();
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------- drain
        const int t = tid - 128;  // TMEM lane == query row of each tile
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        uint32_t items = 0;
        for (int i = blockIdx.x; !failed; i += gridDim.x, ++items) {
            DqsItem it;
            if (!dqs_item(p, i, it)) break;
            const uint32_t b = items & 1;
            bool ok = true;
            if (lane == 0) {
                if (p.stall == tc::kStallConsumer && warp == 4 && items == 0)
                    ok = tc::mbar_wait(bar(bNever), 0, abort_flag, p.stall_budget);
                if (ok) ok = tc::mbar_wait(bar(bAccFull + b), (items >> 1) & 1, abort_flag);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) { fail(); break; }
            tc::fence_after_sync();
            // A thread holds its query row; lanes trade 32-byte pieces within quads (a
            // two-bit transpose of (lane, piece) by xor shuffles), so that each store
            // instruction writes 8 rows' whole 128-byte lines of a 32-column chunk
            // instead of 16 bytes of 32 rows.
            const int m = lane & 3;
            for (int u = 0; u < (it.has1 ? 2 : 1); ++u) {
#pragma unroll
                for (int c32 = 0; c32 < 4; ++c32) {
                    uint32_t r[32];  // pieces 0-3: columns 8q .. 8q + 7 of the chunk
                    tc::tmem_ld32(tmem + lane_base + 256 * b + 128 * u + 32 * c32, r);
                    tc::tmem_wait_ld_dep(r);
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * p.scale);
#pragma unroll
                    for (int bit = 1; bit <= 2; bit <<= 1) {  // lane 4k + q ends with piece q of rows 4k .. 4k + 3
#pragma unroll
                        for (int q0 = 0; q0 < 4; ++q0) {
                            if (q0 & bit) continue;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const uint32_t send = (m & bit) ? r[8 * q0 + j] : r[8 * (q0 | bit) + j];
                                const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, bit);
                                if (m & bit) r[8 * q0 + j] = recv; else r[8 * (q0 | bit) + j] = recv;
                            }
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int r_in = 256 * it.pair + 128 * u + (t - lane) + (lane & ~3) + e;  // row within the sample
                        if (r_in >= it.L) continue;
                        float* const d = p.dyhat + ((size_t)(it.seg0 + r_in) * p.H + it.h) * kD + 32 * c32 + 8 * m;
                        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                                     ::"l"(d), "r"(r[8 * e]), "r"(r[8 * e + 1]), "r"(r[8 * e + 2]), "r"(r[8 * e + 3]),
                                     "r"(r[8 * e + 4]), "r"(r[8 * e + 5]), "r"(r[8 * e + 6]), "r"(r[8 * e + 7])
                                     : "memory");
                    }
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                tc::mbar_arrive(bar(bAccEmpty + b));
                // this warp's scale * dq^ rows of the item are stored: the row warps may read them
                asm volatile("red.release.cta.shared::cta.add.u32 [%0], 1;" :: "r"(drained) : "memory");
            }
        }
    } else if (warp >= 8) {
        // ------------------------------------- row backward (RoPE^-1 + RMSNorm): first
        // the k tiles (scale * dk^ is complete when the launch starts; CTA c takes
        // units c, c + G, ...), then the q tiles of this CTA's own items, each once the
        // drain has stored its rows.  The 8 warps run one unit at a time, joined by
        // named barrier 1; only warp 8 polls the drain count and the others take its
        // answer from shared memory, so all 8 leave together when it gives up.
        RopeTable& srt = *reinterpret_cast<RopeTable*>(smem + kOffRows);
        float* red = reinterpret_cast<float*>(smem + kOffRows + sizeof(RopeTable));
        const int w8 = warp - 8;
        auto sync = [] { asm volatile("bar.sync 1, 256;" ::: "memory"); };
        rope_to_smem(rt, srt, tid - 256, 256);
        sync();
        const int units = p.H * p.plan.cum128[p.seq.n];
        for (int u = blockIdx.x; u < units; u += gridDim.x) rows_unit(srt, rp, 1, u / p.H, u % p.H, w8, lane, red, sync);
        uint32_t items = 0;
        for (int i = blockIdx.x;; i += gridDim.x, ++items) {
            DqsItem it;
            if (!dqs_item(p, i, it)) break;
            if (warp == 8 && lane == 0) {
                const uint32_t target = 4 * (items + 1);
                const long long t0 = clock64();
                int ok = 1;
                while (true) {
                    uint32_t v;
                    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(drained) : "memory");
                    if (v >= target) break;
                    if (*abort_flag || clock64() - t0 > tc::kWaitBudget) { ok = 0; break; }
                    __nanosleep(64);
                }
                row_ok[items & 1] = ok;
            }
            sync();
            if (!row_ok[items & 1]) {  // the same answer in every row warp
                if (warp == 8 && lane == 0) fail();
                break;
            }
            const int t0 = p.plan.cum128[it.rank] + 2 * it.pair;
            rows_unit(srt, rp, 0, t0, it.h, w8, lane, red, sync);
            if (it.has1) rows_unit(srt, rp, 0, t0 + 1, it.h, w8, lane, red, sync);
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
bool encode_rows_b(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int H, int S, int rows) {
    const cuuint64_t dims[2] = {(cuuint64_t)H * kD, (cuuint64_t)S};
    const cuuint64_t strides[1] = {(cuuint64_t)H * kD * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)rows};
    const cuuint32_t es[2] = {1, 1};
    return tensor_map_encoder()(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct BwdMaps {
    CUtensorMap q, k, v, dout;
};

// q^ and dO streamed in 64-row blocks with k^, v as 128-row tiles (dkdv), or
// the other way round (dq).
bool encode_all(BwdMaps& m, const Problem& p, const Workspace& ws, const __nv_bfloat16* dout, int qrows, int krows) {
    return encode_rows_b(&m.q, ws.qhat, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p.H, p.seq.S, qrows) &&
           encode_rows_b(&m.k, ws.khat, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p.H, p.seq.S, krows) &&
           encode_rows_b(&m.v, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.H, p.seq.S, krows) &&
           encode_rows_b(&m.dout, dout, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.H, p.seq.S, qrows);
}
}  // namespace

cudaError_t set_bwd_attributes() {
    cudaError_t e = cudaFuncSetAttribute(dkdv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kvt::kSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dqt::kSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(dq_ds_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dqs::kSmem);
    return e;
}

static BwdTcParams bwd_params(const Problem& p, const Workspace& ws, const float* lse) {
    BwdTcParams b;
    b.seq = p.seq;
    b.plan = ws.plan;
    b.H = p.H;
    b.scale = p.scale;
    b.lse = lse;
    b.delta = ws.delta;
    b.ds = ws.ds;
    b.ds_blocks = ws.ds_blocks;
    b.dv_align32 = 0;
    b.stall = 0;
    b.stall_budget = p.stall.budget;
    return b;
}

cudaError_t launch_bwd_dkdv(const Problem& p, const Workspace& ws, const float* lse,
                            const __nv_bfloat16* dout, __nv_bfloat16* dk, __nv_bfloat16* dv, cudaStream_t st) {
    BwdMaps m;
    if (!encode_all(m, p, ws, dout, 128, 128)) return cudaErrorInvalidValue;
    BwdTcParams b = bwd_params(p, ws, lse);
    b.dv = dv;
    b.dv_align32 = (reinterpret_cast<uintptr_t>(dv) & 31u) == 0;
    b.dyhat = ws.dkhat32;
    if (p.stall.kernel == kStallKernelDkdv) b.stall = p.stall.role;
    const int sms = device_sms();
    if (sms < 1) return cudaErrorNotSupported;
    dkdv_tc_kernel<<<sms, kvt::kThreads, kvt::kSmem, st>>>(m.q, m.k, m.v, m.dout, b);
    return cudaGetLastError();
}

cudaError_t launch_bwd_dq(const Problem& p, const Workspace& ws, const float* lse, const __nv_bfloat16* dout,
                          const RopeTable* rope, __nv_bfloat16* dq, __nv_bfloat16* dk, cudaStream_t st) {
    BwdMaps m;
    if (!encode_all(m, p, ws, dout, 128, 128)) return cudaErrorInvalidValue;
    BwdTcParams b = bwd_params(p, ws, lse);
    const int sms = device_sms();
    if (sms < 1) return cudaErrorNotSupported;
    b.dv = nullptr;
    b.dyhat = ws.dqhat32;
    if (p.stall.kernel == kStallKernelDq) b.stall = p.stall.role;
    if (ws.ds) {  // dS was stored by the dK/dV kernel: dQ is one product per block
        // a block is [32-query chunk][key][32 queries] (query in chunk, key, chunk, block);
        // a box of 2 chunks lands in shared memory in the same order, 64-byte swizzled
        CUtensorMap mds;
        const cuuint64_t dims[4] = {32, 128, 4, (cuuint64_t)ws.ds_blocks};
        const cuuint64_t strides[3] = {32 * 2, 128 * 32 * 2, 128 * 128 * 2};
        const cuuint32_t box[4] = {32, 128, 2, 1};
        const cuuint32_t es[4] = {1, 1, 1, 1};
        if (tensor_map_encoder()(&mds, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, ws.ds, dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        // the row backward's cos / sin table first: the dQ kernel runs those rows too
        const cudaError_t e = launch_rope_table(p, ws, rope, st);
        if (e != cudaSuccess) return e;
        dq_ds_kernel<<<sms, dqs::kThreads, dqs::kSmem, st>>>(mds, m.k, b, *rope, make_rows_params(p, ws, dq, dk));
        return cudaGetLastError();
    }
    dq_tc_kernel<<<sms, dqt::kThreads, dqt::kSmem, st>>>(m.q, m.k, m.v, m.dout, b);
    return cudaGetLastError();
}

}  // namespace h3
