// prologue.cu -- the q/k norm + RoPE prologue (K1).
//
// The prologue rotates and normalises q and k once per (token, head) into the
// fp16 workspaces q^ and k^ that the attention kernels stream with TMA or
// cp.async.  It is bound by HBM bandwidth: 8 bytes moved per q/k element pair
// read + written (2 B read and 2 B written for each of q and k).
#include "common.cuh"
#include "rowops.cuh"

namespace h3 {

// ------------------------------------------------------------------ K1

constexpr int kProWarps = 8;
constexpr int kProCtas = 4;   // resident CTAs per SM (the register budget)
constexpr int kProBatch = 4;  // heads per half-iteration; the next batch's rows load while one is computed

__global__ void __launch_bounds__(kProWarps * 32, kProCtas)
prologue_kernel(Problem p, __half* __restrict__ qhat, __half* __restrict__ khat,
                const __grid_constant__ RopeTable rt, unsigned* err) {
    __shared__ RopeTable srt;
    rope_to_smem(rt, srt, threadIdx.x, blockDim.x);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int tok = blockIdx.x * kProWarps + (threadIdx.x >> 5);
    if (tok >= p.seq.S) return;
    const __nv_bfloat16* __restrict__ q = p.q;
    const __nv_bfloat16* __restrict__ k = p.k;
    const int H = p.H;
    const size_t base = (size_t)tok * H * kD + 4 * lane;
    const size_t src = p.rowmap ? (size_t)p.rowmap[tok] * H * kD + 4 * lane : base;
    // the lane's four bf16 channels of head h of q and k, as they are in memory
    auto load = [&](int h, uint2& rq, uint2& rk) {
        if (h < H) {
            rq = *reinterpret_cast<const uint2*>(q + src + (size_t)h * kD);
            rk = *reinterpret_cast<const uint2*>(k + src + (size_t)h * kD);
        }
    };
    uint2 aq[kProBatch], ak[kProBatch], bq[kProBatch], bk[kProBatch];
#pragma unroll
    for (int b = 0; b < kProBatch; ++b) load(b, aq[b], ak[b]);
    // the lane's rotary entries, the token's angles and the weights while the first rows load
    const LaneRope lr = lane_rope(srt, lane);
    const RowAngles ang = row_angles(lr, p.seq.pos_t[tok], p.seq.pos_h[tok], p.seq.pos_w[tok]);
    float wq[4], wk[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) { wq[e] = p.wq[4 * lane + e]; wk[e] = p.wk[4 * lane + e]; }
    bool ok = true;
    auto rotate = [&](int h, uint2 rq, uint2 rk) {
        if (h >= H) return;
        float x[4], y[4];
        x[0] = bf16_lo(rq.x); x[1] = bf16_hi(rq.x); x[2] = bf16_lo(rq.y); x[3] = bf16_hi(rq.y);
        row_norm_rope(x, wq, ang, lr, p.eps, y);
        ok &= store_row4_f16(qhat + base + (size_t)h * kD, y);
        x[0] = bf16_lo(rk.x); x[1] = bf16_hi(rk.x); x[2] = bf16_lo(rk.y); x[3] = bf16_hi(rk.y);
        row_norm_rope(x, wk, ang, lr, p.eps, y);
        ok &= store_row4_f16(khat + base + (size_t)h * kD, y);
    };
    // software pipeline: the next kProBatch heads' rows load while these are computed
    for (int h0 = 0; h0 < H; h0 += 2 * kProBatch) {
#pragma unroll
        for (int b = 0; b < kProBatch; ++b) load(h0 + kProBatch + b, bq[b], bk[b]);
#pragma unroll
        for (int b = 0; b < kProBatch; ++b) rotate(h0 + b, aq[b], ak[b]);
#pragma unroll
        for (int b = 0; b < kProBatch; ++b) load(h0 + 2 * kProBatch + b, aq[b], ak[b]);
#pragma unroll
        for (int b = 0; b < kProBatch; ++b) rotate(h0 + kProBatch + b, bq[b], bk[b]);
    }
    if (!ok) atomicOr(err, kErrRange);
}

cudaError_t launch_prologue(const Problem& p, const Workspace& ws, const RopeTable* rope, cudaStream_t st) {
    if (p.seq.S == 0) return cudaSuccess;
    const int blocks = (p.seq.S + kProWarps - 1) / kProWarps;
    prologue_kernel<<<blocks, kProWarps * 32, 0, st>>>(p, ws.qhat, ws.khat, *rope, ws.plan.err);
    return cudaGetLastError();
}

}  // namespace h3
