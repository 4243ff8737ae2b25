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
constexpr int kProBatch = 4;  // heads loaded ahead per warp

__global__ void __launch_bounds__(kProWarps * 32, 4)
prologue_kernel(Problem p, __half* __restrict__ qhat, __half* __restrict__ khat,
                const __grid_constant__ RopeTable rt, unsigned* err) {
    __shared__ RopeTable srt;
    rope_to_smem(rt, srt, threadIdx.x, blockDim.x);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int tok = blockIdx.x * kProWarps + (threadIdx.x >> 5);
    if (tok >= p.seq.S) return;
    const LaneRope lr = lane_rope(srt, lane);
    const RowAngles ang = row_angles(lr, p.seq.pos_t[tok], p.seq.pos_h[tok], p.seq.pos_w[tok]);
    float wq[4], wk[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) { wq[e] = p.wq[4 * lane + e]; wk[e] = p.wk[4 * lane + e]; }
    const __nv_bfloat16* __restrict__ q = p.q;
    const __nv_bfloat16* __restrict__ k = p.k;
    const size_t base = (size_t)tok * p.H * kD + 4 * lane;
    const size_t src = p.rowmap ? (size_t)p.rowmap[tok] * p.H * kD + 4 * lane : base;
    bool ok = true;
    for (int h0 = 0; h0 < p.H; h0 += kProBatch) {
        float xq[kProBatch][4], xk[kProBatch][4];
#pragma unroll
        for (int b = 0; b < kProBatch; ++b)
            if (h0 + b < p.H) {
                load_row4(q + src + (size_t)(h0 + b) * kD, xq[b]);
                load_row4(k + src + (size_t)(h0 + b) * kD, xk[b]);
            }
#pragma unroll
        for (int b = 0; b < kProBatch; ++b)
            if (h0 + b < p.H) {
                float y[4];
                row_norm_rope(xq[b], wq, ang, lr, p.eps, y);
                ok &= store_row4_f16(qhat + base + (size_t)(h0 + b) * kD, y);
                row_norm_rope(xk[b], wk, ang, lr, p.eps, y);
                ok &= store_row4_f16(khat + base + (size_t)(h0 + b) * kD, y);
            }
    }
    if (!ok) atomicOr(err, kErrRange);
}

cudaError_t launch_prologue(const Problem& p, const Workspace& ws, const RopeTable* rope, cudaStream_t st) {
    if (p.seq.S == 0) return cudaSuccess;
    int blocks = (p.seq.S + kProWarps - 1) / kProWarps;
    prologue_kernel<<<blocks, kProWarps * 32, 0, st>>>(p, ws.qhat, ws.khat, *rope, ws.plan.err);
    return cudaGetLastError();
}

}  // namespace h3
