// prologue.cu -- per-call plan and the q/k norm + RoPE prologue (K1).
//
// The plan kernel checks the segment offsets on the device and orders the
// samples longest first (so the attention kernels start their longest work
// first); the order only decides which CTA runs a tile, never the arithmetic.
//
// The prologue rotates and normalises q and k once per (token, head) into the
// fp16 workspaces q^ and k^ that the attention kernels stream with TMA or
// cp.async.  It is bound by HBM bandwidth: 8 bytes moved per q/k element pair
// read + written (2 B read and 2 B written for each of q and k).
#include "common.cuh"
#include "rowops.cuh"

namespace h3 {

constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(Seq seq, Plan plan) {
    const int n = seq.n;
    const int tid = threadIdx.x;
    __shared__ int bad;
    __shared__ int scan64[kPlanThreads], scan128[kPlanThreads], scan256[kPlanThreads], scansq[kPlanThreads];
    if (tid == 0) bad = (seq.seg[0] != 0) || (seq.seg[n] != seq.S);
    __syncthreads();
    for (int s = tid; s < n; s += kPlanThreads)
        if (seq.seg[s + 1] <= seq.seg[s]) atomicOr(&bad, 1);
    __syncthreads();
    if (bad) {
        if (tid == 0) atomicOr(plan.err, kErrBadOffsets);
        for (int r = tid; r <= n; r += kPlanThreads) {
            plan.cum64[r] = 0;
            plan.cum128[r] = 0;
            plan.cum256[r] = 0;
            plan.cumsq[r] = 0;
        }
        return;
    }
    // rank: longer samples first, ties by index
    for (int s = tid; s < n; s += kPlanThreads) {
        int L = seq.seg[s + 1] - seq.seg[s];
        int rank = 0;
        for (int u = 0; u < n; ++u) {
            int Lu = seq.seg[u + 1] - seq.seg[u];
            rank += (Lu > L) || (Lu == L && u < s);
        }
        plan.order[rank] = s;
        plan.rank_of[s] = rank;
    }
    __syncthreads();
    // exclusive prefix sums of tile counts in rank order (integer: exact)
    const int chunk = (n + kPlanThreads - 1) / kPlanThreads;
    const int r0 = min(n, tid * chunk), r1 = min(n, r0 + chunk);
    int c64 = 0, c128 = 0, c256 = 0, csq = 0;
    for (int r = r0; r < r1; ++r) {
        int s = plan.order[r];
        int L = seq.seg[s + 1] - seq.seg[s];
        c64 += (L + 63) / 64;
        c128 += (L + 127) / 128;
        c256 += (L + 255) / 256;
        csq += ((L + 127) / 128) * ((L + 127) / 128);
    }
    scan64[tid] = c64;
    scan128[tid] = c128;
    scan256[tid] = c256;
    scansq[tid] = csq;
    __syncthreads();
    for (int off = 1; off < kPlanThreads; off <<= 1) {
        int a = tid >= off ? scan64[tid - off] : 0;
        int b = tid >= off ? scan128[tid - off] : 0;
        int c = tid >= off ? scan256[tid - off] : 0;
        int d = tid >= off ? scansq[tid - off] : 0;
        __syncthreads();
        scan64[tid] += a;
        scan128[tid] += b;
        scan256[tid] += c;
        scansq[tid] += d;
        __syncthreads();
    }
    c64 = scan64[tid] - c64;
    c128 = scan128[tid] - c128;
    c256 = scan256[tid] - c256;
    csq = scansq[tid] - csq;
    for (int r = r0; r < r1; ++r) {
        int s = plan.order[r];
        int L = seq.seg[s + 1] - seq.seg[s];
        plan.cum64[r] = c64;
        plan.cum128[r] = c128;
        plan.cum256[r] = c256;
        plan.cumsq[r] = csq;
        c64 += (L + 63) / 64;
        c128 += (L + 127) / 128;
        c256 += (L + 255) / 256;
        csq += ((L + 127) / 128) * ((L + 127) / 128);
    }
    if (tid == kPlanThreads - 1) {
        plan.cum64[n] = scan64[tid];
        plan.cum128[n] = scan128[tid];
        plan.cum256[n] = scan256[tid];
        plan.cumsq[n] = scansq[tid];
    }
}

cudaError_t launch_plan(const Problem& p, const Workspace& ws, cudaStream_t st) {
    plan_kernel<<<1, kPlanThreads, 0, st>>>(p.seq, ws.plan);
    return cudaGetLastError();
}

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
