// plan.cu -- the per-call plan.
//
// The plan kernel checks the segment offsets on the device and orders the
// samples longest first (so the attention kernels start their longest work
// first); the order only decides which CTA runs a tile, never the arithmetic.
// It also writes, in that order, the prefix sums of each sample's tiles of 64,
// 128 and 256 tokens and of its squared 128-token tile count (the 128 x 128
// score blocks of one head), which the kernels use to map a work item to its
// sample and the stored dS blocks to their place.
#include "common.cuh"

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

}  // namespace h3
