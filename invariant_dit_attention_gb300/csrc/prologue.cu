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
//
// One warp per token, two rows (heads) at a time, one per half-warp.  Lane j of a
// half holds channels 4j .. 4j + 3 (group A) and 4j + 64 .. 4j + 67 (group B):
// the two groups that lanes j and j + 16 hold in the one-row-per-warp layout of
// rowops.cuh.  The row's sum of squares therefore keeps that layout's tree - its
// first butterfly step (lanes 16 apart) is the lane's own sum of its two groups,
// the remaining steps (8, 4, 2, 1) stay inside the half - so q^ / k^ are the same
// bits as the one-row-per-warp form and the fused QKV epilogue.  Half the
// reduction steps and half the 1/sqrt evaluations per row, and group B needs no
// partner exchange when no channel above 64 is rotated (the 16/24/24 sections).

constexpr int kProWarps = 8;
// resident CTAs per SM (the register budget) and head pairs per half-iteration (the
// next batch's rows load while one is computed), per rotary layout (kMode below)
template <int kMode>
struct ProCfg {
    static constexpr int ctas = 2, batch = 2;
};
template <>
struct ProCfg<0> {
    static constexpr int ctas = 3, batch = 1;
};

namespace {
// where a group finds its rotary partner: the partner's half-lane and group
struct PairSrc {
    int lane;   // lane of the partner (same half-warp)
    bool in_b;  // the partner is that lane's group B
};

__device__ __forceinline__ PairSrc pair_src(const RopeTable& rt, int group, int half) {
    const int pg = rt.partner[group];
    return PairSrc{16 * half + (pg & 15), pg >= 16};
}

// sum of squares of the row, its tree as warp_sum's over the one-row-per-warp layout
__device__ __forceinline__ float half_row_sumsq(const float (&a)[4], const float (&b)[4]) {
    float v = sq4(a[0], a[1], a[2], a[3]) + sq4(b[0], b[1], b[2], b[3]);
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    return v;
}

// the rotation of one group from its normed values z and its partner's zp
__device__ __forceinline__ void rope_group(const float (&z)[4], const float (&zp)[4], const LaneRope& lr,
                                           const RowAngles& a, float (&y)[4]) {
    if (lr.axis < 0) {
#pragma unroll
        for (int e = 0; e < 4; ++e) y[e] = z[e];
    } else if (!lr.second) {
#pragma unroll
        for (int e = 0; e < 4; ++e) y[e] = rope_u(z[e], zp[e], a.c[e], a.s[e]);
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) y[e] = rope_v(zp[e], z[e], a.c[e], a.s[e]);
    }
}

__device__ __forceinline__ void unpack4(uint2 u, float (&x)[4]) {
    x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
}

__device__ __forceinline__ void store4_f16(__half* p, const float (&y)[4]) {
    uint2 u;
    u.x = pack_f16(y[0], y[1]);
    u.y = pack_f16(y[2], y[3]);
    *reinterpret_cast<uint2*>(p) = u;
}

// false if the four values are finite and one of them is beyond the fp16 range
// (non-finite values are not range errors); y - y is 0 for a finite y, else NaN
__device__ __forceinline__ bool f16_range_ok(const float (&y)[4]) {
    const float m = fmaxf(fmaxf(fabsf(y[0]), fabsf(y[1])), fmaxf(fabsf(y[2]), fabsf(y[3])));
    const float t = ((y[0] - y[0]) + (y[1] - y[1])) + ((y[2] - y[2]) + (y[3] - y[3]));
    return m <= 65504.f || t != 0.f;
}
}  // namespace

// kMode: 0 = no channel above 64 rotated, 1 = some are, pairs inside each group,
// 2 = a section crosses channel 64 (a partner may sit in the other group)
template <int kMode>
__global__ void __launch_bounds__(kProWarps * 32, ProCfg<kMode>::ctas)
prologue_kernel(Problem p, __half* __restrict__ qhat, __half* __restrict__ khat,
                const __grid_constant__ RopeTable rt, unsigned* err) {
    __shared__ RopeTable srt;
    rope_to_smem(rt, srt, threadIdx.x, blockDim.x);
    __syncthreads();
    const int lane = threadIdx.x & 31, half = lane >> 4, j = lane & 15;
    const int tok = blockIdx.x * kProWarps + (threadIdx.x >> 5);
    if (tok >= p.seq.S) return;
    const __nv_bfloat16* __restrict__ q = p.q;
    const __nv_bfloat16* __restrict__ k = p.k;
    const int H = p.H;
    // the half's head of pair i is 2 i + half; its row at base (+ h * 128)
    const size_t base = (size_t)tok * H * kD + 4 * j;
    const size_t src = p.rowmap ? (size_t)p.rowmap[tok] * H * kD + 4 * j : base;
    // the lane's two groups of head 2 i + half of q and k, as they are in memory
    auto load = [&](int i, uint2 (&rq)[2], uint2 (&rk)[2]) {
        const int h = 2 * i + half;
        if (h < H) {
            const size_t o = src + (size_t)h * kD;
            rq[0] = *reinterpret_cast<const uint2*>(q + o);
            rq[1] = *reinterpret_cast<const uint2*>(q + o + 64);
            rk[0] = *reinterpret_cast<const uint2*>(k + o);
            rk[1] = *reinterpret_cast<const uint2*>(k + o + 64);
        }
    };
    const int pairs = (H + 1) / 2;
    uint2 aq[ProCfg<kMode>::batch][2], ak[ProCfg<kMode>::batch][2], bq[ProCfg<kMode>::batch][2], bk[ProCfg<kMode>::batch][2];
#pragma unroll
    for (int b = 0; b < ProCfg<kMode>::batch; ++b) load(b, aq[b], ak[b]);
    // the lanes' rotary entries, the token's angles and the weights while the first rows load
    const LaneRope la = lane_rope(srt, j);
    LaneRope lb = lane_rope(srt, j + 16);
    if (kMode == 0) lb.axis = -1;
    const PairSrc sa = pair_src(srt, j, half), sb = pair_src(srt, j + 16, half);
    const int pt = p.seq.pos_t[tok], ph = p.seq.pos_h[tok], pw = p.seq.pos_w[tok];
    const RowAngles ga = row_angles(la, pt, ph, pw), gb = row_angles(lb, pt, ph, pw);
    float wq[2][4], wk[2][4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        wq[0][e] = p.wq[4 * j + e]; wq[1][e] = p.wq[4 * j + 64 + e];
        wk[0][e] = p.wk[4 * j + e]; wk[1][e] = p.wk[4 * j + 64 + e];
    }
    // The rows are normed to at most sqrt(128) per channel and the rotations keep a
    // pair's length, so |q^|, |k^| <= sqrt(128) max|w| (to rounding): below 16 max|w|
    // < 60000 no value can leave the fp16 range and the per-value check is skipped.
    float mw = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e)
        mw = fmaxf(mw, fmaxf(fmaxf(fabsf(wq[0][e]), fabsf(wq[1][e])), fmaxf(fabsf(wk[0][e]), fabsf(wk[1][e]))));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, o));
    const bool check = !(16.f * mw < 60000.f);
    bool ok = true;
    auto rotate_row = [&](const uint2 (&r)[2], const float (&w)[2][4], __half* out, bool live) {
        float xa[4], xb[4];
        unpack4(r[0], xa);
        unpack4(r[1], xb);
        const float rs = rstd_of(half_row_sumsq(xa, xb), p.eps);
        float za[4], zb[4], pa[4], pb[4], ya[4], yb[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) { za[e] = norm_w(xa[e], rs, w[0][e]); zb[e] = norm_w(xb[e], rs, w[1][e]); }
        if (kMode != 2) {
#pragma unroll
            for (int e = 0; e < 4; ++e) pa[e] = __shfl_sync(0xffffffffu, za[e], sa.lane);
            if (kMode == 1) {
#pragma unroll
                for (int e = 0; e < 4; ++e) pb[e] = __shfl_sync(0xffffffffu, zb[e], sb.lane);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) pb[e] = zb[e];
            }
        } else {  // a section crosses channel 64: a partner may sit in the other group
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float a0 = __shfl_sync(0xffffffffu, za[e], sa.lane), a1 = __shfl_sync(0xffffffffu, zb[e], sa.lane);
                const float b0 = __shfl_sync(0xffffffffu, za[e], sb.lane), b1 = __shfl_sync(0xffffffffu, zb[e], sb.lane);
                pa[e] = sa.in_b ? a1 : a0;
                pb[e] = sb.in_b ? b1 : b0;
            }
        }
        rope_group(za, pa, la, ga, ya);
        rope_group(zb, pb, lb, gb, yb);
        if (live) {
            store4_f16(out, ya);
            store4_f16(out + 64, yb);
            if (check) ok &= f16_range_ok(ya) && f16_range_ok(yb);
        }
    };
    auto rotate = [&](int i, const uint2 (&rq)[2], const uint2 (&rk)[2]) {
        if (i >= pairs) return;
        const int h = 2 * i + half;
        rotate_row(rq, wq, qhat + base + (size_t)h * kD, h < H);
        rotate_row(rk, wk, khat + base + (size_t)h * kD, h < H);
    };
    // software pipeline: the next batch of head pairs loads while this one is computed
    for (int i0 = 0; i0 < pairs; i0 += 2 * ProCfg<kMode>::batch) {
#pragma unroll
        for (int b = 0; b < ProCfg<kMode>::batch; ++b) load(i0 + ProCfg<kMode>::batch + b, bq[b], bk[b]);
#pragma unroll
        for (int b = 0; b < ProCfg<kMode>::batch; ++b) rotate(i0 + b, aq[b], ak[b]);
#pragma unroll
        for (int b = 0; b < ProCfg<kMode>::batch; ++b) load(i0 + 2 * ProCfg<kMode>::batch + b, aq[b], ak[b]);
#pragma unroll
        for (int b = 0; b < ProCfg<kMode>::batch; ++b) rotate(i0 + ProCfg<kMode>::batch + b, bq[b], bk[b]);
    }
    if (!ok) atomicOr(err, kErrRange);
}

cudaError_t launch_prologue(const Problem& p, const Workspace& ws, const RopeTable* rope, cudaStream_t st) {
    if (p.seq.S == 0) return cudaSuccess;
    const int blocks = (p.seq.S + kProWarps - 1) / kProWarps;
    // the layout of the rotary sections over the lanes' two groups (channel c and c + 64)
    bool rot_b = false, crossed = false;
    for (int g = 0; g < 32; ++g) {
        rot_b |= g >= 16 && rope->axis[g] >= 0;
        crossed |= (g < 16) != (rope->partner[g] < 16);
    }
    const int mode = crossed ? 2 : (rot_b ? 1 : 0);
    if (mode == 0)
        prologue_kernel<0><<<blocks, kProWarps * 32, 0, st>>>(p, ws.qhat, ws.khat, *rope, ws.plan.err);
    else if (mode == 1)
        prologue_kernel<1><<<blocks, kProWarps * 32, 0, st>>>(p, ws.qhat, ws.khat, *rope, ws.plan.err);
    else
        prologue_kernel<2><<<blocks, kProWarps * 32, 0, st>>>(p, ws.qhat, ws.khat, *rope, ws.plan.err);
    return cudaGetLastError();
}

}  // namespace h3
