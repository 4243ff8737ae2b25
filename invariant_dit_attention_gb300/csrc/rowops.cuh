// rowops.cuh -- per-(token, head) q/k prologue and its backward, one warp per row.
//
// Lane l of the warp owns channels 4l..4l+3 of the 128-wide head.
//
// Forward (q_norm/k_norm then rope_q/rope_k of an H3 block, "ws1_one_h3_block"
// page, Bindings table):
//   n = x / sqrt(mean_c x_c^2 + eps),  z = n * w,
//   for a rotated pair (u, v) = (z[o+j], z[o+j+n_a/2]) with angle a = p_axis * f_j:
//   (u, v) -> (u cos a - v sin a, u sin a + v cos a); other channels unchanged.
// All of it in FP32 with one final rounding to fp16 (11-bit significand: the
// rotated rows are bounded by sqrt(128) * max|w|, far inside fp16's range).
//
// Backward, for the gradient dy at the rotated output:
//   g = R(a)^T dy,  dn = g * w,  dx = r (dn - n mean_c(dn_c n_c)),  dw += g * n,
// with r = 1/sqrt(mean x^2 + eps) recomputed from x.
#pragma once

#include "common.cuh"

namespace h3 {

struct RowAngles {
    float c[4], s[4];
};

// The lane's view of the rotary table, read once (the table lives in the
// constant bank, where lanes reading different entries would serialise).
struct LaneRope {
    float f[4];   // frequencies of the lane's four channels
    int axis;     // 0/1/2 = t/h/w, -1 = not rotated
    int partner;  // lane holding the paired channels
    int second;   // 1 if the lane's channels are the second half of their section
};

// Copies the rotary table into shared memory (call with the whole block, then
// __syncthreads); lanes then read their entries from there instead of issuing
// per-lane indexed reads of the kernel-parameter bank.
__device__ __forceinline__ void rope_to_smem(const RopeTable& rt, RopeTable& dst, int tid, int nthreads) {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(&rt);
    uint32_t* d = reinterpret_cast<uint32_t*>(&dst);
    for (int i = tid; i < (int)(sizeof(RopeTable) / 4); i += nthreads) d[i] = src[i];
}

__device__ __forceinline__ LaneRope lane_rope(const RopeTable& rt, int lane) {
    LaneRope r;
#pragma unroll
    for (int e = 0; e < 4; ++e) r.f[e] = rt.inv_freq[4 * lane + e];
    r.axis = rt.axis[lane];
    r.partner = rt.partner[lane];
    r.second = rt.second[lane];
    return r;
}

// cos/sin of the lane's four channels for one token (identity if not rotated).
__device__ __forceinline__ RowAngles row_angles(const LaneRope& lr, int pt, int ph, int pw) {
    RowAngles a;
    if (lr.axis < 0) {
#pragma unroll
        for (int e = 0; e < 4; ++e) { a.c[e] = 1.f; a.s[e] = 0.f; }
        return a;
    }
    const float p = static_cast<float>(lr.axis == 0 ? pt : (lr.axis == 1 ? ph : pw));
#pragma unroll
    for (int e = 0; e < 4; ++e) sincosf(__fmul_rn(p, lr.f[e]), &a.s[e], &a.c[e]);
    return a;
}

// The forward's roundings, spelled out operation by operation (no contraction
// left to the compiler), so that every kernel computing q^ / k^ - the prologue
// here, one warp per row, and the QKV projection's epilogue, one thread per
// row - gets the same bits from the same bf16 row.
//   sum of squares of four channels (a lane's share of the row)
__device__ __forceinline__ float sq4(float x0, float x1, float x2, float x3) {
    return __fmaf_rn(x3, x3, __fmaf_rn(x2, x2, __fmaf_rn(x1, x1, __fmul_rn(x0, x0))));
}
//   1 / sqrt(mean of squares + eps) from the row's sum of squares, correctly
//   rounded (one rounding)
__device__ __forceinline__ float rstd_of(float ss, float eps) { return __frsqrt_rn(__fmaf_rn(ss, 1.0f / kD, eps)); }
//   z = (x r) w
__device__ __forceinline__ float norm_w(float x, float r, float w) { return __fmul_rn(__fmul_rn(x, r), w); }
//   the rotated pair (u, v) -> (u cos - v sin, u sin + v cos)
__device__ __forceinline__ float rope_u(float u, float v, float c, float s) { return __fmaf_rn(u, c, -__fmul_rn(v, s)); }
__device__ __forceinline__ float rope_v(float u, float v, float c, float s) { return __fmaf_rn(u, s, __fmul_rn(v, c)); }

// 1/sqrt(mean of squares + eps) of the row held 4 channels per lane.
__device__ __forceinline__ float row_rstd(const float (&x)[4], float eps) {
    return rstd_of(warp_sum(sq4(x[0], x[1], x[2], x[3])), eps);
}

// y = RoPE(RMSNorm(x) * w) for one row.
__device__ __forceinline__ void row_norm_rope(const float (&x)[4], const float (&w)[4], const RowAngles& a,
                                              const LaneRope& lr, float eps, float (&y)[4]) {
    float r = row_rstd(x, eps);
    float z[4], zp[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) z[e] = norm_w(x[e], r, w[e]);
#pragma unroll
    for (int e = 0; e < 4; ++e) zp[e] = __shfl_sync(0xffffffffu, z[e], lr.partner);
    if (lr.axis < 0) {
#pragma unroll
        for (int e = 0; e < 4; ++e) y[e] = z[e];
    } else if (!lr.second) {  // (u, v) = (own, partner): u cos - v sin
#pragma unroll
        for (int e = 0; e < 4; ++e) y[e] = rope_u(z[e], zp[e], a.c[e], a.s[e]);
    } else {                         // (u, v) = (partner, own): u sin + v cos
#pragma unroll
        for (int e = 0; e < 4; ++e) y[e] = rope_v(zp[e], z[e], a.c[e], a.s[e]);
    }
}

// Backward of row_norm_rope.  dy: gradient at the rotated output; x: the raw
// input row.  Writes dx and adds g*n into dw_acc.
__device__ __forceinline__ void row_norm_rope_bwd(const float (&dy)[4], const float (&x)[4], const float (&w)[4],
                                                  const RowAngles& a, const LaneRope& lr, float eps,
                                                  float (&dx)[4], float (&dw_acc)[4]) {
    float dyp[4], g[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) dyp[e] = __shfl_sync(0xffffffffu, dy[e], lr.partner);
    if (lr.axis < 0) {
#pragma unroll
        for (int e = 0; e < 4; ++e) g[e] = dy[e];
    } else if (!lr.second) {  // g_u = dy_u cos + dy_v sin
#pragma unroll
        for (int e = 0; e < 4; ++e) g[e] = dy[e] * a.c[e] + dyp[e] * a.s[e];
    } else {                         // g_v = -dy_u sin + dy_v cos
#pragma unroll
        for (int e = 0; e < 4; ++e) g[e] = dy[e] * a.c[e] - dyp[e] * a.s[e];
    }
    float r = row_rstd(x, eps);
    float n[4], dn[4];
    float t = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        n[e] = x[e] * r;
        dn[e] = g[e] * w[e];
        t += dn[e] * n[e];
    }
    t = warp_sum(t) * (1.0f / kD);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        dx[e] = r * (dn[e] - n[e] * t);
        dw_acc[e] += g[e] * n[e];
    }
}

__device__ __forceinline__ void load_row4(const __nv_bfloat16* p, float (&x)[4]) {
    uint2 u = *reinterpret_cast<const uint2*>(p);
    x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
}

// Rounds the row to fp16 and stores it; returns false if the four values are
// finite and one of them is beyond the fp16 range (non-finite inputs are not
// range errors).  y - y is 0 for a finite y and NaN otherwise.
__device__ __forceinline__ bool store_row4_f16(__half* p, const float (&y)[4]) {
    uint2 u;
    u.x = pack_f16(y[0], y[1]);
    u.y = pack_f16(y[2], y[3]);
    *reinterpret_cast<uint2*>(p) = u;
    const float m = fmaxf(fmaxf(fabsf(y[0]), fabsf(y[1])), fmaxf(fabsf(y[2]), fabsf(y[3])));
    const float t = ((y[0] - y[0]) + (y[1] - y[1])) + ((y[2] - y[2]) + (y[3] - y[3]));
    return m <= 65504.f || t != 0.f;
}

__device__ __forceinline__ void store_row4(__nv_bfloat16* p, const float (&y)[4]) {
    uint2 u;
    u.x = pack_bf16(y[0], y[1]);
    u.y = pack_bf16(y[2], y[3]);
    *reinterpret_cast<uint2*>(p) = u;
}

}  // namespace h3
