// rows_bwd.cuh -- one unit of the row backward: RoPE^-1 + RMSNorm backward of the
// 128 rows of a (128-token tile, head) for q or k, and the tile's norm-weight
// partial (the per-leaf gradients of the "ws1_one_h3_block" page of RL-Kernel,
// PR #539, Results and Tests; the 128-element norm-weight gradient of its Status
// section).  Run by 8 warps: by its own CTA (rows_bwd_kernel) or by 8 warps of
// the dQ kernel beside its products.
#pragma once
#include "common.cuh"
#include "rowops.cuh"

namespace h3 {

struct RowsParams {
    Seq seq;
    Plan plan;
    int H;
    float eps;
    const float* rope_cs;          // [S][cos 128 | sin 128] per token
    const int32_t* rowmap;         // canonical order: packed row of x and dx (null = identity)
    const float* dyhat[2];         // scale * dq^, scale * dk^: FP32 [S, H, 128]
    const __nv_bfloat16* x[2];     // raw q, k
    const float* w[2];             // q_norm_w, k_norm_w
    __nv_bfloat16* dx[2];          // dq, dk
    float* dw_part[2];             // [tiles128, H, 128]
};

// dx = RMSNorm-backward(RoPE^-1(dy)) per row (one warp per row, rows w8, w8 + 8,
// ... with four rows' loads in flight per warp), and the tile's norm-weight
// partial sum_rows g * n, reduced rows-by-warp then warps in a fixed order (the
// same order whichever warps run the unit).  srt: the rotary table in shared
// memory; red: 8 x 128 floats of shared memory; sync(): a barrier of the 8 warps.
// Returns false (nothing done) for a tile past the plan's last.
template <class Sync>
__device__ __forceinline__ bool rows_unit(const RopeTable& srt, const RowsParams& p, int which, int tile, int h,
                                          int w8, int lane, float* red, Sync sync) {
    int sample, row0, row_end, local;
    if (!plan_tile(p.plan.cum128, p.plan.order, p.seq.seg, p.seq.n, 128, tile, sample, row0, row_end, local)) return false;
    const float* dyhat = p.dyhat[which];
    const __nv_bfloat16* x = p.x[which];
    __nv_bfloat16* dx = p.dx[which];
    const LaneRope lr = lane_rope(srt, lane);
    float wl[4], acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 4; ++e) wl[e] = p.w[which][4 * lane + e];
    const int nvalid = min(128, row_end - row0);
    bool nonfinite = false;
    for (int r0 = w8; r0 < nvalid; r0 += 32) {
        float dy[4][4], xr[4][4];
        RowAngles a[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int row = row0 + min(r0 + 8 * u, nvalid - 1);
            const size_t off = ((size_t)row * p.H + h) * kD + 4 * lane;
            const float4 d4 = *reinterpret_cast<const float4*>(dyhat + off);
            dy[u][0] = d4.x; dy[u][1] = d4.y; dy[u][2] = d4.z; dy[u][3] = d4.w;
            const size_t xoff = p.rowmap ? ((size_t)p.rowmap[row] * p.H + h) * kD + 4 * lane : off;
            load_row4(x + xoff, xr[u]);
            const float4 c4 = *reinterpret_cast<const float4*>(p.rope_cs + (size_t)row * 2 * kD + 4 * lane);
            const float4 s4 = *reinterpret_cast<const float4*>(p.rope_cs + (size_t)row * 2 * kD + kD + 4 * lane);
            a[u].c[0] = c4.x; a[u].c[1] = c4.y; a[u].c[2] = c4.z; a[u].c[3] = c4.w;
            a[u].s[0] = s4.x; a[u].s[1] = s4.y; a[u].s[2] = s4.z; a[u].s[3] = s4.w;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int r = r0 + 8 * u;
            if (r >= nvalid) break;
            float d[4];
            row_norm_rope_bwd(dy[u], xr[u], wl, a[u], lr, p.eps, d, acc);
            nonfinite |= !(isfinite(d[0]) && isfinite(d[1]) && isfinite(d[2]) && isfinite(d[3]));
            const size_t orow = p.rowmap ? (size_t)p.rowmap[row0 + r] : (size_t)(row0 + r);
            store_row4(dx + (orow * p.H + h) * kD + 4 * lane, d);
        }
    }
    // a non-finite gradient row from finite inputs means an fp16 operand (dS) overflowed
    if (nonfinite) atomicOr(p.plan.err, kErrRange);
#pragma unroll
    for (int e = 0; e < 4; ++e) red[w8 * kD + 4 * lane + e] = acc[e];
    sync();
    const int c = 32 * w8 + lane;
    if (c < kD) {
        float sum = 0.f;
#pragma unroll
        for (int wi = 0; wi < 8; ++wi) sum += red[wi * kD + c];
        p.dw_part[which][((size_t)tile * p.H + h) * kD + c] = sum;
    }
    sync();  // red is rewritten by the next unit
    return true;
}

inline RowsParams make_rows_params(const Problem& p, const Workspace& ws, __nv_bfloat16* dq, __nv_bfloat16* dk) {
    RowsParams r;
    r.seq = p.seq;
    r.plan = ws.plan;
    r.H = p.H;
    r.eps = p.eps;
    r.dyhat[0] = ws.dqhat32;
    r.dyhat[1] = ws.dkhat32;
    r.x[0] = p.q;
    r.x[1] = p.k;
    r.w[0] = p.wq;
    r.w[1] = p.wk;
    r.dx[0] = dq;
    r.dx[1] = dk;
    r.dw_part[0] = ws.dwq_part;
    r.dw_part[1] = ws.dwk_part;
    r.rope_cs = ws.rope_cs;
    r.rowmap = p.rowmap;
    return r;
}

}  // namespace h3
