// bwd_mma.cu -- backward of the attention core (K3..K6, warp-MMA version).
//
// Gradients of sum(out * dout) (the per-leaf gradient checks of the
// "ws1_one_h3_block" page, Results and Tests; the 128-element norm-weight
// gradient of its Status section):
//   Delta_i = sum_c dO_ic O_ic                                    (K3)
//   P_ij = exp(scale q^_i.k^_j - lse_i),  dP_ij = dO_i . v_j,
//   dS_ij = P_ij (dP_ij - Delta_i),
//   dV_j = sum_i P_ij dO_i,  dk^_j = scale sum_i dS_ij q^_i          (K4, per key tile)
//   dq^_i = scale sum_j dS_ij k^_j                                  (K5, per query tile)
// then the RoPE and RMSNorm backward in the epilogues of K4/K5, with per-tile
// partial sums of the norm-weight gradients reduced in a fixed order (K6).
// No atomics in any sum: K4 and K5 each recompute S and P, and every sum runs
// over tiles anchored at the sample start in ascending order.  Operand types:
// S = q^ k^T on fp16 (the prologue's rounding), dS rounded to fp16 for the
// dq^ = dS k^ and dk^ = dS^T q^ products, P and dO (bf16) for dV, dO and v
// (bf16) for dP.
#include "common.cuh"
#include "mma.cuh"
#include "rowops.cuh"

namespace h3 {

namespace bwdm {
constexpr int kWarps = 4;
constexpr int kThreads = 128;
constexpr int kRows = 64;     // rows of the tile a CTA owns (queries in K5, keys in K4)
constexpr int kStep = 32;     // rows streamed per inner step (keys in K5, queries in K4)
constexpr int kBig = kRows * kD * 2;   // 16 KB
constexpr int kSmall = kStep * kD * 2;  // 8 KB
constexpr int kSmem = 2 * kBig + 4 * kSmall + 2 * 2 * kStep * 4;  // + lse/Delta per stage
constexpr float kLog2e = 1.4426950408889634f;
}  // namespace bwdm

// ------------------------------------------------------------------ K3

__global__ void __launch_bounds__(256) delta_kernel(const __nv_bfloat16* __restrict__ out,
                                                    const __nv_bfloat16* __restrict__ dout, int S, int H,
                                                    float* __restrict__ delta) {
    const int lane = threadIdx.x & 31;
    const long row = (long)blockIdx.x * 8 + (threadIdx.x >> 5);  // (token, head)
    if (row >= (long)S * H) return;
    float o[4], d[4];
    load_row4(out + row * kD + 4 * lane, o);
    load_row4(dout + row * kD + 4 * lane, d);
    float acc = o[0] * d[0] + o[1] * d[1] + o[2] * d[2] + o[3] * d[3];
    acc = warp_sum(acc);
    if (lane == 0) delta[(long)(row % H) * S + row / H] = acc;
}

// Shared epilogue: rows of a staged fp32 [64][128] tile of d(x^) through the
// prologue backward; writes bf16 dx rows and the tile's weight-gradient partial.
__device__ __forceinline__ void norm_rope_bwd_tile(const float* stage, const __nv_bfloat16* __restrict__ x,
                                                   const float* __restrict__ w, const Seq& seq, int H, int h,
                                                   int row0, int row_end, float eps, const RopeTable& rt,
                                                   __nv_bfloat16* __restrict__ dx, float* __restrict__ dw_part,
                                                   float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float wl[4], acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 4; ++e) wl[e] = w[4 * lane + e];
    for (int r = warp; r < bwdm::kRows; r += bwdm::kWarps) {
        const int row = row0 + r;
        if (row >= row_end) break;
        float dy[4], xr[4], d[4];
        const float4 s4 = *reinterpret_cast<const float4*>(stage + r * kD + 4 * lane);
        dy[0] = s4.x; dy[1] = s4.y; dy[2] = s4.z; dy[3] = s4.w;
        load_row4(x + ((size_t)row * H + h) * kD + 4 * lane, xr);
        RowAngles a = row_angles(rt, lane, seq.pos_t[row], seq.pos_h[row], seq.pos_w[row]);
        row_norm_rope_bwd(dy, xr, wl, a, rt, lane, eps, d, acc);
        store_row4(dx + ((size_t)row * H + h) * kD + 4 * lane, d);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) red[warp * kD + 4 * lane + e] = acc[e];
    __syncthreads();
    if (threadIdx.x < kD) {
        float s = 0.f;
#pragma unroll
        for (int wi = 0; wi < bwdm::kWarps; ++wi) s += red[wi * kD + threadIdx.x];
        dw_part[threadIdx.x] = s;
    }
}

// ------------------------------------------------------------------ K5: dQ

__global__ void __launch_bounds__(bwdm::kThreads)
dq_kernel(const __half* __restrict__ qhat, const __half* __restrict__ khat,
          const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ dout,
          const __nv_bfloat16* __restrict__ q, const float* __restrict__ wq,
          const float* __restrict__ lse, const float* __restrict__ delta, Seq seq, Plan plan, int H,
          float scale, float eps, const __grid_constant__ RopeTable rt,
          __nv_bfloat16* __restrict__ dq, float* __restrict__ dw_part) {
    using namespace bwdm;
    extern __shared__ __align__(1024) uint8_t smem[];
    int sample, row0, row_end, local;
    if (!plan_tile(plan.cum64, plan.order, seq.seg, seq.n, 64, blockIdx.x, sample, row0, row_end, local)) return;
    const int h = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int seg0 = seq.seg[sample];
    const uint32_t sQ = smem_u32(smem), sO = sQ + kBig;
    const uint32_t sK[2] = {sQ + 2 * kBig, sQ + 2 * kBig + 2 * kSmall};
    const uint32_t sV[2] = {sQ + 2 * kBig + kSmall, sQ + 2 * kBig + 3 * kSmall};
    const float scale_log2 = scale * kLog2e;
    const int nkv = (row_end - seg0 + kStep - 1) / kStep;

    load_tile_async<kRows, kThreads>(sQ, qhat, H, h, row0, row_end, tid);
    load_tile_async<kRows, kThreads>(sO, dout, H, h, row0, row_end, tid);
    load_tile_async<kStep, kThreads>(sK[0], khat, H, h, seg0, row_end, tid);
    load_tile_async<kStep, kThreads>(sV[0], v, H, h, seg0, row_end, tid);
    cp_async_commit();

    float lse2[2], dlt[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        int row = min(row0 + warp * 16 + g + 8 * r, row_end - 1);
        lse2[r] = lse[(size_t)h * seq.S + row] * kLog2e;
        dlt[r] = delta[(size_t)h * seq.S + row];
    }
    float acc[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    uint32_t qa[8][4], oa[8][4];
    bool range_ok = true;

    for (int j = 0; j < nkv; ++j) {
        const int buf = j & 1;
        if (j + 1 < nkv) {
            load_tile_async<kStep, kThreads>(sK[buf ^ 1], khat, H, h, seg0 + (j + 1) * kStep, row_end, tid);
            load_tile_async<kStep, kThreads>(sV[buf ^ 1], v, H, h, seg0 + (j + 1) * kStep, row_end, tid);
        }
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        if (j == 0) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                ldsm_a(qa[kk], sQ, warp * 16, kk, lane);
                ldsm_a(oa[kk], sO, warp * 16, kk, lane);
            }
        }
        float s[4][4], dp[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[i][e] = dp[i][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                uint32_t b[4];
                ldsm_b_nk(b, sK[buf], np * 16, kk, lane);
                mma16816_f16(s[2 * np], qa[kk], b[0], b[1]);
                mma16816_f16(s[2 * np + 1], qa[kk], b[2], b[3]);
                ldsm_b_nk(b, sV[buf], np * 16, kk, lane);
                mma16816(dp[2 * np], oa[kk], b[0], b[1]);
                mma16816(dp[2 * np + 1], oa[kk], b[2], b[3]);
            }
        const int key0 = seg0 + j * kStep;
        uint32_t da[2][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            float ds[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = e >> 1;
                const int key = key0 + nt * 8 + 2 * t + (e & 1);
                float p = ex2(fmaf(s[nt][e], scale_log2, -lse2[r]));
                p = key < row_end ? p : 0.f;
                ds[e] = p * (dp[nt][e] - dlt[r]);
                range_ok &= !(fabsf(ds[e]) > 65504.f);
            }
            da[nt >> 1][(nt & 1) * 2 + 0] = pack_f16(ds[0], ds[1]);
            da[nt >> 1][(nt & 1) * 2 + 1] = pack_f16(ds[2], ds[3]);
        }
#pragma unroll
        for (int kc = 0; kc < 2; ++kc)
#pragma unroll
            for (int dpi = 0; dpi < 8; ++dpi) {
                uint32_t b[4];
                ldsm_b_kn(b, sK[buf], kc * 16, dpi * 16, lane);
                mma16816_f16(acc[2 * dpi], da[kc], b[0], b[1]);
                mma16816_f16(acc[2 * dpi + 1], da[kc], b[2], b[3]);
            }
        __syncthreads();
    }
    cp_async_wait<0>();
    __syncthreads();

    // stage scale * dq^ as fp32 [64][128] over the K/V buffers, then the row epilogue
    float* stage = reinterpret_cast<float*>(smem + 2 * kBig);
    float* red = reinterpret_cast<float*>(smem);  // over the Q tile: 4 x 128 floats
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int rr = warp * 16 + g + 8 * r;
#pragma unroll
        for (int dt = 0; dt < 16; ++dt)
            *reinterpret_cast<float2*>(stage + rr * kD + dt * 8 + 2 * t) =
                make_float2(acc[dt][2 * r] * scale, acc[dt][2 * r + 1] * scale);
    }
    __syncthreads();
    norm_rope_bwd_tile(stage, q, wq, seq, H, h, row0, row_end, eps, rt, dq,
                       dw_part + ((size_t)blockIdx.x * H + h) * kD, red);
    if (!range_ok) atomicOr(plan.err, kErrRange);
}

// ------------------------------------------------------------- K4: dK, dV

__global__ void __launch_bounds__(bwdm::kThreads)
dkdv_kernel(const __half* __restrict__ qhat, const __half* __restrict__ khat,
            const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ dout,
            const __nv_bfloat16* __restrict__ k, const float* __restrict__ wk,
            const float* __restrict__ lse, const float* __restrict__ delta, Seq seq, Plan plan, int H,
            float scale, float eps, const __grid_constant__ RopeTable rt,
            __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, float* __restrict__ dw_part) {
    using namespace bwdm;
    extern __shared__ __align__(1024) uint8_t smem[];
    int sample, row0, row_end, local;
    if (!plan_tile(plan.cum64, plan.order, seq.seg, seq.n, 64, blockIdx.x, sample, row0, row_end, local)) return;
    const int h = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int seg0 = seq.seg[sample];
    const uint32_t sK = smem_u32(smem), sV = sK + kBig;
    const uint32_t sQ[2] = {sK + 2 * kBig, sK + 2 * kBig + 2 * kSmall};
    const uint32_t sO[2] = {sK + 2 * kBig + kSmall, sK + 2 * kBig + 3 * kSmall};
    float* sL = reinterpret_cast<float*>(smem + 2 * kBig + 4 * kSmall);  // [2][kStep] lse2, [2][kStep] delta
    const float scale_log2 = scale * kLog2e;
    const int nq = (row_end - seg0 + kStep - 1) / kStep;

    auto load_step = [&](int i, int buf) {
        const int qr0 = seg0 + i * kStep;
        load_tile_async<kStep, kThreads>(sQ[buf], qhat, H, h, qr0, row_end, tid);
        load_tile_async<kStep, kThreads>(sO[buf], dout, H, h, qr0, row_end, tid);
        if (tid < kStep) {
            const int row = min(qr0 + tid, row_end - 1);
            sL[buf * kStep + tid] = lse[(size_t)h * seq.S + row] * kLog2e;
            sL[2 * kStep + buf * kStep + tid] = delta[(size_t)h * seq.S + row];
        }
    };
    load_tile_async<kRows, kThreads>(sK, khat, H, h, row0, row_end, tid);
    load_tile_async<kRows, kThreads>(sV, v, H, h, row0, row_end, tid);
    load_step(0, 0);
    cp_async_commit();

    float adv[16][4], adk[16][4];
    bool range_ok = true;
#pragma unroll
    for (int i = 0; i < 16; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) adv[i][e] = adk[i][e] = 0.f;

    for (int i = 0; i < nq; ++i) {
        const int buf = i & 1;
        if (i + 1 < nq) {
            __syncthreads();  // previous readers of sL[buf ^ 1] are done
            load_step(i + 1, buf ^ 1);
        }
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        float s[4][4], dp[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[a][e] = dp[a][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t ka[4], va[4];
            ldsm_a(ka, sK, warp * 16, kk, lane);
            ldsm_a(va, sV, warp * 16, kk, lane);
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                uint32_t b[4];
                ldsm_b_nk(b, sQ[buf], np * 16, kk, lane);
                mma16816_f16(s[2 * np], ka, b[0], b[1]);
                mma16816_f16(s[2 * np + 1], ka, b[2], b[3]);
                ldsm_b_nk(b, sO[buf], np * 16, kk, lane);
                mma16816(dp[2 * np], va, b[0], b[1]);
                mma16816(dp[2 * np + 1], va, b[2], b[3]);
            }
        }
        const int q0 = seg0 + i * kStep;
        uint32_t pa[2][4], da[2][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            float p[4], ds[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c = nt * 8 + 2 * t + (e & 1);  // query column
                float pe = ex2(fmaf(s[nt][e], scale_log2, -sL[buf * kStep + c]));
                pe = q0 + c < row_end ? pe : 0.f;
                p[e] = pe;
                ds[e] = pe * (dp[nt][e] - sL[2 * kStep + buf * kStep + c]);
                range_ok &= !(fabsf(ds[e]) > 65504.f);
            }
            pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(p[0], p[1]);
            pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(p[2], p[3]);
            da[nt >> 1][(nt & 1) * 2 + 0] = pack_f16(ds[0], ds[1]);
            da[nt >> 1][(nt & 1) * 2 + 1] = pack_f16(ds[2], ds[3]);
        }
#pragma unroll
        for (int kc = 0; kc < 2; ++kc)
#pragma unroll
            for (int dpi = 0; dpi < 8; ++dpi) {
                uint32_t b[4];
                ldsm_b_kn(b, sO[buf], kc * 16, dpi * 16, lane);
                mma16816(adv[2 * dpi], pa[kc], b[0], b[1]);
                mma16816(adv[2 * dpi + 1], pa[kc], b[2], b[3]);
                ldsm_b_kn(b, sQ[buf], kc * 16, dpi * 16, lane);
                mma16816_f16(adk[2 * dpi], da[kc], b[0], b[1]);
                mma16816_f16(adk[2 * dpi + 1], da[kc], b[2], b[3]);
            }
    }
    cp_async_wait<0>();
    __syncthreads();

    // dV rows straight to bf16
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int row = row0 + warp * 16 + g + 8 * r;
        if (row >= row_end) continue;
        __nv_bfloat16* dst = dv + ((size_t)row * H + h) * kD + 2 * t;
#pragma unroll
        for (int dt = 0; dt < 16; ++dt)
            *reinterpret_cast<uint32_t*>(dst + dt * 8) = pack_bf16(adv[dt][2 * r], adv[dt][2 * r + 1]);
    }
    float* stage = reinterpret_cast<float*>(smem + 2 * kBig);
    float* red = reinterpret_cast<float*>(smem);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int rr = warp * 16 + g + 8 * r;
#pragma unroll
        for (int dt = 0; dt < 16; ++dt)
            *reinterpret_cast<float2*>(stage + rr * kD + dt * 8 + 2 * t) =
                make_float2(adk[dt][2 * r] * scale, adk[dt][2 * r + 1] * scale);
    }
    __syncthreads();
    norm_rope_bwd_tile(stage, k, wk, seq, H, h, row0, row_end, eps, rt, dk,
                       dw_part + ((size_t)blockIdx.x * H + h) * kD, red);
    if (!range_ok) atomicOr(plan.err, kErrRange);
}

// ------------------------------------------------------------------ K6

// Per-sample weight gradient: sum over the sample's 64-token tiles (ascending)
// and heads (ascending), split over two fixed interleaved halves then added.
__global__ void __launch_bounds__(256)
dw_sample_kernel(const float* __restrict__ part_q, const float* __restrict__ part_k, Seq seq, Plan plan, int H,
                 float* __restrict__ dwq_s, float* __restrict__ dwk_s) {
    const int s = blockIdx.x;
    const float* part = blockIdx.y == 0 ? part_q : part_k;
    float* dst = blockIdx.y == 0 ? dwq_s : dwk_s;
    const int c = threadIdx.x & 127, grp = threadIdx.x >> 7;
    __shared__ float half[128];
    const int r = plan.rank_of[s];
    const int t0 = plan.cum64[r], t1 = plan.cum64[r + 1];
    float acc = 0.f;
    for (int tt = t0 + grp; tt < t1; tt += 2)
        for (int h = 0; h < H; ++h) acc += part[((size_t)tt * H + h) * kD + c];
    if (grp == 1) half[c] = acc;
    __syncthreads();
    if (grp == 0) dst[(size_t)s * kD + c] = acc + half[c];
}

__global__ void dw_total_kernel(const float* __restrict__ dwq_s, const float* __restrict__ dwk_s, int n,
                                float* __restrict__ dwq, float* __restrict__ dwk) {
    const int c = threadIdx.x & 127;
    const float* src = threadIdx.x < 128 ? dwq_s : dwk_s;
    float acc = 0.f;
    for (int s = 0; s < n; ++s) acc += src[(size_t)s * kD + c];
    (threadIdx.x < 128 ? dwq : dwk)[c] = acc;
}

cudaError_t init_bwd_attributes() {
    using namespace bwdm;
    cudaError_t e = cudaFuncSetAttribute(dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    return e;
}

cudaError_t launch_bwd_delta(const Problem& p, const Workspace& ws, const __nv_bfloat16* out,
                             const __nv_bfloat16* dout, cudaStream_t st) {
    const long rows = (long)p.seq.S * p.H;
    delta_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(out, dout, p.seq.S, p.H, ws.delta);
    return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(const Problem& p, const Workspace& ws, const RopeTable* rope, const float* lse,
                            const __nv_bfloat16* dout, __nv_bfloat16* dk, __nv_bfloat16* dv, cudaStream_t st) {
    using namespace bwdm;
    dim3 grid((p.seq.S + kRows - 1) / kRows + p.seq.n, p.H);
    dkdv_kernel<<<grid, kThreads, kSmem, st>>>(ws.qhat, ws.khat, p.v, dout, p.k, p.wk, lse, ws.delta, p.seq,
                                               ws.plan, p.H, p.scale, p.eps, *rope, dk, dv, ws.dwk_part);
    return cudaGetLastError();
}

cudaError_t launch_bwd_dq(const Problem& p, const Workspace& ws, const RopeTable* rope, const float* lse,
                          const __nv_bfloat16* dout, __nv_bfloat16* dq, cudaStream_t st) {
    using namespace bwdm;
    dim3 grid((p.seq.S + kRows - 1) / kRows + p.seq.n, p.H);
    dq_kernel<<<grid, kThreads, kSmem, st>>>(ws.qhat, ws.khat, p.v, dout, p.q, p.wq, lse, ws.delta, p.seq,
                                             ws.plan, p.H, p.scale, p.eps, *rope, dq, ws.dwq_part);
    return cudaGetLastError();
}

cudaError_t launch_bwd_dw(const Problem& p, const Workspace& ws, float* dwq, float* dwk, float* dwq_s,
                          float* dwk_s, cudaStream_t st) {
    float* qs = dwq_s ? dwq_s : ws.dwq_sample;
    float* ks = dwk_s ? dwk_s : ws.dwk_sample;
    dw_sample_kernel<<<dim3(p.seq.n, 2), 256, 0, st>>>(ws.dwq_part, ws.dwk_part, p.seq, ws.plan, p.H, qs, ks);
    dw_total_kernel<<<1, 256, 0, st>>>(qs, ks, p.seq.n, dwq, dwk);
    return cudaGetLastError();
}

}  // namespace h3
