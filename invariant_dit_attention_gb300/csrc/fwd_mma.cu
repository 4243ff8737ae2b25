// fwd_mma.cu -- forward attention over q^, k^ (K2, warp-MMA version).
//
// One CTA = one (sample, 64-query tile, head).  Four warps own 16 query rows
// each.  Key/value tiles of 64 tokens anchored at the sample start are streamed
// in ascending order with cp.async (double buffered); rows past the sample end
// are zero-filled and their scores replaced (select, not add) by -inf.  S = q^ k^T
// runs on fp16 operands (the prologue's rounding), PV on bf16 P and v.  Online
// softmax keeps a running max m and sum l per row in FP32; P is rounded once to
// bf16 for the PV product; O accumulates in FP32 and is rounded once at the end.
//
// Non-causal attention within each packed sample: the attention node of the
// "ws1_one_h3_block" page (RL-Kernel PR #539), Bindings table.
#include "common.cuh"
#include "mma.cuh"

namespace h3 {

namespace fwdm {
constexpr int kBM = 64;
constexpr int kBN = 64;
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kTileBytes = kBM * kD * 2;  // 16 KB
constexpr int kSmem = kTileBytes * 5;     // Q + 2 x (K, V)
}  // namespace fwdm

__global__ void __launch_bounds__(fwdm::kThreads)
fwd_mma_kernel(const __half* __restrict__ qhat, const __half* __restrict__ khat,
               const __nv_bfloat16* __restrict__ v, Seq seq, Plan plan, int H, float scale_log2,
               __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
    using namespace fwdm;
    extern __shared__ __align__(1024) uint8_t smem[];
    int sample, row0, row_end, local;
    if (!plan_tile(plan.cum64, plan.order, seq.seg, seq.n, 64, blockIdx.x, sample, row0, row_end, local)) return;
    const int h = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int seg0 = seq.seg[sample];
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sK[2] = {sQ + kTileBytes, sQ + 3 * kTileBytes};
    const uint32_t sV[2] = {sQ + 2 * kTileBytes, sQ + 4 * kTileBytes};
    const int nkv = (row_end - seg0 + kBN - 1) / kBN;

    load_tile_async<kBM, kThreads>(sQ, qhat, H, h, row0, row_end, tid);
    load_tile_async<kBN, kThreads>(sK[0], khat, H, h, seg0, row_end, tid);
    load_tile_async<kBN, kThreads>(sV[0], v, H, h, seg0, row_end, tid);
    cp_async_commit();

    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    uint32_t qa[8][4];

    for (int j = 0; j < nkv; ++j) {
        const int buf = j & 1;
        if (j + 1 < nkv) {
            load_tile_async<kBN, kThreads>(sK[buf ^ 1], khat, H, h, seg0 + (j + 1) * kBN, row_end, tid);
            load_tile_async<kBN, kThreads>(sV[buf ^ 1], v, H, h, seg0 + (j + 1) * kBN, row_end, tid);
        }
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        if (j == 0) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) ldsm_a(qa[kk], sQ, warp * 16, kk, lane);
        }
        // S = Q K^T for this warp's 16 rows x 64 keys
        float s[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t b[4];
                ldsm_b_nk(b, sK[buf], np * 16, kk, lane);
                mma16816_f16(s[2 * np], qa[kk], b[0], b[1]);
                mma16816_f16(s[2 * np + 1], qa[kk], b[2], b[3]);
            }
        }
        // mask keys past the sample end
        const int key0 = seg0 + j * kBN;
        if (key0 + kBN > row_end) {
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int key = key0 + nt * 8 + 2 * (lane & 3) + (e & 1);
                    s[nt][e] = key < row_end ? s[nt][e] : -INFINITY;
                }
        }
        // online softmax; rows g (e = 0, 1) and g + 8 (e = 2, 3)
        float mx[2] = {m[0], m[1]};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            mx[0] = fmaxf(mx[0], fmaxf(s[nt][0], s[nt][1]));
            mx[1] = fmaxf(mx[1], fmaxf(s[nt][2], s[nt][3]));
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        }
        float alpha[2], mneg[2], rs[2] = {0.f, 0.f};
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            alpha[r] = ex2((m[r] - mx[r]) * scale_log2);
            m[r] = mx[r];
            mneg[r] = -mx[r] * scale_log2;
        }
        uint32_t pa[4][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            float p0 = ex2(fmaf(s[nt][0], scale_log2, mneg[0]));
            float p1 = ex2(fmaf(s[nt][1], scale_log2, mneg[0]));
            float p2 = ex2(fmaf(s[nt][2], scale_log2, mneg[1]));
            float p3 = ex2(fmaf(s[nt][3], scale_log2, mneg[1]));
            rs[0] += p0 + p1;
            rs[1] += p2 + p3;
            pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(p0, p1);
            pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(p2, p3);
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 1);
            rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 2);
            l[r] = l[r] * alpha[r] + rs[r];
        }
#pragma unroll
        for (int dt = 0; dt < 16; ++dt) {
            o[dt][0] *= alpha[0]; o[dt][1] *= alpha[0];
            o[dt][2] *= alpha[1]; o[dt][3] *= alpha[1];
        }
        // O += P V   (pa[kc]: a0 = rows g keys 2t.., a1 = rows g+8, a2/a3 = keys +8)
#pragma unroll
        for (int kc = 0; kc < 4; ++kc) {
            uint32_t a[4] = {pa[kc][0], pa[kc][1], pa[kc][2], pa[kc][3]};
#pragma unroll
            for (int dp = 0; dp < 8; ++dp) {
                uint32_t b[4];
                ldsm_b_kn(b, sV[buf], kc * 16, dp * 16, lane);
                mma16816(o[2 * dp], a, b[0], b[1]);
                mma16816(o[2 * dp + 1], a, b[2], b[3]);
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    // epilogue: O / l -> bf16, lse = (m * scale_log2 + log2 l) * ln 2
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int row = row0 + warp * 16 + g + 8 * r;
        if (row >= row_end) continue;
        const float inv = 1.0f / l[r];
        __nv_bfloat16* dst = out + ((size_t)row * H + h) * kD + 2 * t;
#pragma unroll
        for (int dt = 0; dt < 16; ++dt)
            *reinterpret_cast<uint32_t*>(dst + dt * 8) = pack_bf16(o[dt][2 * r] * inv, o[dt][2 * r + 1] * inv);
        if (lse && t == 0) lse[(size_t)h * seq.S + row] = (m[r] * scale_log2 + log2f(l[r])) * 0.69314718055994531f;
    }
}

cudaError_t init_fwd_attributes() {
    return cudaFuncSetAttribute(fwd_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, fwdm::kSmem);
}

cudaError_t launch_fwd(const Problem& p, const Workspace& ws, __nv_bfloat16* out, float* lse, cudaStream_t st) {
    using namespace fwdm;
    dim3 grid((p.seq.S + kBM - 1) / kBM + p.seq.n, p.H);
    fwd_mma_kernel<<<grid, kThreads, kSmem, st>>>(ws.qhat, ws.khat, p.v, p.seq, ws.plan, p.H,
                                                 p.scale * 1.4426950408889634f, out, lse);
    return cudaGetLastError();
}

}  // namespace h3
