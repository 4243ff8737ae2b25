// bwd_rows.cu -- the backward's row-wise kernels around the tensor-core ones:
//   delta_kernel      Delta_i = sum_c dO_ic O_ic per (token, head)
//   rope_table_kernel cos / sin of every channel's rotary angle per token
//   rows_bwd_kernel   dx = RMSNorm-backward(RoPE^-1(scale * dx^)) per row, for q
//                     and k, and the norm-weight partial of every 128-token tile
//                     (the units of rows_bwd.cuh; with stored dS the dQ kernel
//                     runs them instead)
//   dw_head_kernel, dw_sample_kernel, dw_total_kernel
//                     the norm-weight gradient per (sample, head), then per
//                     sample over heads, then over samples
// (the per-leaf gradients of the "ws1_one_h3_block" page of RL-Kernel, PR #539,
// Results and Tests; the 128-element norm-weight gradient of its Status
// section).  Every sum runs in one fixed order, with no atomics.
#include "common.cuh"
#include "rows_bwd.cuh"
#include "rowops.cuh"

namespace h3 {

// ------------------------------------------------------------------ Delta

// Four (token, head) rows per warp: half a warp per row, each lane's 16-byte
// loads of out and dout (8 channels) for two rows in flight at once; a lane's
// eight products are added in channel order, then the 16 lanes of a row in a
// fixed butterfly.
__global__ void __launch_bounds__(256) delta_kernel(const __nv_bfloat16* __restrict__ out,
                                                    const __nv_bfloat16* __restrict__ dout, int S, int H,
                                                    const int32_t* __restrict__ out_map, float* __restrict__ delta) {
    const int lane = threadIdx.x & 31, half = lane >> 4, l16 = lane & 15;
    const long rows = (long)S * H;
    const long base = ((long)blockIdx.x * 8 + (threadIdx.x >> 5)) * 4;  // the warp's first row
    uint4 o[2], d[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const long row = base + 2 * u + half;
        o[u] = d[u] = make_uint4(0u, 0u, 0u, 0u);
        if (row < rows) {
            // out is read through the canonical order's map (its packed row), dout is not
            const long orow = out_map ? (long)out_map[row / H] * H + row % H : row;
            o[u] = *reinterpret_cast<const uint4*>(out + orow * kD + 8 * l16);
            d[u] = *reinterpret_cast<const uint4*>(dout + row * kD + 8 * l16);
        }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const long row = base + 2 * u + half;
        const uint32_t ow[4] = {o[u].x, o[u].y, o[u].z, o[u].w}, dw[4] = {d[u].x, d[u].y, d[u].z, d[u].w};
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            acc = __fmaf_rn(bf16_lo(ow[e]), bf16_lo(dw[e]), acc);
            acc = __fmaf_rn(bf16_hi(ow[e]), bf16_hi(dw[e]), acc);
        }
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (l16 == 0 && row < rows) delta[(row % H) * S + row / H] = acc;
    }
}

// ------------------------------------------- RoPE^-1 + RMSNorm backward rows



// cos / sin of every channel's rotary angle per token, [S][cos 128 | sin 128]:
// the same FP32 sincosf(p_axis * f_c) as row_angles, computed once per token
// instead of once per (token, head) row; channels outside the sections get
// (1, 0).
__global__ void __launch_bounds__(256)
rope_table_kernel(const __grid_constant__ RopeTable rt, Seq seq, float* __restrict__ cs) {
    __shared__ RopeTable srt;
    rope_to_smem(rt, srt, threadIdx.x, 256);
    __syncthreads();
    const long i = (long)blockIdx.x * 256 + threadIdx.x;
    if (i >= (long)seq.S * kD) return;
    const int token = (int)(i / kD), ch = (int)(i % kD);
    const int axis = srt.axis[ch >> 2];
    float c = 1.f, sn = 0.f;
    if (axis >= 0) {
        const int pos = axis == 0 ? seq.pos_t[token] : (axis == 1 ? seq.pos_h[token] : seq.pos_w[token]);
        sincosf(__fmul_rn(static_cast<float>(pos), srt.inv_freq[ch]), &sn, &c);
    }
    cs[(size_t)token * 2 * kD + ch] = c;
    cs[(size_t)token * 2 * kD + kD + ch] = sn;
}

// One CTA per (128-token tile of a sample, head) and per q / k (blockIdx.y): the
// unit of rows_unit (rows_bwd.cuh) with the CTA's 256 threads.
__global__ void __launch_bounds__(256, 3)
rows_bwd_kernel(const __grid_constant__ RopeTable rt, const RowsParams p) {
    __shared__ RopeTable srt;
    __shared__ float red[8 * kD];
    rope_to_smem(rt, srt, threadIdx.x, 256);
    __syncthreads();
    rows_unit(srt, p, blockIdx.y, blockIdx.x / p.H, blockIdx.x % p.H, threadIdx.x >> 5, threadIdx.x & 31, red,
              [] { __syncthreads(); });
}

// -------------------------------------------------------- weight gradients

// The norm-weight gradient is reduced in three fixed orders:
//   per (sample, head): the sample's 128-token tile partials in ascending order;
//   per sample: those (sample, head) partials over heads in ascending order;
//   in total: the per-sample sums in ascending sample order.
// A (sample, head) partial depends only on that head's rows of that sample, so
// when the heads are split across GPUs (each GPU running its heads as a handle
// of its own) and the partials are gathered in head order, the same two last
// reductions give the same bits whatever the number of GPUs.

// Per (sample, head) partial: dst[s][h][c] = sum over the sample's tiles t, in
// ascending order, of part[t][h][c].  One thread per (sample, head, channel):
// CTAs of 128 threads over (sample, head, q / k).
__global__ void __launch_bounds__(128)
dw_head_kernel(const float* __restrict__ part_q, const float* __restrict__ part_k, Plan plan, int n, int H,
               float* __restrict__ dst_q, float* __restrict__ dst_k) {
    const int s = blockIdx.x, h = blockIdx.y, c = threadIdx.x;
    const float* part = blockIdx.z == 0 ? part_q : part_k;
    float* dst = blockIdx.z == 0 ? dst_q : dst_k;
    const int r = plan.rank_of[s];
    const int t0 = plan.cum128[r], t1 = plan.cum128[r + 1];
    const size_t hc = (size_t)h * kD + c;
    float acc = 0.f;
    for (int t = t0; t < t1; ++t) acc += part[(size_t)t * H * kD + hc];
    dst[(size_t)s * H * kD + hc] = acc;
}

// Up to two reductions side by side (blockIdx.y): q_norm_w's and k_norm_w's.
struct DwCombine {
    const float* part[2];  // [n][H][128] per (sample, head) partials
    float* per_sample[2];  // [n][128]
    float* total[2];       // [128]
};

// Per sample over heads: per_sample[s][c] = sum over h ascending of part[s][h][c].
// One CTA of 128 threads per sample.
__global__ void __launch_bounds__(128) dw_sample_kernel(const __grid_constant__ DwCombine d, int H) {
    const int s = blockIdx.x, c = threadIdx.x, y = blockIdx.y;
    const float* p = d.part[y] + (size_t)s * H * kD + c;
    float acc = 0.f;
    for (int h = 0; h < H; ++h) acc += p[(size_t)h * kD];
    d.per_sample[y][(size_t)s * kD + c] = acc;
}

// Over samples in ascending order.
__global__ void __launch_bounds__(128) dw_total_kernel(const __grid_constant__ DwCombine d, int n) {
    const int c = threadIdx.x, y = blockIdx.y;
    float acc = 0.f;
    for (int s = 0; s < n; ++s) acc += d.per_sample[y][(size_t)s * kD + c];
    d.total[y][c] = acc;
}

// ------------------------------------------------------------------ host

cudaError_t launch_bwd_delta(const Problem& p, const Workspace& ws, const __nv_bfloat16* out,
                             const __nv_bfloat16* dout, cudaStream_t st) {
    const long rows = (long)p.seq.S * p.H;
    delta_kernel<<<(unsigned)((rows + 31) / 32), 256, 0, st>>>(out, dout, p.seq.S, p.H, p.rowmap, ws.delta);
    return cudaGetLastError();
}

cudaError_t launch_rope_table(const Problem& p, const Workspace& ws, const RopeTable* rope, cudaStream_t st) {
    const long cells = (long)p.seq.S * kD;
    if (cells == 0) return cudaSuccess;
    rope_table_kernel<<<(unsigned)((cells + 255) / 256), 256, 0, st>>>(*rope, p.seq, ws.rope_cs);
    return cudaGetLastError();
}

cudaError_t launch_bwd_rows(const Problem& p, const Workspace& ws, const RopeTable* rope, __nv_bfloat16* dq,
                            __nv_bfloat16* dk, cudaStream_t st) {
    if (ws.ds) return cudaSuccess;  // the dQ kernel from the stored dS ran these rows beside its products
    const RowsParams r = make_rows_params(p, ws, dq, dk);
    cudaError_t e = launch_rope_table(p, ws, rope, st);
    if (e != cudaSuccess) return e;
    // an upper bound of the 128-token tiles (every sample adds at most one partial
    // tile); CTAs past the plan's last tile return at once
    const long tiles = (long)(p.seq.S + 127) / 128 + p.seq.n;
    rows_bwd_kernel<<<dim3((unsigned)(tiles * p.H), 2), 256, 0, st>>>(*rope, r);
    return cudaGetLastError();
}

namespace {
cudaError_t combine(const DwCombine& d, int pairs, int n, int H, cudaStream_t st) {
    dw_sample_kernel<<<dim3(n, pairs), kD, 0, st>>>(d, H);
    dw_total_kernel<<<dim3(1, pairs), kD, 0, st>>>(d, n);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_dw_combine(const float* partials, int n, int H, float* per_sample, float* total,
                              cudaStream_t st) {
    DwCombine d = {{partials, partials}, {per_sample, per_sample}, {total, total}};
    return combine(d, 1, n, H, st);
}

cudaError_t launch_bwd_dw(const Problem& p, const Workspace& ws, float* dwq, float* dwk, float* dwq_s,
                          float* dwk_s, cudaStream_t st) {
    const int n = p.seq.n, H = p.H;
    dw_head_kernel<<<dim3(n, H, 2), kD, 0, st>>>(ws.dwq_part, ws.dwk_part, ws.plan, n, H, ws.dwq_head, ws.dwk_head);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    DwCombine d = {{ws.dwq_head, ws.dwk_head}, {dwq_s ? dwq_s : ws.dwq_sample, dwk_s ? dwk_s : ws.dwk_sample},
                   {dwq, dwk}};
    return combine(d, 2, n, H, st);
}

}  // namespace h3
