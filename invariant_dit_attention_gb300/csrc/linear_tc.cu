// linear_tc.cu -- y = x W^T (+ b): the row-invariant projection GEMM on either
// side of the attention core (the QKV projection feeding the q/k norms and
// the output projection after it; the "ws1_one_h3_block" page of RL-Kernel,
// PR #539, Bindings table: the block's projection nodes, and its Prior art
// section: an interim Triton GEMM there).
//
// x bf16 [rows, K] row-major, W bf16 [N, K] row-major (the [out, in] layout of
// a linear layer), b FP32 [N] or none, y bf16 [rows, N].  FP32 accumulation in
// tensor memory over K in ascending 64-column steps (K = 16 per MMA, fixed
// order inside), one rounding to bf16 after the bias: every output row's bits
// depend only on that row of x and on W, never on the number of rows or on the
// row's position in a tile (no split-K, no atomics).
//
// Persistent kernel, one CTA per SM, 256 threads: warp 0 TMA producer (A box
// 128 rows x 64, B box 256 rows x 64, 128-byte swizzle, 4-stage ring of 48 KB),
// warp 1 single-thread tcgen05 issuer (M = 128, N = 256, K = 16: four MMAs per
// stage into one of two 256-column TMEM accumulators), warps 4-7 the epilogue
// (thread = output row: TMEM -> + b -> bf16 -> global), which drains one
// accumulator while the other one fills.  Tiles are visited in groups of 16
// row tiles with the column tiles inside, so the operands a wave of CTAs works
// on stay in L2.
//
// The QKV form (h3attn_qkv_forward) runs the same kernel with a wider
// epilogue: W's rows are the q, k and v heads in that order, and each
// 128-column half of a tile is one head of one of them.  The epilogue writes
// the bf16 q, k, v rows and, for q and k, also the normalised and rotated
// fp16 rows q^ / k^ that the attention kernels read - the prologue's work done
// while the row is still on chip.  It computes them from the rounded bf16 row
// with the prologue's operations in the prologue's order (its lane partial
// sums of squares, the warp butterfly seen from one lane, then the same
// per-channel products and rotations, with the angles' cos / sin taken from
// the per-token table, which holds the prologue's own sincosf values), so the
// results are bitwise those of the projection followed by the separate
// prologue.
#include <cudaTypedefs.h>

#include "../../include/h3attn.h"
#include "common.cuh"
#include "host.cuh"
#include "rowops.cuh"
#include "tc.cuh"

namespace h3 {

namespace lint {
constexpr int kThreads = 256;
constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kRing = 4;
constexpr int kABytes = kBM * kBK * 2;          // 16 KB
constexpr int kBBytes = kBN * kBK * 2;          // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;  // 48 KB
constexpr int kOffBar = kRing * kStageBytes;
constexpr int kSmem = kOffBar + 256;            // the dynamic shared memory base is 1024-aligned (checked)
// QKV form: one head of the thread's row as bf16 pairs (65 words per row: the
// odd stride keeps the rows' words in different banks), then the rotary table
constexpr int kRowWords = 65;
constexpr int kOffRows = kSmem;
constexpr int kOffRope = kOffRows + kBM * kRowWords * 4;
constexpr int kOffWn = kOffRope + (int)sizeof(RopeTable);  // q_norm_w, k_norm_w
constexpr int kSmemQkv = kOffWn + 2 * kD * 4;
static_assert(kThreads == 2 * kD, "one thread per norm weight when staging them");
static_assert(kSmemQkv <= 232448, "shared memory of the QKV form");
static_assert(sizeof(RopeTable) % 16 == 0, "norm weights stay 16-byte aligned");
constexpr int kGroupM = 16;                     // row tiles per raster group
enum { bFull = 0, bEmpty = bFull + kRing, bAccFull = bEmpty + kRing, bAccEmpty = bAccFull + 2, bDone = bAccEmpty + 2,
       bNever, bCount };
}  // namespace lint

struct QkvParams {
    int H, D;                    // heads, D = H * 128 (q, k and v each D columns of y)
    float eps;
    const float* wn[2];          // q_norm_w, k_norm_w
    const int32_t* pos[3];       // t, h, w positions of each row
    __nv_bfloat16* out[3];       // q, k, v rows [rows, H, 128]
    __half* hat[2];              // q^, k^ rows [rows, H, 128]
    const float* rope_cs;        // [rows][cos 128 | sin 128]: the angles' cos / sin per token
    RopeTable rope;
};

struct LinearParams {
    int rows, N, K;
    int tiles_m, tiles_n;
    const float* bias;
    __nv_bfloat16* y;
    unsigned* err;
    int stall;               // tc::StallRole stalled once on the CTA's first tile (tests), else 0
    long long stall_budget;  // clock cycles of that stall's bounded wait
    QkvParams qkv;  // QKV form only
};

// Tile t of the raster: groups of kGroupM row tiles, column tiles inside a group.
__device__ __forceinline__ void linear_tile(const LinearParams& p, int t, int& tm, int& tn) {
    const int per_group = lint::kGroupM * p.tiles_n;
    const int g = t / per_group, r = t % per_group;
    const int gm0 = g * lint::kGroupM;
    const int gsize = min(lint::kGroupM, p.tiles_m - gm0);
    tm = gm0 + r % gsize;
    tn = r / gsize;
}

// Channel c of the staged bf16 row (two per 32-bit word, element 0 low).
__device__ __forceinline__ float staged(const uint32_t* row, int c) {
    const uint32_t w = row[c >> 1];
    return (c & 1) ? bf16_hi(w) : bf16_lo(w);
}

// The QKV epilogue of one tile for one thread (row): both 128-column heads of
// the tile, from the TMEM accumulator columns at acc.  A q or k head is staged
// in shared memory as bf16, normalised and rotated pair by pair (each rotated
// pair once, both outputs from one cos / sin), written back into the staging
// row as fp16 in place (a pair's inputs are not needed by any other pair) and
// then copied out.  Returns false if a q^ / k^ value left the fp16 range.
__device__ __forceinline__ bool qkv_epilogue(const LinearParams& p, uint8_t* smem, uint32_t acc, int row_in, int row,
                                             bool row_ok, int tn) {
    using namespace lint;
    const QkvParams& q = p.qkv;
    uint32_t* srow = reinterpret_cast<uint32_t*>(smem + kOffRows) + row_in * kRowWords;
    __half* srow16 = reinterpret_cast<__half*>(srow);
    const RopeTable& rt = *reinterpret_cast<const RopeTable*>(smem + kOffRope);
    bool in_range = true;
    for (int hh = 0; hh < 2; ++hh) {
        const int col0 = tn * kBN + 128 * hh;
        if (col0 >= p.N) break;
        const int which = col0 / q.D, head = (col0 - which * q.D) >> 7;
        __syncwarp();  // the TMEM loads below are warp-collective
        float part[32];  // the lanes' sums of squares in the prologue's layout (lane l: channels 4l..4l+3)
#pragma unroll
        for (int c32 = 0; c32 < 4; ++c32) {
            uint32_t r[32];
            tc::tmem_ld32(acc + 128 * hh + 32 * c32, r);
            tc::tmem_wait_ld_dep(r);
            float v[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
            if (p.bias) {
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    const float4 b4 = *reinterpret_cast<const float4*>(p.bias + col0 + 32 * c32 + e);
                    v[e] += b4.x; v[e + 1] += b4.y; v[e + 2] += b4.z; v[e + 3] += b4.w;
                }
            }
            uint32_t u[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) u[e] = pack_bf16(v[2 * e], v[2 * e + 1]);
            if (row_ok) {
                uint4* dst = reinterpret_cast<uint4*>(q.out[which] + ((size_t)row * q.H + head) * kD + 32 * c32);
#pragma unroll
                for (int e = 0; e < 4; ++e) dst[e] = make_uint4(u[4 * e], u[4 * e + 1], u[4 * e + 2], u[4 * e + 3]);
            }
            if (which < 2) {
#pragma unroll
                for (int e = 0; e < 16; ++e) srow[16 * c32 + e] = u[e];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    part[8 * c32 + j] =
                        sq4(bf16_lo(u[2 * j]), bf16_hi(u[2 * j]), bf16_lo(u[2 * j + 1]), bf16_hi(u[2 * j + 1]));
            }
        }
        if (which == 2 || !row_ok) continue;
        // warp_sum's butterfly (offsets 16, 8, 4, 2, 1) as lane 0 sees it
        float a16[16], a8[8], a4[4];
#pragma unroll
        for (int j = 0; j < 16; ++j) a16[j] = part[j] + part[j + 16];
#pragma unroll
        for (int j = 0; j < 8; ++j) a8[j] = a16[j] + a16[j + 8];
#pragma unroll
        for (int j = 0; j < 4; ++j) a4[j] = a8[j] + a8[j + 4];
        const float rs = rstd_of((a4[0] + a4[2]) + (a4[1] + a4[3]), q.eps);
        const float* wn = reinterpret_cast<const float*>(smem + kOffWn) + kD * which;
        const float* csr = q.rope_cs + (size_t)row * 2 * kD;  // the prologue's sincosf values, per token
        uint32_t notfit = 0, nonfinite = 0;  // per group of four channels (a prologue lane), as its check
        auto note = [&](float y, int g) {
            notfit |= (uint32_t)!(fabsf(y) <= 65504.f) << g;
            nonfinite |= (uint32_t)!isfinite(y) << g;
        };
        for (int g = 0; g < 32; ++g) {
            if (rt.axis[g] < 0) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c = 4 * g + e;
                    const float y = norm_w(staged(srow, c), rs, wn[c]);
                    note(y, g);
                    srow16[c] = __float2half_rn(y);
                }
            } else if (!rt.second[g]) {  // the pair (4g + e, 4pg + e); the second half's groups are done here
                const int pg = rt.partner[g];
                const float4 c4 = *reinterpret_cast<const float4*>(csr + 4 * g);
                const float4 s4 = *reinterpret_cast<const float4*>(csr + kD + 4 * g);
                const float cs[4] = {c4.x, c4.y, c4.z, c4.w}, sn[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int cu = 4 * g + e, cv = 4 * pg + e;
                    const float zu = norm_w(staged(srow, cu), rs, wn[cu]);
                    const float zv = norm_w(staged(srow, cv), rs, wn[cv]);
                    const float yu = rope_u(zu, zv, cs[e], sn[e]), yv = rope_v(zu, zv, cs[e], sn[e]);
                    note(yu, g);
                    note(yv, pg);
                    srow16[cu] = __float2half_rn(yu);
                    srow16[cv] = __float2half_rn(yv);
                }
            }
        }
        in_range &= (notfit & ~nonfinite) == 0;
        uint4* hat = reinterpret_cast<uint4*>(q.hat[which] + ((size_t)row * q.H + head) * kD);
#pragma unroll 4
        for (int w16 = 0; w16 < 16; ++w16)
            hat[w16] = make_uint4(srow[4 * w16], srow[4 * w16 + 1], srow[4 * w16 + 2], srow[4 * w16 + 3]);
    }
    return in_range;
}

template <bool kQkv>
__global__ void __launch_bounds__(lint::kThreads, 1)
linear_tc_kernel(const __grid_constant__ CUtensorMap ma, const __grid_constant__ CUtensorMap mb,
                 const __grid_constant__ LinearParams p) {
    using namespace lint;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {  // the layout below needs a 1024-byte aligned base
        if (threadIdx.x == 0) atomicOr(p.err, kErrTimeout);
        return;
    }
    uint8_t* smem = smem_raw;
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) { return sbase + kOffBar + 8u * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * bCount);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + 8 * bCount + 4);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_tiles = p.tiles_m * p.tiles_n, n_k = p.K / kBK;

    if (tid == 0) {
        for (int i = 0; i < kRing; ++i) {
            tc::mbar_init(bar(bFull + i), 1);
            tc::mbar_init(bar(bEmpty + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(bar(bAccFull + i), 1);
            tc::mbar_init(bar(bAccEmpty + i), 4);
        }
        tc::mbar_init(bar(bDone), 1);
        tc::mbar_init(bar(bNever), 1);  // nothing arrives: the target of a test's stall
        *abort_flag = 0;
        tc::fence_mbar_init();
        tc::prefetch_map(&ma);
        tc::prefetch_map(&mb);
    }
    if constexpr (kQkv) {
        rope_to_smem(p.qkv.rope, *reinterpret_cast<RopeTable*>(smem + kOffRope), tid, kThreads);
        reinterpret_cast<float*>(smem + kOffWn)[tid] = p.qkv.wn[tid / kD][tid % kD];  // kThreads == 2 * kD
    }
    if (warp == 1) {
        tc::tmem_alloc(smem_u32(tmem_slot), 512);
        tc::tmem_relinquish();
        tc::fence_before_sync();
    }
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    bool failed = false;
    auto fail = [&]() {
        failed = true;
        *abort_flag = 1;
        atomicOr(p.err, kErrTimeout);
    };

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0;  // stages armed (each completed by its two copies)
            for (int t = blockIdx.x; t < n_tiles && !failed; t += gridDim.x) {
                int tm, tn;
                linear_tile(p, t, tm, tn);
                for (int ks = 0; ks < n_k; ++ks, ++it) {
                    const uint32_t s = it % kRing;
                    if (p.stall == tc::kStallProducer && it == 0 &&
                        !tc::mbar_wait(bar(bNever), 0, abort_flag, p.stall_budget)) {
                        fail();
                        break;
                    }
                    if (!tc::mbar_wait(bar(bEmpty + s), ((it / kRing) & 1) ^ 1, abort_flag)) { fail(); break; }
                    const uint32_t dst = sbase + s * kStageBytes;
                    tc::mbar_expect_tx(bar(bFull + s), kStageBytes);
                    tc::tma_load_2d(dst, &ma, ks * kBK, tm * kBM, bar(bFull + s));
                    tc::tma_load_2d(dst + kABytes, &mb, ks * kBK, tn * kBN, bar(bFull + s));
                }
            }
            // every copy issued has landed before the CTA's shared memory is released
            if (!tc::drain_ring(bar(bFull), kRing, it)) atomicOr(p.err, kErrTimeout);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t id = tc::idesc_f16(true, false, kBM, kBN);  // bf16 x bf16, K-major A and B
            const uint64_t da = tc::smem_desc_sw128(sbase, 16, 1024);
            const uint64_t db = tc::smem_desc_sw128(sbase + kABytes, 16, 1024);
            uint32_t it = 0, tc_n = 0;
            for (int t = blockIdx.x; t < n_tiles && !failed; t += gridDim.x, ++tc_n) {
                const uint32_t b = tc_n & 1;
                // the epilogue has drained this accumulator (two tiles ago)
                if (tc_n >= 2 && !tc::mbar_wait(bar(bAccEmpty + b), ((tc_n >> 1) - 1) & 1, abort_flag)) { fail(); break; }
                tc::fence_after_sync();
                for (int ks = 0; ks < n_k; ++ks, ++it) {
                    const uint32_t s = it % kRing;
                    if (!tc::mbar_wait(bar(bFull + s), (it / kRing) & 1, abort_flag)) { fail(); break; }
                    tc::fence_after_sync();
                    const uint32_t so = (s * kStageBytes) >> 4;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        tc::mma_ss(tmem + kBN * b, da + so + ((kk * 32) >> 4), db + so + ((kk * 32) >> 4), id,
                                   (ks > 0) || (kk > 0));
                    tc::mma_commit(bar(bEmpty + s));
                    if (p.stall == tc::kStallMma && it == 0 &&
                        !tc::mbar_wait(bar(bNever), 0, abort_flag, p.stall_budget)) {
                        fail();
                        break;
                    }
                }
                if (failed) break;
                tc::mma_commit(bar(bAccFull + b));
            }
            // every issued MMA has completed before TMEM is released (also on an abort)
            tc::mma_commit(bar(bDone));
            if (!tc::mbar_drain(bar(bDone), 0)) fail();
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------- epilogue
        const int row_in = tid - 128;  // TMEM lane == row of the tile
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        uint32_t tc_n = 0;
        for (int t = blockIdx.x; t < n_tiles && !failed; t += gridDim.x, ++tc_n) {
            int tm, tn;
            linear_tile(p, t, tm, tn);
            const uint32_t b = tc_n & 1;
            bool ok = true;
            if (lane == 0) {
                if (p.stall == tc::kStallConsumer && warp == 4 && tc_n == 0)
                    ok = tc::mbar_wait(bar(bNever), 0, abort_flag, p.stall_budget);
                if (ok) ok = tc::mbar_wait(bar(bAccFull + b), (tc_n >> 1) & 1, abort_flag);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) { fail(); break; }
            tc::fence_after_sync();
            const int row = tm * kBM + row_in;
            const bool row_ok = row < p.rows;
            if constexpr (kQkv) {
                if (!qkv_epilogue(p, smem, tmem + lane_base + kBN * b, row_in, row, row_ok, tn)) atomicOr(p.err, kErrRange);
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(bar(bAccEmpty + b));
                continue;
            }
            __nv_bfloat16* dst = p.y + (size_t)row * p.N + tn * kBN;
            for (int c32 = 0; c32 < kBN / 32; ++c32) {
                uint32_t r[32];
                tc::tmem_ld32(tmem + lane_base + kBN * b + 32 * c32, r);
                tc::tmem_wait_ld_dep(r);
                const int col0 = tn * kBN + 32 * c32;
                if (row_ok && col0 < p.N) {
                    float v[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
                    if (p.bias) {
#pragma unroll
                        for (int e = 0; e < 32; e += 4) {
                            const float4 b4 = *reinterpret_cast<const float4*>(p.bias + col0 + e);
                            v[e] += b4.x; v[e + 1] += b4.y; v[e + 2] += b4.z; v[e + 3] += b4.w;
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 u;
                        u.x = pack_bf16(v[e], v[e + 1]);
                        u.y = pack_bf16(v[e + 2], v[e + 3]);
                        u.z = pack_bf16(v[e + 4], v[e + 5]);
                        u.w = pack_bf16(v[e + 6], v[e + 7]);
                        *reinterpret_cast<uint4*>(dst + 32 * c32 + e) = u;
                    }
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(bar(bAccEmpty + b));
        }
    }

    // the producer has waited out its copies and the issuer its products
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ host

namespace {
bool encode_2d(CUtensorMap* m, const void* base, int inner, int outer, int box_outer) {
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    const cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
    const cuuint32_t box[2] = {(cuuint32_t)lint::kBK, (cuuint32_t)box_outer};
    const cuuint32_t es[2] = {1, 1};
    return tensor_map_encoder()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                                es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool al16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

cudaError_t set_linear_attributes() {
    cudaError_t e = cudaFuncSetAttribute(linear_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         lint::kSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(linear_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, lint::kSmemQkv);
    return e;
}

}  // namespace h3

using namespace h3;

extern "C" h3attn_status h3attn_linear(const h3attn_bf16* x, int rows, int in_features, const h3attn_bf16* w,
                                       int out_features, const float* bias, h3attn_bf16* y,
                                       uint32_t* device_error_flags, void* stream) {
    if (rows < 0 || in_features < 1 || out_features < 1) return H3ATTN_ERR_INVALID_ARG;
    if (in_features % lint::kBK != 0 || out_features % 32 != 0) return H3ATTN_ERR_UNSUPPORTED;
    if (rows == 0) return H3ATTN_OK;
    if (!al16(x) || !al16(w) || !al16(y) || (bias && !al16(bias)) || !device_error_flags ||
        (reinterpret_cast<uintptr_t>(device_error_flags) & 3u))
        return H3ATTN_ERR_INVALID_ARG;
    if ((long long)rows * in_features >= (1LL << 40) || (long long)out_features * in_features >= (1LL << 40))
        return H3ATTN_ERR_CAPACITY;
    const cudaError_t pe = prepare_device();
    if (pe != cudaSuccess) return pe == cudaErrorNotSupported ? H3ATTN_ERR_UNSUPPORTED : H3ATTN_ERR_CUDA;
    const int sms = device_sms();
    CUtensorMap ma, mb;
    if (!encode_2d(&ma, x, in_features, rows, lint::kBM) || !encode_2d(&mb, w, in_features, out_features, lint::kBN))
        return H3ATTN_ERR_INVALID_ARG;
    LinearParams p;
    p.rows = rows;
    p.N = out_features;
    p.K = in_features;
    p.tiles_m = (rows + lint::kBM - 1) / lint::kBM;
    p.tiles_n = (out_features + lint::kBN - 1) / lint::kBN;
    p.bias = bias;
    p.y = reinterpret_cast<__nv_bfloat16*>(y);
    p.err = device_error_flags;
    p.stall = 0;
    p.stall_budget = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(device_error_flags, 0, 4, s) != cudaSuccess) return H3ATTN_ERR_CUDA;
    const int tiles = p.tiles_m * p.tiles_n;
    linear_tc_kernel<false><<<tiles < sms ? tiles : sms, lint::kThreads, lint::kSmem, s>>>(ma, mb, p);
    return cudaGetLastError() == cudaSuccess ? H3ATTN_OK : H3ATTN_ERR_CUDA;
}

namespace h3 {

// The QKV form: y = x W^T + b with W [3 H 128, in_features] (q, k, v heads),
// written as the q, k, v rows plus q^ / k^ into the workspace.
cudaError_t launch_qkv(const Problem& p, const Workspace& ws, const RopeTable* rope, const __nv_bfloat16* x,
                       int in_features, const __nv_bfloat16* w, const float* bias, __nv_bfloat16* q, __nv_bfloat16* k,
                       __nv_bfloat16* v, cudaStream_t st) {
    if (p.seq.S == 0) return cudaSuccess;
    const int sms = device_sms();
    if (sms < 1) return cudaErrorNotSupported;
    const int D = p.H * kD, N = 3 * D;
    CUtensorMap ma, mb;
    if (!encode_2d(&ma, x, in_features, p.seq.S, lint::kBM) || !encode_2d(&mb, w, in_features, N, lint::kBN))
        return cudaErrorInvalidValue;
    LinearParams lp;
    lp.rows = p.seq.S;
    lp.N = N;
    lp.K = in_features;
    lp.tiles_m = (lp.rows + lint::kBM - 1) / lint::kBM;
    lp.tiles_n = (N + lint::kBN - 1) / lint::kBN;
    lp.bias = bias;
    lp.y = nullptr;
    lp.err = ws.plan.err;
    lp.stall = p.stall.kernel == kStallKernelQkv ? p.stall.role : 0;
    lp.stall_budget = p.stall.budget;
    lp.qkv.H = p.H;
    lp.qkv.D = D;
    lp.qkv.eps = p.eps;
    lp.qkv.wn[0] = p.wq;
    lp.qkv.wn[1] = p.wk;
    lp.qkv.pos[0] = p.seq.pos_t;
    lp.qkv.pos[1] = p.seq.pos_h;
    lp.qkv.pos[2] = p.seq.pos_w;
    lp.qkv.out[0] = q;
    lp.qkv.out[1] = k;
    lp.qkv.out[2] = v;
    lp.qkv.hat[0] = ws.qhat;
    lp.qkv.hat[1] = ws.khat;
    lp.qkv.rope_cs = ws.rope_cs;
    lp.qkv.rope = *rope;
    const int tiles = lp.tiles_m * lp.tiles_n;
    linear_tc_kernel<true><<<tiles < sms ? tiles : sms, lint::kThreads, lint::kSmemQkv, st>>>(ma, mb, lp);
    return cudaGetLastError();
}

}  // namespace h3
