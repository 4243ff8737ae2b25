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
#include <cudaTypedefs.h>

#include "../../include/h3attn.h"
#include "common.cuh"
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
constexpr int kGroupM = 16;                     // row tiles per raster group
enum { bFull = 0, bEmpty = bFull + kRing, bAccFull = bEmpty + kRing, bAccEmpty = bAccFull + 2, bDone = bAccEmpty + 2,
       bCount };
}  // namespace lint

struct LinearParams {
    int rows, N, K;
    int tiles_m, tiles_n;
    const float* bias;
    __nv_bfloat16* y;
    unsigned* err;
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

__global__ void __launch_bounds__(lint::kThreads, 1)
linear_tc_kernel(const __grid_constant__ CUtensorMap ma, const __grid_constant__ CUtensorMap mb, const LinearParams p) {
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
        *abort_flag = 0;
        tc::fence_mbar_init();
        tc::prefetch_map(&ma);
        tc::prefetch_map(&mb);
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
            uint32_t it = 0;
            for (int t = blockIdx.x; t < n_tiles && !failed; t += gridDim.x) {
                int tm, tn;
                linear_tile(p, t, tm, tn);
                for (int ks = 0; ks < n_k; ++ks, ++it) {
                    const uint32_t s = it % kRing;
                    if (!tc::mbar_wait(bar(bEmpty + s), ((it / kRing) & 1) ^ 1, abort_flag)) { fail(); break; }
                    const uint32_t dst = sbase + s * kStageBytes;
                    tc::mbar_expect_tx(bar(bFull + s), kStageBytes);
                    tc::tma_load_2d(dst, &ma, ks * kBK, tm * kBM, bar(bFull + s));
                    tc::tma_load_2d(dst + kABytes, &mb, ks * kBK, tn * kBN, bar(bFull + s));
                }
            }
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
                }
                if (failed) break;
                tc::mma_commit(bar(bAccFull + b));
            }
            tc::mma_commit(bar(bDone));
            if (!tc::mbar_wait(bar(bDone), 0, abort_flag) && !failed) fail();
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
            if (lane == 0) ok = tc::mbar_wait(bar(bAccFull + b), (tc_n >> 1) & 1, abort_flag);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) { fail(); break; }
            tc::fence_after_sync();
            const int row = tm * kBM + row_in;
            const bool row_ok = row < p.rows;
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

    __syncthreads();
    if (warp == 0 && lane == 0 && *abort_flag) {
        // let any TMA still in flight land before the CTA's shared memory goes away
        const long long t0 = clock64();
        while (clock64() - t0 < 20000000LL) {
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ host

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode_l = nullptr;
int g_sms_l = 0;
int g_dev_l = -1;

bool encode_2d(CUtensorMap* m, const void* base, int inner, int outer, int box_outer) {
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    const cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
    const cuuint32_t box[2] = {(cuuint32_t)lint::kBK, (cuuint32_t)box_outer};
    const cuuint32_t es[2] = {1, 1};
    return g_encode_l(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

h3attn_status init_linear(int dev) {
    if (!g_encode_l) {
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", reinterpret_cast<void**>(&g_encode_l),
                                                         12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !g_encode_l) return H3ATTN_ERR_CUDA;
    }
    if (g_dev_l != dev) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return H3ATTN_ERR_CUDA;
        if (!(prop.major == 10 && prop.minor == 3)) return H3ATTN_ERR_UNSUPPORTED;
        if (cudaFuncSetAttribute(linear_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, lint::kSmem) !=
            cudaSuccess)
            return H3ATTN_ERR_CUDA;
        g_sms_l = prop.multiProcessorCount;
        g_dev_l = dev;
    }
    return H3ATTN_OK;
}

bool al16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

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
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return H3ATTN_ERR_CUDA;
    const h3attn_status st = init_linear(dev);
    if (st != H3ATTN_OK) return st;
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
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(device_error_flags, 0, 4, s) != cudaSuccess) return H3ATTN_ERR_CUDA;
    const int tiles = p.tiles_m * p.tiles_n;
    linear_tc_kernel<<<tiles < g_sms_l ? tiles : g_sms_l, lint::kThreads, lint::kSmem, s>>>(ma, mb, p);
    return cudaGetLastError() == cudaSuccess ? H3ATTN_OK : H3ATTN_ERR_CUDA;
}
