// common.cuh -- shared device helpers and launch parameters of libh3attn.
//
// Layout conventions (all kernels): bf16 tensors are token-major [S, H, 128];
// element (i, h, c) sits at (i * H + h) * 128 + c.  Samples are addressed by
// the segment offsets; every tile of queries or keys is anchored at its sample's
// first token, never at a global tile boundary, so that a sample's arithmetic
// is the same whether it runs alone or packed with others.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace h3 {

constexpr int kD = 128;  // head dim

// Bits of the device error word.
constexpr unsigned kErrBadOffsets = 1u;
constexpr unsigned kErrTimeout = 2u;
constexpr unsigned kErrRange = 4u;  // a rotated q^/k^ or dS value left the fp16 range

// Rotary layout, per channel group of 4 (lane l of a warp owns channels 4l..4l+3).
// A section of n channels pairs channel o+j with o+j+n/2, so with n a multiple
// of 8 the partner of a group is another whole group.
struct RopeTable {
    float inv_freq[kD];       // frequency of the pair channel c belongs to (0 if not rotated)
    int8_t axis[32];          // 0/1/2 = t/h/w, -1 = not rotated
    int8_t partner[32];       // lane holding the paired channels
    int8_t second[32];        // 1 if this group is the second half of its section
    int8_t pad[32];           // keeps the size a multiple of 16 bytes
};

// Per-call plan written on the device from seg_offsets: samples ordered by
// decreasing length (ties by index) and cumulative tile counts in that order.
struct Plan {
    int* order;      // [max_samples] sample index of rank r
    int* cum64;      // [max_samples + 1] tiles of 64 tokens before rank r
    int* cum128;     // [max_samples + 1] tiles of 128 tokens before rank r
    int* cum256;     // [max_samples + 1] blocks of 256 tokens before rank r
    int* rank_of;    // [max_samples] rank of sample s
    int* cumsq;      // [max_samples + 1] sum of (tiles of 128 tokens)^2 before rank r: the
                     //   128 x 128 score blocks of one head of the samples before it
    unsigned* err;   // device error word
};

struct Seq {
    const int32_t* seg;   // [n + 1] offsets
    const int32_t* pos_t;
    const int32_t* pos_h;
    const int32_t* pos_w;
    int n;                // samples
    int S;                // tokens
};

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);  // round to nearest even
    return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 r = __floats2half2_rn(lo, hi);  // round to nearest even
    return *reinterpret_cast<uint32_t*>(&r);
}

// 2^x on the SFU (MUFU.EX2); results below 2^-126 flush to zero.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed pairs of FP32 values for the f32x2 FMA / ADD / MUL instructions of
// sm_100-class SMs (one instruction does two lanes' worth of the same op).
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2unpack(uint64_t v, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Column-pair steps of the softmax gradient on 64-bit register pairs (two FP32
// values), written as single asm blocks so that the halves of a pair are plain
// register views and no moves are needed between the packed and scalar forms.
//   p2 = 2^(s2 * c2 + n2) per half (ex2.approx, flush-to-zero below 2^-126)
__device__ __forceinline__ uint64_t exp2_pair(uint64_t s2, uint64_t c2, uint64_t n2) {
    uint64_t p2;
    asm("{\n.reg .b64 t;\n.reg .f32 a0, a1, q0, q1;\n"
        "fma.rn.f32x2 t, %1, %2, %3;\n"
        "mov.b64 {a0, a1}, t;\n"
        "ex2.approx.ftz.f32 q0, a0;\n"
        "ex2.approx.ftz.f32 q1, a1;\n"
        "mov.b64 %0, {q0, q1};\n}"
        : "=l"(p2) : "l"(s2), "l"(c2), "l"(n2));
    return p2;
}
//   p2 = 2^(s2 * c2 + n2) per half on the FMA pipe instead of the SFU (the
//   softmax needs one 2^x per score; a kernel can move a fixed share of its
//   columns off the SFU with this - measured slower on this GPU, so the
//   kernels' shares are zero, and h3attn_debug_exp2 keeps it tested):
//   x = s c + n, clamped to >= -127;  n = floor(x) exactly (a
//   round-toward-minus-infinity addition of 1.5 * 2^23 leaves floor(x) in the
//   low mantissa bits) and f = x - n rounded once (exact unless -1 < x < 0 is
//   small, where the rounding moves 2^f by at most 2^-25 ln 2 relative);  2^f = p(f) = 1 + c1 f + ... + c5 f^5 by Horner with
//   fused multiply-adds, the minimax polynomial of relative error with p(0) = 1
//   (Remez exchange; coefficients from csrc/fit_exp2_poly.py, max relative
//   error 1.4e-7 evaluated in float32, about the SFU's own);  2^n from the
//   exponent field ((floor(x) + 127) << 23, which is +0 for x < -126: results
//   below 2^-126 are 0, as with the flush-to-zero SFU instruction).  Valid for
//   x <= 127; the softmax passes x <= 8.
__device__ __forceinline__ uint64_t exp2_poly_pair(uint64_t s2, uint64_t c2, uint64_t n2) {
    uint64_t r;
    asm("{\n.reg .b64 x, t, n, f, p, e, k;\n.reg .f32 x0, x1;\n.reg .b32 t0, t1, e0, e1;\n"
        "fma.rn.f32x2 x, %1, %2, %3;\n"
        "mov.b64 {x0, x1}, x;\n"
        "max.f32 x0, x0, 0fC2FE0000;\n"          // -127
        "max.f32 x1, x1, 0fC2FE0000;\n"
        "mov.b64 x, {x0, x1};\n"
        "mov.b64 k, {0f4B400000, 0f4B400000};\n"  // 1.5 * 2^23
        "add.rm.f32x2 t, x, k;\n"
        "sub.rn.f32x2 n, t, k;\n"
        "sub.rn.f32x2 f, x, n;\n"
        "mov.b64 p, {0f3AF4BA7D, 0f3AF4BA7D};\n"  // c5
        "mov.b64 k, {0f3C13BC2B, 0f3C13BC2B};\n"  // c4
        "fma.rn.f32x2 p, p, f, k;\n"
        "mov.b64 k, {0f3D648E73, 0f3D648E73};\n"  // c3
        "fma.rn.f32x2 p, p, f, k;\n"
        "mov.b64 k, {0f3E75EDAB, 0f3E75EDAB};\n"  // c2
        "fma.rn.f32x2 p, p, f, k;\n"
        "mov.b64 k, {0f3F31725D, 0f3F31725D};\n"  // c1
        "fma.rn.f32x2 p, p, f, k;\n"
        "mov.b64 k, {0f3F800000, 0f3F800000};\n"  // 1
        "fma.rn.f32x2 p, p, f, k;\n"
        "mov.b64 {t0, t1}, t;\n"
        "shl.b32 e0, t0, 23;\n"
        "shl.b32 e1, t1, 23;\n"
        "add.u32 e0, e0, 0x3F800000;\n"
        "add.u32 e1, e1, 0x3F800000;\n"
        "mov.b64 e, {e0, e1};\n"
        "mul.rn.f32x2 %0, p, e;\n}"
        : "=l"(r) : "l"(s2), "l"(c2), "l"(n2));
    return r;
}
// max(a, b, c) in one instruction
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// the two halves of a pair
__device__ __forceinline__ float pair_lo(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float pair_hi(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }
// bf16x2 of a pair, low half first (round to nearest even)
__device__ __forceinline__ uint32_t bf16_pair(uint64_t p2) {
    uint32_t r;
    asm("{\n.reg .f32 a0, a1;\nmov.b64 {a0, a1}, %1;\ncvt.rn.bf16x2.f32 %0, a1, a0;\n}" : "=r"(r) : "l"(p2));
    return r;
}
//   dS = p2 * (d2 + n2) per half, as f16x2, low half first (round to nearest even)
__device__ __forceinline__ uint32_t ds_f16_pair(uint64_t p2, uint64_t d2, uint64_t n2) {
    uint32_t r;
    asm("{\n.reg .b64 t;\n.reg .f32 a0, a1;\n"
        "add.rn.f32x2 t, %2, %3;\n"
        "mul.rn.f32x2 t, %1, t;\n"
        "mov.b64 {a0, a1}, t;\n"
        "cvt.rn.f16x2.f32 %0, a1, a0;\n}"
        : "=r"(r) : "l"(p2), "l"(d2), "l"(n2));
    return r;
}
// Zeroes the halves of a pair whose column (col, col + 1) is not below `valid`.
__device__ __forceinline__ uint64_t mask_pair(uint64_t p2, int col, int valid) {
    float a, b;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(p2));
    a = col < valid ? a : 0.f;
    b = col + 1 < valid ? b : 0.f;
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}

// Item of a persistent CTA's k-th turn: turn k deals items [k G, k G + G) to the
// G CTAs, in CTA order on even turns and in reverse on odd ones.  The items come
// longest sample first, so alternating the direction evens out the per-CTA
// totals that plain round-robin tilts toward the low CTA indices (13539-token
// pack, H = 48: the largest forward share falls from 3.6% to 2.6% above the
// mean).  Every role of a CTA walks the same sequence.
__device__ __forceinline__ int turn_item(int k) {
    const int c = (k & 1) ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x;
    return k * (int)gridDim.x + c;
}

__device__ __forceinline__ float warp_sum(float v) {
    // fixed butterfly: every lane ends with the same, order-fixed sum
    v += __shfl_xor_sync(0xffffffffu, v, 16);
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    return v;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Maps a tile index of the plan (tiles of `tile` tokens, samples in rank order)
// to its sample and the tile's first token.  Returns false past the last tile.
__device__ __forceinline__ bool plan_tile(const int* __restrict__ cum, const int* __restrict__ order,
                                          const int32_t* __restrict__ seg, int n, int tile, int t,
                                          int& sample, int& row0, int& row_end, int& local) {
    if (t >= cum[n]) return false;
    int lo = 0, hi = n;  // find rank r with cum[r] <= t < cum[r+1]
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (cum[mid] <= t) lo = mid; else hi = mid;
    }
    sample = order[lo];
    local = t - cum[lo];
    row0 = seg[sample] + local * tile;
    row_end = seg[sample + 1];
    return true;
}

// ------------------------------------------------------- launch interface

struct Workspace {
    __half* qhat;            // [max_tokens, H, 128] rotated, normalised q (fp16)
    __half* khat;            // [max_tokens, H, 128] rotated, normalised k (fp16)
    float* delta;            // [H, max_tokens]
    float* dqhat32;          // [max_tokens, H, 128] scale * dq^ (FP32), backward only
    float* dkhat32;          // [max_tokens, H, 128] scale * dk^ (FP32), backward only
    float* rope_cs;          // [max_tokens, 2, 128] cos / sin of the rotary angles, backward only
    float* dwq_part;         // [max_tiles64, H, 128]
    float* dwk_part;         // [max_tiles64, H, 128]
    float* dwq_sample;       // [max_samples, 128]
    float* dwk_sample;       // [max_samples, 128]
    float* dwq_head;         // [max_samples, H, 128] per (sample, head) partials of the last backward
    float* dwk_head;         // [max_samples, H, 128]
    Plan plan;
    // canonical key order only (null otherwise)
    int32_t* perm;           // [max_tokens] packed index of canonical slot c
    int32_t* pos_c;          // [3, max_tokens] positions in canonical order
    float* lse_c;            // [H, max_tokens] softmax row terms in canonical order
    __nv_bfloat16* rows_c[4];  // [max_tokens, H, 128] each, canonical order: v, out, dout, dv
    uint4* keys;             // [max_tokens] sort keys of the canonical order
    // stored dS (null if the handle recomputes it in the dQ kernel): fp16 128 x 128
    // blocks of dS^T laid out [32-query chunk][key][32 queries], block (sample of rank
    // r, head h, key tile j, query tile i) at H cumsq[r] + h nq^2 + j nq + i, nq = the
    // sample's 128-token tiles
    __half* ds;
    long long ds_blocks;     // capacity in blocks
};

// A test's request that one kernel of the next call stall one of its roles
// once, on a bounded wait that nothing completes (see tc::StallRole), to
// exercise the kernel's unwinding.  kernel 0 = none.
enum StallKernel { kStallKernelNone = 0, kStallKernelFwd = 1, kStallKernelDkdv = 2, kStallKernelDq = 3,
                   kStallKernelQkv = 4 };
struct StallRequest {
    int kernel = 0;
    int role = 0;
    long long budget = 0;  // clock cycles
};

struct Problem {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const float* wq;
    const float* wk;
    Seq seq;
    int H;
    float eps;
    float scale;
    // Canonical key order: packed row of the token in canonical slot i (null =
    // identity).  Kernels that address the caller's q, k or out rows one token
    // at a time (prologue, Delta, row backward) read and write them through it.
    const int32_t* rowmap = nullptr;
    StallRequest stall;  // tests only
};

// Stages of one call, in launch order (timed separately when stage timing is on).
// Values match the h3attn_stage enum of the C ABI.
enum Stage { kStagePlan = 0, kStagePrologue, kStageFwd, kStageDelta, kStageDkdv, kStageDq, kStageDw, kStageRows,
             kStageOrder, kStagePermute, kStageQkv, kStages };

cudaError_t launch_plan(const Problem& p, const Workspace& ws, cudaStream_t st);
cudaError_t launch_prologue(const Problem& p, const Workspace& ws, const RopeTable* rope, cudaStream_t st);
cudaError_t launch_fwd(const Problem& p, const Workspace& ws, __nv_bfloat16* out, float* lse, cudaStream_t st);
cudaError_t launch_bwd_delta(const Problem& p, const Workspace& ws, const __nv_bfloat16* out,
                             const __nv_bfloat16* dout, cudaStream_t st);
cudaError_t launch_bwd_dkdv(const Problem& p, const Workspace& ws, const float* lse,
                            const __nv_bfloat16* dout, __nv_bfloat16* dk, __nv_bfloat16* dv, cudaStream_t st);
// dQ; with the stored dS (ws.ds) also the row backward of q and k (dq, dk), so
// launch_bwd_rows then has nothing left to do
cudaError_t launch_bwd_dq(const Problem& p, const Workspace& ws, const float* lse, const __nv_bfloat16* dout,
                          const RopeTable* rope, __nv_bfloat16* dq, __nv_bfloat16* dk, cudaStream_t st);
cudaError_t launch_bwd_rows(const Problem& p, const Workspace& ws, const RopeTable* rope, __nv_bfloat16* dq,
                            __nv_bfloat16* dk, cudaStream_t st);
cudaError_t launch_order(const Problem& p, const __nv_bfloat16* dout, uint4* keys, int32_t* perm, unsigned* err,
                         cudaStream_t st);
// Gather (canonical copy row c <- packed row perm[c]) or scatter (the reverse) of
// up to six [S, H, 128] bf16 tensors, the [H, S] row terms (either may be
// absent) and, gathering only, the three position rows.
cudaError_t launch_permute(const int32_t* perm, int S, int H, int ntensors, const void* const* src, void* const* dst,
                           const float* lse_src, float* lse_dst, const int32_t* const pos_src[3], int32_t* pos_dst[3],
                           bool scatter, unsigned* err, cudaStream_t st);
// cos / sin of every channel's rotary angle per token into ws.rope_cs (bwd_rows.cu).
cudaError_t launch_rope_table(const Problem& p, const Workspace& ws, const RopeTable* rope, cudaStream_t st);
// The fused QKV projection (linear_tc.cu): q, k, v rows and the workspace's q^, k^
// (reads the rotary table launch_rope_table wrote).
cudaError_t launch_qkv(const Problem& p, const Workspace& ws, const RopeTable* rope, const __nv_bfloat16* x,
                       int in_features, const __nv_bfloat16* w, const float* bias, __nv_bfloat16* q, __nv_bfloat16* k,
                       __nv_bfloat16* v, cudaStream_t st);
cudaError_t launch_bwd_dw(const Problem& p, const Workspace& ws, float* dwq, float* dwk, float* dwq_s,
                          float* dwk_s, cudaStream_t st);
// The fixed-order reduction of per-(sample, head) norm-weight partials [n][H][128]:
// per sample over heads ascending into per_sample [n][128], then over samples
// ascending into total [128] (bwd_rows.cu).
cudaError_t launch_dw_combine(const float* partials, int n, int H, float* per_sample, float* total,
                              cudaStream_t st);

}  // namespace h3
