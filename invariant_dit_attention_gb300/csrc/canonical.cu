// canonical.cu -- the canonical token order and the row permutations around it.
//
// The attention core sums keys (forward, dQ) and queries (dK, dV, the weight
// gradients) in the order the tokens sit in memory, so permuting a sample's
// packed rows together with their positions changes output bits: control H-C3
// in the Results of the "ws1_one_h3_block" page of RL-Kernel (PR #539).  With
// the canonical key order a call first sorts each sample's tokens by
//   1. position (t, h, w) as signed integers, t first,
//   2. the k, v, q (and, in the backward, dout) rows, all heads in memory
//      order, compared as sequences of bf16 bit patterns read as unsigned
//      16-bit integers,
//   3. packed index (tokens equal up to here are identical in every input),
// runs the same kernels on the tokens in that order (gathering or mapping each
// per-token input) and scatters the per-token outputs back.  What the kernels
// see then depends only on each sample's multiset of tokens, and they are
// deterministic with tiles anchored at the sample start, so every output bit
// is independent of the packed order.
//
// The sort is a rank count: the rank of token i is the number of tokens of its
// sample that come before it.  A sample of L tokens costs L^2 comparisons of a
// 16-byte key (position plus the first two bf16 of the k row); equal keys fall
// back to comparing the rows in global memory.
// The permutations are plain row copies, bound by HBM bandwidth; the kernels
// that address q, k and out one row at a time read and write them through the
// order instead (Problem::rowmap), so only the rows that other kernels move by
// TMA or store as tiles are copied: v and dout in, out and dv back.
#include "common.cuh"

namespace h3 {

namespace {

constexpr int kOrdThreads = 256;
constexpr int kOrdTokens = kOrdThreads / 32;  // one warp per token

struct OrderArgs {
    const int32_t* seg;
    int n, S;
    const int32_t* pos[3];
    const uint4* rows[4];  // k, v, q, dout (dout may be absent)
    int nrows;
    int row_vecs;  // 16-byte vectors per token row: H * 128 * 2 / 16
    ulonglong2* keys;  // [S] sort keys
    int32_t* perm;
    unsigned* err;
};

// Order-preserving map of int32 onto uint32.
__device__ __forceinline__ uint64_t ukey(int32_t x) { return static_cast<uint32_t>(x) ^ 0x80000000u; }

// Sort key of every token as two 64-bit words compared in turn: (t, h) and
// (w, first two bf16 of the k row; element 0 is the low half of the first
// 32-bit word, so it is rotated to the high half).  Also starts perm as the
// identity, so that slots an invalid seg_offsets array leaves unranked still
// name a token of the batch.
__global__ void __launch_bounds__(256) key_kernel(const __grid_constant__ OrderArgs A) {
    const int j = blockIdx.x * 256 + threadIdx.x;
    if (j >= A.S) return;
    const uint32_t w = reinterpret_cast<const uint32_t*>(A.rows[0] + (size_t)j * A.row_vecs)[0];
    A.keys[j] = make_ulonglong2((ukey(A.pos[0][j]) << 32) | ukey(A.pos[1][j]),
                                (ukey(A.pos[2][j]) << 32) | ((w << 16) | (w >> 16)));
    A.perm[j] = j;
}

// Two bf16 in memory order: element 0 in the low half.
__device__ __forceinline__ int cmp_pair(uint32_t a, uint32_t b) {
    if (a == b) return 0;
    const uint32_t al = a & 0xffffu, bl = b & 0xffffu;
    if (al != bl) return al < bl ? -1 : 1;
    return (a >> 16) < (b >> 16) ? -1 : 1;
}

// Rows of tokens j and i, lexicographically over k, v, q (, dout).
__device__ int cmp_rows(const OrderArgs& A, int j, int i) {
    for (int r = 0; r < A.nrows; ++r) {
        const uint4* __restrict__ x = A.rows[r] + (size_t)j * A.row_vecs;
        const uint4* __restrict__ y = A.rows[r] + (size_t)i * A.row_vecs;
        for (int e = 0; e < A.row_vecs; ++e) {
            const uint4 a = x[e], b = y[e];
            int c = cmp_pair(a.x, b.x);
            if (!c) c = cmp_pair(a.y, b.y);
            if (!c) c = cmp_pair(a.z, b.z);
            if (!c) c = cmp_pair(a.w, b.w);
            if (c) return c;
        }
    }
    return 0;
}

// One warp per token: its lanes stride over the token's sample comparing keys
// (read through L1: the warps of a block share a sample's keys) and add their
// counts at the end.
__global__ void __launch_bounds__(kOrdThreads) order_kernel(const __grid_constant__ OrderArgs A) {
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * kOrdTokens + (threadIdx.x >> 5);
    if (i >= A.S) return;  // whole warps leave together
    int lo = 0, hi = A.n;  // sample of token i: the last s with seg[s] <= i
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (A.seg[mid] <= i) lo = mid; else hi = mid;
    }
    const int a = max(A.seg[lo], 0), b = min(A.seg[lo + 1], A.S);
    if (!(a <= i && i < b)) {
        if (lane == 0) atomicOr(A.err, kErrBadOffsets);
        return;
    }
    const ulonglong2* __restrict__ K = A.keys;
    const ulonglong2 mine = K[i];
    int rank = 0;
#pragma unroll 4
    for (int j = a + lane; j < b; j += 32) {
        const ulonglong2 kj = __ldg(K + j);
        rank += (kj.x < mine.x) | ((kj.x == mine.x) & (kj.y < mine.y));
        if (kj.x == mine.x && kj.y == mine.y && j != i) {
            const int c = cmp_rows(A, j, i);
            rank += c < 0 || (c == 0 && j < i);
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
    if (lane == 0) {
        if (a + rank < b) A.perm[a + rank] = i;
        else atomicOr(A.err, kErrBadOffsets);
    }
}

constexpr int kPermWarps = 8;
constexpr int kMaxPermTensors = 6;

struct PermArgs {
    const uint4* src[kMaxPermTensors];
    uint4* dst[kMaxPermTensors];
};

// Row c of the canonical copy <-> row perm[c] of the packed tensor; one warp
// per (row, tensor).  A perm value outside [0, S) (only after bad offsets)
// is reported and skipped.
__global__ void __launch_bounds__(kPermWarps * 32)
permute_rows_kernel(const __grid_constant__ PermArgs P, const int32_t* __restrict__ perm, int S, int row_vecs, int scatter, unsigned* err) {
    const int lane = threadIdx.x & 31;
    const int c = blockIdx.x * kPermWarps + (threadIdx.x >> 5);
    if (c >= S) return;
    const int t = perm[c];
    if (t < 0 || t >= S) {
        if (lane == 0) atomicOr(err, kErrBadOffsets);
        return;
    }
    const size_t from = (size_t)(scatter ? c : t) * row_vecs, to = (size_t)(scatter ? t : c) * row_vecs;
    const uint4* __restrict__ s = P.src[blockIdx.y] + from;
    uint4* __restrict__ d = P.dst[blockIdx.y] + to;
#pragma unroll 4
    for (int e = lane; e < row_vecs; e += 32) d[e] = __ldcs(s + e);
}

// The [H, S] softmax row terms (gather or scatter) and, when gathering, the
// three position rows.
__global__ void __launch_bounds__(256)
permute_small_kernel(const int32_t* __restrict__ perm, int S, int H, const float* __restrict__ lse_src,
                     float* __restrict__ lse_dst, const int32_t* p0, const int32_t* p1, const int32_t* p2,
                     int32_t* d0, int32_t* d1, int32_t* d2, int scatter) {
    const long total = (long)(H + 1) * S;
    for (long x = blockIdx.x * (long)blockDim.x + threadIdx.x; x < total; x += (long)gridDim.x * blockDim.x) {
        const int r = (int)(x / S), c = (int)(x % S);
        const int t = perm[c];
        if (t < 0 || t >= S) continue;  // reported by permute_rows_kernel
        if (r < H) {
            if (lse_src) {
                if (scatter) lse_dst[(size_t)r * S + t] = lse_src[(size_t)r * S + c];
                else lse_dst[(size_t)r * S + c] = lse_src[(size_t)r * S + t];
            }
        } else if (d0) {
            d0[c] = p0[t];
            d1[c] = p1[t];
            d2[c] = p2[t];
        }
    }
}

}  // namespace

cudaError_t launch_order(const Problem& p, const __nv_bfloat16* dout, uint4* keys, int32_t* perm, unsigned* err,
                         cudaStream_t st) {
    if (p.seq.S == 0) return cudaSuccess;
    OrderArgs A;
    A.seg = p.seq.seg;
    A.n = p.seq.n;
    A.S = p.seq.S;
    A.pos[0] = p.seq.pos_t;
    A.pos[1] = p.seq.pos_h;
    A.pos[2] = p.seq.pos_w;
    A.rows[0] = reinterpret_cast<const uint4*>(p.k);
    A.rows[1] = reinterpret_cast<const uint4*>(p.v);
    A.rows[2] = reinterpret_cast<const uint4*>(p.q);
    A.rows[3] = reinterpret_cast<const uint4*>(dout);
    A.nrows = dout ? 4 : 3;
    A.row_vecs = p.H * kD * 2 / 16;
    A.keys = reinterpret_cast<ulonglong2*>(keys);
    A.perm = perm;
    A.err = err;
    key_kernel<<<(p.seq.S + 255) / 256, 256, 0, st>>>(A);
    order_kernel<<<(p.seq.S + kOrdTokens - 1) / kOrdTokens, kOrdThreads, 0, st>>>(A);
    return cudaGetLastError();
}

cudaError_t launch_permute(const int32_t* perm, int S, int H, int ntensors, const void* const* src, void* const* dst,
                           const float* lse_src, float* lse_dst, const int32_t* const pos_src[3], int32_t* pos_dst[3],
                           bool scatter, unsigned* err, cudaStream_t st) {
    if (S == 0) return cudaSuccess;
    if (ntensors < 0 || ntensors > kMaxPermTensors) return cudaErrorInvalidValue;
    if (ntensors > 0) {
        PermArgs P;
        for (int t = 0; t < kMaxPermTensors; ++t) {
            P.src[t] = t < ntensors ? static_cast<const uint4*>(src[t]) : nullptr;
            P.dst[t] = t < ntensors ? static_cast<uint4*>(dst[t]) : nullptr;
        }
        dim3 grid((S + kPermWarps - 1) / kPermWarps, ntensors);
        permute_rows_kernel<<<grid, kPermWarps * 32, 0, st>>>(P, perm, S, H * kD * 2 / 16, scatter ? 1 : 0, err);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const bool pos = pos_src && pos_dst && !scatter;
    if (!lse_src && !pos) return cudaSuccess;
    const long total = (long)(H + 1) * S;
    const int blocks = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
    permute_small_kernel<<<blocks, 256, 0, st>>>(perm, S, H, lse_src, lse_dst, pos ? pos_src[0] : nullptr,
                                                 pos ? pos_src[1] : nullptr, pos ? pos_src[2] : nullptr,
                                                 pos ? pos_dst[0] : nullptr, pos ? pos_dst[1] : nullptr,
                                                 pos ? pos_dst[2] : nullptr, scatter ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace h3
