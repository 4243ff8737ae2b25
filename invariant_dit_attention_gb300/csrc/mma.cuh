// mma.cuh -- warp-level bf16/fp16 MMA (m16n8k16), ldmatrix and cp.async helpers
// with a 128-byte XOR swizzle for [rows][128] bf16 tiles in shared memory.
#pragma once

#include "common.cuh"

namespace h3 {

// Byte offset of 16-byte chunk `ch` (0..15) of row `r` in a [rows][128] bf16
// tile: rows are 256 bytes, chunk index XORed with the row's low 3 bits so
// that 8 consecutive rows at one chunk hit 8 different bank groups.
__device__ __forceinline__ uint32_t swz(int r, int ch) { return (uint32_t)(r * 256 + ((ch ^ (r & 7)) << 4)); }

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma16816_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

// 16-byte async copy; src_bytes = 0 writes zeros (used for rows past a sample's end).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" :: "r"(dst), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" :: "n"(N)); }

// Loads rows [row0, row0 + ROWS) of head h of a [S, H, 128] tensor into a
// swizzled tile; rows at or past row_end are zero-filled.  All threads of the
// block take part.
template <int ROWS, int THREADS, class T>
__device__ __forceinline__ void load_tile_async(uint32_t tile, const T* __restrict__ g, int H, int h,
                                                int row0, int row_end, int tid) {
    static_assert(sizeof(T) == 2, "16-bit elements");
#pragma unroll
    for (int i = tid; i < ROWS * 16; i += THREADS) {
        int r = i >> 4, ch = i & 15;
        int row = row0 + r;
        bool ok = row < row_end;
        const T* src = g + ((size_t)(ok ? row : row0) * H + h) * kD + ch * 8;
        cp_async16(tile + swz(r, ch), src, ok ? 16 : 0);
    }
}

// A fragments (16 rows x 16 k) of rows [r0, r0+16), k-chunk kk (16 columns).
__device__ __forceinline__ void ldsm_a(uint32_t (&a)[4], uint32_t tile, int r0, int kk, int lane) {
    int r = r0 + (lane & 15);
    int ch = kk * 2 + (lane >> 4);
    ldsm_x4(a, tile + swz(r, ch));
}

// B fragments for two n-tiles (rows n0..n0+15 of a [n][k] tile), k-chunk kk:
// b[0], b[1] for n-tile n0..n0+7 and b[2], b[3] for n0+8..n0+15.
__device__ __forceinline__ void ldsm_b_nk(uint32_t (&b)[4], uint32_t tile, int n0, int kk, int lane) {
    int r = n0 + (lane & 7) + ((lane >> 4) << 3);
    int ch = kk * 2 + ((lane >> 3) & 1);
    ldsm_x4(b, tile + swz(r, ch));
}

// B fragments from a [k][n] tile (k rows, n contiguous): k rows k0..k0+15,
// n columns n0..n0+15 (two n-tiles), via ldmatrix.trans.
__device__ __forceinline__ void ldsm_b_kn(uint32_t (&b)[4], uint32_t tile, int k0, int n0, int lane) {
    int r = k0 + (lane & 7) + (((lane >> 3) & 1) << 3);
    int ch = (n0 >> 3) + (lane >> 4);
    ldsm_x4_t(b, tile + swz(r, ch));
}

}  // namespace h3
