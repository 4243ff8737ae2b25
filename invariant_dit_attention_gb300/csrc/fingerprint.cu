// fingerprint.cu -- a 64-bit fingerprint of a device buffer's bytes, computed on
// the GPU, so that runs can be compared without copying their outputs to the
// host (the "ws1_full_h3_transformer" page of RL-Kernel, PR #571, Status: the
// rollout and training trajectories are compared twice each with GPU-side
// checksum fingerprints).
//
// Definition.  The buffer is read as little-endian 64-bit words w_0 .. w_{m-1}
// (the last word zero-padded when the size is not a multiple of 8).  With
// mix() the finaliser of the splitmix64 generator (Steele, Lea and Flood,
// "Fast splittable pseudorandom number generators", OOPSLA 2014, in the
// variant with shifts 30, 27, 31 published with Vigna's splitmix64):
//   fingerprint = mix( sum_i mix(w_i + (i + 1) * G) + bytes )  mod 2^64,
// G = 0x9e3779b97f4a7c15.  Each word is salted with its index, so moving a
// value changes the fingerprint; the sum is an integer sum mod 2^64, whose
// value does not depend on the order in which the GPU's threads add it up, so
// the fingerprint is a pure function of the bytes.
#include "../../include/h3attn.h"
#include "common.cuh"
#include "host.cuh"

namespace h3 {
namespace {

constexpr uint64_t kGolden = 0x9e3779b97f4a7c15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

// Sum of the salted, mixed words (grid-stride), added into *acc.
__global__ void __launch_bounds__(256)
fingerprint_sum_kernel(const uint8_t* __restrict__ data, uint64_t bytes, unsigned long long* acc) {
    const uint64_t words = bytes / 8, tail = bytes % 8;
    const uint64_t* w = reinterpret_cast<const uint64_t*>(data);
    uint64_t sum = 0;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < words; i += stride)
        sum += mix64(__ldg(w + i) + (i + 1) * kGolden);
    if (tail && blockIdx.x == 0 && threadIdx.x == 0) {
        uint64_t last = 0;
        for (uint64_t b = 0; b < tail; ++b) last |= (uint64_t)data[words * 8 + b] << (8 * b);
        sum += mix64(last + (words + 1) * kGolden);
    }
    // integer sums mod 2^64: exact, so the order of the additions does not matter
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    __shared__ uint64_t red[8];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint64_t s = 0;
        for (int k = 0; k < 8; ++k) s += red[k];
        atomicAdd(acc, (unsigned long long)s);
    }
}

__global__ void fingerprint_final_kernel(unsigned long long* acc, uint64_t bytes) {
    *acc = mix64((uint64_t)*acc + bytes);
}

}  // namespace
}  // namespace h3

using namespace h3;

extern "C" h3attn_status h3attn_fingerprint(const void* data, uint64_t bytes, uint64_t* fingerprint, void* stream) {
    if (!fingerprint || (reinterpret_cast<uintptr_t>(fingerprint) & 7u)) return H3ATTN_ERR_INVALID_ARG;
    if (bytes > 0 && (!data || (reinterpret_cast<uintptr_t>(data) & 7u))) return H3ATTN_ERR_INVALID_ARG;
    const cudaError_t pe = prepare_device();
    if (pe != cudaSuccess) return pe == cudaErrorNotSupported ? H3ATTN_ERR_UNSUPPORTED : H3ATTN_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned long long* acc = reinterpret_cast<unsigned long long*>(fingerprint);
    if (cudaMemsetAsync(acc, 0, 8, s) != cudaSuccess) return H3ATTN_ERR_CUDA;
    if (bytes > 0) {
        const uint64_t words = (bytes + 7) / 8;
        const uint64_t want = (words + 255) / 256;
        const int cap = 4 * device_sms();
        const unsigned blocks = (unsigned)(want < (uint64_t)cap ? want : (uint64_t)cap);
        fingerprint_sum_kernel<<<blocks < 1 ? 1 : blocks, 256, 0, s>>>(static_cast<const uint8_t*>(data), bytes, acc);
    }
    fingerprint_final_kernel<<<1, 1, 0, s>>>(acc, bytes);
    return cudaGetLastError() == cudaSuccess ? H3ATTN_OK : H3ATTN_ERR_CUDA;
}
