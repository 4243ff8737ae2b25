// exp2_check.cu -- test hook: the attention kernels' two 2^x paths (the SFU
// instruction and the FMA-pipe polynomial of exp2_poly_pair) evaluated on
// caller-given arguments, so that tests can check the polynomial's bits and
// its error against the SFU on the GPU itself.
#include "../../include/h3attn.h"
#include "common.cuh"
#include "host.cuh"

namespace h3 {
namespace {
__global__ void exp2_check_kernel(const float* __restrict__ x, float* __restrict__ y, int n, int path) {
    const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (i >= n) return;
    const float a = x[i], b = i + 1 < n ? x[i + 1] : 0.f;
    // 2^(x * 1 + 0), as the softmax forms its argument
    const uint64_t x2 = f2pack(a, b), one = f2pack(1.f, 1.f), zero = f2pack(0.f, 0.f);
    const uint64_t r = path == 1 ? exp2_poly_pair(x2, one, zero) : exp2_pair(x2, one, zero);
    y[i] = pair_lo(r);
    if (i + 1 < n) y[i + 1] = pair_hi(r);
}
}  // namespace
}  // namespace h3

using namespace h3;

extern "C" h3attn_status h3attn_debug_exp2(const float* x, float* y, int n, int path, void* stream) {
    if (n < 0 || (path != 0 && path != 1)) return H3ATTN_ERR_INVALID_ARG;
    if (n == 0) return H3ATTN_OK;
    if (!x || !y || (reinterpret_cast<uintptr_t>(x) & 3u) || (reinterpret_cast<uintptr_t>(y) & 3u))
        return H3ATTN_ERR_INVALID_ARG;
    const cudaError_t pe = prepare_device();
    if (pe != cudaSuccess) return pe == cudaErrorNotSupported ? H3ATTN_ERR_UNSUPPORTED : H3ATTN_ERR_CUDA;
    const int pairs = (n + 1) / 2;
    exp2_check_kernel<<<(pairs + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, y, n, path);
    return cudaGetLastError() == cudaSuccess ? H3ATTN_OK : H3ATTN_ERR_CUDA;
}
