// forward_noalloc.cu -- h3attn_forward_static: the forward for callers that
// cannot allocate device memory.
//
// Some hosts forbid device allocation once they are running: a plugin inside an
// inference server that owns every byte of the GPU through its own pool, code
// that runs under a memory budget enforced by the host process, or callers that
// must never hit cudaMalloc's implicit device synchronisation on a hot path.
// This entry point needs no handle and allocates nothing: its scratch (the
// rotated q^/k^ rows, the per-call sample plan and the device error word) lives
// in one file-scope __device__ array below, which every GPU that loads the
// library keeps for the life of the process.
//
// The arithmetic is exactly h3attn_forward's (same plan, prologue and
// attention kernels), only the scratch pointers differ.
#include <mutex>
#include <string.h>

#include "../../include/h3attn.h"
#include "common.cuh"
#include "host.cuh"

using namespace h3;

namespace {

constexpr size_t kPlanBytes = 64u << 10;  // order, rank, four cumulative tables, error word
constexpr size_t kRowBytes = (size_t)H3ATTN_STATIC_MAX_TOKEN_HEADS * kD * 2;  // one fp16 [S, H, 128] buffer
constexpr size_t kScratchBytes = kPlanBytes + 2 * kRowBytes;
static_assert((H3ATTN_STATIC_MAX_SAMPLES + 1) * 4 * 6 + 16 <= kPlanBytes, "plan region too small");

// The shared scratch.  Host code must not use this name as an address: it is
// resolved per device with cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_static_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
uint8_t* g_scratch_ptr[kMaxDevices];  // device address of g_static_scratch, per device

// Once per device, with that device current: prepare the device (kernel
// attributes, SM count) and resolve the scratch's device address.  Allocates
// nothing.
h3attn_status setup_device(int dev, uint8_t** out) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        const cudaError_t pe = prepare_device();
        if (pe != cudaSuccess) return pe == cudaErrorNotSupported ? H3ATTN_ERR_UNSUPPORTED : H3ATTN_ERR_CUDA;
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) return H3ATTN_ERR_CUDA;
        g_scratch_ptr[dev] = static_cast<uint8_t*>(ptr);
    }
    *out = g_scratch_ptr[dev];
    return H3ATTN_OK;
}

bool al16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool al4(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" h3attn_status h3attn_forward_static(const h3attn_config* cfg, const h3attn_bf16* q, const h3attn_bf16* k,
                                               const h3attn_bf16* v, const float* q_norm_w, const float* k_norm_w,
                                               const int32_t* const pos_ids[3], const int32_t* seg_offsets,
                                               int num_samples, int total_tokens, h3attn_bf16* out, float* lse,
                                               uint32_t* device_error_flags, void* stream) {
    if (!cfg) return H3ATTN_ERR_INVALID_ARG;
    if (cfg->num_heads < 1 || !(cfg->eps >= 0.f) || !(cfg->rope_theta > 0.f) || !(cfg->softmax_scale >= 0.f))
        return H3ATTN_ERR_INVALID_ARG;
    if (cfg->head_dim != kD || cfg->rope_pairing != 0 || cfg->key_order != H3ATTN_KEY_ORDER_PACKED)
        return H3ATTN_ERR_UNSUPPORTED;
    RopeTable rt;
    if (!build_rope_table(cfg->rope_sections, cfg->rope_theta, rt)) return H3ATTN_ERR_UNSUPPORTED;
    if (total_tokens < 0 || num_samples < 0) return H3ATTN_ERR_INVALID_ARG;
    if (total_tokens == 0) return H3ATTN_OK;
    if (num_samples < 1 || num_samples > total_tokens) return H3ATTN_ERR_INVALID_ARG;
    if ((long long)total_tokens * cfg->num_heads > H3ATTN_STATIC_MAX_TOKEN_HEADS ||
        num_samples > H3ATTN_STATIC_MAX_SAMPLES)
        return H3ATTN_ERR_CAPACITY;
    if (!al16(q) || !al16(k) || !al16(v) || !al16(q_norm_w) || !al16(k_norm_w) || !al16(out))
        return H3ATTN_ERR_INVALID_ARG;
    if (!pos_ids || !al4(pos_ids[0]) || !al4(pos_ids[1]) || !al4(pos_ids[2]) || !al4(seg_offsets) ||
        (lse && !al4(lse)) || (device_error_flags && !al4(device_error_flags)))
        return H3ATTN_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return H3ATTN_ERR_CUDA;
    if (dev >= kMaxDevices) return H3ATTN_ERR_UNSUPPORTED;
    uint8_t* base = nullptr;
    const h3attn_status st = setup_device(dev, &base);
    if (st != H3ATTN_OK) return st;

    const int n1 = H3ATTN_STATIC_MAX_SAMPLES + 1;
    int* ints = reinterpret_cast<int*>(base);
    Workspace ws;
    memset(&ws, 0, sizeof ws);
    ws.plan.order = ints;
    ws.plan.rank_of = ints + n1;
    ws.plan.cum64 = ints + 2 * n1;
    ws.plan.cum128 = ints + 3 * n1;
    ws.plan.cum256 = ints + 4 * n1;
    ws.plan.cumsq = ints + 5 * n1;
    ws.plan.err = reinterpret_cast<unsigned*>(ints + 6 * n1);
    ws.qhat = reinterpret_cast<__half*>(base + kPlanBytes);
    ws.khat = reinterpret_cast<__half*>(base + kPlanBytes + kRowBytes);

    Problem p;
    p.q = reinterpret_cast<const __nv_bfloat16*>(q);
    p.k = reinterpret_cast<const __nv_bfloat16*>(k);
    p.v = reinterpret_cast<const __nv_bfloat16*>(v);
    p.wq = q_norm_w;
    p.wk = k_norm_w;
    p.seq.seg = seg_offsets;
    p.seq.pos_t = pos_ids[0];
    p.seq.pos_h = pos_ids[1];
    p.seq.pos_w = pos_ids[2];
    p.seq.n = num_samples;
    p.seq.S = total_tokens;
    p.H = cfg->num_heads;
    p.eps = cfg->eps;
    p.scale = cfg->softmax_scale == 0.f ? 1.0f / sqrtf((float)kD) : cfg->softmax_scale;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the error word is the only scratch that must start at zero
    if (cudaMemsetAsync(ws.plan.err, 0, sizeof(unsigned), s) != cudaSuccess) return H3ATTN_ERR_CUDA;
    if (launch_plan(p, ws, s) != cudaSuccess || launch_prologue(p, ws, &rt, s) != cudaSuccess ||
        launch_fwd(p, ws, reinterpret_cast<__nv_bfloat16*>(out), lse, s) != cudaSuccess)
        return H3ATTN_ERR_CUDA;
    if (device_error_flags &&
        cudaMemcpyAsync(device_error_flags, ws.plan.err, sizeof(unsigned), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return H3ATTN_ERR_CUDA;
    return H3ATTN_OK;
}
