// host.cu -- host-side state shared by the launchers (see host.cuh).
#include <math.h>
#include <mutex>
#include <string.h>

#include "host.cuh"

namespace h3 {

namespace {
std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
int g_sms[kMaxDevices];  // 0 until the device is prepared
}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    std::call_once(g_encode_once, [] {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

cudaError_t prepare_device() {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorNotSupported;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (g_sms[dev] > 0) return cudaSuccess;
    cudaDeviceProp prop;
    if ((e = cudaGetDeviceProperties(&prop, dev)) != cudaSuccess) return e;
    if (!(prop.major == 10 && prop.minor == 3)) return cudaErrorNotSupported;
    if (!tensor_map_encoder()) return cudaErrorNotSupported;
    if ((e = set_fwd_attributes()) != cudaSuccess || (e = set_bwd_attributes()) != cudaSuccess ||
        (e = set_linear_attributes()) != cudaSuccess)
        return e;
    g_sms[dev] = prop.multiProcessorCount;
    return cudaSuccess;
}

int device_sms() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    return g_sms[dev];
}

bool build_rope_table(const int sections[3], float theta, RopeTable& rt) {
    memset(&rt, 0, sizeof rt);
    for (int g = 0; g < 32; ++g) { rt.axis[g] = -1; rt.partner[g] = (int8_t)g; rt.second[g] = 0; }
    int off = 0;
    for (int a = 0; a < 3; ++a) {
        const int n = sections[a];
        if (n < 0 || n % 8 != 0 || off + n > kD) return false;
        const int half = n / 2;
        for (int j = 0; j < half; ++j) {
            // frequency of pair j of an n-channel axis: theta^(-2j/n)
            const float f = (float)pow((double)theta, -2.0 * j / (double)n);
            rt.inv_freq[off + j] = f;
            rt.inv_freq[off + j + half] = f;
        }
        // channel groups of 4 (one lane each): a section of n channels pairs group
        // g of its first half with group g + n/8 of its second half
        for (int grp = off / 4; grp < (off + n) / 4; ++grp) {
            const bool second = grp * 4 - off >= half;
            rt.axis[grp] = (int8_t)a;
            rt.second[grp] = second ? 1 : 0;
            rt.partner[grp] = (int8_t)(second ? grp - half / 4 : grp + half / 4);
        }
        off += n;
    }
    return true;
}

}  // namespace h3
