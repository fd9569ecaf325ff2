// Status strings, version and the host helpers of launch.h.
#include <cuda_runtime.h>

#include <mutex>

#include "launch.h"

namespace pa {

int elem_bytes(int dtype) {
    switch (dtype) {
    case PA_F16:
    case PA_BF16: return 2;
    case PA_FP8_E4M3: return 1;
    default: return 0;
    }
}

pa_status check_cache(const pa_kv_cache* c) {
    if (c == nullptr || c->k_cache == nullptr || c->v_cache == nullptr) return PA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(c->k_cache) & 15u) || (reinterpret_cast<uintptr_t>(c->v_cache) & 15u))
        return PA_ERR_INVALID_ARG;
    if (c->num_blocks <= 0 || c->num_blocks > INT32_MAX || c->block_size <= 0 ||
        c->num_kv_heads <= 0 || c->head_size <= 0)
        return PA_ERR_INVALID_ARG;
    if (elem_bytes(c->kv_dtype) == 0) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

namespace {
constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices];
int g_smem[kMaxDevices];
std::mutex g_mu;

bool query(int* dev) {
    if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_sms[*dev] == 0) {
        int sms = 0, smem = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, *dev) != cudaSuccess)
            return false;
        g_smem[*dev] = smem;
        g_sms[*dev] = sms;
    }
    return true;
}
}  // namespace

int device_sm_count() {
    int dev;
    return query(&dev) ? g_sms[dev] : 0;
}

int current_device() {
    int dev;
    return cudaGetDevice(&dev) == cudaSuccess ? dev : -1;
}

int device_max_smem_optin() {
    int dev;
    return query(&dev) ? g_smem[dev] : 0;
}

}  // namespace pa

extern "C" const char* pa_status_str(pa_status s) {
    switch (s) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported configuration";
    case PA_ERR_OOM: return "out of free blocks";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_TIMEOUT: return "device wait timed out";
    case PA_ERR_BAD_BLOCK: return "block id or slot outside the cache";
    default: return "unknown status";
    }
}

extern "C" int32_t pa_version(void) { return 100; }
