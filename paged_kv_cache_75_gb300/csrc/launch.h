// Host-side helpers shared by the entry points: argument checks and device
// queries.  Host code only.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <utility>

#include "pa_kv.h"

namespace pa {

// bytes of one element of a storage dtype (0 for an unknown code)
int elem_bytes(int dtype);

// Checks a cache descriptor: non-null 16-byte-aligned pointers, positive
// sizes, a known dtype.
pa_status check_cache(const pa_kv_cache* cache);

// SM count of the current device (cached per device); 0 on failure.
int device_sm_count();

// Largest dynamic shared memory a block may opt into on the current device.
int device_max_smem_optin();

// Current device ordinal, -1 on failure.
int current_device();

// Per-kernel launch facts cached across calls, so that a launch costs no
// attribute or occupancy query after the first one: the dynamic-smem opt-in
// is raised once per device, and the last (device, smem) -> blocks-per-SM
// answer is remembered.
struct LaunchCache {
    std::atomic<uint64_t> optin_devices{0};  // bit d: attribute set on device d
    std::atomic<uint64_t> occ{0};            // device << 48 | smem << 16 | blocks
};

template <typename Kernel>
int blocks_per_sm(Kernel kern, int threads, int smem, LaunchCache& c) {
    const int dev = current_device();
    if (dev < 0 || dev >= 64 || smem < 0 || smem >= (1 << 24)) return 0;
    const uint64_t bit = 1ull << dev;
    if (!(c.optin_devices.load(std::memory_order_relaxed) & bit)) {
        // opt in to everything the block may use next to its static smem
        cudaFuncAttributes attr;
        if (cudaFuncGetAttributes(&attr, kern) != cudaSuccess) return 0;
        const int room = device_max_smem_optin() - static_cast<int>(attr.sharedSizeBytes);
        if (room < smem ||
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, room) != cudaSuccess)
            return 0;
        c.optin_devices.fetch_or(bit);
    }
    const uint64_t key = (static_cast<uint64_t>(dev) << 48) | (static_cast<uint64_t>(smem) << 16);
    const uint64_t v = c.occ.load(std::memory_order_relaxed);
    if ((v & ~0xffffull) == key && (v & 0xffffull) != 0) return static_cast<int>(v & 0xffffull);
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem) != cudaSuccess) return 0;
    c.occ.store(key | static_cast<uint64_t>(n & 0xffff), std::memory_order_relaxed);
    return n;
}


// Launch with programmatic stream serialization: the kernel's blocks may be
// scheduled while the previous kernel on the stream drains, which hides the
// launch gap between back-to-back calls.  Every kernel launched this way calls
// pdl_wait() before touching global memory.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kern)(Params...), int grid, int block, int smem, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(block));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace pa
