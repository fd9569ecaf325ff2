// Block swap between the device cache and page-locked host memory.
//
// "Как работает paged attention? (детально)" 4.3 Preemption: when physical
// blocks run out, a request is chosen, its KV cache is saved to CPU memory
// and its blocks are freed; when it resumes its blocks are restored from CPU
// (swap-based preemption).  vLLM paper summary (easyvpn24.com/25506.html),
// section 5 (scheduling and preemption): a CPU block allocator manages the
// blocks swapped to CPU RAM, and swapping is bounded by the bandwidth between
// CPU memory and GPU memory.
//
// One launch moves every (device block, host block) pair of a swap: K and V
// of all KV heads, each block one contiguous num_kv_heads*block_size*head_size
// run on both sides.  Threads copy 16-byte chunks through the host buffer's
// device-mapped address (page-locked memory on a unified address space), so a
// swap of many scattered blocks is one kernel rather than one copy per block.
#include "common.cuh"
#include "launch.h"

namespace pa {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
swap_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, uint4* __restrict__ host_k,
                   uint4* __restrict__ host_v, const int32_t* __restrict__ pairs, int64_t num_blocks,
                   int64_t num_host_blocks, int64_t chunks_per_block, int32_t to_host, int32_t* status) {
    const int64_t dev = pairs[2 * blockIdx.y], host = pairs[2 * blockIdx.y + 1];
    if (dev < 0 || dev >= num_blocks || host < 0 || host >= num_host_blocks) {
        if (blockIdx.x == 0 && threadIdx.x == 0) report(status, PA_ERR_BAD_BLOCK);
        return;
    }
    uint4* dk = k_cache + dev * chunks_per_block;
    uint4* dv = v_cache + dev * chunks_per_block;
    uint4* hk = host_k + host * chunks_per_block;
    uint4* hv = host_v + host * chunks_per_block;
    for (int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; c < chunks_per_block;
         c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        if (to_host) {
            const uint4 a = __ldcs(dk + c), b = __ldcs(dv + c);
            hk[c] = a;
            hv[c] = b;
        } else {
            const uint4 a = hk[c], b = hv[c];
            dk[c] = a;
            dv[c] = b;
        }
    }
}

// The device address of page-locked host memory; nullptr for anything else.
void* mapped_host(void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) return nullptr;
    return a.devicePointer;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" pa_status pa_swap_blocks(const pa_kv_cache* cache, void* host_k, void* host_v,
                                    int64_t num_host_blocks, const int32_t* pairs, int32_t n,
                                    int32_t to_host, int32_t* dev_status, pa_stream_t stream) {
    pa_status st = check_cache(cache);
    if (st != PA_OK) return st;
    if (n < 0 || num_host_blocks < 0) return PA_ERR_INVALID_ARG;
    if (n == 0) return PA_OK;
    if (n > 65535) return PA_ERR_INVALID_ARG;  // one grid row per pair
    if (pairs == nullptr || host_k == nullptr || host_v == nullptr) return PA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(host_k) & 15u) || (reinterpret_cast<uintptr_t>(host_v) & 15u))
        return PA_ERR_INVALID_ARG;
    void* mk = mapped_host(host_k);
    void* mv = mapped_host(host_v);
    if (mk == nullptr || mv == nullptr) return PA_ERR_INVALID_ARG;  // not page-locked host memory
    const int64_t block_bytes = static_cast<int64_t>(cache->num_kv_heads) * cache->block_size *
                                cache->head_size * elem_bytes(cache->kv_dtype);
    if (block_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    const int64_t chunks = block_bytes / 16;
    const int64_t per_block = (chunks + kThreads - 1) / kThreads;
    const dim3 grid(static_cast<unsigned>(per_block < 8 ? per_block : 8), static_cast<unsigned>(n));
    swap_blocks_kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4*>(cache->k_cache), static_cast<uint4*>(cache->v_cache), static_cast<uint4*>(mk),
        static_cast<uint4*>(mv), pairs, cache->num_blocks, num_host_blocks, chunks, to_host ? 1 : 0,
        dev_status);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
