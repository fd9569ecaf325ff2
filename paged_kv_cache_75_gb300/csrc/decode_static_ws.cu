// pa_decode_static_ws: paged decode for callers that cannot allocate device
// memory.
//
// Who needs it: code that runs inside a host program which owns all device
// memory through its own allocator (a plugin, an embedded runtime) and may not
// call cudaMalloc, and latency-critical serving loops that must not call
// cudaMalloc / cudaFree because those calls can synchronise the device.  Such
// callers cannot provide the split-K workspace that pa_decode asks for, so
// this entry point brings its own: one fixed-size array of device memory that
// is part of the library image and lives on every GPU that loads the library
// until the process exits.
//
// The array is shared by every call on a device and keeps whatever the last
// call left in it.  pa_decode writes every partial result it later reads, so
// nothing has to be cleared between calls; but two calls whose kernels
// overlap on the GPU (different streams, no ordering between them) race on
// the array and give wrong results.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "launch.h"
#include "pa_kv.h"

namespace {

// the scratch itself: host code must not use this name as a device address
static __device__ __align__(256) unsigned char g_decode_scratch[PA_DECODE_STATIC_WS_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];
CUcontext g_scratch_ctx[kMaxDevices];

// The context current on this thread (the device's primary context unless the
// caller made another one current), or null if it cannot be read.
CUcontext current_context() {
    using GetCurrent = CUresult (*)(CUcontext*);
    static GetCurrent fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<GetCurrent>(nullptr);
        return reinterpret_cast<GetCurrent>(f);
    }();
    CUcontext c = nullptr;
    if (fn == nullptr || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

// Device address of the scratch on the current device.  Looked up with
// cudaGetSymbolAddress (that device current) the first time a device is used,
// and again whenever the context current on the device has changed since (a
// cudaDeviceReset, or a context the caller created, loads the library's
// module at a new address); otherwise the remembered address is returned.
pa_status scratch_on_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
    const CUcontext ctx = current_context();
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_addr[dev] == nullptr || ctx == nullptr || ctx != g_scratch_ctx[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return PA_ERR_CUDA;
        g_scratch_addr[dev] = p;
        // read again: the lookup makes the device's context current if none was
        g_scratch_ctx[dev] = current_context();
    }
    *out = g_scratch_addr[dev];
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_static_ws(void* out, const void* q, pa_dtype q_dtype,
                                         const pa_kv_cache* cache, const int32_t* block_table,
                                         int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                         int32_t num_seqs, int32_t max_seq_len, int32_t num_heads,
                                         float scale, int32_t partition_size, int32_t* dev_status,
                                         pa_stream_t stream) {
    if (cache == nullptr) return PA_ERR_INVALID_ARG;
    // the automatic partition is resolved here, so that the size check and the
    // launch use the same one (pa_decode_workspace_size would answer for 512)
    int32_t P = partition_size;
    if (P == 0 && num_seqs > 0) {
        P = pa_decode_partition_size(num_seqs, num_heads, cache->num_kv_heads, max_seq_len);
        if (P <= 0) P = 0;  // arguments pa_decode rejects: let it say why
    }
    const size_t need = pa_decode_workspace_size(num_seqs, num_heads, cache->head_size, max_seq_len,
                                                 cache->block_size, P);
    if (need > PA_DECODE_STATIC_WS_BYTES) return PA_ERR_UNSUPPORTED;  // beyond the built-in scratch
    void* ws = nullptr;
    if (need > 0) {
        const pa_status st = scratch_on_current_device(&ws);
        if (st != PA_OK) return st;
    }
    return pa_decode(out, q, q_dtype, cache, block_table, max_blocks_per_seq, seq_lens, num_seqs,
                     max_seq_len, num_heads, scale, P, ws,
                     need > 0 ? static_cast<size_t>(PA_DECODE_STATIC_WS_BYTES) : 0, dev_status, stream);
}
