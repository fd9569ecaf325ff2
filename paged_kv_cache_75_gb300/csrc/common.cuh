// Device-side helpers shared by the kernels of the library: PTX wrappers for
// mbarriers and bulk (TMA) copies, bounded waits, error reporting and the
// number-format conversions the kernels need.  sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_kv.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "this library targets sm_103a (Blackwell) only"
#endif

namespace pa {

// ---------------------------------------------------------------------------
// error reporting: the first error code wins, later ones are dropped
// ---------------------------------------------------------------------------
__device__ __forceinline__ void report(int32_t* status, int code) {
    if (status != nullptr) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------------------
// shared-memory addresses, mbarriers, bulk copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait limit for every mbarrier wait in the library.  A wait that runs out
// reports PA_ERR_TIMEOUT and returns false instead of spinning forever.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Bounded wait on an mbarrier phase.  Also gives up (returning false) as soon
// as *abort is set by another warp of the block; a phase already complete is
// taken without reading the flag (its data has landed), so the common case
// costs one try_wait.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t* status,
                                          volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                report(status, PA_ERR_TIMEOUT);
                *abort = 1;
                return false;
            }
        }
    }
}

// 1-D bulk copy global -> shared (no tensor map), completion counted on `bar`.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Same with an L2 eviction-priority hint (`policy` from createpolicy).
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
        "[%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// producer side of a named barrier: counts this warp's threads without waiting
__device__ __forceinline__ void named_bar_arrive(int id, int nthreads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Programmatic dependent launch.  The library launches its kernels with
// programmatic stream serialization, so a kernel may become resident while the
// previous kernel on the stream is still finishing.  pdl_wait() blocks until
// every grid this one depends on has completed and its memory operations are
// visible; each kernel calls it before its first global load or store.
// pdl_trigger() lets the next launch's blocks be scheduled early (they still
// wait in their own pdl_wait() for this grid to complete).  Both are no-ops for
// a launch without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Snake order of a persistent grid over a work list: in round r a CTA takes
// item r*grid + blockIdx.x when r is even and r*grid + (grid-1-blockIdx.x)
// when r is odd; -1 once past the list.  Over a list sorted longest first this
// evens out the CTAs' totals.
__device__ __forceinline__ int snake_item(int r, int n_items) {
    const int64_t base = static_cast<int64_t>(r) * gridDim.x;
    const int64_t i = base + ((r & 1) ? static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x)
                                      : static_cast<int>(blockIdx.x));
    return i < n_items ? static_cast<int>(i) : -1;
}

// ---------------------------------------------------------------------------
// conversions
// ---------------------------------------------------------------------------
// two packed 16-bit floats -> two floats
__device__ __forceinline__ float2 f16x2_to_f2(uint32_t w) {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    return __half22float2(h);
}
// bf16 -> f32 is exact: the bf16 bits are the top half of the f32 bits
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
// two E4M3 codes (low 16 bits of w) -> two floats, exact via half2
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t w) {
    __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xffffu),
                                                __NV_E4M3);
    __half2 h = *reinterpret_cast<__half2*>(&hr);
    return __half22float2(h);
}

template <int KV>
__device__ __forceinline__ float2 kv_pair(uint32_t w);
template <>
__device__ __forceinline__ float2 kv_pair<PA_F16>(uint32_t w) { return f16x2_to_f2(w); }
template <>
__device__ __forceinline__ float2 kv_pair<PA_BF16>(uint32_t w) { return bf16x2_to_f2(w); }

template <int T>
struct dtype_traits;
template <>
struct dtype_traits<PA_F16> {
    using storage = __half;
    static constexpr int bytes = 2;
    __device__ static float to_f(storage x) { return __half2float(x); }
    __device__ static storage from_f(float x) { return __float2half_rn(x); }
};
template <>
struct dtype_traits<PA_BF16> {
    using storage = __nv_bfloat16;
    static constexpr int bytes = 2;
    __device__ static float to_f(storage x) { return __bfloat162float(x); }
    __device__ static storage from_f(float x) { return __float2bfloat16_rn(x); }
};
template <>
struct dtype_traits<PA_FP8_E4M3> {
    using storage = uint8_t;
    static constexpr int bytes = 1;
};

}  // namespace pa
