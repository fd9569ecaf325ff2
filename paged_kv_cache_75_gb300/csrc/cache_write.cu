// Cache write (new K/V rows into their slots) and whole-block copies.
//
// "Paged 어텐션" (data-sketchers.com transformers paged-attention wiki),
// Decode 경로: the paged cache is updated in place through the block table.
// "Как работает paged attention? (детально)" 4.1 step 5: the new token's KV
// is written to its position inside the physical block; 3.3: a shared block
// is copied before a sequence writes into it (copy-on-write).
// vLLM paper summary (easyvpn24.com/25506.html) §3: new KV goes to the free
// slot of the last block, or to a newly mapped block.
//
// Both kernels are HBM-bound scatters/copies: every byte is read once and
// written once, 16 bytes per thread access.
#include "common.cuh"
#include "launch.h"

namespace pa {
namespace {

constexpr int kThreads = 256;

// Same-dtype write: one thread moves one 16-byte chunk (8 elements) of K and
// the matching chunk of V.
__global__ void __launch_bounds__(kThreads)
cache_write_copy16(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                   const uint4* __restrict__ k, const uint4* __restrict__ v,
                   const int64_t* __restrict__ slot_mapping, int64_t num_tokens,
                   int64_t token_stride_chunks, int32_t num_kv_heads, int32_t chunks_per_row,
                   int32_t block_size, int64_t num_slots, int32_t* status) {
    pdl_wait();
    pdl_trigger();
    const int64_t chunks_per_token = static_cast<int64_t>(num_kv_heads) * chunks_per_row;
    const int64_t total = num_tokens * chunks_per_token;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / chunks_per_token;
        const int64_t r = i - t * chunks_per_token;  // head * chunks_per_row + chunk
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            report(status, PA_ERR_BAD_BLOCK);
            continue;
        }
        const int64_t blk = slot / block_size, off = slot - blk * block_size;
        const int64_t h = r / chunks_per_row, c = r - h * chunks_per_row;
        const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * chunks_per_row + c;
        const int64_t src = t * token_stride_chunks + r;
        const uint4 kv = __ldcs(k + src);
        const uint4 vv = __ldcs(v + src);
        k_cache[dst] = kv;
        v_cache[dst] = vv;
    }
}

__device__ __forceinline__ uint32_t quantize_pair(float a, float b, float scale) {
    // IEEE binary32 division, then round-to-nearest-even with saturation
    const float2 x = make_float2(__fdiv_rn(a, scale), __fdiv_rn(b, scale));
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(x, __NV_SATFINITE, __NV_E4M3));
}

// E4M3 write: one thread converts 8 input elements (16 bytes) into 8 codes.
template <int IN>
__global__ void __launch_bounds__(kThreads)
cache_write_e4m3(uint2* __restrict__ k_cache, uint2* __restrict__ v_cache,
                 const uint4* __restrict__ k, const uint4* __restrict__ v,
                 const int64_t* __restrict__ slot_mapping, int64_t num_tokens,
                 int64_t token_stride_chunks, int32_t num_kv_heads, int32_t chunks_per_row,
                 int32_t block_size, int64_t num_slots, float k_scale, float v_scale,
                 int32_t* status) {
    pdl_wait();
    pdl_trigger();
    const int64_t chunks_per_token = static_cast<int64_t>(num_kv_heads) * chunks_per_row;
    const int64_t total = num_tokens * chunks_per_token;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / chunks_per_token;
        const int64_t r = i - t * chunks_per_token;
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            report(status, PA_ERR_BAD_BLOCK);
            continue;
        }
        const int64_t blk = slot / block_size, off = slot - blk * block_size;
        const int64_t h = r / chunks_per_row, c = r - h * chunks_per_row;
        const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * chunks_per_row + c;
        const int64_t src = t * token_stride_chunks + r;
        const uint4 kin = __ldcs(k + src);
        const uint4 vin = __ldcs(v + src);
        const uint32_t kw[4] = {kin.x, kin.y, kin.z, kin.w};
        const uint32_t vw[4] = {vin.x, vin.y, vin.z, vin.w};
        uint32_t ko[2], vo[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float2 k0 = kv_pair<IN>(kw[2 * j]), k1 = kv_pair<IN>(kw[2 * j + 1]);
            const float2 v0 = kv_pair<IN>(vw[2 * j]), v1 = kv_pair<IN>(vw[2 * j + 1]);
            ko[j] = quantize_pair(k0.x, k0.y, k_scale) | (quantize_pair(k1.x, k1.y, k_scale) << 16);
            vo[j] = quantize_pair(v0.x, v0.y, v_scale) | (quantize_pair(v1.x, v1.y, v_scale) << 16);
        }
        k_cache[dst] = make_uint2(ko[0], ko[1]);
        v_cache[dst] = make_uint2(vo[0], vo[1]);
    }
}

// Element-wise fallback for rows that are not 16-byte aligned.
template <int IN, int KV>
__global__ void __launch_bounds__(kThreads)
cache_write_scalar(void* __restrict__ k_cache, void* __restrict__ v_cache,
                   const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                   const int64_t* __restrict__ slot_mapping, int64_t num_tokens,
                   int64_t token_stride, int32_t num_kv_heads, int32_t head_size,
                   int32_t block_size, int64_t num_slots, float k_scale, float v_scale,
                   int32_t* status) {
    pdl_wait();
    pdl_trigger();
    const int64_t per_token = static_cast<int64_t>(num_kv_heads) * head_size;
    const int64_t total = num_tokens * per_token;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / per_token;
        const int64_t r = i - t * per_token;
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_slots) {
            report(status, PA_ERR_BAD_BLOCK);
            continue;
        }
        const int64_t blk = slot / block_size, off = slot - blk * block_size;
        const int64_t h = r / head_size, d = r - h * head_size;
        const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * head_size + d;
        const uint16_t kb = k[t * token_stride + r], vb = v[t * token_stride + r];
        if constexpr (KV == PA_FP8_E4M3) {
            const float kf = kv_pair<IN>(kb).x, vf = kv_pair<IN>(vb).x;
            static_cast<uint8_t*>(k_cache)[dst] = static_cast<uint8_t>(quantize_pair(kf, 0.f, k_scale) & 0xff);
            static_cast<uint8_t*>(v_cache)[dst] = static_cast<uint8_t>(quantize_pair(vf, 0.f, v_scale) & 0xff);
        } else {
            static_cast<uint16_t*>(k_cache)[dst] = kb;
            static_cast<uint16_t*>(v_cache)[dst] = vb;
        }
    }
}

// Copy whole blocks: blockIdx.y = pair index, x-dimension strides the block.
__global__ void __launch_bounds__(kThreads)
copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                   const int32_t* __restrict__ pairs, int64_t num_blocks, int64_t chunks_per_block,
                   int32_t* status) {
    const int64_t src = pairs[2 * blockIdx.y], dst = pairs[2 * blockIdx.y + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (blockIdx.x == 0 && threadIdx.x == 0) report(status, PA_ERR_BAD_BLOCK);
        return;
    }
    for (int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
         c < chunks_per_block; c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        k_cache[dst * chunks_per_block + c] = k_cache[src * chunks_per_block + c];
        v_cache[dst * chunks_per_block + c] = v_cache[src * chunks_per_block + c];
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" pa_status pa_kv_cache_write(const pa_kv_cache* cache, const void* k, const void* v,
                                       pa_dtype in_dtype, int64_t num_tokens,
                                       int64_t token_stride, const int64_t* slot_mapping,
                                       int32_t* dev_status, pa_stream_t stream) {
    pa_status st = check_cache(cache);
    if (st != PA_OK) return st;
    if (num_tokens < 0) return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (k == nullptr || v == nullptr || slot_mapping == nullptr) return PA_ERR_INVALID_ARG;
    if (in_dtype != PA_F16 && in_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (cache->kv_dtype != PA_FP8_E4M3 && cache->kv_dtype != in_dtype) return PA_ERR_UNSUPPORTED;
    const int64_t row = static_cast<int64_t>(cache->num_kv_heads) * cache->head_size;
    if (token_stride < row) return PA_ERR_INVALID_ARG;
    if (cache->kv_dtype == PA_FP8_E4M3 && !(cache->k_scale > 0.f && cache->v_scale > 0.f))
        return PA_ERR_INVALID_ARG;

    const int64_t num_slots = cache->num_blocks * cache->block_size;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool vec = aligned16(k) && aligned16(v) && (token_stride % 8) == 0 &&
                     (cache->head_size % 8) == 0;
    const int sms = device_sm_count();
    if (sms <= 0) return PA_ERR_CUDA;
    if (vec) {
        cudaError_t st = cudaSuccess;
        const int32_t chunks_per_row = cache->head_size / 8;
        const int64_t total = num_tokens * cache->num_kv_heads * chunks_per_row;
        const int64_t want = (total + kThreads - 1) / kThreads;
        const int grid = static_cast<int>(want < sms * 16 ? want : sms * 16);
        if (cache->kv_dtype == PA_FP8_E4M3) {
            if (in_dtype == PA_F16)
                st = launch_pdl(cache_write_e4m3<PA_F16>, grid, kThreads, 0, s,
                    static_cast<uint2*>(cache->k_cache), static_cast<uint2*>(cache->v_cache),
                    static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping,
                    num_tokens, token_stride / 8, cache->num_kv_heads, chunks_per_row,
                    cache->block_size, num_slots, cache->k_scale, cache->v_scale, dev_status);
            else
                st = launch_pdl(cache_write_e4m3<PA_BF16>, grid, kThreads, 0, s,
                    static_cast<uint2*>(cache->k_cache), static_cast<uint2*>(cache->v_cache),
                    static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping,
                    num_tokens, token_stride / 8, cache->num_kv_heads, chunks_per_row,
                    cache->block_size, num_slots, cache->k_scale, cache->v_scale, dev_status);
        } else {
            st = launch_pdl(cache_write_copy16, grid, kThreads, 0, s,
                static_cast<uint4*>(cache->k_cache), static_cast<uint4*>(cache->v_cache),
                static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping,
                num_tokens, token_stride / 8, cache->num_kv_heads, chunks_per_row,
                cache->block_size, num_slots, dev_status);
        }
        if (st != cudaSuccess) return PA_ERR_CUDA;
    } else {
        const int64_t total = num_tokens * row;
        const int64_t want = (total + kThreads - 1) / kThreads;
        const int grid = static_cast<int>(want < sms * 16 ? want : sms * 16);
        const uint16_t* kk = static_cast<const uint16_t*>(k);
        const uint16_t* vv = static_cast<const uint16_t*>(v);
#define PA_SCALAR(IN, KV)                                                                     \
    cache_write_scalar<IN, KV><<<grid, kThreads, 0, s>>>(                                     \
        cache->k_cache, cache->v_cache, kk, vv, slot_mapping, num_tokens, token_stride,       \
        cache->num_kv_heads, cache->head_size, cache->block_size, num_slots, cache->k_scale, \
        cache->v_scale, dev_status)
        if (cache->kv_dtype == PA_FP8_E4M3) {
            if (in_dtype == PA_F16) PA_SCALAR(PA_F16, PA_FP8_E4M3);
            else PA_SCALAR(PA_BF16, PA_FP8_E4M3);
        } else if (in_dtype == PA_F16) {
            PA_SCALAR(PA_F16, PA_F16);
        } else {
            PA_SCALAR(PA_BF16, PA_BF16);
        }
#undef PA_SCALAR
    }
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

extern "C" pa_status pa_copy_blocks(const pa_kv_cache* cache, const int32_t* src_dst_pairs,
                                    int32_t n, int32_t* dev_status, pa_stream_t stream) {
    pa_status st = check_cache(cache);
    if (st != PA_OK) return st;
    if (n < 0 || (n > 0 && src_dst_pairs == nullptr)) return PA_ERR_INVALID_ARG;
    if (n == 0) return PA_OK;
    if (n > 65535) return PA_ERR_INVALID_ARG;  // one grid row per pair
    const int64_t bytes = static_cast<int64_t>(cache->num_kv_heads) * cache->block_size *
                          cache->head_size * elem_bytes(cache->kv_dtype);
    if (bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    const int64_t chunks = bytes / 16;
    const int64_t want = (chunks + kThreads - 1) / kThreads;
    dim3 grid(static_cast<unsigned>(want < 64 ? want : 64), static_cast<unsigned>(n));
    copy_blocks_kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4*>(cache->k_cache), static_cast<uint4*>(cache->v_cache), src_dst_pairs,
        cache->num_blocks, chunks, dev_status);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
