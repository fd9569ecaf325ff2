// Host-side launch of the paged decode kernels for one (q dtype, KV dtype,
// block size); included by the per-configuration translation units.
#pragma once

#include "decode_impl.cuh"
#include "launch.h"

namespace pa {

// ring depth: as many stages as fit next to the rest of the block's shared
// memory when `ctas` blocks share an SM (228 KB, 1 KB reserved per block),
// at most 48 KB and 8 stages, at least 2.  48 KB per block (144 KB in flight
// per SM) is where the copy stream runs best: the fp16 single-head decode
// moved 0.975 of the measured copy rate with three 16 KB stages and 0.94 with
// four, and two stages fell to 0.93.
inline int decode_stages(int stage_bytes, int other_bytes, int ctas) {
    int room = (228 * 1024) / ctas - 1024 - 1024 - other_bytes;
    if (room > 48 * 1024) room = 48 * 1024;
    int s = room / stage_bytes;
    return s < 2 ? 2 : (s > 8 ? 8 : s);
}

template <int QDT, int KVDT, int D, int G, int BS>
pa_status launch_decode_t(DecodeParams p, cudaStream_t stream) {
    using C = DecodeCfg<QDT, KVDT, D, G, BS>;
    const int other = static_cast<int>(DecodeSmem::make(0, C::STAGE_BYTES, C::QBYTES, C::MERGE_FLOATS,
                                                        p.num_seqs).total) + 2 * 8 * 8 + 64;
    // CTAs an SM holds under the register cap (65536 registers per SM)
    constexpr int kCtas = 65536 / (C::THREADS * C::MAX_REGS) < 1 ? 1
                          : (65536 / (C::THREADS * C::MAX_REGS) > 4 ? 4 : 65536 / (C::THREADS * C::MAX_REGS));
    p.stages = decode_stages(C::STAGE_BYTES, other, kCtas);
    const DecodeSmem L = DecodeSmem::make(p.stages, C::STAGE_BYTES, C::QBYTES, C::MERGE_FLOATS, p.num_seqs);
    const int smem = static_cast<int>(L.total) + 1024;  // slack for the 1 KB base alignment
    if (smem > device_max_smem_optin()) return PA_ERR_UNSUPPORTED;
    const bool append = p.k_new != nullptr;
    auto kern = append ? paged_decode_kernel<QDT, KVDT, D, G, BS, true> : paged_decode_kernel<QDT, KVDT, D, G, BS, false>;
    static LaunchCache cache, cache_append;
    const int per_sm = blocks_per_sm(kern, C::THREADS, smem, append ? cache_append : cache);
    if (per_sm <= 0) return PA_ERR_CUDA;
    const int sms = device_sm_count();
    const int64_t max_items = static_cast<int64_t>(p.num_seqs) * p.num_kv_heads * p.max_parts;
    const int64_t cap = static_cast<int64_t>(sms) * per_sm;
    const int grid = static_cast<int>(max_items < cap ? max_items : cap);
    if (grid <= 0) return PA_OK;
    if (launch_pdl(kern, grid, C::THREADS, smem, stream, p) != cudaSuccess) return PA_ERR_CUDA;
    if (p.max_parts > 1) {
        // group mode: the merge runs over the batch's members
        DecodeParams r = p;
        if (r.vm > 0) {
            r.vm = 0;
            r.num_seqs = r.num_members;
        }
        // warps per (sequence, head): more when pairs have many partitions
        const int64_t pairs = static_cast<int64_t>(r.num_seqs) * r.num_heads;
        const int wpp = p.max_parts >= 32 ? 8 : p.max_parts >= 8 ? 4 : p.max_parts >= 3 ? 2 : 1;
        const int rgrid = static_cast<int>((pairs * wpp + 7) / 8);
        cudaError_t e;
        if (wpp == 8) e = launch_pdl(paged_decode_reduce_kernel<QDT, D, 8>, rgrid, 256, 0, stream, r);
        else if (wpp == 4) e = launch_pdl(paged_decode_reduce_kernel<QDT, D, 4>, rgrid, 256, 0, stream, r);
        else if (wpp == 2) e = launch_pdl(paged_decode_reduce_kernel<QDT, D, 2>, rgrid, 256, 0, stream, r);
        else e = launch_pdl(paged_decode_reduce_kernel<QDT, D, 1>, rgrid, 256, 0, stream, r);
        if (e != cudaSuccess) return PA_ERR_CUDA;
    }
    return PA_OK;
}

template <int QDT, int KVDT, int BS>
pa_status launch_decode_bs(const DecodeParams& p, int head_size, int group, cudaStream_t s) {
#define PA_CASE(D, G) \
    if (head_size == D && group == G) return launch_decode_t<QDT, KVDT, D, G, BS>(p, s);
    PA_CASE(128, 1) PA_CASE(128, 2) PA_CASE(128, 4) PA_CASE(128, 8)
    PA_CASE(64, 1) PA_CASE(64, 2) PA_CASE(64, 4) PA_CASE(64, 8)
#undef PA_CASE
    return PA_ERR_UNSUPPORTED;
}

// one per translation unit: (KV dtype, block size); E4M3 units take both q dtypes
#define PA_DECLARE_DECODE(NAME) \
    pa_status NAME(const DecodeParams& p, int q_dtype, int head_size, int group, cudaStream_t s);
PA_DECLARE_DECODE(launch_decode_f16_bs16)
PA_DECLARE_DECODE(launch_decode_f16_bs32)
PA_DECLARE_DECODE(launch_decode_f16_bs64)
PA_DECLARE_DECODE(launch_decode_bf16_bs16)
PA_DECLARE_DECODE(launch_decode_bf16_bs32)
PA_DECLARE_DECODE(launch_decode_bf16_bs64)
PA_DECLARE_DECODE(launch_decode_fp8_bs16)
PA_DECLARE_DECODE(launch_decode_fp8_bs32)
PA_DECLARE_DECODE(launch_decode_fp8_bs64)
#undef PA_DECLARE_DECODE

}  // namespace pa
