// pa_decode / pa_decode_workspace_size: argument checks and dispatch.
#include <cmath>

#include "decode_launch.cuh"

namespace pa {
namespace {

// Automatic partition: the longest of 2048 (1024 when a KV head serves four or
// more query heads, whose items already carry more fixed work) halved down to
// 512 tokens while the (sequence, KV head, partition) items would not fill two
// rounds of resident blocks.  Fewer, longer items save the partials and the
// merge; the balanced schedule keeps long items from leaving blocks idle.
int auto_partition(int64_t num_seqs, int num_kv_heads, int max_seq_len, int group) {
    int p = group >= 4 ? 1024 : 2048;
    const int64_t ctas = 3ll * device_sm_count();  // resident decode blocks
    const int64_t pairs = num_seqs * num_kv_heads;
    auto items = [&](int q) { return pairs * ((max_seq_len + q - 1) / q); };
    // Few (sequence, KV head) pairs over long contexts: every partition costs a
    // query load and a merge of its warps' partials, so longer partitions go
    // faster while the items still give each resident block four or more (the
    // E4M3 decode of 8 sequences of 32k-128k tokens moved 0.77 of the copy rate
    // with 512-token partitions, 0.86 with 1024 and 0.92 with 4096).
    if (pairs < ctas) {
        while (2 * p <= 8192 && items(2 * p) >= 4 * ctas) p <<= 1;
    } else if (group >= 4) {
        // many pairs through the tensor-core consumer: 1536 tokens (the GQA
        // decode of 256 sequences, lengths log-normal around 1000, moved 0.71
        // of the copy rate at 768, 0.74 at 1024, 0.75 at 1536, 0.74 at 2048)
        p = 1536;
    }
    // Shorter ones while the items would not fill the GPU twice, never below
    // 512 (the workspace size query answers for 512).
    while (p / 2 >= 512 && items(p) < 2 * ctas) p >>= 1;
    return p;  // 512 .. 8192, a multiple of every block size
}

int resolve_partition(int partition_size, int64_t num_seqs, int num_kv_heads, int max_seq_len, int group) {
    return partition_size > 0 ? partition_size : auto_partition(num_seqs, num_kv_heads, max_seq_len, group);
}

// Workspace sizes hold for any automatic choice: it never goes below 512.
int ws_partition(int partition_size) { return partition_size > 0 ? partition_size : 512; }

int max_parts_of(int max_seq_len, int partition) {
    return max_seq_len <= partition ? 1 : (max_seq_len + partition - 1) / partition;
}

struct WsLayout {
    size_t lse_off, o_off, bytes;
};

WsLayout ws_layout(int64_t num_seqs, int64_t num_heads, int64_t head_size, int max_parts) {
    WsLayout w{0, 0, 0};
    if (max_parts <= 1) return w;
    const size_t rows = static_cast<size_t>(num_seqs) * num_heads * max_parts;
    w.lse_off = 0;
    w.o_off = (rows * 4 + 255) & ~static_cast<size_t>(255);
    w.bytes = w.o_off + rows * head_size * 4;
    return w;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t head_size,
                                           int32_t max_seq_len, int32_t block_size,
                                           int32_t partition_size) {
    if (num_seqs <= 0 || num_heads <= 0 || head_size <= 0 || max_seq_len < 0 || block_size <= 0 ||
        partition_size < 0)
        return 0;
    const int P = ws_partition(partition_size);
    return ws_layout(num_seqs, num_heads, head_size, max_parts_of(max_seq_len, P)).bytes;
}

namespace pa {
namespace {

// pa_decode, and pa_decode_append when k_new / v_new are given
pa_status decode_entry(void* out, const void* q, pa_dtype q_dtype, const pa_kv_cache* cache,
                       const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                       int32_t num_seqs, int32_t max_seq_len, int32_t num_heads, float scale,
                       int32_t partition_size, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                       pa_stream_t stream, const void* k_new, const void* v_new,
                       const int32_t* cu_seq_lens_k = nullptr, const int32_t* cu_groups = nullptr,
                       const int32_t* shared_lens = nullptr, int32_t num_groups = 0, bool group_mode = false,
                       int32_t max_group_size = 0, bool no_copies = false) {
    pa_status st = check_cache(cache);
    if (st != PA_OK) return st;
    if (num_seqs < 0 || num_heads <= 0 || max_blocks_per_seq <= 0 || max_seq_len < 0 ||
        partition_size < 0 || !std::isfinite(scale))
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (out == nullptr || q == nullptr || block_table == nullptr || (seq_lens == nullptr && cu_seq_lens_k == nullptr))
        return PA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(out) & 15u) || (reinterpret_cast<uintptr_t>(q) & 15u))
        return PA_ERR_INVALID_ARG;
    if ((k_new == nullptr) != (v_new == nullptr)) return PA_ERR_INVALID_ARG;
    if (k_new != nullptr &&
        ((reinterpret_cast<uintptr_t>(k_new) & 15u) || (reinterpret_cast<uintptr_t>(v_new) & 15u)))
        return PA_ERR_INVALID_ARG;
    if (num_heads % cache->num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    const int group = num_heads / cache->num_kv_heads;
    const int D = cache->head_size, bs = cache->block_size;
    if (D != 64 && D != 128) return PA_ERR_UNSUPPORTED;
    if (bs != 16 && bs != 32 && bs != 64) return PA_ERR_UNSUPPORTED;
    if (group != 1 && group != 2 && group != 4 && group != 8) return PA_ERR_UNSUPPORTED;
    if (q_dtype != PA_F16 && q_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (cache->kv_dtype != PA_FP8_E4M3 && cache->kv_dtype != q_dtype) return PA_ERR_UNSUPPORTED;
    if (cache->kv_dtype == PA_FP8_E4M3 &&
        !(cache->k_scale > 0.f && std::isfinite(cache->k_scale) && cache->v_scale > 0.f &&
          std::isfinite(cache->v_scale)))
        return PA_ERR_INVALID_ARG;
    const int P = resolve_partition(partition_size, num_seqs, cache->num_kv_heads, max_seq_len, group);
    if (P % bs != 0) return PA_ERR_INVALID_ARG;
    if (num_seqs > 16384) return PA_ERR_UNSUPPORTED;
    if (cu_groups != nullptr && (shared_lens == nullptr || num_groups <= 0 || k_new != nullptr))
        return PA_ERR_INVALID_ARG;
    // group mode (the cascade in one launch): 8 / group members per launched
    // sequence fill the eight query rows of the G = 8 kernel over their group's
    // shared tokens, then every member's own tokens as sequences of their own
    const int vm = group_mode ? 8 / group : 0;
    const int64_t vpg = group_mode ? (max_group_size + vm - 1) / vm : 0;
    if (group_mode && (cu_groups == nullptr || max_group_size < 1)) return PA_ERR_INVALID_ARG;
    if (group_mode && num_groups * vpg + num_seqs > 16384) return PA_ERR_UNSUPPORTED;
    // cascade: the prefix's parts (ceil(s0/P)) and the suffix's (parts_of(L-s0))
    // never exceed parts_of(L) + 1
    const int max_parts = max_parts_of(max_seq_len, P) + (cu_groups != nullptr ? 1 : 0);
    const WsLayout w = ws_layout(num_seqs, num_heads, D, max_parts);
    if (w.bytes > 0 && (workspace == nullptr || workspace_bytes < w.bytes ||
                        (reinterpret_cast<uintptr_t>(workspace) & 15u)))
        return PA_ERR_INVALID_ARG;

    DecodeParams p{};
    p.out = out;
    p.q = q;
    p.k_cache = static_cast<const uint8_t*>(cache->k_cache);
    p.v_cache = static_cast<const uint8_t*>(cache->v_cache);
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.cu_seq_lens_k = cu_seq_lens_k;
    p.ws_lse = w.bytes ? reinterpret_cast<float*>(static_cast<char*>(workspace) + w.lse_off) : nullptr;
    p.ws_o = w.bytes ? reinterpret_cast<float*>(static_cast<char*>(workspace) + w.o_off) : nullptr;
    p.status = dev_status;
    p.num_blocks = cache->num_blocks;
    p.block_size = bs;
    p.num_kv_heads = cache->num_kv_heads;
    p.num_heads = num_heads;
    p.num_seqs = num_seqs;
    p.max_blocks = max_blocks_per_seq;
    p.max_seq_len = max_seq_len;
    p.partition = P;
    p.max_parts = max_parts;
    const float k_scale = cache->kv_dtype == PA_FP8_E4M3 ? cache->k_scale : 1.f;
    p.qk_scale = scale * k_scale * 1.4426950408889634f;
    p.v_scale = cache->kv_dtype == PA_FP8_E4M3 ? cache->v_scale : 1.f;
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_scale_w = cache->k_scale;
    p.v_scale_w = cache->v_scale;
    p.cu_groups = cu_groups;
    p.shared_lens = shared_lens;
    p.num_groups = num_groups;
    p.num_members = num_seqs;
    p.no_copies = no_copies ? 1 : 0;
    int kgroup = group;
    if (group_mode) {
        p.vm = vm;
        p.vpg = static_cast<int32_t>(vpg);
        p.vcount = static_cast<int32_t>(num_groups * vpg);
        p.g_real = group;
        p.num_seqs = p.vcount + num_seqs;
        kgroup = 8;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
#define PA_BS(KV)                                                       \
    if (bs == 16) return launch_decode_##KV##_bs16(p, q_dtype, D, kgroup, s); \
    if (bs == 32) return launch_decode_##KV##_bs32(p, q_dtype, D, kgroup, s); \
    return launch_decode_##KV##_bs64(p, q_dtype, D, kgroup, s);
    if (cache->kv_dtype == PA_F16) { PA_BS(f16) }
    if (cache->kv_dtype == PA_BF16) { PA_BS(bf16) }
    PA_BS(fp8)
#undef PA_BS
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_decode(void* out, const void* q, pa_dtype q_dtype, const pa_kv_cache* cache,
                               const int32_t* block_table, int32_t max_blocks_per_seq,
                               const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                               int32_t num_heads, float scale, int32_t partition_size,
                               void* workspace, size_t workspace_bytes, int32_t* dev_status,
                               pa_stream_t stream) {
    return pa::decode_entry(out, q, q_dtype, cache, block_table, max_blocks_per_seq, seq_lens, num_seqs,
                            max_seq_len, num_heads, scale, partition_size, workspace, workspace_bytes, dev_status,
                            stream, nullptr, nullptr);
}

extern "C" pa_status pa_decode_append(void* out, const void* q, const void* k_new, const void* v_new,
                                      pa_dtype q_dtype, const pa_kv_cache* cache, const int32_t* block_table,
                                      int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
                                      int32_t max_seq_len, int32_t num_heads, float scale,
                                      int32_t partition_size, void* workspace, size_t workspace_bytes,
                                      int32_t* dev_status, pa_stream_t stream) {
    if (k_new == nullptr || v_new == nullptr) return num_seqs == 0 ? PA_OK : PA_ERR_INVALID_ARG;
    if (cache != nullptr && cache->kv_dtype == PA_FP8_E4M3 &&
        !(cache->k_scale > 0.f && cache->v_scale > 0.f))
        return PA_ERR_INVALID_ARG;
    return pa::decode_entry(out, q, q_dtype, cache, block_table, max_blocks_per_seq, seq_lens, num_seqs,
                            max_seq_len, num_heads, scale, partition_size, workspace, workspace_bytes, dev_status,
                            stream, k_new, v_new);
}

extern "C" pa_status pa_decode_test_wait_timeout(void* out, const void* q, pa_dtype q_dtype,
                                                 const pa_kv_cache* cache, const int32_t* block_table,
                                                 int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                                 int32_t num_seqs, int32_t max_seq_len, int32_t num_heads,
                                                 float scale, int32_t partition_size, void* workspace,
                                                 size_t workspace_bytes, int32_t* dev_status, pa_stream_t stream) {
    return pa::decode_entry(out, q, q_dtype, cache, block_table, max_blocks_per_seq, seq_lens, num_seqs,
                            max_seq_len, num_heads, scale, partition_size, workspace, workspace_bytes, dev_status,
                            stream, nullptr, nullptr, nullptr, nullptr, nullptr, 0, false, 0, true);
}

extern "C" int32_t pa_decode_partition_size(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                            int32_t max_seq_len) {
    if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || max_seq_len < 0)
        return 0;
    return auto_partition(num_seqs, num_kv_heads, max_seq_len, num_heads / num_kv_heads);
}

extern "C" size_t pa_decode_cascade_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t head_size,
                                                   int32_t max_seq_len, int32_t block_size,
                                                   int32_t partition_size) {
    if (num_seqs <= 0 || num_heads <= 0 || head_size <= 0 || max_seq_len < 0 || block_size <= 0 ||
        partition_size < 0)
        return 0;
    const int P = ws_partition(partition_size);
    return ws_layout(num_seqs, num_heads, head_size, max_parts_of(max_seq_len, P) + 1).bytes;
}

extern "C" pa_status pa_decode_cascade(void* out, const void* q, pa_dtype q_dtype, const pa_kv_cache* cache,
                                       const int32_t* block_table, int32_t max_blocks_per_seq,
                                       const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                                       int32_t num_heads, float scale, const int32_t* cu_groups,
                                       const int32_t* shared_lens, int32_t num_groups, int32_t max_group_size,
                                       int32_t max_shared_len, int32_t partition_size, void* workspace,
                                       size_t workspace_bytes, int32_t* dev_status, pa_stream_t stream) {
    pa_status st = check_cache(cache);
    if (st != PA_OK) return st;
    if (num_seqs < 0 || num_groups < 0 || num_heads <= 0 || max_blocks_per_seq <= 0 || max_seq_len < 0 ||
        partition_size < 0 || !std::isfinite(scale))
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (num_groups == 0 || cu_groups == nullptr || shared_lens == nullptr || seq_lens == nullptr ||
        out == nullptr || q == nullptr || block_table == nullptr || workspace == nullptr)
        return PA_ERR_INVALID_ARG;
    if (num_heads % cache->num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    const int group = num_heads / cache->num_kv_heads;
    const int bs = cache->block_size;
    if (group != 1 && group != 2 && group != 4 && group != 8) return PA_ERR_UNSUPPORTED;
    if (max_group_size < 1) return PA_ERR_INVALID_ARG;
    if (max_shared_len < 0 || max_shared_len > max_seq_len || max_shared_len % bs != 0) return PA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 15u)) return PA_ERR_INVALID_ARG;
    const int P = resolve_partition(partition_size, num_seqs, cache->num_kv_heads, max_seq_len, group);
    if (P <= 0 || P % bs != 0) return PA_ERR_INVALID_ARG;
    const int max_parts = max_parts_of(max_seq_len, P) + 1;
    const WsLayout w = ws_layout(num_seqs, num_heads, cache->head_size, max_parts);
    if (workspace_bytes < w.bytes) return PA_ERR_INVALID_ARG;
    // One decode launch in group mode: a group's members side by side as the
    // query rows of one sequence over the group's shared blocks (read once per
    // 8 / group members, partials into parts 0 .. ceil(s0/P)-1) and every
    // member's own tokens (partials after those) share one work list; then the
    // log-sum-exp merge of all parts
    return decode_entry(out, q, q_dtype, cache, block_table, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                        num_heads, scale, P, workspace, workspace_bytes, dev_status, stream, nullptr, nullptr,
                        nullptr, cu_groups, shared_lens, num_groups, true, max_group_size);
}

extern "C" size_t pa_varlen_mixed_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t head_size,
                                                 int32_t max_seqlen_k, int32_t block_size) {
    return pa_decode_workspace_size(num_seqs, num_heads, head_size, max_seqlen_k, block_size, 0);
}

extern "C" pa_status pa_varlen_mixed(void* out, const void* q, pa_dtype q_dtype, const pa_kv_cache* cache,
                                     const int32_t* block_table, int32_t max_blocks_per_seq,
                                     const int32_t* cu_seq_lens_q, const int32_t* cu_seq_lens_k,
                                     const int32_t* host_cu_seq_lens_q, int32_t num_seqs, int32_t max_seqlen_q,
                                     int32_t max_seqlen_k, int32_t num_heads, float scale, int32_t causal,
                                     void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                     pa_stream_t stream) {
    if (num_seqs < 0 || max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (host_cu_seq_lens_q == nullptr || cache == nullptr) return PA_ERR_INVALID_ARG;
    // the trailing run of one-token sequences goes to the decode kernel
    int n_dec = 0;
    while (n_dec < num_seqs &&
           host_cu_seq_lens_q[num_seqs - n_dec] - host_cu_seq_lens_q[num_seqs - n_dec - 1] == 1)
        ++n_dec;
    const int n_pre = num_seqs - n_dec;
    if (n_pre > 0) {
        const pa_status st = pa_prefill_varlen(out, q, q_dtype, cache, block_table, max_blocks_per_seq,
                                               cu_seq_lens_q, cu_seq_lens_k, n_pre, max_seqlen_q, max_seqlen_k,
                                               num_heads, scale, causal, dev_status, stream);
        if (st != PA_OK) return st;
    }
    if (n_dec > 0) {
        // one query per sequence: causal or not, it sees all of its keys
        const int64_t r0 = host_cu_seq_lens_q[n_pre];
        const int64_t row_bytes = static_cast<int64_t>(num_heads) * cache->head_size * 2;
        return decode_entry(static_cast<char*>(out) + r0 * row_bytes, static_cast<const char*>(q) + r0 * row_bytes,
                            q_dtype, cache, block_table + static_cast<int64_t>(n_pre) * max_blocks_per_seq,
                            max_blocks_per_seq, nullptr, n_dec, max_seqlen_k, num_heads, scale, 0, workspace,
                            workspace_bytes, dev_status, stream, nullptr, nullptr, cu_seq_lens_k + n_pre);
    }
    return PA_OK;
}
