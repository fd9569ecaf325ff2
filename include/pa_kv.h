/*
 * pa_kv.h -- C ABI of the paged KV-cache attention library (libpa_kv.so).
 *
 * PagedAttention keeps each sequence's keys and values in fixed-size blocks
 * of `block_size` tokens per KV head; the blocks sit at arbitrary physical
 * block ids and a per-sequence block table maps logical block j (tokens
 * j*block_size .. (j+1)*block_size-1) to its physical id.  Sources:
 *   - vLLM PagedAttention design doc ("分页注意力机制", vllm.ooos.top):
 *     sections 输入参数 (q, k_cache, v_cache, out), 概念 (sequence, context,
 *     block), QK, Softmax, Value, Output.
 *   - "Paged 어텐션" (data-sketchers.com transformers paged-attention wiki):
 *     "Decode 경로" (block_table [batch, max_blocks_per_seq], -1 =
 *     unallocated, cache_seqlens, in-place cache update) and "Varlen 경로"
 *     (cu_seq_lens_q / cu_seq_lens_k, max_seqlen_q / max_seqlen_k).
 *   - "Как работает paged attention? (детально)" (aivaro.ru answers/837):
 *     sections 3.2 BlockManager, 3.3 copy-on-write, 4.1-4.2 allocation and
 *     deallocation, 5.1 block-wise attention.
 *   - vLLM paper summary (easyvpn24.com/25506.html): sections 2-4.
 *
 * Conventions for every call below:
 *   - Device pointers point to memory the caller owns (e.g. torch tensors);
 *     the device calls allocate nothing.  All device work is queued on
 *     `stream` (a cudaStream_t; NULL = the legacy default stream) and is
 *     asynchronous; the call returns once the work is queued.
 *   - Arguments are checked on the host before anything is launched; a bad
 *     argument returns PA_ERR_INVALID_ARG or PA_ERR_UNSUPPORTED and launches
 *     nothing.  A failed launch returns PA_ERR_CUDA.
 *   - Errors that depend on device data (a block id outside the pool, a slot
 *     outside the cache, a length above the stated maximum, a wait that ran
 *     out of time) are written to *dev_status (a device int32 the caller
 *     zeroes; may be NULL): the first error code wins.  The kernels never trap.
 *   - Cache layout (both K and V): [num_blocks][num_kv_heads][block_size]
 *     [head_size], row-major, so one (block, kv head) page is one contiguous
 *     block_size*head_size run.
 *   - GQA: query head h reads KV head h / (num_heads / num_kv_heads);
 *     num_heads must be a multiple of num_kv_heads.
 *   - Pool handles (pa_pool_*) hold host memory only and are not thread-safe.
 */
#ifndef PA_KV_H
#define PA_KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* the same type as cudaStream_t */
typedef struct CUstream_st* pa_stream_t;

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,  /* bad pointer, size, shape or length */
    PA_ERR_UNSUPPORTED = 2,  /* valid, but a head size / dtype / block size not built */
    PA_ERR_OOM = 3,          /* the block pool has too few free blocks */
    PA_ERR_CUDA = 4,         /* a CUDA launch or query failed */
    PA_ERR_TIMEOUT = 5,      /* device: a bounded wait ran out (dev_status only) */
    PA_ERR_BAD_BLOCK = 6     /* device: block id or slot outside the cache */
} pa_status;

typedef enum {
    PA_F16 = 0,       /* IEEE binary16 */
    PA_BF16 = 1,      /* bfloat16 */
    PA_FP8_E4M3 = 2   /* OCP FP8 E4M3 (finite-only "fn"), KV cache only */
} pa_dtype;

/* Description of one layer's paged KV cache (device memory owned by the
 * caller).  k_cache / v_cache: [num_blocks][num_kv_heads][block_size]
 * [head_size] elements of kv_dtype, 16-byte aligned.  For PA_FP8_E4M3 a
 * stored code c means the value c * k_scale (keys) or c * v_scale (values);
 * the scales are ignored for 16-bit caches. ("FP8 KV Cache" in the vLLM
 * feature list on "ChunkLlama", docsearch.algolia.com.) */
typedef struct {
    void* k_cache;
    void* v_cache;
    int64_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_size;
    pa_dtype kv_dtype;
    float k_scale;
    float v_scale;
} pa_kv_cache;

/* Human-readable name of a status code (static string). */
const char* pa_status_str(pa_status s);

/* Library version, major*10000 + minor*100 + patch. */
int32_t pa_version(void);

/* ---------------------------------------------------------------------------
 * Write new K/V rows into their cache slots.
 * "Paged 어텐션", Decode 경로 (the cache is updated in place through the
 * block table); "Как работает paged attention?" 4.1 step 5 (the new token's
 * KV goes to its position in the physical block); vLLM paper summary §3.
 *
 * k, v: device, [num_tokens][num_kv_heads][head_size] of in_dtype (F16 or
 *   BF16); consecutive tokens are token_stride elements apart (>=
 *   num_kv_heads*head_size; lets k/v be views into a fused qkv buffer).
 * slot_mapping: device int64 [num_tokens]; slot s means physical block
 *   s / block_size, offset s % block_size; s < 0 skips the token (padding).
 *   A slot >= num_blocks*block_size is skipped and reported as
 *   PA_ERR_BAD_BLOCK in *dev_status.
 * A 16-bit cache must have kv_dtype == in_dtype: the bits are moved
 *   unchanged.  An E4M3 cache stores e4m3_satfinite(round-to-nearest-even(
 *   (float)x / scale)), the division done in IEEE binary32.
 * Several tokens with the same slot: which one lands is unspecified.
 * ------------------------------------------------------------------------- */
pa_status pa_kv_cache_write(const pa_kv_cache* cache, const void* k, const void* v,
                            pa_dtype in_dtype, int64_t num_tokens, int64_t token_stride,
                            const int64_t* slot_mapping, int32_t* dev_status, pa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Copy whole physical blocks (all KV heads, K and V): the device half of
 * copy-on-write ("Как работает paged attention?" 3.3: a shared block is
 * copied before a sequence writes into it).
 * src_dst_pairs: device int32 [n][2] = (source id, destination id).  A pair
 * with an id outside [0, num_blocks) is skipped and reported as
 * PA_ERR_BAD_BLOCK.  Destinations must be distinct and not also sources.
 * ------------------------------------------------------------------------- */
pa_status pa_copy_blocks(const pa_kv_cache* cache, const int32_t* src_dst_pairs, int32_t n,
                         int32_t* dev_status, pa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Single-query decode attention over the paged cache.
 * vLLM PagedAttention design doc (whole walk-through: QK, Softmax, Value,
 * Output; the grid axis over context partitions); "Paged 어텐션" Decode 경로.
 *
 * For every sequence b and query head h, with L = seq_lens[b] and
 * kvh = h / (num_heads / num_kv_heads):
 *     s_t = scale * sum_d q[b][h][d] * K_b[t][d]      for t < L
 *     out[b][h][:] = sum_t softmax(s)_t * V_b[t][:]
 * where K_b[t] = k_cache[block_table[b][t / block_size]][kvh][t % block_size]
 * (times k_scale for E4M3), V_b likewise.  L = 0 gives out = 0.  Positions
 * t >= L take no part (they may hold anything, NaN included).
 *
 * out, q: device [num_seqs][num_heads][head_size] of q_dtype (F16 or BF16),
 *   16-byte aligned.  q_dtype must equal kv_dtype for 16-bit caches; an E4M3
 *   cache takes F16 or BF16 queries.  out is rounded to nearest even.
 * block_table: device int32 [num_seqs][max_blocks_per_seq]; only the first
 *   ceil(L / block_size) entries of a row are read; each must be in
 *   [0, num_blocks), otherwise PA_ERR_BAD_BLOCK is reported and that page is
 *   left out.
 * seq_lens: device int32 [num_seqs], the attended lengths ("cache_seqlens"
 *   counting the token just written).  Each must be <= max_seq_len and
 *   <= max_blocks_per_seq*block_size, otherwise PA_ERR_INVALID_ARG is
 *   reported and the sequence's output is 0.
 * partition_size: tokens per context partition (a multiple of block_size),
 *   0 = automatic (pa_decode_partition_size: 2048, or 1024 when num_heads /
 *   num_kv_heads >= 4; with fewer (sequence, KV head) pairs than resident
 *   decode blocks, doubled up to 8192 while the work items of max_seq_len
 *   still number four or more per block; with more pairs and num_heads /
 *   num_kv_heads >= 4, 1536; then halved, not below 512, while the items
 *   would not fill the GPU twice over; the workspace size query answers for
 *   512, which covers every automatic choice).  A
 *   sequence longer than one partition is split; the
 *   partitions' partial results go to `workspace` and a second kernel merges
 *   them by their log-sum-exp.
 * workspace: device scratch of at least pa_decode_workspace_size(...) bytes,
 *   16-byte aligned (may be NULL when that size is 0).
 * Supported: head_size 64 or 128; block_size 16, 32 or 64;
 *   num_heads / num_kv_heads in {1, 2, 4, 8}.
 * ------------------------------------------------------------------------- */
size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t head_size,
                                int32_t max_seq_len, int32_t block_size, int32_t partition_size);

/* The partition size pa_decode takes for partition_size = 0 on the current
 * device (host call, no launch); 0 for invalid arguments. */
int32_t pa_decode_partition_size(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                 int32_t max_seq_len);

pa_status pa_decode(void* out, const void* q, pa_dtype q_dtype, const pa_kv_cache* cache,
                    const int32_t* block_table, int32_t max_blocks_per_seq,
                    const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                    int32_t num_heads, float scale, int32_t partition_size, void* workspace,
                    size_t workspace_bytes, int32_t* dev_status, pa_stream_t stream);

/* ---------------------------------------------------------------------------
 * pa_decode for callers that cannot allocate device memory.  (The pages have
 * no counterpart: this is a property of the library, not of the method.)
 *
 * Some callers cannot call cudaMalloc: a plugin or embedded runtime whose host
 * program owns all device memory through its own allocator, or a serving loop
 * that must not call cudaMalloc/cudaFree because they can synchronise the
 * device.  This call takes the same arguments as pa_decode minus the
 * workspace: the split-K partial results go to a scratch array of
 * PA_DECODE_STATIC_WS_BYTES that is built into the library and held by every
 * GPU that loads it until the process exits.  It allocates nothing.
 *   - partition_size 0 is resolved first (pa_decode_partition_size) and the
 *     resolved partition is the one both the size check and the launch use.
 *   - A call whose pa_decode_workspace_size(..., resolved partition) exceeds
 *     PA_DECODE_STATIC_WS_BYTES returns PA_ERR_UNSUPPORTED and launches
 *     nothing (use pa_decode with a workspace of your own instead).
 *   - The first call on a device looks up the scratch's device address
 *     (cudaGetSymbolAddress, with that device current) and remembers it
 *     together with the context then current; a call that finds another
 *     context current (after cudaDeviceReset, or in a context the caller
 *     created) looks it up again.  Make the first call on a device, and in
 *     each such new context, before any stream capture.
 *   - Every call on a device shares the one array and finds the previous
 *     call's data in it; nothing needs clearing, but calls whose kernels
 *     overlap on the GPU (e.g. on two unordered streams) race and give wrong
 *     results.  Order them on one stream.
 * ------------------------------------------------------------------------- */
#define PA_DECODE_STATIC_WS_BYTES (16u * 1024u * 1024u)

pa_status pa_decode_static_ws(void* out, const void* q, pa_dtype q_dtype, const pa_kv_cache* cache,
                              const int32_t* block_table, int32_t max_blocks_per_seq,
                              const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                              int32_t num_heads, float scale, int32_t partition_size,
                              int32_t* dev_status, pa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Varlen prefill (and mixed prefill + decode) attention over the paged cache.
 * "Paged 어텐션" Varlen 경로 (cu_seq_lens_q/k index a batch of sequences of
 * different lengths; max_seqlen_q/k bound them); keys and values are read
 * from the paged cache through block_table as in the Decode 경로; causal
 * masking per block as in "Как работает paged attention?" 5.1.
 *
 * Sequence b owns query rows cu_seq_lens_q[b] .. cu_seq_lens_q[b+1]-1 of q
 * and has Lk = cu_seq_lens_k[b+1] - cu_seq_lens_k[b] keys at logical
 * positions 0..Lk-1 of its block-table row (the new tokens' K/V must already
 * be in the cache, e.g. by pa_kv_cache_write).  With Lq query rows, query i
 * sits at position Lk - Lq + i; with causal != 0 it sees keys j <= Lk - Lq + i
 * (bottom-right alignment), otherwise all Lk keys.  A row that sees no key
 * outputs 0.
 * q, out: device [total_q][num_heads][head_size] of q_dtype (BF16 or F16,
 *   equal to kv_dtype), total_q = cu_seq_lens_q[num_seqs], 16-byte aligned.
 * cu_seq_lens_q, cu_seq_lens_k: device int32 [num_seqs + 1], non-decreasing,
 *   starting at 0.  max_seqlen_q / max_seqlen_k must bound the lengths (a
 *   sequence that breaks them is reported as PA_ERR_INVALID_ARG and its rows
 *   are not written).  A block id outside [0, num_blocks) among the entries
 *   a sequence needs is reported as PA_ERR_BAD_BLOCK; that sequence's rows are
 *   then unspecified.
 * Supported: head_size 128; block_size 16, 32 or 64;
 *   num_heads / num_kv_heads in {1, 2, 4, 8}; 16-bit caches.
 * ------------------------------------------------------------------------- */
pa_status pa_prefill_varlen(void* out, const void* q, pa_dtype q_dtype, const pa_kv_cache* cache,
                            const int32_t* block_table, int32_t max_blocks_per_seq,
                            const int32_t* cu_seq_lens_q, const int32_t* cu_seq_lens_k,
                            int32_t num_seqs, int32_t max_seqlen_q, int32_t max_seqlen_k,
                            int32_t num_heads, float scale, int32_t causal, int32_t* dev_status,
                            pa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Swap whole blocks between the device cache and page-locked host memory:
 * the data move of swap-based preemption ("Как работает paged attention?"
 * 4.3: the preempted request's KV cache goes to CPU memory and comes back
 * when it resumes; vLLM paper summary, section 5: a CPU block allocator
 * holds the swapped blocks).  Which requests to preempt, and the host-side
 * block ids, are the caller's (a scheduler's) business.
 *
 * host_k, host_v: page-locked host memory (cudaHostAlloc / cudaMallocHost /
 *   cudaHostRegister, or a pinned torch tensor), 16-byte aligned, laid out
 *   like the cache: [num_host_blocks][num_kv_heads][block_size][head_size]
 *   of the cache's dtype.  Pageable memory is rejected (PA_ERR_INVALID_ARG).
 * pairs: device int32 [n][2] = (device block id, host block id), n <= 65535.
 *   to_host != 0 copies device -> host (swap out), 0 copies host -> device
 *   (swap in).  A pair with an id out of range is skipped and reported as
 *   PA_ERR_BAD_BLOCK.  Destinations must be distinct.
 * Asynchronous on `stream`; the host buffers must stay valid (and, for swap
 * out, unread) until the stream reaches this point.
 * ------------------------------------------------------------------------- */
pa_status pa_swap_blocks(const pa_kv_cache* cache, void* host_k, void* host_v, int64_t num_host_blocks,
                         const int32_t* pairs, int32_t n, int32_t to_host, int32_t* dev_status,
                         pa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Fused cache write + decode: for every sequence b with L = seq_lens[b] >= 1,
 * the new token's K/V (k_new[b], v_new[b]) is stored at position L-1 -- the
 * slot block_table[b][(L-1)/block_size]*block_size + (L-1)%block_size, as
 * pa_kv_cache_write would store it -- and the query attends over all L
 * tokens including it, in one launch.  Results and cache contents are
 * bit-identical to pa_kv_cache_write followed by pa_decode ("Paged 어텐션",
 * Decode 경로: the kernel updates the cache in place; the worked example's
 * new tokens at positions 30, 32, 70).  The new token's page is read only up
 * to the row before it.
 *
 * k_new, v_new: device [num_seqs][num_kv_heads][head_size] of q_dtype,
 *   16-byte aligned.  E4M3 caches store e4m3_satfinite(rne(x / scale)).
 * The block holding position L-1 must already be in the table (an id out of
 *   range is reported as PA_ERR_BAD_BLOCK and nothing is written for it).
 * Everything else as pa_decode (same workspace size).
 * ------------------------------------------------------------------------- */
pa_status pa_decode_append(void* out, const void* q, const void* k_new, const void* v_new, pa_dtype q_dtype,
                           const pa_kv_cache* cache, const int32_t* block_table, int32_t max_blocks_per_seq,
                           const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len, int32_t num_heads,
                           float scale, int32_t partition_size, void* workspace, size_t workspace_bytes,
                           int32_t* dev_status, pa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Shared-prefix ("cascade") decode.  "Как работает paged attention?
 * (детально)" §3.3: sequences of parallel sampling or beam search refer to the
 * same physical blocks for their common prefix (copy-on-write on change); §7:
 * requests with the same prefix reuse its physical blocks (prefix caching);
 * the vLLM paper summary lists parallel sampling and shared prefixes among its
 * decoding scenarios.  The pages give no kernel for it; this entry point
 * computes exactly what pa_decode computes (the same softmax(q K^T scale) V per
 * sequence and head, up to fp32 rounding order) but reads a group's shared
 * blocks once per 8 / (num_heads / num_kv_heads) members: one decode launch
 * attends every member's query to the shared tokens (those members' heads side
 * by side as the eight query rows of one sequence) and each member's own
 * tokens, all in partitions of one work list, and the log-sum-exp merge of
 * pa_decode combines all partitions.
 *
 * cu_groups: device int32 [num_groups+1], 0 = cu_groups[0] <= ... <=
 *   cu_groups[num_groups] = num_seqs; sequences cu_groups[g] .. cu_groups[g+1]-1
 *   form group g (consecutive rows of q, out, block_table and seq_lens).
 * shared_lens: device int32 [num_groups]: group g's first shared_lens[g] tokens
 *   are whole blocks (a multiple of block_size) that every member's block-table
 *   row names identically and every member attends (shared_lens[g] <= each
 *   member's length).  The blocks are read through the group's first row; a
 *   member whose row differs there, or a shared length that breaks these rules,
 *   is reported as PA_ERR_INVALID_ARG in dev_status.
 * max_group_size: the largest group (host bound, >= 1).  max_shared_len: host
 *   bound on shared_lens (a multiple of block_size, <= max_seq_len).
 * workspace: pa_decode_cascade_workspace_size(...) bytes, 16-byte aligned (never
 *   0: every (sequence, head) keeps a prefix and a suffix partial).
 * Supported: the shapes and types of pa_decode (fp16/bf16 caches with q of the
 *   same type, or E4M3 caches; head_size 64 or 128; block sizes 16/32/64;
 *   num_heads / num_kv_heads in {1, 2, 4, 8}); others return PA_ERR_UNSUPPORTED
 *   with nothing launched.  Everything else as pa_decode.
 * ------------------------------------------------------------------------- */
size_t pa_decode_cascade_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t head_size,
                                        int32_t max_seq_len, int32_t block_size, int32_t partition_size);
pa_status pa_decode_cascade(void* out, const void* q, pa_dtype q_dtype, const pa_kv_cache* cache,
                            const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                            int32_t num_seqs, int32_t max_seq_len, int32_t num_heads, float scale,
                            const int32_t* cu_groups, const int32_t* shared_lens, int32_t num_groups,
                            int32_t max_group_size, int32_t max_shared_len, int32_t partition_size,
                            void* workspace, size_t workspace_bytes, int32_t* dev_status, pa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Mixed batch dispatcher: a varlen batch (as pa_prefill_varlen) whose
 * trailing sequences have one query token each is split -- the leading
 * sequences go to the varlen tensor-core kernel, the trailing one-token run
 * to the decode kernel, which reads each length as cu_seq_lens_k[b+1] -
 * cu_seq_lens_k[b] ("Paged 어텐션": the decode path is the faster one for
 * single-query sequences, the varlen path takes the prefills).  A single
 * query sees all of its keys, causal or not, so the split computes the same
 * attention.
 *
 * host_cu_seq_lens_q: host int32 [num_seqs+1], a copy of cu_seq_lens_q (the
 *   split is decided on the host; nothing is read back from the device).
 * workspace: device scratch of pa_varlen_mixed_workspace_size(...) bytes,
 *   16-byte aligned (NULL if that is 0), for the decode kernel's partitions.
 * Everything else as pa_prefill_varlen; head_size 64 is only served when
 * every sequence is a one-token sequence.
 * ------------------------------------------------------------------------- */
size_t pa_varlen_mixed_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t head_size,
                                      int32_t max_seqlen_k, int32_t block_size);
pa_status pa_varlen_mixed(void* out, const void* q, pa_dtype q_dtype, const pa_kv_cache* cache,
                          const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* cu_seq_lens_q,
                          const int32_t* cu_seq_lens_k, const int32_t* host_cu_seq_lens_q, int32_t num_seqs,
                          int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t num_heads, float scale,
                          int32_t causal, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                          pa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Varlen attention over packed K/V: "Paged 어텐션", Varlen 경로 -- the batch's
 * keys and values are contiguous tensors [Σk][num_kv_heads][head_size]
 * indexed by cu_seq_lens_k (no cache, no block table), queries as in
 * pa_prefill_varlen.  Same arithmetic and causal alignment as
 * pa_prefill_varlen (bottom-right; rows without a visible key give 0).
 *
 * k, v: device, total_k rows of num_kv_heads*head_size elements of dtype (F16
 *   or BF16, the same as q and out), 16-byte aligned; may be NULL when
 *   total_k == 0.  cu_seq_lens_k[b+1] must be <= total_k, otherwise
 *   PA_ERR_INVALID_ARG is reported in *dev_status and that sequence's rows are
 *   unspecified.
 * Supported: head_size 128; num_heads / num_kv_heads in {1, 2, 4, 8};
 *   num_seqs <= 6144.
 * ------------------------------------------------------------------------- */
pa_status pa_prefill_varlen_packed(void* out, const void* q, const void* k, const void* v, pa_dtype dtype,
                                   const int32_t* cu_seq_lens_q, const int32_t* cu_seq_lens_k, int32_t num_seqs,
                                   int32_t max_seqlen_q, int32_t max_seqlen_k, int64_t total_k, int32_t num_heads,
                                   int32_t num_kv_heads, int32_t head_size, float scale, int32_t causal,
                                   int32_t* dev_status, pa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Slots of new tokens from a block table (host arrays): "Как работает paged
 * attention?" 4.1 (logical block = pos / block_size, offset pos % block_size);
 * vLLM paper summary §3.  For token i of sequence seq_idx[i] at position
 * pos[i]: slot = block_table[seq][pos / block_size] * block_size
 * + pos % block_size.  An entry < 0 (unallocated) or a position past the row
 * gives slot -1.  block_table: host int32 [num_seqs][max_blocks]; seq_idx:
 * host int32 [n] in [0, num_seqs); pos: host int64 [n] >= 0; slots_out: host
 * int64 [n].  Returns PA_ERR_INVALID_ARG for a bad sequence index or position.
 * ------------------------------------------------------------------------- */
pa_status pa_slot_mapping(const int32_t* block_table, int32_t num_seqs, int32_t max_blocks,
                          int32_t block_size, const int32_t* seq_idx, const int64_t* pos, int64_t n,
                          int64_t* slots_out);

/* ---------------------------------------------------------------------------
 * Host block pool ("Как работает paged attention?" 3.2 BlockManager, 3.3,
 * 4.1, 4.2; vLLM paper summary §2-4).  Host memory only.
 *
 * The free list is FIFO: allocation takes its head, a freed block goes to
 * its tail.  free_order (nullable, a permutation of 0..num_blocks-1) sets the
 * initial order; NULL means 0, 1, 2, ...
 * pa_pool_append(seq, n): positions len .. len+n-1 get slots; a position in a
 *   logical block not yet mapped gets a new block (reference count 1).  If the
 *   last block is shared (reference count > 1) and not full, it is first
 *   replaced by a private block taken from the free list: the (old, new) pair
 *   is written to cow_pairs_out (room for 2 int32) and *n_cow_out = 1; the
 *   caller copies it with pa_copy_blocks before writing the slots.  If the
 *   free list cannot supply every block the append needs, nothing changes and
 *   PA_ERR_OOM is returned.  slots_out: host int64 [n].
 * pa_pool_fork(parent, child): the child shares all of the parent's blocks
 *   (each reference count + 1) and its length.
 * pa_pool_free_seq: each block's reference count - 1, in logical order; a
 *   block reaching 0 goes to the tail of the free list.
 * pa_pool_block_table: host int32 [n][max_blocks] rows, -1 padded, and host
 *   int32 lens_out[n] (nullable).  A sequence with more blocks than
 *   max_blocks gives PA_ERR_INVALID_ARG.
 * Sequence ids are arbitrary int64 keys; an unknown id gives
 * PA_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------- */
pa_status pa_pool_create(int64_t num_blocks, int32_t block_size, const int32_t* free_order,
                         void** pool_out);
void pa_pool_destroy(void* pool);
pa_status pa_pool_add_seq(void* pool, int64_t seq_id);
pa_status pa_pool_append(void* pool, int64_t seq_id, int32_t n_tokens, int64_t* slots_out,
                         int32_t* cow_pairs_out, int32_t* n_cow_out);
pa_status pa_pool_fork(void* pool, int64_t parent, int64_t child);
pa_status pa_pool_free_seq(void* pool, int64_t seq_id);
pa_status pa_pool_block_table(void* pool, const int64_t* seq_ids, int32_t n, int32_t max_blocks,
                              int32_t* table_out, int32_t* lens_out);
int64_t pa_pool_num_free(void* pool);
int32_t pa_pool_ref_count(void* pool, int64_t block);
int32_t pa_pool_seq_len(void* pool, int64_t seq_id);

/* ---------------------------------------------------------------------------
 * Test hook for the decode's wait timeout.  (Not on the pages: every wait of
 * the library's kernels is bounded, so that a stalled copy ends in an error
 * status instead of a hung GPU.)
 *
 * Same arguments and host checks as pa_decode, but the launched decode's
 * producer warp issues no copy at all: no page and no query ever lands, so
 * every consumer wait runs out after the library's wait limit (2 s) with
 * nothing in flight, PA_ERR_TIMEOUT (5) is written to *dev_status, and the
 * kernel returns.  The output and workspace contents are unspecified
 * afterwards (within their stated sizes); the device stays usable.  For the
 * library's own tests; a serving path has no use for it.
 * ------------------------------------------------------------------------- */
pa_status pa_decode_test_wait_timeout(void* out, const void* q, pa_dtype q_dtype, const pa_kv_cache* cache,
                                      const int32_t* block_table, int32_t max_blocks_per_seq,
                                      const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                                      int32_t num_heads, float scale, int32_t partition_size, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status, pa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_KV_H */
