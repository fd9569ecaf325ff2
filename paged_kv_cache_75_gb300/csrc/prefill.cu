// Varlen (prefill / mixed) attention over the paged KV cache on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// "Paged 어텐션" (data-sketchers.com transformers paged-attention wiki),
// Varlen 경로: a batch of sequences of different lengths is indexed by the
// cumulative lengths cu_seq_lens_q / cu_seq_lens_k (bounded by max_seqlen_q /
// max_seqlen_k); here the keys and values come from the paged cache through
// block_table (Decode 경로) instead of packed K/V tensors.
// "Как работает paged attention? (детально)" 5.1: attention runs block by
// block over the physical blocks, with the causal mask applied per block.
// Softmax by max subtraction as in the vLLM PagedAttention design doc
// (section Softmax), kept online across key tiles.
//
// Work item = (sequence, tile of TQ = 128/G query tokens, KV head): its 128
// rows are the G query heads of the KV head for TQ tokens (row = t*G + g), so
// one key/value tile serves the whole GQA group.  Items are sorted by their
// key-tile count and dealt to the persistent blocks in snake order.  Per
// item, key tiles of 128 keys stream through a 3-stage K ring and a 2-stage
// V ring:
//   warps 0, 2  load pages with TMA tensor copies (128B swizzle), through the
//               block table (or 3-D boxes of packed K/V): warp 0 the K ring,
//               warp 2 the V ring;
//   warp 3      loads each item's 128 query rows into shared memory in the
//               layout of a K tile once the previous item's last QK is done
//               (two 3-D TMA boxes; at the batch's end 16-byte asynchronous
//               copies, zero past the sequence);
//   warp 1      allocates tensor memory and issues every MMA from one thread:
//               S[t & 1] = Q K(t)^T from shared memory, then
//               O[c] += P V(t) with the weights P written over S[t & 1]; two
//               O buffers (c alternates per item) let one item's epilogue run
//               beside the next item's first PV;
//   warps 4..7, two softmax warpgroups that split the 128 key columns of each
//   8..11       tile (a thread: 64 columns of one row, its tensor-memory
//               lane).  They take weights against a shared reference max and
//               vote at a barrier whether any row's sum would pass 2^64; only
//               then (and on an item's first tile) is the true max taken,
//               exchanged through shared memory, O rescaled in tensor memory
//               and the weights recomputed.  Weights go to tensor memory as
//               bf16 hi + lo (both truncated, ~16 bits together; two PV
//               passes) or one fp16.  An item's epilogue (O / l) is written
//               once the next item's first weights are out.
// Causal alignment is bottom-right: query i of a sequence with Lq queries and
// Lk keys sits at position Lk - Lq + i.  Every wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace pa {
namespace {

constexpr int kD = 128;              // head size
constexpr int kBN = 128;             // keys per tile
constexpr int kRows = 128;           // MMA M: query rows per item
constexpr int kStages = 3;           // depth of the K ring
constexpr int kStagesV = 2;          // depth of the V ring
constexpr int kThreads = 384;        // 12 warps
constexpr int kSoftWarp0 = 4;        // softmax warpgroups = warps 4..7 and 8..11
constexpr uint32_t kTmemCols = 512;
// tensor-memory columns: S[b] (fp32 scores of the key tiles t with t & 1 = b,
// later overwritten by the 16-bit weights P) and O[c] (fp32 accumulators of
// the items with key tiles, c = their count & 1: one item's O is written out
// while the next item's first PV goes to the other)
constexpr uint32_t kColS = 0;    // S[b] at b * kBN
constexpr uint32_t kColO = 256;  // O[c] at kColO + c * kD

// shared memory layout (bytes from the 1 KB-aligned base)
constexpr int kBlkBytes = kBN * 128;           // 16 KB: one 64-column block of a K or V tile
constexpr int kTileBytes = 2 * kBlkBytes;      // 32 KB: a K or a V tile
constexpr int kOffK = 0;                       // K ring
constexpr int kOffV = kOffK + kStages * kTileBytes;  // V ring
constexpr int kOffQ = kOffV + kStagesV * kTileBytes; // the item's 128 query rows, laid out like a K tile
constexpr int kOffBar = kOffQ + kTileBytes;
constexpr int kNumBars = 2 * kStages + 2 * kStagesV + 3 * 2 + 3;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kOffXch = kOffMisc + 64;                   // [2 slots][2 warpgroups][128 rows] floats
constexpr int kOffPend = kOffXch + 2 * 2 * kRows * 4;  // [256] int64 row offsets, then [256] float row sums
constexpr int kItemCache = 64;                          // a CTA's first items, worked out once
constexpr int kOffItems = kOffPend + 256 * 12;          // [kItemCache] Work
constexpr int kSmemBytes = kOffItems + kItemCache * 32;
constexpr int kMaxSeqs = 6144;                           // prefix of query tiles: (B + 1) ints

struct PrefillParams {
    void* out;
    const uint16_t* q;
    const int32_t* block_table;
    const int32_t* cu_q;
    const int32_t* cu_k;
    int32_t* status;
    int64_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t num_heads;
    int32_t group;  // num_heads / num_kv_heads
    int32_t tq;     // query tokens per item (128 / group)
    int32_t num_seqs;
    int32_t max_blocks;
    int32_t max_q;
    int32_t max_k;
    int32_t causal;
    float scale_log2;  // scale * log2(e)
    int64_t total_k;   // packed K/V: rows of K and V (Σ key lengths); -1 for the paged cache
    int32_t order_cap; // query tiles the shared-memory work order holds (set by the launch)
    int32_t q_rows;    // token extent of the query tensor map: min(num_seqs * max_seqlen_q, INT32_MAX)
};

// ---------------------------------------------------------------------------
// PTX wrappers (tcgen05, TMA)
// ---------------------------------------------------------------------------
// shared-memory matrix descriptor, 128-byte swizzle
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = static_cast<uint64_t>((addr >> 4) & 0x3FFF);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32;
    d |= 1ull << 46;  // descriptor version
    d |= 2ull << 61;  // SWIZZLE_128B
    return d;
}
// instruction descriptor, kind::f16, fp32 accumulate; fmt 0 = f16, 1 = bf16
__host__ __device__ constexpr uint32_t mma_idesc(int fmt, int M, int N, int b_mn_major) {
    return (1u << 4) | (static_cast<uint32_t>(fmt) << 7) | (static_cast<uint32_t>(fmt) << 10) |
           (static_cast<uint32_t>(b_mn_major) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}
// A from tensor memory (row per lane, two 16-bit elements per column), B from shared memory
__device__ __forceinline__ void mma_f16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t db, uint32_t idesc,
                                           uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(db), "r"(idesc), "r"(acc));
}
// A and B from shared memory
__device__ __forceinline__ void mma_f16_ss(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(da), "l"(db), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's tensor-memory lane
__device__ __forceinline__ void tmem_ld32(uint32_t addr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(addr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32(uint32_t addr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(addr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 64 consecutive fp32 columns of this thread's tensor-memory lane, one wait
__device__ __forceinline__ void tmem_ld64(uint32_t addr, float (&v)[64]) {
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,"
        "%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(addr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}
// 16 consecutive 32-bit columns of this thread's lane (completion: tmem_wait_st)
__device__ __forceinline__ void tmem_st16(uint32_t addr, const uint32_t (&w)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            addr),
        "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]), "r"(w[8]), "r"(w[9]),
        "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// two fp32 -> their upper halves (bf16 by truncation), x in the low half
__device__ __forceinline__ uint32_t hi_halves(float x, float y) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(d) : "r"(__float_as_uint(x)), "r"(__float_as_uint(y)));
    return d;
}
// packed fp32 pairs: one instruction for both halves
__device__ __forceinline__ uint64_t f2pack(float x, float y) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}
__device__ __forceinline__ float2 f2unpack(uint64_t r) {
    float2 f;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(r));
    return f;
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// named barrier over n threads that also ORs a predicate across them
__device__ __forceinline__ bool bar_red_or(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "barrier.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// 2-D tiled TMA load into shared memory, completion counted on `bar`
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// 16-byte asynchronous copy global -> shared; src_bytes 0 writes zeros and
// reads nothing
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// one 32-byte global store (dst 32-byte aligned)
__device__ __forceinline__ void st_global_v8(void* dst, const uint32_t* w) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(reinterpret_cast<uint64_t>(dst)),
                 "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// 3-D tiled TMA load (packed K/V: {element, KV head, token})
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// byte offset of (row, 16-byte chunk) in a [rows][128 B] region with 128B swizzle
__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

template <int DT>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (DT == PA_BF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}

// lengths of sequence b; false if they break the stated bounds
__device__ __forceinline__ bool seq_lens_ok(const PrefillParams& p, int b, int& lq, int& lk) {
    const int q0 = __ldg(p.cu_q + b), q1 = __ldg(p.cu_q + b + 1);
    const int k0 = __ldg(p.cu_k + b);
    const int k1 = __ldg(p.cu_k + b + 1);
    lq = q1 - q0;
    lk = k1 - k0;
    const bool fits = p.total_k >= 0 ? (k0 >= 0 && static_cast<int64_t>(k1) <= p.total_k)
                                     : static_cast<int64_t>(lk) <= static_cast<int64_t>(p.max_blocks) * p.block_size;
    return lq >= 0 && lk >= 0 && lq <= p.max_q && lk <= p.max_k && fits;
}

struct Work {
    int b, i0, kvh, lq, lk, kend, ntiles;
    int q0;  // cu_q[b]: the sequence's first query row
};
static_assert(sizeof(Work) == 32, "the item cache holds 32-byte entries");

// Work order.  An item's cost is its number of key tiles, which under the
// causal mask grows along a sequence's query tiles and differs widely between
// sequences.  When the query tiles fit the shared-memory order array, every
// CTA sorts them by cost class (64 classes, most key tiles first, ties in
// list order) and deals the items out in snake order (snake_item): the
// CTAs' totals then stay within about 1 % of each other on a mixed batch,
// where round-robin in sequence order left the busiest 11 % above the mean.
// Otherwise the items keep sequence order.
__device__ __forceinline__ int tile_seq(const PrefillParams& p, const int32_t* prefix, int tile) {
    int lo = 0, hi = p.num_seqs - 1;  // largest b with prefix[b] <= tile
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= tile) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ int tile_class(const PrefillParams& p, const int32_t* prefix, int tile) {
    const int b = tile_seq(p, prefix, tile);
    int lq, lk;
    seq_lens_ok(p, b, lq, lk);
    const int i0 = (tile - prefix[b]) * p.tq;
    int kend = lk;
    if (p.causal) kend = min(lk, lk - lq + min(i0 + p.tq, lq));
    const int maxt = (p.max_k + kBN - 1) / kBN;
    const int nt = kend > 0 ? min(maxt, (kend + kBN - 1) / kBN) : 0;
    return 63 - static_cast<int>((static_cast<int64_t>(nt) * 64) / (maxt + 1));  // 0 = most key tiles
}

// Stable counting sort of the n query tiles by class: each warp counts a
// contiguous chunk (lanes of equal class found by match.any), warp 0 turns
// the [warp][class] counts into class-major offsets, each warp then places its
// chunk in order.  All threads of the block take part; hist holds 12*64 ints.
__device__ void build_tile_order(const PrefillParams& p, const int32_t* prefix, int n, int32_t* order,
                                 int32_t* hist) {
    constexpr int NW = kThreads / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunk = ((n + NW - 1) / NW + 31) & ~31;
    const int t0 = warp * chunk, t1 = min(n, t0 + chunk);
    int32_t* h = hist + warp * 64;
    h[lane] = 0;
    h[lane + 32] = 0;
    __syncwarp();
    for (int c0 = t0; c0 < t1; c0 += 32) {
        const int t = c0 + lane;
        const int key = t < t1 ? tile_class(p, prefix, t) : 64;
        const unsigned same = __match_any_sync(0xffffffffu, key);
        if (t < t1 && lane == __ffs(same) - 1) h[key] += __popc(same);
        __syncwarp();
    }
    __syncthreads();
    if (warp == 0) {
        int tot0 = 0, tot1 = 0;
        for (int w = 0; w < NW; ++w) {
            tot0 += hist[w * 64 + 2 * lane];
            tot1 += hist[w * 64 + 2 * lane + 1];
        }
        int incl = tot0 + tot1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += x;
        }
        int base0 = incl - tot0 - tot1, base1 = incl - tot1;
        for (int w = 0; w < NW; ++w) {
            const int x0 = hist[w * 64 + 2 * lane], x1 = hist[w * 64 + 2 * lane + 1];
            hist[w * 64 + 2 * lane] = base0;
            hist[w * 64 + 2 * lane + 1] = base1;
            base0 += x0;
            base1 += x1;
        }
    }
    __syncthreads();
    for (int c0 = t0; c0 < t1; c0 += 32) {
        const int t = c0 + lane;
        const int key = t < t1 ? tile_class(p, prefix, t) : 64;
        const unsigned same = __match_any_sync(0xffffffffu, key);
        if (t < t1) order[h[key] + __popc(same & ((1u << lane) - 1u))] = t;
        __syncwarp();
        if (t < t1 && lane == __ffs(same) - 1) h[key] += __popc(same);
        __syncwarp();
    }
    __syncthreads();
}

__device__ __forceinline__ Work work_item(const PrefillParams& p, const int32_t* prefix, const int32_t* order,
                                          int item) {
    Work w;
    int tile_id = item / p.num_kv_heads;
    w.kvh = item - tile_id * p.num_kv_heads;
    if (order != nullptr) tile_id = order[tile_id];
    int lo = 0, hi = p.num_seqs - 1;  // largest b with prefix[b] <= tile_id
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= tile_id) lo = mid;
        else hi = mid - 1;
    }
    w.b = lo;
    seq_lens_ok(p, lo, w.lq, w.lk);
    w.q0 = __ldg(p.cu_q + lo);
    w.i0 = (tile_id - prefix[lo]) * p.tq;
    const int shift = w.lk - w.lq;
    w.kend = w.lk;
    if (p.causal) w.kend = min(w.lk, shift + min(w.i0 + p.tq, w.lq));
    w.ntiles = w.kend > 0 ? (w.kend + kBN - 1) / kBN : 0;
    return w;
}

// PACKED: K and V are contiguous [Σk][num_kv_heads][head_size] tensors indexed
// by cu_seq_lens_k (no cache, no block table); otherwise the paged cache.
template <int DT, bool PACKED>
__global__ void __launch_bounds__(kThreads, 1)
paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                        const __grid_constant__ CUtensorMap map_q,
                        const PrefillParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 128B-swizzled tiles need 1 KB alignment; the launch adds 1 KB of slack
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sK = smem + kOffK;
    uint8_t* sV = smem + kOffV;
    uint8_t* sQ = smem + kOffQ;
    const uint32_t bar0 = smem_addr(smem + kOffBar);
    const uint32_t k_full = bar0;                       // [kStages] TMA bytes of a K tile
    const uint32_t k_empty = k_full + 8 * kStages;      // [kStages] MMA commit after QK
    const uint32_t v_full = k_empty + 8 * kStages;      // [kStagesV] TMA bytes of a V tile
    const uint32_t v_empty = v_full + 8 * kStagesV;     // [kStagesV] MMA commit after PV
    const uint32_t s_full = v_empty + 8 * kStagesV;     // [2] MMA commit after QK into S[b]
    const uint32_t p_full = s_full + 16;           // [2] the 8 softmax warps: P[b] written
    const uint32_t o_done = p_full + 16;           // [2] MMA commit after PV number g, on o_done[g & 1]
    const uint32_t q_full = o_done + 16;           // the query loader warp: an item's Q in shared memory
    const uint32_t q_empty = q_full + 8;           // MMA commit after an item's last QK
    const uint32_t mma_done = q_empty + 8;         // MMA commit at the very end
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
    volatile int* snap = reinterpret_cast<volatile int*>(smem + kOffMisc + 8);  // [2] abort snapshots
    float* xch = reinterpret_cast<float*>(smem + kOffXch);
    int64_t* pend_off = reinterpret_cast<int64_t*>(smem + kOffPend);        // pending epilogue: out offset (-1: no row)
    float* pend_l = reinterpret_cast<float*>(smem + kOffPend + 256 * 8);     // and partial row sum, per thread
    int32_t* prefix = reinterpret_cast<int32_t*>(smem + kSmemBytes);  // B + 1 ints past the fixed layout
    __shared__ int32_t scan_scratch[kThreads / 32];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = p.num_seqs;

    pdl_wait();
    pdl_trigger();
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(k_full + 8 * s, 1);
            mbar_init(k_empty + 8 * s, 1);
        }
        for (int s = 0; s < kStagesV; ++s) {
            mbar_init(v_full + 8 * s, 1);
            mbar_init(v_empty + 8 * s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(s_full + 8 * s, 1);
            mbar_init(p_full + 8 * s, 8);
            mbar_init(o_done + 8 * s, 1);
        }
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        snap[0] = 0;
        snap[1] = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }

    // ---- per-sequence prefix of query tiles ----
    {
        const int chunk = (B + kThreads - 1) / kThreads;
        const int b0 = tid * chunk, b1 = min(B, b0 + chunk);
        int local = 0;
        for (int b = b0; b < b1; ++b) {
            int lq, lk;
            if (seq_lens_ok(p, b, lq, lk)) local += (lq + p.tq - 1) / p.tq;
            else report(p.status, PA_ERR_INVALID_ARG);
        }
        int v = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += n;
        }
        if (lane == 31) scan_scratch[warp] = v;
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            int run = 0;
            for (int w = 0; w < kThreads / 32; ++w) {
                const int x = scan_scratch[w];
                scan_scratch[w] = run;
                run += x;
            }
            prefix[B] = run;
        }
        __syncthreads();
        int run = scan_scratch[warp] + v - local;
        for (int b = b0; b < b1; ++b) {
            prefix[b] = run;
            int lq, lk;
            if (seq_lens_ok(p, b, lq, lk)) run += (lq + p.tq - 1) / p.tq;
        }
        __syncthreads();
    }
    // ---- work order of the query tiles ----
    const int32_t* order = nullptr;
    if (p.order_cap > 0 && prefix[B] <= p.order_cap) {
        int32_t* ord = prefix + B + 1;
        build_tile_order(p, prefix, prefix[B], ord, ord + p.order_cap);
        order = ord;
    }
    const uint32_t tmem = *tmem_slot;
    const int n_items = prefix[B] * p.num_kv_heads;
    // this CTA's first kItemCache items, worked out once: every role's item
    // loop reads them from here (item_work) instead of searching the tile
    // prefix and reading the sequence lengths at each item boundary
    Work* item_cache = reinterpret_cast<Work*>(smem + kOffItems);
    if (tid < kItemCache) {
        const int item = snake_item(tid, n_items);
        if (item >= 0) item_cache[tid] = work_item(p, prefix, order, item);
    }
    __syncthreads();
    auto item_work = [&](int rnd, int item) -> Work {
        return rnd < kItemCache ? item_cache[rnd] : work_item(p, prefix, order, item);
    };
    if (warp == 0 || warp == 2) {
        // ------------------------------- loaders -------------------------------
        // K (warp 0) and V (warp 2) have rings and loader warps of their own: a
        // K stage is free again once its QK is done, long before the PV of the
        // same tile has used V, and each warp issues only half of a tile's
        // copies (a tile of block-size-16 pages is 16 copies of K and 16 of V,
        // issued lane by lane).
        const int kv = warp == 0 ? 0 : 1;
        const uint32_t full0 = kv == 0 ? k_full : v_full;
        const uint32_t empty0 = kv == 0 ? k_empty : v_empty;
        const uint32_t ring = smem_addr(kv == 0 ? sK : sV);
        const CUtensorMap* map = kv == 0 ? &map_k : &map_v;
        const uint32_t nst = kv == 0 ? kStages : kStagesV;  // ring depth
        uint32_t fill = 0, stage = 0, phase = 0;
        bool ok = true;
        if constexpr (PACKED) {
            // a tile is 128 consecutive rows of one KV head: one 3-D box per
            // 64-column half (rows past the tensor read as zero; rows past the
            // sequence are masked / zeroed by the softmax warps)
            for (int rnd = 0, item; ok && (item = snake_item(rnd, n_items)) >= 0; ++rnd) {
                const Work w = item_work(rnd, item);
                const int row0 = __ldg(p.cu_k + w.b);
                for (int t = 0; t < w.ntiles && ok; ++t) {
                    const uint32_t full = full0 + 8 * stage;
                    if (lane == 0) ok = mbar_wait(empty0 + 8 * stage, phase ^ 1u, p.status, abort_flag);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    if (lane == 0) {
                        mbar_expect_tx(full, kTileBytes);
                        const uint32_t dst = ring + stage * kTileBytes;
                        tma_load_3d(dst, map, 0, w.kvh, row0 + t * kBN, full);
                        tma_load_3d(dst + kBlkBytes, map, 64, w.kvh, row0 + t * kBN, full);
                    }
                    __syncwarp();
                    ++fill;
                    if (++stage == nst) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        } else {
            const int ppt = kBN / p.block_size;  // pages per tile (2, 4 or 8)
            for (int rnd = 0, item; ok && (item = snake_item(rnd, n_items)) >= 0; ++rnd) {
                const Work w = item_work(rnd, item);
                const int32_t* bt_row = p.block_table + static_cast<int64_t>(w.b) * p.max_blocks;
                // page ids come in batches of 32 (one per lane, -1: past Lk, -2:
                // bad id), so the table's latency is paid once per batch
                const int pages = (w.ntiles * kBN + p.block_size - 1) / p.block_size;
                int32_t id = -1;
                for (int t = 0; t < w.ntiles && ok; ++t) {
                    const int pg0 = t * ppt;  // first page of this tile
                    if ((pg0 & 31) == 0) {
                        const int pg = pg0 + lane;
                        id = -1;
                        if (pg < pages && pg * p.block_size < w.lk) {
                            id = __ldg(bt_row + pg);
                            if (id < 0 || id >= p.num_blocks) {
                                // both loader warps read the id; one reports it
                                if (kv == 0) report(p.status, PA_ERR_BAD_BLOCK);
                                id = -2;
                            }
                        }
                    }
                    // lane k < ppt holds the id of page k of this tile
                    const int my_id = __shfl_sync(0xffffffffu, id, (pg0 + (lane & 7)) & 31);
                    const bool have = lane < ppt && my_id >= 0;
                    const uint32_t bytes =
                        static_cast<uint32_t>(__popc(__ballot_sync(0xffffffffu, have))) * 2u * p.block_size * kD;
                    const int row = (my_id * p.num_kv_heads + w.kvh) * p.block_size;
                    const uint32_t off = lane * p.block_size * 128;  // page lane's rows in a 64-column block
                    const uint32_t full = full0 + 8 * stage;
                    if (lane == 0) ok = mbar_wait(empty0 + 8 * stage, phase ^ 1u, p.status, abort_flag);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    if (lane == 0) {
                        if (bytes) mbar_expect_tx(full, bytes);
                        else mbar_arrive(full);
                    }
                    __syncwarp();
                    if (have) {
                        const uint32_t dst = ring + stage * kTileBytes + off;
                        tma_load_2d(dst, map, 0, row, full);
                        tma_load_2d(dst + kBlkBytes, map, 64, row, full);
                    }
                    ++fill;
                    if (++stage == nst) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        // after an abort, wait (bounded) for this ring's copies still landing
        if (lane == 0 && *abort_flag) {
            const uint64_t t0 = global_timer_ns();
            const uint32_t first = fill > nst ? fill - nst : 0u;
            for (uint32_t f = first; f < fill; ++f)
                while (!mbar_try_wait(full0 + 8 * (f % nst), (f / nst) & 1u))
                    if (global_timer_ns() - t0 > kWaitLimitNs) break;
        }
    } else if (warp == 3) {
        // ----------------------------- query loader -----------------------------
        // an item's 128 query rows (row = token * G + head) as a K-major,
        // 128B-swizzled operand, the layout of a K tile, once the previous
        // item's last QK has released the buffer: two TMA boxes when the
        // item's tokens end inside the batch and inside the map's extent
        // (rows past the sequence then hold the next sequence's queries:
        // every key is masked for them and they are never written out), else
        // 16-byte copies zero-filled past the sequence, handed to the async
        // proxy (also when a sequence before it broke max_seqlen_q and pushed
        // its rows past num_seqs * max_seqlen_q)
        const int64_t total_q = __ldg(p.cu_q + p.num_seqs);
        uint32_t qn = 0;
        bool ok = true;
        for (int rnd = 0, item; ok && (item = snake_item(rnd, n_items)) >= 0; ++rnd) {
            const Work w = item_work(rnd, item);
            if (w.ntiles == 0) continue;
            if (lane == 0) ok = mbar_wait(q_empty, (qn & 1u) ^ 1u, p.status, abort_flag);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            const int64_t tok0 = static_cast<int64_t>(w.q0) + w.i0;
            const uint32_t dst0 = smem_addr(sQ);
            if (tok0 + p.tq <= total_q && tok0 + p.tq <= p.q_rows) {
                if (lane == 0) {
                    mbar_expect_tx(q_full, kTileBytes);
                    tma_load_3d(dst0, &map_q, 0, w.kvh * p.group, static_cast<int>(tok0), q_full);
                    tma_load_3d(dst0 + kBlkBytes, &map_q, 64, w.kvh * p.group, static_cast<int>(tok0), q_full);
                }
                __syncwarp();
                ++qn;
                continue;
            }
            // (the buffer's previous contents may have come through the async proxy)
            fence_async_smem();
            for (int i = lane; i < kRows * 16; i += 32) {
                const int r = i >> 4, c = i & 15;  // row, 16-byte chunk of the row
                const int t_row = r / p.group, g_row = r - t_row * p.group;
                const bool valid = w.i0 + t_row < w.lq;
                const uint16_t* src =
                    valid ? p.q + ((tok0 + t_row) * p.num_heads + w.kvh * p.group + g_row) * kD + c * 8 : p.q;
                cp_async16(dst0 + (c >> 3) * kBlkBytes + sw128(r, c & 7), src, valid ? 16u : 0u);
            }
            cp_async_wait_all();
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_full);
            ++qn;
        }
        // after an abort, wait (bounded) for a query copy still landing (one
        // at most: each load waits for the buffer's release)
        if (lane == 0 && *abort_flag && qn > 0) {
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(q_full, (qn - 1u) & 1u))
                if (global_timer_ns() - t0 > kWaitLimitNs) break;
        }
    } else if (warp == 1) {
        // -------------------------------- MMA ---------------------------------
        // per item: S[0] = Q K(0)^T, S[1] = Q K(1)^T, then for each tile t:
        // O[c] (+)= P[t&1] V(t) once both softmax warpgroups have written P over S, followed
        // by S[t&1] = Q K(t+2)^T.  One thread issues everything, so the tensor
        // pipe sees each PV before the QK that overwrites its P, and a commit
        // after QK(t+2) also covers PV(t).  The commit after an item's last QK
        // releases the query buffer to the query loader.
        const uint32_t id_qk = mma_idesc(DT == PA_BF16 ? 1 : 0, kRows, kBN, 0);
        const uint32_t id_pv = mma_idesc(DT == PA_BF16 ? 1 : 0, kRows, kD, 1);
        // descriptors are built once; a k-step only adds a constant to the
        // start-address field (bits 0..13, in 16-byte units)
        const uint64_t dk = smem_desc(smem_addr(sK), 16, 1024);
        const uint64_t dv = smem_desc(smem_addr(sV), kBlkBytes, 1024);
        const uint64_t dq = smem_desc(smem_addr(sQ), 16, 1024);
        uint32_t k_stage = 0, k_phase = 0;  // K ring position of the next QK
        uint32_t v_stage = 0, v_phase = 0;  // V ring position of the next PV
        uint32_t p_use[2] = {0, 0};         // P[b] handed over so far
        uint32_t pv_count = 0;              // PVs issued so far (all items)
        uint32_t q_cnt = 0;                 // items with tiles
        bool ok = true;
        auto issue_qk = [&](int t, bool last) -> bool {
            if (!mbar_wait(k_full + 8 * k_stage, k_phase, p.status, abort_flag)) return false;
            tc_fence_after();
            if (lane == 0) {
                const uint64_t dks = dk + k_stage * (kTileBytes >> 4);
#pragma unroll
                for (int k = 0; k < kD / 16; ++k) {
                    // Q and K: 32 bytes per k-step in a 64-column block
                    const uint32_t step = (k / 4) * (kBlkBytes >> 4) + (k % 4) * 2;
                    mma_f16_ss(tmem + kColS + (t & 1) * kBN, dq + step, dks + step, id_qk, k > 0 ? 1u : 0u);
                }
                mma_commit(s_full + 8 * (t & 1));
                mma_commit(k_empty + 8 * k_stage);
                if (last) mma_commit(q_empty);
            }
            __syncwarp();
            if (++k_stage == kStages) {
                k_stage = 0;
                k_phase ^= 1u;
            }
            return true;
        };
        // the next item's bookkeeping is done after an item's first QKs, while
        // the softmax warps work on its first tile, not between two items
        int item = snake_item(0, n_items);
        Work w_next{};
        if (item >= 0) w_next = item_work(0, item);
        for (int rnd = 0; ok && item >= 0; ++rnd) {
            const Work w = w_next;
            const int item2 = snake_item(rnd + 1, n_items);
            if (w.ntiles == 0) {
                item = item2;
                if (item >= 0) w_next = item_work(rnd + 1, item);
                continue;
            }
            ok = mbar_wait(q_full, q_cnt & 1u, p.status, abort_flag);
            const uint32_t col_o = tmem + kColO + (q_cnt & 1u) * kD;  // this item's O
            ++q_cnt;
            if (ok) ok = issue_qk(0, w.ntiles == 1);
            if (ok && w.ntiles > 1) ok = issue_qk(1, w.ntiles == 2);
            item = item2;
            if (item >= 0) w_next = item_work(rnd + 1, item);
            for (int t = 0; t < w.ntiles && ok; ++t) {
                const int y = t & 1;
                ok = mbar_wait(p_full + 8 * y, p_use[y] & 1u, p.status, abort_flag) &&
                     mbar_wait(v_full + 8 * v_stage, v_phase, p.status, abort_flag);
                if (!ok) break;
                ++p_use[y];
                tc_fence_after();
                if (lane == 0) {
                    const uint64_t dvs = dv + v_stage * (kTileBytes >> 4);
                    constexpr int kParts = DT == PA_BF16 ? 2 : 1;  // bf16: hi and lo weights
#pragma unroll
                    for (int part = 0; part < kParts; ++part) {
#pragma unroll
                        for (int j = 0; j < kBN / 16; ++j) {
                            // keys 16j..16j+15: P at 8 columns of half j/4 (hi at +0, lo at +32);
                            // V: 2048 bytes per 16 keys
                            mma_f16_ts(col_o, tmem + kColS + y * kBN + (j / 4) * 64 + part * 32 + (j % 4) * 8,
                                       dvs + j * (2048 >> 4), id_pv, (t > 0 || part > 0 || j > 0) ? 1u : 0u);
                        }
                    }
                    mma_commit(v_empty + 8 * v_stage);
                    mma_commit(o_done + 8 * (pv_count & 1u));
                }
                __syncwarp();
                ++pv_count;
                if (++v_stage == kStagesV) {
                    v_stage = 0;
                    v_phase ^= 1u;
                }
                if (t + 2 < w.ntiles) ok = issue_qk(t + 2, t + 3 == w.ntiles);
            }
        }
        // every MMA this warp issued is complete before tensor memory is freed
        if (lane == 0) mma_commit(mma_done);
        __syncwarp();
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(mma_done, 0u))
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                report(p.status, PA_ERR_TIMEOUT);
                break;
            }
    } else if (warp >= kSoftWarp0) {
        // ------------------------------ softmax -------------------------------
        // Both warpgroups work on every key tile: warpgroup x takes keys
        // 64x .. 64x+63 of S[t&1] and the value columns 64x .. 64x+63 of O, row
        // r = its tensor-memory lane.  Both use one reference max m per row.
        // Fast path: weights against the current m, and a barrier that ORs
        // "this row's partial sum left the safe range" over all 256 threads;
        // only then (and on an item's first tile, where m is -inf) do both
        // warpgroups take the tile's true row max, swap it through shared
        // memory, move m, rescale O and recompute.  Between such events the
        // weights may grow up to 2^58 against m, well inside fp32 and bf16
        // range, so no precision is lost.  Every thread of both warpgroups
        // passes the same barriers whatever its waits returned, and stops only
        // on an abort snapshot taken right after the previous barrier.
        // An item's epilogue (O / l out of its O buffer) is deferred to the top
        // of the next item's second key tile (or the end of its first, if it
        // has one): the tensor cores meanwhile run that item's first PV into
        // the other O buffer.
        const int x = (warp - kSoftWarp0) >> 2;   // warpgroup
        const int u = tid - kSoftWarp0 * 32;       // 0..255 over both warpgroups
        const int r = u & 127;                     // row of the tile = tensor-memory lane
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t sbuf = tmem + kColS + 64 * x + lane_base;   // + b * kBN
        const uint32_t tmem_o0 = tmem + kColO + 64 * x + lane_base;  // + c * kD: O[c]
        uint32_t s_use[2] = {0, 0};
        uint32_t n_tiled = 0;  // items with key tiles so far (O[n_tiled & 1] is the current item's)
        uint32_t nbar = 0;     // barriers passed (same count in all 256 threads)
        uint32_t tiles = 0;    // key tiles (= PVs) before the current item
        constexpr float kSafe = 18446744073709551616.f;  // 2^64: partial sums below it need no new max
        // after every barrier among the 256: the abort snapshot of the previous one
        auto snapshot = [&]() -> bool {
            const int stop = snap[(nbar + 1) & 1];
            if (u == 0) snap[nbar & 1] = *abort_flag;
            ++nbar;
            return stop != 0;
        };
        bool stop = false;
        // this row's query row and head in q / out for item w
        auto row_of = [&](const Work& w, bool& valid) -> int64_t {
            const int t_row = r / p.group, g_row = r - t_row * p.group;
            const int qi = w.i0 + t_row;  // query index of this row in its sequence
            valid = qi < w.lq;
            const int qrow = w.q0 + qi;
            const int head = w.kvh * p.group + g_row;
            return (static_cast<int64_t>(qrow) * p.num_heads + head) * kD;
        };
        // the pending epilogue: the previous item with key tiles, not yet
        // written out; its per-thread row offset and partial sum wait in
        // shared memory (pend_off[u], pend_l[u])
        bool pend = false, pend_ok = false;
        // all 256 threads: the pending item's O / l out of O buffer o_col (this
        // thread's columns), its last PV number g; false once an abort
        // snapshot says stop.  These threads saw an S committed after the
        // item's last PV (the next item's first QK) or, when no item follows,
        // after the PV before it (the item's last QK); and the PV two after it
        // needs weights not written yet: the wait neither aliases nor passes early.
        auto finish = [&](uint32_t o_col, uint32_t g) -> bool {
            pend = false;
            bool okf = pend_ok && mbar_wait(o_done + 8 * (g & 1u), (g >> 1) & 1u, p.status, abort_flag);
            okf = __all_sync(0xffffffffu, okf);
            const float my_l = pend_l[u];
            const int64_t my_off = pend_off[u];
            xch[((nbar & 1) * 2 + x) * kRows + r] = my_l;
            named_bar_sync(3, 256);
            if (snapshot()) return false;
            if (okf) {
                tc_fence_after();
                const float L = my_l + xch[((((nbar - 1) & 1) * 2) + (x ^ 1)) * kRows + r];
                const float inv = L > 0.f ? 1.f / L : 0.f;
                uint16_t* dst_e = static_cast<uint16_t*>(p.out) + my_off + 64 * x;
                // 32-byte stores (whole sectors) when out allows them: a row's
                // 16 columns start at a multiple of 32 bytes from out
                const bool wide = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0;
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 32) {
                    float o[32];
                    tmem_ld32(o_col + c0, o);
                    if (my_off >= 0) {
                        uint32_t wv[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) wv[j] = pack2<DT>(o[2 * j] * inv, o[2 * j + 1] * inv);
                        if (wide) {
#pragma unroll
                            for (int j = 0; j < 2; ++j) st_global_v8(dst_e + c0 + 16 * j, wv + 8 * j);
                        } else {
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                *reinterpret_cast<uint4*>(dst_e + c0 + 8 * j) =
                                    make_uint4(wv[4 * j], wv[4 * j + 1], wv[4 * j + 2], wv[4 * j + 3]);
                        }
                    }
                }
                // a later item's first PV overwrites this O buffer: its p_full
                // arrival orders that after these reads
                tc_fence_before();
            }
            return true;
        };
        for (int rnd = 0, item; !stop && (item = snake_item(rnd, n_items)) >= 0; ++rnd) {
            const Work w = item_work(rnd, item);
            const int shift = w.lk - w.lq;
            const int t_row = r / p.group;
            const int qi = w.i0 + t_row;  // query index of this row in its sequence
            bool row_valid;
            const int64_t row_off = row_of(w, row_valid);
            const int lim = p.causal ? min(w.lk, shift + qi + 1) : w.lk;  // keys [0, lim) visible
            uint16_t* dst = static_cast<uint16_t*>(p.out) + row_off + 64 * x;
            if (w.ntiles == 0) {
                // no visible key for any row of the item: output 0
                if (row_valid) {
                    for (int c = 0; c < 64; c += 8)
                        *reinterpret_cast<uint4*>(dst + c) = make_uint4(0u, 0u, 0u, 0u);
                }
                continue;
            }
            const uint32_t tmem_o = tmem_o0 + (n_tiled & 1u) * kD;  // this item's O
            ++n_tiled;
            float m = -INFINITY, l = 0.f;  // reference max (same in both warpgroups), own partial sum
            bool ok = true;
            const uint64_t sc2 = f2pack(p.scale_log2, p.scale_log2);
            for (int t = 0; t < w.ntiles; ++t) {
                // the previous item's O is the other buffer; its last PV is
                // the one before this item's first
                if (t == 1 && pend && !finish(tmem_o0 + (n_tiled & 1u) * kD, tiles - 1)) {
                    stop = true;
                    break;
                }
                const int b = t & 1;
                const int key0 = t * kBN + 64 * x;  // first key of this thread's 64 columns
                const int vis = row_valid ? lim - key0 : 0;  // visible keys of these columns: [0, vis)
                ok = ok && mbar_wait(s_full + 8 * b, s_use[b] & 1u, p.status, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                ++s_use[b];
                float e[64];
                float sum = 0.f;
                bool over = false;
                if (ok) {
                    tc_fence_after();
                    tmem_ld64(sbuf + b * kBN, e);
                    if (vis < 64) {
#pragma unroll
                        for (int i = 0; i < 64; ++i)
                            if (i >= vis) e[i] = -INFINITY;
                    }
                    if (m == -INFINITY) {
                        // no reference yet: the slow path, unless these columns
                        // are all masked for this row (weights 0)
                        over = vis > 0;
#pragma unroll
                        for (int i = 0; i < 64; ++i) e[i] = 0.f;
                    } else {
                        // p = 2^(s*scale - m): one packed FFMA per pair and one exp2
                        // per score (masked scores are -inf and give 0)
                        const uint64_t nb2 = f2pack(-m, -m);
#pragma unroll
                        for (int i = 0; i < 64; i += 2) {
                            const float2 a = f2unpack(f2fma(f2pack(e[i], e[i + 1]), sc2, nb2));
                            e[i] = ex2(a.x);
                            e[i + 1] = ex2(a.y);
                        }
                        uint64_t s8[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            s8[j] = f2add(f2add(f2pack(e[2 * j], e[2 * j + 1]), f2pack(e[2 * j + 8], e[2 * j + 9])),
                                          f2add(f2pack(e[2 * j + 16], e[2 * j + 17]), f2pack(e[2 * j + 24], e[2 * j + 25])));
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            s8[j] = f2add(s8[j], f2add(f2add(f2pack(e[2 * j + 32], e[2 * j + 33]), f2pack(e[2 * j + 40], e[2 * j + 41])),
                                                       f2add(f2pack(e[2 * j + 48], e[2 * j + 49]), f2pack(e[2 * j + 56], e[2 * j + 57]))));
                        const float2 s01 = f2unpack(f2add(f2add(s8[0], s8[1]), f2add(s8[2], s8[3])));
                        sum = s01.x + s01.y;
                        over = !(sum < kSafe);  // also catches inf and NaN
                    }
                }
                const bool any = bar_red_or(2, 256, over);
                if (snapshot()) {
                    stop = true;
                    break;
                }
                if (any) {
                    // slow path (all 256 threads): the tile's true row max over both
                    // halves, a new reference, O and l rescaled, weights recomputed
                    float mx = -INFINITY;
                    if (ok) {
                        tmem_ld64(sbuf + b * kBN, e);
                        if (vis < 64) {
#pragma unroll
                            for (int i = 0; i < 64; ++i)
                                if (i >= vis) e[i] = -INFINITY;
                        }
                        float m8[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) m8[j] = fmax3(e[8 * j], e[8 * j + 1], e[8 * j + 2]);
#pragma unroll
                        for (int j = 0; j < 8; ++j) m8[j] = fmax3(m8[j], e[8 * j + 3], e[8 * j + 4]);
#pragma unroll
                        for (int j = 0; j < 8; ++j) m8[j] = fmax3(m8[j], e[8 * j + 5], e[8 * j + 6]);
#pragma unroll
                        for (int j = 0; j < 8; ++j) m8[j] = fmaxf(m8[j], e[8 * j + 7]);
                        mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
                    }
                    xch[((nbar & 1) * 2 + x) * kRows + r] = mx;
                    named_bar_sync(3, 256);
                    if (snapshot()) {
                        stop = true;
                        break;
                    }
                    if (!ok) continue;
                    // scale > 0: the max commutes with it
                    mx = fmaxf(mx, xch[((((nbar - 1) & 1) * 2) + (x ^ 1)) * kRows + r]) * p.scale_log2;
                    const bool grow = mx > m;
                    const float a = grow ? ex2(m - mx) : 1.f;  // 0 when m = -inf
                    // O holds PV(0..t-1) against m: rescale it (warp-wide accesses,
                    // factor 1 for other rows) once PV(t-1) is complete.  PV number g
                    // completes a phase of o_done[g & 1]; the previous phase of that
                    // barrier belongs to PV(t-3), complete since it precedes QK(t).
                    if (__any_sync(0xffffffffu, grow) && t > 0) {
                        const uint32_t g = tiles + t - 1;
                        ok = mbar_wait(o_done + 8 * (g & 1u), (g >> 1) & 1u, p.status, abort_flag);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) continue;
                        tc_fence_after();
#pragma unroll
                        for (int c0 = 0; c0 < 64; c0 += 32) {
                            float o[32];
                            tmem_ld32(tmem_o + c0, o);
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] *= a;
                            tmem_st32(tmem_o + c0, o);
                        }
                    }
                    if (grow) {
                        l *= a;
                        m = mx;
                    }
                    const float nb = m == -INFINITY ? 0.f : -m;
                    const uint64_t nb2 = f2pack(nb, nb);
#pragma unroll
                    for (int i = 0; i < 64; i += 2) {
                        const float2 q2 = f2unpack(f2fma(f2pack(e[i], e[i + 1]), sc2, nb2));
                        e[i] = ex2(q2.x);
                        e[i + 1] = ex2(q2.y);
                    }
                    float r8[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) r8[j] = (e[j] + e[j + 8]) + (e[j + 16] + e[j + 24]);
#pragma unroll
                    for (int j = 0; j < 8; ++j) r8[j] += (e[j + 32] + e[j + 40]) + (e[j + 48] + e[j + 56]);
                    sum = ((r8[0] + r8[1]) + (r8[2] + r8[3])) + ((r8[4] + r8[5]) + (r8[6] + r8[7]));
                }
                if (!ok) continue;
                l += sum;
                // values past Lk in the last tile may hold anything: zero those
                // V rows (after the tile landed) so zero weights never meet NaN
                if (t * kBN + kBN > w.lk) {
                    const uint32_t f = tiles + t;
                    ok = mbar_wait(v_full + 8 * (f % kStagesV), (f / kStagesV) & 1u, p.status, abort_flag);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) continue;
                    uint8_t* vt = sV + (f % kStagesV) * kTileBytes;
                    const int first = max(0, w.lk - t * kBN);
                    for (int ci = u; ci < (kBN - first) * 16; ci += 256) {
                        const int rr = first + (ci >> 4), c = ci & 15;
                        *reinterpret_cast<uint4*>(vt + (c >> 3) * kBlkBytes + sw128(rr, c & 7)) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_async_smem();
                }
                // P over S in tensor memory as 16-bit pairs (bf16: hi at columns
                // 0..31 of this warpgroup's 64 and the remainder lo at 32..63, both
                // truncated, ~16 bits together)
#pragma unroll
                for (int h = 0; h < 2; ++h) {  // keys 32h .. 32h+31 = columns 16h .. 16h+15
                    uint32_t hw[16], lw[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float a = e[32 * h + 2 * j], c = e[32 * h + 2 * j + 1];
                        if constexpr (DT == PA_BF16) {
                            hw[j] = hi_halves(a, c);
                            const float2 lo = f2unpack(f2add(f2pack(a, c), f2pack(-__uint_as_float(hw[j] << 16),
                                                                                -__uint_as_float(hw[j] & 0xffff0000u))));
                            lw[j] = hi_halves(lo.x, lo.y);
                        } else {
                            hw[j] = pack2<DT>(a, c);
                        }
                    }
                    tmem_st16(sbuf + b * kBN + 16 * h, hw);
                    if constexpr (DT == PA_BF16) tmem_st16(sbuf + b * kBN + 32 + 16 * h, lw);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full + 8 * b);
            }
            if (stop) break;
            // an item with one key tile reaches no second tile: the previous
            // item's epilogue comes here, after its only weights are out
            if (pend && !finish(tmem_o0 + (n_tiled & 1u) * kD, tiles - 1)) break;
            tiles += w.ntiles;
            pend = true;
            pend_ok = ok;
            pend_l[u] = l;
            pend_off[u] = row_valid ? row_off : -1;
        }
        // the last item: its O buffer is the current one, its last PV the last of all
        if (pend && !stop) finish(tmem_o0 + ((n_tiled - 1u) & 1u) * kD, tiles - 1);
    }
    // ---- teardown: every role is done; free tensor memory ----
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

// ---------------------------------------------------------------------------
// host: tensor maps (driver entry point, no link-time dependency on libcuda)
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// the cache as a 2-D tensor of rows (num_blocks * kv_heads * block_size) x head_size
bool make_cache_map(CUtensorMap* map, const void* base, int64_t rows, int dtype, int block_size) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(block_size)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                          2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// packed K or V as a 3-D tensor {head_size, num_kv_heads, total rows}; a box
// is 64 elements x 1 head x 128 rows
bool make_packed_map(CUtensorMap* map, const void* base, int64_t total_k, int num_kv_heads, int dtype) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(num_kv_heads),
                                static_cast<cuuint64_t>(total_k)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 2,
                                   static_cast<cuuint64_t>(num_kv_heads) * kD * 2};
    const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kBN)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                          3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// q as a 3-D tensor {head_size, num_heads, tokens}; a box is 64 elements x G
// heads x 128/G tokens: one item's rows in the layout of a K tile.  The token
// extent is num_seqs * max_seqlen_q, a bound on the real count (which only
// the device knows): boxes are loaded only for items whose tokens end before
// the real count and inside this extent, so no copy reaches past the real rows.
int32_t q_map_rows(int num_seqs, int max_q) {
    const int64_t bound = static_cast<int64_t>(num_seqs) * max_q;
    return static_cast<int32_t>(bound < INT32_MAX ? bound : INT32_MAX);
}
bool make_q_map(CUtensorMap* map, const void* q, int num_heads, int group, int num_seqs, int max_q, int dtype) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(num_heads),
                                static_cast<cuuint64_t>(q_map_rows(num_seqs, max_q))};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 2, static_cast<cuuint64_t>(num_heads) * kD * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(kRows / group)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                          3, const_cast<void*>(q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// launch shared by the paged and packed entry points (p filled in, maps built)
template <bool PACKED>
pa_status launch_prefill(const PrefillParams& p, pa_dtype dtype, const CUtensorMap& map_k,
                         const CUtensorMap& map_v, const CUtensorMap& map_q, pa_stream_t stream) {
    // shared memory past the fixed layout: the tile prefix (B+1 ints), the
    // work order (up to every query tile the bounds allow, within what the
    // device offers) and the sort's [12 warps][64 classes] counts
    const int base = kSmemBytes + (p.num_seqs + 1) * 4 + 1024;
    if (base > device_max_smem_optin()) return PA_ERR_UNSUPPORTED;
    const int64_t tiles_bound = static_cast<int64_t>(p.num_seqs) * ((p.max_q + p.tq - 1) / p.tq);
    // (2 KB kept back for the kernel's static shared memory)
    const int64_t room = (device_max_smem_optin() - 2048 - base) / 4 - (kThreads / 32) * 64;
    PrefillParams q = p;
    q.order_cap = static_cast<int32_t>(room <= 0 ? 0 : (tiles_bound < room ? tiles_bound : room));
    const int smem = base + (q.order_cap > 0 ? (q.order_cap + (kThreads / 32) * 64) * 4 : 0);
    static LaunchCache cache_bf16, cache_f16;
    auto kern = dtype == PA_BF16 ? paged_prefill_tc_kernel<PA_BF16, PACKED> : paged_prefill_tc_kernel<PA_F16, PACKED>;
    const int per_sm = blocks_per_sm(kern, kThreads, smem, dtype == PA_BF16 ? cache_bf16 : cache_f16);
    if (per_sm <= 0) return PA_ERR_CUDA;
    const int64_t max_items =
        static_cast<int64_t>(p.num_seqs) * ((p.max_q + p.tq - 1) / p.tq) * p.num_kv_heads;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * per_sm;
    const int grid = static_cast<int>(max_items < cap ? max_items : cap);
    if (grid <= 0) return PA_OK;
    return launch_pdl(kern, grid, kThreads, smem, reinterpret_cast<cudaStream_t>(stream), map_k, map_v, map_q, q) ==
                   cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" pa_status pa_prefill_varlen(void* out, const void* q, pa_dtype q_dtype,
                                       const pa_kv_cache* cache, const int32_t* block_table,
                                       int32_t max_blocks_per_seq, const int32_t* cu_seq_lens_q,
                                       const int32_t* cu_seq_lens_k, int32_t num_seqs,
                                       int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t num_heads,
                                       float scale, int32_t causal, int32_t* dev_status,
                                       pa_stream_t stream) {
    pa_status st = check_cache(cache);
    if (st != PA_OK) return st;
    if (num_seqs < 0 || num_heads <= 0 || max_blocks_per_seq <= 0 || max_seqlen_q < 0 ||
        max_seqlen_k < 0 || !(scale == scale))
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0 || max_seqlen_q == 0) return PA_OK;
    if (out == nullptr || q == nullptr || block_table == nullptr || cu_seq_lens_q == nullptr ||
        cu_seq_lens_k == nullptr)
        return PA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(out) & 15u) || (reinterpret_cast<uintptr_t>(q) & 15u))
        return PA_ERR_INVALID_ARG;
    if (num_heads % cache->num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    const int group = num_heads / cache->num_kv_heads;
    if (cache->head_size != kD) return PA_ERR_UNSUPPORTED;
    if (group != 1 && group != 2 && group != 4 && group != 8) return PA_ERR_UNSUPPORTED;
    if (q_dtype != PA_F16 && q_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (cache->kv_dtype != q_dtype) return PA_ERR_UNSUPPORTED;
    const int bs = cache->block_size;
    if (bs != 16 && bs != 32 && bs != 64) return PA_ERR_UNSUPPORTED;
    if (num_seqs > kMaxSeqs) return PA_ERR_UNSUPPORTED;
    const int64_t rows = cache->num_blocks * cache->num_kv_heads * bs;
    if (rows > INT32_MAX) return PA_ERR_UNSUPPORTED;

    PrefillParams p{};
    p.out = out;
    p.q = static_cast<const uint16_t*>(q);
    p.block_table = block_table;
    p.cu_q = cu_seq_lens_q;
    p.cu_k = cu_seq_lens_k;
    p.status = dev_status;
    p.num_blocks = cache->num_blocks;
    p.block_size = bs;
    p.num_kv_heads = cache->num_kv_heads;
    p.num_heads = num_heads;
    p.group = group;
    p.tq = kRows / group;
    p.num_seqs = num_seqs;
    p.max_blocks = max_blocks_per_seq;
    p.max_q = max_seqlen_q;
    p.max_k = max_seqlen_k;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.total_k = -1;

    CUtensorMap map_k, map_v;
    if (!make_cache_map(&map_k, cache->k_cache, rows, q_dtype, bs) ||
        !make_cache_map(&map_v, cache->v_cache, rows, q_dtype, bs))
        return PA_ERR_CUDA;
    CUtensorMap map_q;
    if (!make_q_map(&map_q, q, num_heads, group, num_seqs, max_seqlen_q, q_dtype)) return PA_ERR_CUDA;
    p.q_rows = q_map_rows(num_seqs, max_seqlen_q);
    return launch_prefill<false>(p, q_dtype, map_k, map_v, map_q, stream);
}

extern "C" pa_status pa_prefill_varlen_packed(void* out, const void* q, const void* k, const void* v,
                                              pa_dtype dtype, const int32_t* cu_seq_lens_q,
                                              const int32_t* cu_seq_lens_k, int32_t num_seqs,
                                              int32_t max_seqlen_q, int32_t max_seqlen_k, int64_t total_k,
                                              int32_t num_heads, int32_t num_kv_heads, int32_t head_size,
                                              float scale, int32_t causal, int32_t* dev_status,
                                              pa_stream_t stream) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || max_seqlen_q < 0 || max_seqlen_k < 0 ||
        total_k < 0 || !(scale == scale))
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0 || max_seqlen_q == 0) return PA_OK;
    if (out == nullptr || q == nullptr || cu_seq_lens_q == nullptr || cu_seq_lens_k == nullptr)
        return PA_ERR_INVALID_ARG;
    if (total_k > 0 && (k == nullptr || v == nullptr)) return PA_ERR_INVALID_ARG;
    for (const void* ptr : {static_cast<const void*>(out), q, k, v})
        if (reinterpret_cast<uintptr_t>(ptr) & 15u) return PA_ERR_INVALID_ARG;
    if (num_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    const int group = num_heads / num_kv_heads;
    if (head_size != kD) return PA_ERR_UNSUPPORTED;
    if (group != 1 && group != 2 && group != 4 && group != 8) return PA_ERR_UNSUPPORTED;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (num_seqs > kMaxSeqs) return PA_ERR_UNSUPPORTED;
    if (total_k > INT32_MAX - kBN) return PA_ERR_UNSUPPORTED;

    PrefillParams p{};
    p.out = out;
    p.q = static_cast<const uint16_t*>(q);
    p.cu_q = cu_seq_lens_q;
    p.cu_k = cu_seq_lens_k;
    p.status = dev_status;
    p.block_size = kBN;
    p.num_kv_heads = num_kv_heads;
    p.num_heads = num_heads;
    p.group = group;
    p.tq = kRows / group;
    p.num_seqs = num_seqs;
    p.max_q = max_seqlen_q;
    p.max_k = max_seqlen_k;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.total_k = total_k;

    // an empty K/V still needs a valid map: point it at q (never read, every
    // sequence then has no key)
    const int64_t rows = total_k > 0 ? total_k : 1;
    CUtensorMap map_k, map_v;
    if (!make_packed_map(&map_k, total_k > 0 ? k : q, rows, num_kv_heads, dtype) ||
        !make_packed_map(&map_v, total_k > 0 ? v : q, rows, num_kv_heads, dtype))
        return PA_ERR_CUDA;
    CUtensorMap map_q;
    if (!make_q_map(&map_q, q, num_heads, group, num_seqs, max_seqlen_q, dtype)) return PA_ERR_CUDA;
    p.q_rows = q_map_rows(num_seqs, max_seqlen_q);
    return launch_prefill<true>(p, dtype, map_k, map_v, map_q, stream);
}
