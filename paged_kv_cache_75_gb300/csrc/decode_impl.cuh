// Paged single-query decode attention: kernel templates.
//
// What it computes follows the vLLM PagedAttention design doc ("分页注意力机制",
// vllm.ooos.top/design/paged_attention): for one sequence and query head,
// scores s_t = scale * q . K_t over the context tokens reached through the
// block table (section Key), softmax by max subtraction (section Softmax:
// m(x), f(x), l(x)), masked tokens excluded (section qk_max 和 logits), then
// the value-weighted sum (section Value) written per sequence and head
// (section Output).  The doc's grid has a third axis over context partitions
// whose partial outputs are merged afterwards; here that is a log-sum-exp
// merge in a second kernel.  Inputs follow "Paged 어텐션" (Decode 경로):
// block_table [batch, max_blocks_per_seq] and per-sequence cache lengths.
//
// How (GB300 design, not the doc's):
//  * persistent CTAs walk a flattened list of work items (sequence,
//    partition, KV head); every CTA builds the list's per-sequence prefix in
//    shared memory from seq_lens, so short and long sequences share the GPU
//    without a max_num_partitions-shaped grid;
//  * one producer warp streams each (block, KV head) page -- one contiguous
//    block_size*head_size run in the [blocks][kv_heads][block_size][head]
//    layout -- into a ring of shared-memory stages (32 tokens of K and V per
//    stage) with 1-D bulk async copies (cp.async.bulk), completion counted on
//    mbarriers;
//  * four consumer warps split each stage's tokens; all G query heads of a KV
//    head are handled together, so a page is read once per KV head (GQA);
//  * with one or two query heads per KV head, each 8-lane token group keeps
//    its own online softmax in fp32 (exp2 domain, lazy rescale), QK with
//    warp-shuffle reductions; with four or eight, 16-token slices go through
//    tensor-core MMAs (mma.sync, fp32 accumulate) with one softmax state per
//    head; groups and warps are merged once per work item;
//  * the shared-prefix (cascade) decode is this kernel in "group mode": a
//    group's members side by side as one sequence's query rows over their
//    shared blocks, beside every member's own tokens, in one work list;
//  * every mbarrier wait is bounded (PA_ERR_TIMEOUT, no hang).
#pragma once

#include <type_traits>

#include "common.cuh"

namespace pa {

struct DecodeParams {
    void* out;
    const void* q;
    const uint8_t* k_cache;
    const uint8_t* v_cache;
    const int32_t* block_table;
    const int32_t* seq_lens;
    const int32_t* cu_seq_lens_k;  // when set: L_b = cu[b+1] - cu[b] (seq_lens unused)
    float* ws_lse;  // [B*H*max_parts]
    float* ws_o;    // [B*H*max_parts*D]
    int32_t* status;
    int64_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t num_heads;
    int32_t num_seqs;
    int32_t max_blocks;
    int32_t max_seq_len;
    int32_t partition;  // tokens per partition, multiple of block_size
    int32_t max_parts;  // ceil(max_seq_len / partition)
    int32_t stages;     // ring depth
    float qk_scale;     // scale * k_scale * log2(e)
    float v_scale;
    // append mode: the new token of every sequence (position L-1), written to
    // the cache and attended in the same launch; [B][Hkv][D] of the query type
    const void* k_new;
    const void* v_new;
    float k_scale_w, v_scale_w;  // E4M3 cache: the write's scales
    // cascade suffix pass: sequences cu_groups[g] .. cu_groups[g+1]-1 form group
    // g, whose first s0 = shared_lens[g] tokens (whole blocks, the same physical
    // blocks in every member) a prefix pass has attended in parts of
    // `partition` tokens (workspace parts 0 .. ceil(s0/partition)-1); this
    // launch attends tokens [s0, L) and writes its partials after those
    const int32_t* cu_groups;
    const int32_t* shared_lens;
    int32_t num_groups;
    // cascade decode in one launch ("group mode", vm > 0).  Sequence b <
    // vcount of the launch is the members cu_groups[g] + j*vm .. + vm-1 (those
    // that exist) of group g = b / vpg, j = b % vpg, over the group's first
    // shared_lens[g] tokens read through the group's first member's table row:
    // the kernel's G = vm * g_real query rows of a KV head are those members'
    // g_real heads, member after member, and the partials go to the members'
    // workspace parts 0 .. ceil(s0/partition)-1.  Sequence vcount + m is
    // member m alone over its own tokens [s0, L) (query rows past g_real
    // empty), partials after the prefix's.  A merge launch follows.
    // num_members: the batch's real sequence count.
    int32_t vm;
    int32_t vpg;
    int32_t vcount;
    int32_t g_real;
    int32_t num_members;
    // test hook (pa_decode_test_wait_timeout; 0 on every other path): the
    // producer warp issues no copy at all, so every consumer wait runs out
    // with nothing in flight, reports PA_ERR_TIMEOUT and the block returns
    int32_t no_copies;
};

template <int QDT, int KVDT, int D, int G, int BS>
struct DecodeCfg {
    // Four or more query heads per KV head: the QK and PV products of a
    // 16-token slice are dense [16 x D] x [D x G] contractions, run on tensor
    // cores (mma.sync m16n8k16, heads on N) by warps that each hold all G heads.
    // Fewer heads keep the CUDA-core consumer.
    static constexpr bool MMA = G >= 4;
    // query heads per consumer warp (CUDA-core consumer): one or two
    static constexpr int GW = MMA ? G : (G < 2 ? G : 2);
    static constexpr int HG = G / GW;                 // head groups (warp sets)
    static constexpr int TW = 4 / HG;                 // token warps per head group
    static constexpr int NCW = TW * HG;               // consumer warps (4)
    static constexpr int THREADS = (NCW + 1) * 32;    // + one producer warp
    static constexpr int LPT = 8;                     // lanes per token
    static constexpr int TG = 32 / LPT;               // tokens per warp step
    static constexpr int EPL = D / LPT;               // row elements per lane
    static constexpr int KB = dtype_traits<KVDT>::bytes;
    static constexpr int QB = dtype_traits<QDT>::bytes;
    static constexpr int TPI = TW * TG;               // tokens per block step
    static constexpr int VB = (EPL * KB < 16) ? EPL * KB : 16;  // row chunk bytes
    static constexpr int NV = EPL * KB / VB;          // row chunks per lane
    static constexpr int EV = VB / KB;                // elements per chunk
    static constexpr int PL = EPL / 2;                // element pairs per lane
    static constexpr int ROWB = D * KB;               // bytes per token row
    static constexpr int PAGE = BS * ROWB;            // bytes of one (block, KV head) page
    // pages per ring stage: 32 tokens, except 64 for the tensor-core consumer
    // at block size 32, so that each stage holds a 16-token slice for each of
    // the four warps and they finish an item together
    static constexpr int SPAGES = BS >= 64 ? 1 : (BS == 32 ? (MMA ? 2 : 1) : 32 / BS);
    static constexpr int STOK = SPAGES * BS;          // tokens per ring stage
    static constexpr int SUB = STOK / TPI;            // block steps per stage
    static constexpr int STAGE_BYTES = 2 * SPAGES * PAGE;  // K pages, then V pages
    static constexpr int QBYTES = G * D * QB;         // one item's queries
    static constexpr int MERGE_FLOATS = NCW * GW * (D + 2);
    // register cap: three 5-warp CTAs per SM (a block's register share is
    // counted in pairs of warps)
    static constexpr int MAX_REGS = 128;
    static_assert(EPL * KB >= 4 && EPL % 4 == 0, "unsupported head size");
    static_assert(STOK % TPI == 0, "block size must be a multiple of the step");
    // steps handled together: one head per warp has enough independent work
    // per step; several heads gain from interleaving two steps' reductions
    static constexpr int NB = GW == 1 ? 1 : 2;
    static_assert(MMA || SUB % NB == 0, "steps of a stage go in groups of NB");
    // tensor-core consumer: 16-token slices per stage, one warp each
    static constexpr int SLICES = STOK / 16;
    static_assert(!MMA || (SLICES == 2 || SLICES == 4), "stages of 32 or 64 tokens");
};

// shared memory carve-up (byte offsets from the 1 KB-aligned base)
struct DecodeSmem {
    uint32_t ring, qbuf, merge, prefix, order, keys, hist, bars, flags, total;
    __host__ __device__ static DecodeSmem make(int stages, int stage_bytes, int qbytes,
                                               int merge_floats, int num_seqs) {
        DecodeSmem s;
        uint32_t o = 0;
        s.ring = o;
        o += static_cast<uint32_t>(stages) * stage_bytes;
        s.qbuf = o;
        o += 2u * ((qbytes + 127u) & ~127u);
        s.merge = o;
        o += static_cast<uint32_t>(merge_floats) * 4u;
        o = (o + 15u) & ~15u;
        s.prefix = o;
        o += (static_cast<uint32_t>(num_seqs) + 1u) * 4u;
        s.order = o;
        o += static_cast<uint32_t>(num_seqs) * 4u;
        s.hist = o;  // [8 warps][64 classes] ints
        o += 8u * 64u * 4u;
        s.keys = o;  // one class byte per sequence
        o += (static_cast<uint32_t>(num_seqs) + 15u) & ~15u;
        o = (o + 7u) & ~7u;
        s.bars = o;
        o += (2u * stages + 4u) * 8u;
        s.flags = o;
        o += (static_cast<uint32_t>(stages) + 1u) * 4u;
        s.total = (o + 127u) & ~127u;
        return s;
    }
};

// number of partitions a sequence of length L splits into (>= 1)
__device__ __forceinline__ int parts_of(int L, int P) { return L <= P ? 1 : (L + P - 1) / P; }

// cascade: workspace parts the prefix pass filled for a shared length s0
__device__ __forceinline__ int prefix_parts(const DecodeParams& p, int s0) {
    return p.cu_groups != nullptr ? (s0 + p.partition - 1) / p.partition : 0;
}

// Cascade suffix pass: the group of sequence b (largest g with cu_groups[g] <= b).
__device__ __forceinline__ int group_of(const DecodeParams& p, int b) {
    int lo = 0, hi = p.num_groups - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(p.cu_groups + mid) <= b) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Group mode: the members sequence b stands for (m0 .. m0+nm-1; nm = 0 past
// a group's end or for a malformed cu_groups) and whether it is a member's own
// tokens (b >= vcount) rather than its group's shared ones.
struct VSeq {
    int g, m0, nm;
    bool own;
};
__device__ __forceinline__ VSeq vseq(const DecodeParams& p, int b) {
    VSeq v;
    v.own = b >= p.vcount;
    if (v.own) {
        v.g = 0;  // (not needed by the callers)
        v.m0 = b - p.vcount;
        v.nm = 1;
        return v;
    }
    v.g = b / p.vpg;
    const int c0 = __ldg(p.cu_groups + v.g), c1 = min(__ldg(p.cu_groups + v.g + 1), p.num_members);
    v.m0 = c0 + (b - v.g * p.vpg) * p.vm;
    v.nm = c0 < 0 ? 0 : max(0, min(p.vm, c1 - v.m0));
    return v;
}

// First token of sequence b (length L) this launch attends: its group's shared
// length in a cascade suffix pass, else 0.  A shared length that is negative,
// past L or not a whole number of blocks is reported and taken as 0.
__device__ __forceinline__ int seq_start(const DecodeParams& p, int b, int L) {
    if (p.cu_groups == nullptr) return 0;
    if (p.vm > 0) {
        if (b < p.vcount) return 0;  // group mode: a group's shared tokens
        b -= p.vcount;               // a member's own tokens
    }
    const int s0 = __ldg(p.shared_lens + group_of(p, b));
    if (s0 < 0 || s0 > L || s0 % p.block_size != 0) {
        report(p.status, PA_ERR_INVALID_ARG);
        return 0;
    }
    return s0;
}

// A length is usable iff 0 <= L <= max_seq_len and L fits the table row.
__device__ __forceinline__ int checked_len(const DecodeParams& p, int b) {
    if (p.vm > 0 && b >= p.vcount) b -= p.vcount;  // group mode: a member's own tokens
    else if (p.vm > 0) {
        // group mode: the group's shared blocks, for a sequence with members
        const VSeq v = vseq(p, b);
        if (v.nm == 0) return 0;
        const int s0 = __ldg(p.shared_lens + v.g);
        if (s0 < 0 || s0 > p.max_seq_len || s0 % p.block_size != 0 ||
            static_cast<int64_t>(s0) > static_cast<int64_t>(p.max_blocks) * p.block_size)
            return -1;
        return s0;
    }
    // lengths from seq_lens, or as differences of cumulative key lengths
    int L = p.cu_seq_lens_k != nullptr ? __ldg(p.cu_seq_lens_k + b + 1) - __ldg(p.cu_seq_lens_k + b)
                                       : __ldg(p.seq_lens + b);
    if (L < 0 || L > p.max_seq_len || static_cast<int64_t>(L) > static_cast<int64_t>(p.max_blocks) * p.block_size)
        return -1;
    return L;
}

// Work list and its order.  A sequence of length L splits into n = parts_of(L)
// partitions; all but the last hold exactly `partition` tokens ("full"), the
// last holds L - (n-1)*partition.  The list puts every full partition first
// (in sequence order), then the last partitions, longest first (64 length
// classes, ties in sequence order); each entry stands for num_kv_heads items,
// one per KV head.  CTAs deal the items out in snake order (snake_item),
// so the long items spread over all CTAs and the short ones fill the gaps:
// with mixed lengths this keeps the busiest CTA within a few percent of the
// mean, where plain round-robin in sequence order left it 20-35 % above.
//
// prefix[b] = full partitions of sequences < b, prefix[B] = their total F;
// order[k] = the sequence whose last partition is entry F + k.
// All threads of the block take part; scratch holds one int per warp, keys
// one byte per sequence, hist 64 ints per warp.
__device__ __forceinline__ int tail_class(int L, int P) {
    const int t = L - (parts_of(L, P) - 1) * P;  // tokens of the last partition, 0..P
    return static_cast<int>((static_cast<int64_t>(P - t) * 64) / (P + 1));  // 0 = longest
}

__device__ inline void build_schedule(const DecodeParams& p, int32_t* prefix, int32_t* order, int32_t* scratch,
                                      uint8_t* keys, int32_t* hist) {
    const int B = p.num_seqs;
    const int nt = blockDim.x, t = threadIdx.x;
    const int chunk = (B + nt - 1) / nt;
    const int b0 = t * chunk, b1 = min(B, b0 + chunk);
    int local = 0;
    for (int b = b0; b < b1; ++b) {
        int L = checked_len(p, b);
        if (L < 0) report(p.status, PA_ERR_INVALID_ARG);
        L = L < 0 ? 0 : L;
        const int n = L - seq_start(p, b, L);
        local += parts_of(n, p.partition) - 1;
        keys[b] = static_cast<uint8_t>(tail_class(n, p.partition));
    }
    // inclusive scan inside the warp
    const int lane = t & 31, warp = t >> 5;
    int v = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) scratch[warp] = v;
    __syncthreads();
    if (t == 0) {
        int run = 0;
        for (int w = 0; w < (nt + 31) / 32; ++w) {
            int x = scratch[w];
            scratch[w] = run;
            run += x;
        }
        prefix[B] = run;
    }
    __syncthreads();
    int run = scratch[warp] + v - local;
    for (int b = b0; b < b1; ++b) {
        prefix[b] = run;
        int L = checked_len(p, b);
        L = L < 0 ? 0 : L;
        run += parts_of(L - seq_start(p, b, L), p.partition) - 1;
    }
    // last partitions: a stable counting sort by the class bytes, every warp
    // counting a contiguous chunk (lanes of equal class found by match.any),
    // warp 0 turning the [warp][class] counts into class-major offsets, every
    // warp then placing its chunk in order
    const int NW = nt / 32;
    const int wch = ((B + NW - 1) / NW + 31) & ~31;
    const int c0 = warp * wch, c1 = min(B, c0 + wch);
    int32_t* h = hist + warp * 64;
    h[lane] = 0;
    h[lane + 32] = 0;
    __syncwarp();
    for (int cb = c0; cb < c1; cb += 32) {
        const int b = cb + lane;
        const int key = b < c1 ? keys[b] : 64;
        const unsigned same = __match_any_sync(0xffffffffu, key);
        if (b < c1 && lane == __ffs(same) - 1) h[key] += __popc(same);
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
    for (int cb = c0; cb < c1; cb += 32) {
        const int b = cb + lane;
        const int key = b < c1 ? keys[b] : 64;
        const unsigned same = __match_any_sync(0xffffffffu, key);
        if (b < c1) order[h[key] + __popc(same & ((1u << lane) - 1u))] = b;
        __syncwarp();
        if (b < c1 && lane == __ffs(same) - 1) h[key] += __popc(same);
        __syncwarp();
    }
    __syncthreads();
}

struct Item {
    int b, part, kvh, L, s0, t1, j0, j1, nparts;
};

__device__ __forceinline__ Item decode_item(const DecodeParams& p, const int32_t* prefix, const int32_t* order,
                                            int i) {
    Item it;
    const int sp = i / p.num_kv_heads;
    it.kvh = i - sp * p.num_kv_heads;
    const int F = prefix[p.num_seqs];
    int L;
    if (sp < F) {
        int lo = 0, hi = p.num_seqs - 1;  // largest b with prefix[b] <= sp
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (prefix[mid] <= sp) lo = mid;
            else hi = mid - 1;
        }
        it.b = lo;
        it.part = sp - prefix[lo];
        L = checked_len(p, lo);
        it.L = L < 0 ? 0 : L;
        it.s0 = seq_start(p, lo, it.L);
        it.nparts = parts_of(it.L - it.s0, p.partition);
    } else {
        it.b = order[sp - F];
        L = checked_len(p, it.b);
        it.L = L < 0 ? 0 : L;
        it.s0 = seq_start(p, it.b, it.L);
        it.nparts = parts_of(it.L - it.s0, p.partition);
        it.part = it.nparts - 1;
    }
    const int t0 = it.s0 + it.part * p.partition;
    it.t1 = min(it.L, t0 + p.partition);
    it.j0 = t0 / p.block_size;
    it.j1 = it.t1 > t0 ? (it.t1 + p.block_size - 1) / p.block_size : it.j0;
    return it;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// chunk of B bytes (16, 8 or 4) from shared memory into 32-bit words
template <int B>
__device__ __forceinline__ void load_chunk(const uint8_t* src, uint32_t (&w)[4]) {
    if constexpr (B == 16) {
        const uint4 x = *reinterpret_cast<const uint4*>(src);
        w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
    } else if constexpr (B == 8) {
        const uint2 x = *reinterpret_cast<const uint2*>(src);
        w[0] = x.x; w[1] = x.y; w[2] = 0u; w[3] = 0u;
    } else {
        w[0] = *reinterpret_cast<const uint32_t*>(src); w[1] = w[2] = w[3] = 0u;
    }
}

// a0 += q.lo * k.lo, a1 += q.hi * k.hi on packed 16-bit pairs.  A product of
// two 16-bit floats is exact in fp32, so this equals fp32 FMAs on the
// widened values (one rounding per FMA).
template <int DT>
__device__ __forceinline__ void fma_mixed2(float& a0, float& a1, uint32_t q, uint32_t k) {
    if constexpr (DT == PA_BF16) {
        asm("{\n\t.reg .b16 ql, qh, kl, kh;\n\tmov.b32 {ql, qh}, %2;\n\tmov.b32 {kl, kh}, %3;\n\t"
            "fma.rn.f32.bf16 %0, ql, kl, %0;\n\tfma.rn.f32.bf16 %1, qh, kh, %1;\n\t}"
            : "+f"(a0), "+f"(a1) : "r"(q), "r"(k));
    } else {
        asm("{\n\t.reg .b16 ql, qh, kl, kh;\n\tmov.b32 {ql, qh}, %2;\n\tmov.b32 {kl, kh}, %3;\n\t"
            "fma.rn.f32.f16 %0, ql, kl, %0;\n\tfma.rn.f32.f16 %1, qh, kh, %1;\n\t}"
            : "+f"(a0), "+f"(a1) : "r"(q), "r"(k));
    }
}

// two E4M3 codes (low 16 bits of w) -> packed fp16 pair (exact)
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t w) {
    uint32_t h;
    const uint16_t b = static_cast<uint16_t>(w & 0xffffu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(b));
    return h;
}

// Packed fp32 pairs: one 64-bit register pair holds (x, y); fma/mul on both
// halves is one instruction (fma.rn.f32x2 / mul.rn.f32x2).
__device__ __forceinline__ uint64_t pk2(float x, float y) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}
__device__ __forceinline__ uint64_t pk2u(uint32_t x, uint32_t y) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(x), "r"(y));
    return r;
}
__device__ __forceinline__ float2 up2(uint64_t r) {
    float2 f;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(r));
    return f;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// packed 16-bit pair -> fp32 pair
template <int DT>
__device__ __forceinline__ uint64_t pair_of(uint32_t w);
template <>
__device__ __forceinline__ uint64_t pair_of<PA_BF16>(uint32_t w) { return pk2u(w << 16, w & 0xffff0000u); }
template <>
__device__ __forceinline__ uint64_t pair_of<PA_F16>(uint32_t w) {
    const float2 f = f16x2_to_f2(w);
    return pk2(f.x, f.y);
}

// End of a work item: the consumer warps have left their per-warp partials
// (max m and sum l in log2 units, unnormalised outputs) in `merge`, laid out
// [head group][token warp][head][D + 2]; merge them and write the output row
// (unsplit sequence) or the partition's normalised row and log-sum-exp
// (split sequence).  All consumer warps call it; it brackets its work with the
// consumers' named barrier.
template <typename C, int QDT, int D, int G>
__device__ __forceinline__ void store_item(const DecodeParams& p, const Item& it, float* merge) {
    named_bar_sync(1, C::NCW * 32);
    {
        const int tid = threadIdx.x;  // 0 .. NCW*32-1
        const bool direct = it.nparts == 1 && p.cu_groups == nullptr;
        const int part = it.part + prefix_parts(p, it.s0);  // cascade: after the prefix's parts
        // group mode: query row g is head g % g_real of member m0 + g / g_real
        VSeq v{0, it.b, 0, false};
        if (p.vm > 0) {
            v = vseq(p, it.b);
            // a group without shared tokens leaves its members' parts to
            // their own sequences (the same parts, written in this launch)
            if (!v.own && it.L == 0) v.nm = 0;
        }
        // Thread tid takes pairs of one head: g = tid / TPH, columns 2j for j =
        // tid % TPH, + TPH, ...; the head's max over the slots, the slots'
        // weights and the normaliser are taken once per thread.
        constexpr int NT = C::NCW * 32;
        constexpr int TPH = NT / G < 1 ? 1 : NT / G;  // threads per head
        for (int g = tid / TPH; g < G; g += NT / TPH) {
            const int ghg = g / C::GW, gw = g % C::GW;
            float M = -INFINITY;
#pragma unroll
            for (int t = 0; t < C::TW; ++t) M = fmaxf(M, merge[((ghg * C::TW + t) * C::GW + gw) * (D + 2) + D]);
            float wt[C::TW];
            float lsum = 0.f;
#pragma unroll
            for (int t = 0; t < C::TW; ++t) {
                const float* mw = merge + ((ghg * C::TW + t) * C::GW + gw) * (D + 2);
                wt[t] = M == -INFINITY ? 0.f : fast_exp2(mw[D] - M);
                lsum = fmaf(wt[t], mw[D + 1], lsum);
            }
            const float inv = M == -INFINITY ? 0.f : p.v_scale / lsum;
#pragma unroll
            for (int t = 0; t < C::TW; ++t) wt[t] *= inv;
            int h = it.kvh * G + g;
            int64_t bh = static_cast<int64_t>(it.b) * p.num_heads + h;
            if (p.vm > 0) {
                const int mi = g / p.g_real;
                if (mi >= v.nm) continue;
                h = it.kvh * p.g_real + (g - mi * p.g_real);
                bh = static_cast<int64_t>(v.m0 + mi) * p.num_heads + h;
            }
            const int64_t r = bh * p.max_parts + part;
            if (!direct && tid % TPH == 0) p.ws_lse[r] = M == -INFINITY ? -INFINITY : M + __log2f(lsum);
            for (int j = tid % TPH; j < D / 2; j += TPH) {
                const int d = 2 * j;
                float o0 = 0.f, o1 = 0.f;
#pragma unroll
                for (int t = 0; t < C::TW; ++t) {
                    const float2 x = *reinterpret_cast<const float2*>(
                        merge + ((ghg * C::TW + t) * C::GW + gw) * (D + 2) + d);
                    o0 = fmaf(wt[t], x.x, o0);
                    o1 = fmaf(wt[t], x.y, o1);
                }
                if (direct) {
                    using T = typename dtype_traits<QDT>::storage;
                    T* out = static_cast<T*>(p.out) + bh * D + d;
                    out[0] = dtype_traits<QDT>::from_f(o0);
                    out[1] = dtype_traits<QDT>::from_f(o1);
                } else {
                    *reinterpret_cast<float2*>(p.ws_o + r * D + d) = make_float2(o0, o1);
                }
            }
        }
    }
    named_bar_sync(1, C::NCW * 32);
}

// ---------------------------------------------------------------------------
// Tensor-core consumer (G >= 4)
// ---------------------------------------------------------------------------
// One m16n8k16 MMA with fp32 accumulators; MT = PA_F16 or PA_BF16 operands.
template <int MT>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    if constexpr (MT == PA_BF16) {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    } else {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}

// Transpose of an 8x8 matrix of 16-bit elements held one pair per lane (lane
// 4r+c holds row r, columns 2c and 2c+1): afterwards lane 4r+c holds column r,
// rows 2c and 2c+1.
__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// two fp32 values -> packed pair of the MMA operand type (RN)
template <int MT>
__device__ __forceinline__ uint32_t pack_pair(float lo, float hi) {
    if constexpr (MT == PA_BF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}

// Consumer warps of the tensor-core path.  Every stage of 32 (or 64) tokens
// is cut into 16-token slices; slice k of the f-th stage the consumers see
// goes to warp (f*SLICES + k) % 4, which holds all G query heads (all four
// warps still wait for and release every stage).  For a
// slice, with lane = 4*gi + ti:
//  * S^T[16 tokens x 8 heads] = K[16 x D] . Q^T[D x 8]: tokens on M, heads on N
//    (heads G..7 zero), D/16 k-steps.  The contraction order over d is free, so
//    lane ti's k-columns are the d-span [W*ti, W*ti + W) (W = D/4) of its rows:
//    k-step s takes elements 4s..4s+3 of every span, and each A fragment comes
//    straight from 16-byte shared-memory loads of the K rows gi and gi+8;
//  * scores scaled, masked, one online-softmax state per head (the max is
//    reduced over the slice's tokens, so every weight of a head in the MMA
//    below shares one reference; lazy rescale as in the CUDA-core path);
//  * O^T[D x 8] += V^T[D x 16] . P^T[16 x 8]: the weights' C layout (token,
//    head pair) becomes the B layout (token pair, head) by one movmatrix per
//    8 tokens; V rows load like K rows, and a movmatrix per 8x8 tile turns
//    them into V^T A fragments, whose rows (d) then follow the span order:
//    m-tile mt, row r<8 is d = W*(r/2) + 4*mt + r%2 (with the chunk rotation
//    below, the owner's chunk in place of mt/2), row r>=8 that d + 2;
//  * bf16 weights go in as hi + lo so they keep 16 bits; fp16 weights (fp16
//    and E4M3 caches, V exact in fp16) take one MMA.  With four heads the
//    queries fill columns 0..3 and again 4..7, so lanes ti >= 2 carry the
//    same scores and softmax state as lanes ti - 2 and hand in the lo
//    weights in columns 4..7: one MMA per tile takes hi and lo at once, and
//    the two halves of O are added when the item ends.  Otherwise (eight
//    heads) the lo weights take a second MMA.
// Masked tokens (past the item or on a missing page) get weight 0 and their
// V rows are zeroed before the MMA, so stale stage bytes never reach a sum.
template <typename C, int QDT, int KVDT, int D, int G, int BS>
__device__ __forceinline__ void decode_consumer_mma(const DecodeParams& p, uint8_t* ring, const uint8_t* qbuf,
                                                    float* merge, const int32_t* prefix, const int32_t* order,
                                                    int n_items, uint32_t full0, uint32_t empty0, uint32_t qfull0,
                                                    uint32_t qempty0, volatile int* abort_flag,
                                                    volatile int* stage_mask, int warp, int lane) {
    constexpr int MT = C::KB == 2 ? KVDT : PA_F16;  // operand type of both products
    constexpr bool HILO = MT == PA_BF16;
    constexpr bool PACK = HILO && G == 4;  // lo weights in the columns of heads 4..7
    constexpr int W = D / 4;   // d-span of a lane, elements
    constexpr int KS = D / 16; // QK k-steps = PV m-tiles
    constexpr int SL = C::SLICES;
    constexpr uint32_t QSLOT = (C::QBYTES + 127) & ~127;
    constexpr float kTau = 8.f;
    // 16-byte chunks of a lane's span.  With four (16-bit rows of 128), the
    // spans of lanes ti and ti+2 start 128 bytes apart, on the same banks;
    // those lanes take their chunks in an order rotated by two, which halves
    // the bank conflicts of every row load.  The rotation depends on ti only
    // (the owner of the k-columns), so Q and the output rows follow it.
    constexpr int NCH = W * C::KB / 16;
    constexpr bool ROT = NCH == 4;
    const int gi = lane >> 2, ti = lane & 3;
    const int rot = ROT ? 2 * (ti >> 1) : 0;
    const int S = p.stages;
    uint32_t stage = 0, phase = 0, fc = 0, qn = 0;
    for (int rnd = 0, i; (i = snake_item(rnd, n_items)) >= 0; ++rnd, ++qn) {
        const Item it = decode_item(p, prefix, order, i);
        const uint32_t slot = qn & 1u;
        bool ok = __all_sync(0xffffffffu, mbar_wait(qfull0 + 8u * slot, (qn >> 1) & 1u, p.status, abort_flag));
        // ---- Q^T fragments: head gi, span [W*ti, W*ti + W) as pairs ----
        uint32_t qb[KS][2];
        float qk_scale = p.qk_scale;
        {
            const int qh = PACK ? (gi & 3) : gi;  // the head of MMA column gi
            const uint8_t* qs = qbuf + slot * QSLOT + (qh * D + W * ti) * C::QB;
            if constexpr (C::KB == 2) {
#pragma unroll
                for (int c = 0; c < W / 8; ++c) {
                    uint4 x = make_uint4(0u, 0u, 0u, 0u);
                    if (PACK || gi < G) x = *reinterpret_cast<const uint4*>(qs + 16 * ((c + rot) & (NCH - 1)));
                    qb[2 * c][0] = x.x;
                    qb[2 * c][1] = x.y;
                    qb[2 * c + 1][0] = x.z;
                    qb[2 * c + 1][1] = x.w;
                }
            } else {
                // E4M3 cache: queries to fp16 scaled by a power of two so that
                // the largest lands in [2^14, 2^15); the scale is folded back
                // into the score scale
                float qv[W];
                float mx = 0.f;
#pragma unroll
                for (int c = 0; c < W / 2; ++c) {
                    float2 f = make_float2(0.f, 0.f);
                    if (gi < G) f = kv_pair<QDT>(*reinterpret_cast<const uint32_t*>(qs + 4 * c));
                    qv[2 * c] = f.x;
                    qv[2 * c + 1] = f.y;
                    mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
                }
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                int ex = mx > 0.f ? ((__float_as_int(mx) >> 23) & 0xff) - 127 - 14 : 0;
                ex = max(-100, min(100, ex));
                const float down = __int_as_float((127 - ex) << 23), up = __int_as_float((127 + ex) << 23);
                qk_scale *= up;
#pragma unroll
                for (int s2 = 0; s2 < KS; ++s2) {
                    qb[s2][0] = pack_pair<PA_F16>(qv[4 * s2] * down, qv[4 * s2 + 1] * down);
                    qb[s2][1] = pack_pair<PA_F16>(qv[4 * s2 + 2] * down, qv[4 * s2 + 3] * down);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(qempty0 + 8u * slot);

        float o[KS][4];
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // heads 2ti, 2ti+1

        for (int js = it.j0; js < it.j1 && ok; js += C::SPAGES, ++fc) {
            // Every consumer warp waits for every stage and releases it, also
            // when the stage holds no slice of its own: then no warp can fall a
            // whole ring behind the producer, so no parity wait can match an
            // older phase of the same stage, and every copy has landed before
            // the block exits.
            if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8u * stage, phase, p.status, abort_flag))) {
                ok = false;
                break;
            }
            const int k = (warp - static_cast<int>((fc * SL) & 3u)) & 3;  // this warp's slice of the stage
            if (k < SL) {
                const int mask = stage_mask[stage];
                const int tk0 = 16 * k + gi, tk1 = tk0 + 8;  // stage tokens of rows gi and gi+8
                const uint8_t* kr0 = ring + stage * C::STAGE_BYTES + tk0 * C::ROWB + W * ti * C::KB;
                const uint8_t* kr1 = kr0 + 8 * C::ROWB;
                // a stage whose pages are all present and whose tokens all lie
                // before the item's end needs no per-token masks
                const bool full_stage = mask == (1 << C::SPAGES) - 1 && js * BS + C::STOK <= it.t1;
                auto slice = [&](auto full_tag) {
                    constexpr bool FULL = decltype(full_tag)::value;
                    const bool v0 = FULL || (((mask >> (tk0 / BS)) & 1) && js * BS + tk0 < it.t1);
                    const bool v1 = FULL || (((mask >> (tk1 / BS)) & 1) && js * BS + tk1 < it.t1);
                    // ---- S^T = K Q^T (two accumulators: two independent MMA chains) ----
                    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
                    if constexpr (C::KB == 2) {
#pragma unroll
                        for (int c = 0; c < W / 8; ++c) {
                            const int cc = (c + rot) & (NCH - 1);
                            const uint4 x0 = *reinterpret_cast<const uint4*>(kr0 + 16 * cc);
                            const uint4 x1 = *reinterpret_cast<const uint4*>(kr1 + 16 * cc);
                            mma16816<MT>(sa, x0.x, x1.x, x0.y, x1.y, qb[2 * c][0], qb[2 * c][1]);
                            mma16816<MT>(sb, x0.z, x1.z, x0.w, x1.w, qb[2 * c + 1][0], qb[2 * c + 1][1]);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < W / 16; ++c) {
                            const uint4 x0 = *reinterpret_cast<const uint4*>(kr0 + 16 * c);
                            const uint4 x1 = *reinterpret_cast<const uint4*>(kr1 + 16 * c);
                            const uint32_t w0[4] = {x0.x, x0.y, x0.z, x0.w}, w1[4] = {x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                mma16816<MT>((j & 1) ? sb : sa, e4m3x2_to_h2(w0[j]), e4m3x2_to_h2(w1[j]),
                                             e4m3x2_to_h2(w0[j] >> 16), e4m3x2_to_h2(w1[j] >> 16), qb[4 * c + j][0],
                                             qb[4 * c + j][1]);
                        }
                    }
                    // ---- online softmax: c0/c1 = token gi, heads 2ti/2ti+1; c2/c3 = token gi+8 ----
                    const float s0 = v0 ? (sa[0] + sb[0]) * qk_scale : -INFINITY;
                    const float s1 = v0 ? (sa[1] + sb[1]) * qk_scale : -INFINITY;
                    const float s2 = v1 ? (sa[2] + sb[2]) * qk_scale : -INFINITY;
                    const float s3 = v1 ? (sa[3] + sb[3]) * qk_scale : -INFINITY;
                    // The reference max of a head moves only when one of its
                    // scores passes it by more than tau; a lane tests its own
                    // four and the warp votes, so the reduction over the slice's
                    // tokens runs only then (an item's first slice, and rarely
                    // after it)
                    if (__any_sync(0xffffffffu, fmaxf(s0, s2) > m0 + kTau || fmaxf(s1, s3) > m1 + kTau)) {
                        float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
                        // (with the lo columns, also over lanes ti and ti^2, whose
                        // scores are the same products in two MMA columns: one
                        // max, so both halves of O always share one reference)
#pragma unroll
                        for (int o2 = PACK ? 2 : 4; o2 < 32; o2 <<= 1) {
                            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o2));
                            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o2));
                        }
                        const bool r0 = mx0 > m0 + kTau, r1 = mx1 > m1 + kTau;
                        const float a0 = r0 ? fast_exp2(m0 - mx0) : 1.f, a1 = r1 ? fast_exp2(m1 - mx1) : 1.f;
                        m0 = r0 ? mx0 : m0;
                        m1 = r1 ? mx1 : m1;
                        l0 *= a0;
                        l1 *= a1;
#pragma unroll
                        for (int mt = 0; mt < KS; ++mt) {
                            o[mt][0] *= a0;
                            o[mt][1] *= a1;
                            o[mt][2] *= a0;
                            o[mt][3] *= a1;
                        }
                    }
                    const float p0 = v0 ? fast_exp2(s0 - m0) : 0.f, p1 = v0 ? fast_exp2(s1 - m1) : 0.f;
                    const float p2 = v1 ? fast_exp2(s2 - m0) : 0.f, p3 = v1 ? fast_exp2(s3 - m1) : 0.f;
                    l0 += p0 + p2;
                    l1 += p1 + p3;
                    // ---- P^T fragments (token pair, head gi) ----
                    uint32_t pb0, pb1;
                    [[maybe_unused]] uint32_t pl0 = 0u, pl1 = 0u;
                    if constexpr (PACK) {
                        // columns 0..3 (lanes ti < 2): hi = the top 16 bits; columns
                        // 4..7 (lanes ti >= 2, the same heads): lo = the rest in bf16
                        const uint32_t u0 = __float_as_uint(p0), u1 = __float_as_uint(p1);
                        const uint32_t u2 = __float_as_uint(p2), u3 = __float_as_uint(p3);
                        uint32_t w0 = __byte_perm(u0, u1, 0x7632), w1 = __byte_perm(u2, u3, 0x7632);
                        if (ti >= 2) {
                            w0 = pack_pair<PA_BF16>(p0 - __uint_as_float(u0 & 0xffff0000u),
                                                    p1 - __uint_as_float(u1 & 0xffff0000u));
                            w1 = pack_pair<PA_BF16>(p2 - __uint_as_float(u2 & 0xffff0000u),
                                                    p3 - __uint_as_float(u3 & 0xffff0000u));
                        }
                        pb0 = movtrans(w0);
                        pb1 = movtrans(w1);
                    } else if constexpr (HILO) {
                        // hi = the top 16 bits (truncation), lo = the rest rounded to bf16
                        const uint32_t u0 = __float_as_uint(p0), u1 = __float_as_uint(p1);
                        const uint32_t u2 = __float_as_uint(p2), u3 = __float_as_uint(p3);
                        pb0 = movtrans(__byte_perm(u0, u1, 0x7632));
                        pb1 = movtrans(__byte_perm(u2, u3, 0x7632));
                        pl0 = movtrans(pack_pair<PA_BF16>(p0 - __uint_as_float(u0 & 0xffff0000u),
                                                          p1 - __uint_as_float(u1 & 0xffff0000u)));
                        pl1 = movtrans(pack_pair<PA_BF16>(p2 - __uint_as_float(u2 & 0xffff0000u),
                                                          p3 - __uint_as_float(u3 & 0xffff0000u)));
                    } else {
                        pb0 = movtrans(pack_pair<MT>(p0, p1));
                        pb1 = movtrans(pack_pair<MT>(p2, p3));
                    }
                    // ---- O^T += V^T P^T (masked rows zeroed) ----
                    const uint8_t* vr0 = kr0 + C::SPAGES * C::PAGE;
                    const uint8_t* vr1 = vr0 + 8 * C::ROWB;
                    if constexpr (C::KB == 2) {
#pragma unroll
                        for (int c = 0; c < W / 8; ++c) {
                            const int cc = (c + rot) & (NCH - 1);
                            uint4 y0 = *reinterpret_cast<const uint4*>(vr0 + 16 * cc);
                            uint4 y1 = *reinterpret_cast<const uint4*>(vr1 + 16 * cc);
                            if (!FULL && !v0) y0 = make_uint4(0u, 0u, 0u, 0u);
                            if (!FULL && !v1) y1 = make_uint4(0u, 0u, 0u, 0u);
                            // pairs 4cc..4cc+3 of the span: m-tiles 2c (pairs 4cc, 4cc+1) and 2c+1
                            const uint32_t ta0 = movtrans(y0.x), tb0 = movtrans(y0.y), tc0 = movtrans(y0.z),
                                           td0 = movtrans(y0.w);
                            const uint32_t ta1 = movtrans(y1.x), tb1 = movtrans(y1.y), tc1 = movtrans(y1.z),
                                           td1 = movtrans(y1.w);
                            mma16816<MT>(o[2 * c], ta0, tb0, ta1, tb1, pb0, pb1);
                            mma16816<MT>(o[2 * c + 1], tc0, td0, tc1, td1, pb0, pb1);
                            if constexpr (HILO && !PACK) {
                                mma16816<MT>(o[2 * c], ta0, tb0, ta1, tb1, pl0, pl1);
                                mma16816<MT>(o[2 * c + 1], tc0, td0, tc1, td1, pl0, pl1);
                            }
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < W / 16; ++c) {
                            uint4 y0 = *reinterpret_cast<const uint4*>(vr0 + 16 * c);
                            uint4 y1 = *reinterpret_cast<const uint4*>(vr1 + 16 * c);
                            if (!FULL && !v0) y0 = make_uint4(0u, 0u, 0u, 0u);
                            if (!FULL && !v1) y1 = make_uint4(0u, 0u, 0u, 0u);
                            const uint32_t w0[4] = {y0.x, y0.y, y0.z, y0.w}, w1[4] = {y1.x, y1.y, y1.z, y1.w};
                            // word j: elements 4j..4j+3 = pairs 2j, 2j+1 of this chunk = m-tile 4c + j
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                mma16816<MT>(o[4 * c + j], movtrans(e4m3x2_to_h2(w0[j])),
                                             movtrans(e4m3x2_to_h2(w0[j] >> 16)), movtrans(e4m3x2_to_h2(w1[j])),
                                             movtrans(e4m3x2_to_h2(w1[j] >> 16)), pb0, pb1);
                        }
                    }
                };
                if (full_stage) slice(std::true_type{});
                else slice(std::false_type{});
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8u * stage);
            if (++stage == static_cast<uint32_t>(S)) {
                stage = 0;
                phase ^= 1u;
            }
        }

        // ---- this warp's partials to the merge area ----
        if constexpr (PACK) {
            // the lo half of each head's sum sits two lanes up (columns 4..7)
#pragma unroll
            for (int mt = 0; mt < KS; ++mt)
#pragma unroll
                for (int r = 0; r < 4; ++r) o[mt][r] += __shfl_xor_sync(0xffffffffu, o[mt][r], 2);
        }
#pragma unroll
        for (int o2 = 4; o2 < 32; o2 <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, o2);
            l1 += __shfl_xor_sync(0xffffffffu, l1, o2);
        }
        {
            float* mw = merge + warp * G * (D + 2);
            const int h0 = 2 * ti, h1 = 2 * ti + 1;
            if (h0 < G) {
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    // rows gi, gi+8 of m-tile mt: the d of the pair the span owner
                    // (lane ti = gi/2 of the V load) held in that tile
                    int da;
                    if constexpr (C::KB == 2) {
                        const int cc = ROT ? ((mt >> 1) + 2 * (gi >> 2)) & (NCH - 1) : (mt >> 1);
                        da = W * (gi >> 1) + 8 * cc + 4 * (mt & 1) + (gi & 1);
                    } else {
                        da = W * (gi >> 1) + 4 * mt + (gi & 1);
                    }
                    const int db = da + 2;
                    mw[h0 * (D + 2) + da] = o[mt][0];
                    mw[h1 * (D + 2) + da] = o[mt][1];
                    mw[h0 * (D + 2) + db] = o[mt][2];
                    mw[h1 * (D + 2) + db] = o[mt][3];
                }
                if (gi == 0) {
                    mw[h0 * (D + 2) + D] = m0;
                    mw[h0 * (D + 2) + D + 1] = l0;
                    mw[h1 * (D + 2) + D] = m1;
                    mw[h1 * (D + 2) + D + 1] = l1;
                }
            }
        }
        store_item<C, QDT, D, G>(p, it, merge);
    }
}

// Append mode, first half: lane c of the producer warp loads its 16-byte
// chunk of the new token's input rows (chunks 0..CH-1 of K, then CH..2CH-1 of
// V; CH = 16-byte chunks per input row) when the item starts, so the stage that
// holds the token does not wait on this load.  Lanes past 2*CH load nothing.
template <typename C, int QDT>
__device__ __forceinline__ uint4 append_prefetch(const DecodeParams& p, const Item& it, int lane) {
    constexpr int D = C::ROWB / C::KB;
    constexpr int CH = D * 2 / 16;  // the input rows are 16-bit
    static_assert(2 * CH <= 32, "one chunk per lane");
    if (lane >= 2 * CH) return make_uint4(0u, 0u, 0u, 0u);
    const bool isv = lane >= CH;
    const int64_t src_row = (static_cast<int64_t>(it.b) * p.num_kv_heads + it.kvh) * D;
    return __ldg(reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(isv ? p.v_new : p.k_new) + src_row * 2) +
                 (isv ? lane - CH : lane));
}

// Append mode, second half: the prefetched chunk `x`, in the cache's type
// (16-bit: the bits; E4M3: IEEE x/scale rounded to nearest even with
// saturation, as pa_kv_cache_write stores it), goes to the cache slot of
// position L-1 and to row (L-1) % BS of the stage page at `page` (K at page,
// V SPAGES pages further).
template <typename C, int QDT, int KVDT>
__device__ __forceinline__ void append_row(const DecodeParams& p, const Item& it, int32_t blk, uint8_t* page,
                                           int lane, uint4 x) {
    constexpr int D = C::ROWB / C::KB;
    constexpr int CH = D * 2 / 16;
    if (lane >= 2 * CH) return;
    const int r = (it.L - 1) % (C::PAGE / C::ROWB);
    const int64_t cache_off = (static_cast<int64_t>(blk) * p.num_kv_heads + it.kvh) * C::PAGE + r * C::ROWB;
    const bool isv = lane >= CH;
    const int cc = isv ? lane - CH : lane;
    uint8_t* srow = page + (isv ? C::SPAGES * C::PAGE : 0) + r * C::ROWB;
    uint8_t* crow = const_cast<uint8_t*>(isv ? p.v_cache : p.k_cache) + cache_off;
    if constexpr (C::KB == 2) {
        *reinterpret_cast<uint4*>(srow + cc * 16) = x;
        *reinterpret_cast<uint4*>(crow + cc * 16) = x;
    } else {
        // E4M3: 8 input elements (16 bytes) -> 8 codes (8 bytes)
        const float sc = isv ? p.v_scale_w : p.k_scale_w;
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        uint32_t codes[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float2 a = kv_pair<QDT>(w[2 * h]), b = kv_pair<QDT>(w[2 * h + 1]);
            const uint32_t lo = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(
                make_float2(__fdiv_rn(a.x, sc), __fdiv_rn(a.y, sc)), __NV_SATFINITE, __NV_E4M3));
            const uint32_t hi = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(
                make_float2(__fdiv_rn(b.x, sc), __fdiv_rn(b.y, sc)), __NV_SATFINITE, __NV_E4M3));
            codes[h] = lo | (hi << 16);
        }
        const uint2 y = make_uint2(codes[0], codes[1]);
        *reinterpret_cast<uint2*>(srow + cc * 8) = y;
        *reinterpret_cast<uint2*>(crow + cc * 8) = y;
    }
}

// APPEND: the new token of every sequence is written and attended in the
// same launch (pa_decode_append); a separate instantiation keeps the plain
// decode's producer loop as lean as it was.
template <int QDT, int KVDT, int D, int G, int BS, bool APPEND>
__global__ void __maxnreg__((DecodeCfg<QDT, KVDT, D, G, BS>::MAX_REGS))
paged_decode_kernel(const DecodeParams p) {
    using C = DecodeCfg<QDT, KVDT, D, G, BS>;
    // the 16-bit type the QK products are taken in: the cache's, or fp16
    // (exact for E4M3 codes) with power-of-two scaled queries for E4M3 caches
    constexpr int KT = C::KB == 2 ? KVDT : PA_F16;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const DecodeSmem L = DecodeSmem::make(p.stages, C::STAGE_BYTES, C::QBYTES, C::MERGE_FLOATS, p.num_seqs);
    uint8_t* ring = smem_raw + L.ring;
    uint8_t* qbuf = smem_raw + L.qbuf;
    float* merge = reinterpret_cast<float*>(smem_raw + L.merge);
    int32_t* prefix = reinterpret_cast<int32_t*>(smem_raw + L.prefix);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + L.bars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + L.flags);
    volatile int* stage_mask = abort_flag + 1;  // bit k: page k of the stage is present
    const int S = p.stages;
    const uint32_t full0 = smem_addr(bars), empty0 = full0 + 8u * S;
    const uint32_t qfull0 = full0 + 16u * S, qempty0 = qfull0 + 16u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr uint32_t QSLOT = (C::QBYTES + 127) & ~127;

    pdl_wait();
    pdl_trigger();
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, C::NCW);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(qfull0 + 8u * s, 1);
            mbar_init(qempty0 + 8u * s, C::NCW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    // merge area doubles as scan scratch before the first item
    int32_t* order = reinterpret_cast<int32_t*>(smem_raw + L.order);
    build_schedule(p, prefix, order, reinterpret_cast<int32_t*>(merge), smem_raw + L.keys,
                   reinterpret_cast<int32_t*>(smem_raw + L.hist));
    const int n_items = (prefix[p.num_seqs] + p.num_seqs) * p.num_kv_heads;

    if (warp == C::NCW) {
        // ------------------------------ producer ------------------------------
        if (p.no_copies) return;
        const uint64_t policy = policy_evict_first();
        uint32_t fill = 0;    // ring stages used so far by this CTA
        uint32_t stage = 0;   // fill % S
        uint32_t phase = 0;   // (fill / S) & 1
        uint32_t issued = 0;  // fills that started copies
        uint32_t qn = 0;      // items issued so far
        bool ok = true;
        for (int rnd = 0, i; ok && (i = snake_item(rnd, n_items)) >= 0; ++rnd, ++qn) {
            const Item it = decode_item(p, prefix, order, i);
            if (lane == 0) {
                const uint32_t slot = qn & 1u;
                if (qn >= 2) ok = mbar_wait(qempty0 + 8u * slot, ((qn >> 1) - 1) & 1u, p.status, abort_flag);
                if (ok && p.vm > 0) {
                    // group mode: each member's g_real heads, zeros for absent members
                    const VSeq v = vseq(p, it.b);
                    const uint32_t mb = static_cast<uint32_t>(p.g_real) * D * C::QB;
                    uint8_t* dst = qbuf + slot * QSLOT;
                    for (uint32_t o = static_cast<uint32_t>(v.nm) * mb; o < C::QBYTES; o += 16)
                        *reinterpret_cast<uint4*>(dst + o) = make_uint4(0u, 0u, 0u, 0u);
                    mbar_expect_tx(qfull0 + 8u * slot, static_cast<uint32_t>(v.nm) * mb);
                    for (int mi = 0; mi < v.nm; ++mi) {
                        const uint8_t* src =
                            static_cast<const uint8_t*>(p.q) +
                            (static_cast<int64_t>(v.m0 + mi) * p.num_heads + it.kvh * p.g_real) * D * C::QB;
                        bulk_g2s(smem_addr(dst + mi * mb), src, mb, qfull0 + 8u * slot);
                    }
                } else if (ok) {
                    const uint8_t* src = static_cast<const uint8_t*>(p.q) +
                                         (static_cast<int64_t>(it.b) * p.num_heads + it.kvh * G) * D * C::QB;
                    mbar_expect_tx(qfull0 + 8u * slot, C::QBYTES);
                    bulk_g2s(smem_addr(qbuf + slot * QSLOT), src, C::QBYTES, qfull0 + 8u * slot);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            // append mode: the item whose last partition holds the new token
            // loads that token's rows now
            uint4 xnew = make_uint4(0u, 0u, 0u, 0u);
            if constexpr (APPEND) {
                if (it.L > 0 && it.t1 == it.L) xnew = append_prefetch<C, QDT>(p, it, lane);
            }
            // (group mode: the group's first member's row, or the member's own)
            const int member = p.vm > 0 && it.b >= p.vcount ? it.b - p.vcount : it.b;
            const int trow = p.vm > 0 && it.b < p.vcount ? __ldg(p.cu_groups + it.b / p.vpg) : member;
            const int32_t* row = p.block_table + static_cast<int64_t>(trow) * p.max_blocks;
            // cascade: the prefix pass read the shared blocks through the group's
            // first row; a member whose row names other blocks there is reported
            if (p.cu_groups != nullptr && it.part == 0 && it.kvh == 0 && it.s0 > 0) {
                const int b0 = __ldg(p.cu_groups + group_of(p, member));
                if (b0 != member) {
                    const int32_t* row0 = p.block_table + static_cast<int64_t>(b0) * p.max_blocks;
                    bool bad = false;
                    for (int j = lane; j < it.s0 / BS; j += 32) bad |= __ldg(row0 + j) != __ldg(row + j);
                    if (__any_sync(0xffffffffu, bad) && lane == 0) report(p.status, PA_ERR_INVALID_ARG);
                }
            }
            const int64_t head_off = static_cast<int64_t>(it.kvh) * C::PAGE;
            const int64_t blk_stride = static_cast<int64_t>(p.num_kv_heads) * C::PAGE;
            // block ids come 32 at a time, one per lane; the next batch's load
            // is issued before this batch's stages are filled, so its latency
            // hides behind them
            // block ids come 32 at a time, one per lane; the next batch's load
            // is issued before this batch's stages are filled, so its latency
            // hides behind them
            int32_t id_next = it.j0 + lane < it.j1 ? __ldg(row + it.j0 + lane) : -1;
            for (int jb = it.j0; jb < it.j1 && ok; jb += 32) {
                const int32_t id = id_next;
                id_next = jb + 32 + lane < it.j1 ? __ldg(row + jb + 32 + lane) : -1;
                const int cnt = min(32, it.j1 - jb);
                for (int k0 = 0; k0 < cnt; k0 += C::SPAGES) {
                    int32_t ids[C::SPAGES];
#pragma unroll
                    for (int k = 0; k < C::SPAGES; ++k) ids[k] = __shfl_sync(0xffffffffu, id, k0 + k);
                    // one lane fills the stage (every stage of a plain decode, and
                    // the stages of an append that do not hold the new token)
                    auto fill_lane0 = [&]() {
                        if (lane == 0) {
                            if (fill >= static_cast<uint32_t>(S))
                                ok = mbar_wait(empty0 + 8u * stage, phase ^ 1u, p.status, abort_flag);
                            if (ok) {
                                const uint32_t bar = full0 + 8u * stage;
                                const uint32_t dst = smem_addr(ring) + stage * C::STAGE_BYTES;
                                int mask = 0;
                                uint32_t bytes = 0;
#pragma unroll
                                for (int k = 0; k < C::SPAGES; ++k) {
                                    if (k0 + k >= cnt) continue;  // past the item's pages
                                    if (ids[k] >= 0 && ids[k] < p.num_blocks) {
                                        mask |= 1 << k;
                                        bytes += 2u * C::PAGE;
                                    } else {
                                        report(p.status, PA_ERR_BAD_BLOCK);
                                    }
                                }
                                stage_mask[stage] = mask;
                                if (bytes) {
                                    mbar_expect_tx(bar, bytes);
#pragma unroll
                                    for (int k = 0; k < C::SPAGES; ++k) {
                                        if (!(mask & (1 << k))) continue;
                                        const int64_t off = ids[k] * blk_stride + head_off;
                                        bulk_g2s_hint(dst + k * C::PAGE, p.k_cache + off, C::PAGE, bar, policy);
                                        bulk_g2s_hint(dst + (C::SPAGES + k) * C::PAGE, p.v_cache + off, C::PAGE, bar,
                                                      policy);
                                    }
                                    issued = fill + 1;
                                } else {
                                    mbar_arrive(bar);
                                }
                            }
                        }
                    };
                    if constexpr (!APPEND) {
                        fill_lane0();
                    } else {
                        // append mode: the page holding the new token (position L-1,
                        // in the item's last partition) copies only the rows before it;
                        // the warp writes the new row into the stage and the cache
                        int pk = -1;  // page of this stage that holds the new token
                        if (it.L > 0 && it.t1 == it.L) {
                            const int jn = (it.L - 1) / BS - (jb + k0);
                            if (jn >= 0 && jn < C::SPAGES && jn < cnt - k0) pk = jn;
                        }
                        if (pk < 0) {
                            fill_lane0();
                        } else {
                            if (lane == 0 && fill >= static_cast<uint32_t>(S))
                                ok = mbar_wait(empty0 + 8u * stage, phase ^ 1u, p.status, abort_flag);
                            ok = __shfl_sync(0xffffffffu, ok, 0);
                            if (ok && pk >= 0 && ids[pk] >= 0 && ids[pk] < p.num_blocks)
                                append_row<C, QDT, KVDT>(p, it, ids[pk], ring + stage * C::STAGE_BYTES + pk * C::PAGE,
                                                         lane, xnew);
                            __syncwarp();
                            if (lane == 0 && ok) {
                                const uint32_t bar = full0 + 8u * stage;
                                const uint32_t dst = smem_addr(ring) + stage * C::STAGE_BYTES;
                                const uint32_t rn = static_cast<uint32_t>((it.L - 1) % BS);  // rows before the new one
                                int mask = 0;
                                uint32_t bytes = 0;
#pragma unroll
                                for (int k = 0; k < C::SPAGES; ++k) {
                                    if (k0 + k >= cnt) continue;  // past the item's pages
                                    if (ids[k] >= 0 && ids[k] < p.num_blocks) {
                                        mask |= 1 << k;
                                        bytes += 2u * (k == pk ? rn * C::ROWB : C::PAGE);
                                    } else {
                                        report(p.status, PA_ERR_BAD_BLOCK);
                                    }
                                }
                                stage_mask[stage] = mask;
                                if (bytes) {
                                    mbar_expect_tx(bar, bytes);
#pragma unroll
                                    for (int k = 0; k < C::SPAGES; ++k) {
                                        if (!(mask & (1 << k))) continue;
                                        const uint32_t n = k == pk ? rn * C::ROWB : C::PAGE;
                                        if (n == 0) continue;
                                        const int64_t off = ids[k] * blk_stride + head_off;
                                        bulk_g2s_hint(dst + k * C::PAGE, p.k_cache + off, n, bar, policy);
                                        bulk_g2s_hint(dst + (C::SPAGES + k) * C::PAGE, p.v_cache + off, n, bar, policy);
                                    }
                                    issued = fill + 1;
                                } else {
                                    mbar_arrive(bar);
                                }
                            }
                        }
                    }
                    ++fill;
                    if (++stage == static_cast<uint32_t>(S)) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                }
            }
        }
        // do not leave while copies may still land: after an abort, wait
        // (bounded) for every stage that was filled but maybe not consumed
        if (lane == 0 && *abort_flag) {
            const uint32_t first = issued > static_cast<uint32_t>(S) ? issued - S : 0u;
            const uint64_t t0 = global_timer_ns();
            for (uint32_t f = first; f < issued; ++f) {
                const uint32_t st = f % S;
                while (!mbar_try_wait(full0 + 8u * st, (f / S) & 1u)) {
                    if (global_timer_ns() - t0 > kWaitLimitNs) break;
                }
            }
        }
        return;
    }

    // ------------------------------- consumers ------------------------------
    if constexpr (C::MMA) {
        decode_consumer_mma<C, QDT, KVDT, D, G, BS>(p, ring, qbuf, merge, prefix, order, n_items, full0, empty0,
                                                    qfull0, qempty0, abort_flag, stage_mask, warp, lane);
        return;
    }
    // Consumer warp w works for head group hg = w / TW (query heads hg*GW ..
    // hg*GW+GW-1 of the KV head) as token warp tw = w % TW.  A warp is TG token
    // groups of LPT lanes; in every TPI-token step of a stage, group tg takes
    // token u*TPI + tw*TG + tg, and lane c of the group owns the row chunks
    // {v*LPT + c} (VB bytes each) of that token's key row (its share of the
    // dot products) and value row (its share of the outputs).  Every group
    // keeps its own online-softmax state, so a step needs no exchange between
    // groups; groups, then warps, are merged once per work item.
    const int hg = warp / C::TW, tw = warp % C::TW;
    const int tg = lane / C::LPT, c = lane % C::LPT;
    constexpr float kTau = 8.f;  // lazy-rescale threshold (log2 units)
    const uint32_t lane_off = (tw * C::TG + tg) * C::ROWB + c * C::VB;
    uint32_t stage = 0, phase = 0;
    uint32_t qn = 0;
    for (int rnd = 0, i; (i = snake_item(rnd, n_items)) >= 0; ++rnd, ++qn) {
        const Item it = decode_item(p, prefix, order, i);
        const uint32_t slot = qn & 1u;
        bool ok = __all_sync(0xffffffffu, mbar_wait(qfull0 + 8u * slot, (qn >> 1) & 1u, p.status, abort_flag));
        // this warp's queries as packed 16-bit pairs in the lane's chunk order
        uint32_t qw[C::GW][C::PL];
        float qk_scale = p.qk_scale;
        {
            const uint8_t* qs = qbuf + slot * QSLOT;
            if constexpr (C::KB == 2) {
#pragma unroll
                for (int g = 0; g < C::GW; ++g)
#pragma unroll
                    for (int v = 0; v < C::NV; ++v)
#pragma unroll
                        for (int e = 0; e < C::EV; e += 2)
                            qw[g][(v * C::EV + e) / 2] = *reinterpret_cast<const uint32_t*>(
                                qs + ((hg * C::GW + g) * D + (v * C::LPT + c) * C::EV + e) * C::QB);
            } else {
                // E4M3 cache: queries to fp16, scaled by a power of two so that
                // the largest lands in [2^14, 2^15) (exact but for components
                // 2^28 times smaller than the largest); the scale is folded
                // back into the score scale
                float qv[C::GW][C::EPL];
                float mx = 0.f;
#pragma unroll
                for (int g = 0; g < C::GW; ++g)
#pragma unroll
                    for (int v = 0; v < C::NV; ++v)
#pragma unroll
                        for (int e = 0; e < C::EV; e += 2) {
                            const float2 f = kv_pair<QDT>(*reinterpret_cast<const uint32_t*>(
                                qs + ((hg * C::GW + g) * D + (v * C::LPT + c) * C::EV + e) * C::QB));
                            qv[g][v * C::EV + e] = f.x;
                            qv[g][v * C::EV + e + 1] = f.y;
                            mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
                        }
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                int ex = mx > 0.f ? ((__float_as_int(mx) >> 23) & 0xff) - 127 - 14 : 0;
                ex = max(-100, min(100, ex));
                const float down = __int_as_float((127 - ex) << 23), up = __int_as_float((127 + ex) << 23);
                qk_scale *= up;
#pragma unroll
                for (int g = 0; g < C::GW; ++g)
#pragma unroll
                    for (int x = 0; x < C::PL; ++x) {
                        const __half2 h = __floats2half2_rn(qv[g][2 * x] * down, qv[g][2 * x + 1] * down);
                        qw[g][x] = *reinterpret_cast<const uint32_t*>(&h);
                    }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(qempty0 + 8u * slot);

        float m[C::GW], l[C::GW];
        uint64_t acc[C::GW][C::PL];
#pragma unroll
        for (int g = 0; g < C::GW; ++g) {
            m[g] = -INFINITY;
            l[g] = 0.f;
#pragma unroll
            for (int x = 0; x < C::PL; ++x) acc[g][x] = 0ull;
        }

        for (int js = it.j0; js < it.j1 && ok; js += C::SPAGES) {
            if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8u * stage, phase, p.status, abort_flag))) {
                ok = false;
                break;
            }
            const int mask = stage_mask[stage];
            const uint8_t* Kp = ring + stage * C::STAGE_BYTES + lane_off;
            const uint8_t* Vp = Kp + C::SPAGES * C::PAGE;
            const int tok0 = js * BS + tw * C::TG + tg;  // this group's first position
            // a stage whose pages are all present and whose tokens all lie
            // before the item's end takes a path without per-token masks
            const bool full_stage = mask == (1 << C::SPAGES) - 1 && js * BS + C::STOK <= it.t1;
            auto stage_steps = [&](auto full_tag) {
                constexpr bool FULL = decltype(full_tag)::value;
                // with several heads per warp, steps go in pairs (NB = 2): both
                // steps' dot products and shuffle reductions interleave (twice the
                // independent chains), and the softmax takes one lazy-rescale
                // decision per pair
#pragma unroll
                for (int u0 = 0; u0 < C::SUB; u0 += C::NB) {
                    bool valid[C::NB];
                    uint32_t vw[C::NB][C::NV][4];
                    float sc[C::NB][C::GW];
#pragma unroll
                    for (int h = 0; h < C::NB; ++h) {
                        const int tis = (u0 + h) * C::TPI;  // step offset inside the stage
                        valid[h] = FULL || (((mask >> ((tis + tw * C::TG + tg) / BS)) & 1) && tok0 + tis < it.t1);
                        // value chunks are loaded up front (unconditionally: the
                        // rows are in shared memory) so the loads overlap the QK math
#pragma unroll
                        for (int v = 0; v < C::NV; ++v) load_chunk<C::VB>(Vp + tis * C::ROWB + v * C::LPT * C::VB, vw[h][v]);
                    }
                    // ---- QK: this lane's chunks of both steps, then butterflies over the group ----
                    {
                        float s0[C::NB][C::GW], s1[C::NB][C::GW];
#pragma unroll
                        for (int h = 0; h < C::NB; ++h)
#pragma unroll
                            for (int g = 0; g < C::GW; ++g) s0[h][g] = s1[h][g] = 0.f;
#pragma unroll
                        for (int h = 0; h < C::NB; ++h) {
                            const uint8_t* krow = Kp + (u0 + h) * C::TPI * C::ROWB;
#pragma unroll
                            for (int v = 0; v < C::NV; ++v) {
                                uint32_t w[4];
                                load_chunk<C::VB>(krow + v * C::LPT * C::VB, w);
#pragma unroll
                                for (int x = 0; x < C::VB / 4; ++x) {
                                    if constexpr (C::KB == 2) {
                                        const int pi = (v * C::EV) / 2 + x;
#pragma unroll
                                        for (int g = 0; g < C::GW; ++g)
                                            fma_mixed2<KT>(s0[h][g], s1[h][g], qw[g][pi], w[x]);
                                    } else {
                                        const uint32_t h0 = e4m3x2_to_h2(w[x]), h1 = e4m3x2_to_h2(w[x] >> 16);
                                        const int pi = (v * C::EV) / 2 + 2 * x;
#pragma unroll
                                        for (int g = 0; g < C::GW; ++g) {
                                            fma_mixed2<KT>(s0[h][g], s1[h][g], qw[g][pi], h0);
                                            fma_mixed2<KT>(s0[h][g], s1[h][g], qw[g][pi + 1], h1);
                                        }
                                    }
                                }
                            }
                        }
                        float t[C::NB][C::GW];
#pragma unroll
                        for (int h = 0; h < C::NB; ++h)
#pragma unroll
                            for (int g = 0; g < C::GW; ++g) t[h][g] = s0[h][g] + s1[h][g];
#pragma unroll
                        for (int o = 1; o < C::LPT; o <<= 1)
#pragma unroll
                            for (int h = 0; h < C::NB; ++h)
#pragma unroll
                                for (int g = 0; g < C::GW; ++g) t[h][g] += __shfl_xor_sync(0xffffffffu, t[h][g], o);
#pragma unroll
                        for (int h = 0; h < C::NB; ++h)
#pragma unroll
                            for (int g = 0; g < C::GW; ++g) sc[h][g] = (FULL || valid[h]) ? t[h][g] * qk_scale : -INFINITY;
                    }
                    // ---- online softmax of this group over the NB steps, lazy rescale (warp-uniform test) ----
                    float smax[C::GW];
#pragma unroll
                    for (int g = 0; g < C::GW; ++g) {
                        smax[g] = sc[0][g];
#pragma unroll
                        for (int h = 1; h < C::NB; ++h) smax[g] = fmaxf(smax[g], sc[h][g]);
                    }
                    bool need = false;
#pragma unroll
                    for (int g = 0; g < C::GW; ++g) need |= smax[g] > m[g] + kTau;
                    if (__any_sync(0xffffffffu, need)) {
#pragma unroll
                        for (int g = 0; g < C::GW; ++g) {
                            const float mx = smax[g];
                            const bool r = mx > m[g] + kTau;
                            const float a = r ? fast_exp2(m[g] - mx) : 1.f;  // 0 when m = -inf
                            m[g] = r ? mx : m[g];
                            l[g] *= a;
                            const uint64_t aa = pk2(a, a);
#pragma unroll
                            for (int x = 0; x < C::PL; ++x) acc[g][x] = fmul2(acc[g][x], aa);
                        }
                    }
                    uint64_t pp[C::NB][C::GW];
#pragma unroll
                    for (int h = 0; h < C::NB; ++h)
#pragma unroll
                        for (int g = 0; g < C::GW; ++g) {
                            const float pr = (FULL || valid[h]) ? fast_exp2(sc[h][g] - m[g]) : 0.f;
                            l[g] += pr;
                            pp[h][g] = pk2(pr, pr);
                        }
                    // ---- PV over this lane's value chunks (masked rows are not read) ----
#pragma unroll
                    for (int h = 0; h < C::NB; ++h) {
                        if (FULL || valid[h]) {
#pragma unroll
                            for (int v = 0; v < C::NV; ++v) {
                                const uint32_t (&w)[4] = vw[h][v];
#pragma unroll
                                for (int x = 0; x < C::VB / 4; ++x) {
                                    if constexpr (C::KB == 2) {
                                        const uint64_t v2 = pair_of<KVDT>(w[x]);
                                        const int pi = (v * C::EV) / 2 + x;
#pragma unroll
                                        for (int g = 0; g < C::GW; ++g) acc[g][pi] = ffma2(pp[h][g], v2, acc[g][pi]);
                                    } else {
                                        const uint64_t v0 = pair_of<PA_F16>(e4m3x2_to_h2(w[x]));
                                        const uint64_t v1 = pair_of<PA_F16>(e4m3x2_to_h2(w[x] >> 16));
                                        const int pi = (v * C::EV) / 2 + 2 * x;
#pragma unroll
                                        for (int g = 0; g < C::GW; ++g) {
                                            acc[g][pi] = ffma2(pp[h][g], v0, acc[g][pi]);
                                            acc[g][pi + 1] = ffma2(pp[h][g], v1, acc[g][pi + 1]);
                                        }
                                    }
                                }
                            }
                        }
                    }
                }
            };
            if (full_stage) stage_steps(std::true_type{});
            else stage_steps(std::false_type{});
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8u * stage);
            if (++stage == static_cast<uint32_t>(S)) {
                stage = 0;
                phase ^= 1u;
            }
        }

        // ---- merge the token groups of this warp, then the token warps ----
        {
            float* mw = merge + warp * C::GW * (D + 2);
#pragma unroll
            for (int g = 0; g < C::GW; ++g) {
                float M = m[g];
#pragma unroll
                for (int o = C::LPT; o < 32; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
                const float f = M == -INFINITY ? 0.f : fast_exp2(m[g] - M);
                float lw = l[g] * f;
#pragma unroll
                for (int o = C::LPT; o < 32; o <<= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
#pragma unroll
                for (int x = 0; x < C::PL; ++x) {
                    float2 a = up2(acc[g][x]);
                    a.x *= f;
                    a.y *= f;
#pragma unroll
                    for (int o = C::LPT; o < 32; o <<= 1) {
                        a.x += __shfl_xor_sync(0xffffffffu, a.x, o);
                        a.y += __shfl_xor_sync(0xffffffffu, a.y, o);
                    }
                    if (tg == 0) {
                        const int k = 2 * x;  // lane-local element index
                        const int e = ((k / C::EV) * C::LPT + c) * C::EV + k % C::EV;
                        mw[g * (D + 2) + e] = a.x;
                        mw[g * (D + 2) + e + 1] = a.y;
                    }
                }
                if (lane == 0) {
                    mw[g * (D + 2) + D] = M;
                    mw[g * (D + 2) + D + 1] = lw;
                }
            }
        }
        store_item<C, QDT, D, G>(p, it, merge);
    }
}

// Log-sum-exp merge of the partitions of every (sequence, head) that was
// split.  WPP warps share one (sequence, head): each takes every WPP-th
// partition (four at a time, so their loads overlap), weighting it by
// exp2(lse - M) against the pair's overall max M; the warps' sums then meet in
// shared memory.  Lanes own D/32 consecutive output columns.  With hundreds of
// partitions per pair (long contexts) one warp per pair left most of the GPU
// idle and each warp waiting on one row load at a time.
template <int QDT, int D, int WPP>
__global__ void __launch_bounds__(256)
paged_decode_reduce_kernel(const DecodeParams p) {
    pdl_wait();
    pdl_trigger();
    constexpr int DL = D / 32;
    constexpr int PPC = 8 / WPP;  // (sequence, head) pairs per block
    __shared__ float red[8][D + 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = warp % WPP;
    const int64_t bh = static_cast<int64_t>(blockIdx.x) * PPC + warp / WPP;
    int np = 0;
    if (bh < static_cast<int64_t>(p.num_seqs) * p.num_heads) {
        const int b = static_cast<int>(bh / p.num_heads);
        const int Lc = checked_len(p, b);
        const int L = Lc < 0 ? 0 : Lc;
        // cascade: the prefix's parts, then the suffix's partitions
        const int s0 = seq_start(p, b, L);
        np = parts_of(L - s0, p.partition) + prefix_parts(p, s0);
    }
    // unsplit pairs were written by the decode kernel (a cascade's all go
    // through the workspace)
    const bool work = np > 1 || (np == 1 && p.cu_groups != nullptr);
    const float* lse = p.ws_lse + bh * p.max_parts;
    float M = -INFINITY;
    if (work) {
        for (int i = lane; i < np; i += 32) M = fmaxf(M, lse[i]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    }
    float acc[DL];
#pragma unroll
    for (int d = 0; d < DL; ++d) acc[d] = 0.f;
    float wsum = 0.f;
    if (work && M != -INFINITY) {
        const float* o = p.ws_o + bh * p.max_parts * D + lane * DL;
        int i = sub;
        for (; i + 3 * WPP < np; i += 4 * WPP) {
            float w[4], v[4][DL];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                w[u] = lse[i + u * WPP];
#pragma unroll
                for (int d = 0; d < DL; ++d) v[u][d] = o[static_cast<int64_t>(i + u * WPP) * D + d];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float x = fast_exp2(w[u] - M);
                wsum += x;
#pragma unroll
                for (int d = 0; d < DL; ++d) acc[d] = fmaf(x, v[u][d], acc[d]);
            }
        }
        for (; i < np; i += WPP) {
            const float x = fast_exp2(lse[i] - M);
            wsum += x;
#pragma unroll
            for (int d = 0; d < DL; ++d) acc[d] = fmaf(x, o[static_cast<int64_t>(i) * D + d], acc[d]);
        }
    }
    if constexpr (WPP > 1) {
#pragma unroll
        for (int d = 0; d < DL; ++d) red[warp][lane * DL + d] = acc[d];
        if (lane == 0) red[warp][D] = wsum;
        __syncthreads();
        if (sub == 0 && work) {
#pragma unroll
            for (int k = 1; k < WPP; ++k) {
#pragma unroll
                for (int d = 0; d < DL; ++d) acc[d] += red[warp + k][lane * DL + d];
                wsum += red[warp + k][D];
            }
        }
    }
    if (sub != 0 || !work) return;
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    using T = typename dtype_traits<QDT>::storage;
    T* out = static_cast<T*>(p.out) + bh * D + lane * DL;
#pragma unroll
    for (int d = 0; d < DL; ++d) out[d] = dtype_traits<QDT>::from_f(acc[d] * inv);
}

}  // namespace pa
