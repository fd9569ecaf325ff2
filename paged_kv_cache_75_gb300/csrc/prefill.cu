// Varlen (prefill / mixed) attention over the paged KV cache.
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
// This translation unit is the tensor-core path built on mma.sync
// (m16n8k16, fp32 accumulate): 4 warps x 16 query rows per CTA, 64-key tiles
// gathered page by page with 16-byte cp.async into XOR-swizzled shared
// memory, double-buffered.  Causal alignment is bottom-right: query i of a
// sequence with Lq queries and Lk keys sits at position Lk - Lq + i.
#include "common.cuh"
#include "launch.h"

namespace pa {
namespace {

constexpr int kD = 128;        // head size
constexpr int kBM = 64;        // query rows per tile
constexpr int kBN = 64;        // keys per tile
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kRowBytes = kD * 2;
constexpr int kTileBytes = kBN * kRowBytes;  // 16 KB
constexpr int kQBytes = kBM * kRowBytes;     // 16 KB

struct PrefillParams {
    void* out;
    const uint16_t* q;
    const uint16_t* k_cache;
    const uint16_t* v_cache;
    const int32_t* block_table;
    const int32_t* cu_q;
    const int32_t* cu_k;
    int32_t* status;
    int64_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t num_heads;
    int32_t num_seqs;
    int32_t max_blocks;
    int32_t max_q;
    int32_t max_k;
    int32_t causal;
    float scale_log2;  // scale * log2(e)
};

// byte offset of (row, 16-byte chunk) inside a swizzled [rows][128] b16 tile
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return static_cast<uint32_t>(row * kRowBytes + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    const int n = valid ? 16 : 0;  // 0 source bytes: zero-fill
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

template <int DT>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if constexpr (DT == PA_BF16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
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

// (lo, hi) weights -> packed 16-bit pair, plus (bf16 only) the packed
// residual pair that the first rounding dropped
template <int DT>
__device__ __forceinline__ void split_pair(float lo, float hi, uint32_t& main, uint32_t& rest) {
    main = pack2<DT>(lo, hi);
    if constexpr (DT == PA_BF16) {
        const float lo_r = __uint_as_float(main << 16), hi_r = __uint_as_float(main & 0xffff0000u);
        rest = pack2<DT>(lo - lo_r, hi - hi_r);
    } else {
        rest = 0u;
    }
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// per-sequence lengths, or -1 if they break the stated bounds
__device__ __forceinline__ bool seq_lens_ok(const PrefillParams& p, int b, int& lq, int& lk) {
    const int q0 = __ldg(p.cu_q + b), q1 = __ldg(p.cu_q + b + 1);
    const int k0 = __ldg(p.cu_k + b), k1 = __ldg(p.cu_k + b + 1);
    lq = q1 - q0;
    lk = k1 - k0;
    return lq >= 0 && lk >= 0 && lq <= p.max_q && lk <= p.max_k &&
           static_cast<int64_t>(lk) <= static_cast<int64_t>(p.max_blocks) * p.block_size;
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 2) paged_prefill_mma_kernel(const PrefillParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* sQ = smem;
    uint8_t* sK[2] = {smem + kQBytes, smem + kQBytes + kTileBytes};
    uint8_t* sV[2] = {smem + kQBytes + 2 * kTileBytes, smem + kQBytes + 3 * kTileBytes};
    int32_t* prefix = reinterpret_cast<int32_t*>(smem + kQBytes + 4 * kTileBytes);
    __shared__ int32_t scan_scratch[kWarps];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = p.num_seqs;

    // ---- per-sequence tile prefix: tiles(b) = ceil(Lq_b / 64) ----
    {
        const int chunk = (B + kThreads - 1) / kThreads;
        const int b0 = tid * chunk, b1 = min(B, b0 + chunk);
        int local = 0;
        for (int b = b0; b < b1; ++b) {
            int lq, lk;
            if (seq_lens_ok(p, b, lq, lk)) local += (lq + kBM - 1) / kBM;
            else report(p.status, PA_ERR_INVALID_ARG);
        }
        int v = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += n;
        }
        if (lane == 31) scan_scratch[warp] = v;
        __syncthreads();
        if (tid == 0) {
            int run = 0;
            for (int w = 0; w < kWarps; ++w) {
                int x = scan_scratch[w];
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
            if (seq_lens_ok(p, b, lq, lk)) run += (lq + kBM - 1) / kBM;
        }
        __syncthreads();
    }
    const int n_items = prefix[B] * p.num_heads;
    const int group = p.num_heads / p.num_kv_heads;
    const int64_t hstride = static_cast<int64_t>(p.num_heads) * kD;  // elements per q/out row

    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int tile_id = item / p.num_heads;
        const int h = item - tile_id * p.num_heads;
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (prefix[mid] <= tile_id) lo = mid;
            else hi = mid - 1;
        }
        const int b = lo;
        int lq, lk;
        seq_lens_ok(p, b, lq, lk);
        const int i0 = (tile_id - prefix[b]) * kBM;
        const int qrow0 = __ldg(p.cu_q + b) + i0;
        const int shift = lk - lq;
        const int kvh = h / group;
        int kend = lk;  // exclusive bound on the keys this tile can see
        if (p.causal) kend = min(lk, shift + min(i0 + kBM, lq));
        const int n_tiles = kend > 0 ? (kend + kBN - 1) / kBN : 0;
        const int32_t* bt_row = p.block_table + static_cast<int64_t>(b) * p.max_blocks;

        // ---- Q tile (rows past Lq are zero-filled) ----
        for (int ci = tid; ci < kBM * 16; ci += kThreads) {
            const int r = ci >> 4, c = ci & 15;
            const bool ok = i0 + r < lq;
            const uint16_t* src = p.q + (static_cast<int64_t>(ok ? qrow0 + r : 0) * hstride + h * kD + c * 8);
            cp_async16(smem_addr(sQ) + swz(r, c), src, ok);
        }
        cp_async_commit();

        auto load_kv = [&](int t, int buf) {
            const int key0 = t * kBN;
            for (int ci = tid; ci < kBN * 16; ci += kThreads) {
                const int r = ci >> 4, c = ci & 15;
                const int key = key0 + r;
                bool ok = key < lk;
                int64_t off = 0;
                if (ok) {
                    const int32_t blk = __ldg(bt_row + key / p.block_size);
                    if (blk < 0 || blk >= p.num_blocks) {
                        report(p.status, PA_ERR_BAD_BLOCK);
                        ok = false;
                    } else {
                        off = ((static_cast<int64_t>(blk) * p.num_kv_heads + kvh) * p.block_size +
                               key % p.block_size) * kD + c * 8;
                    }
                }
                cp_async16(smem_addr(sK[buf]) + swz(r, c), p.k_cache + off, ok);
                cp_async16(smem_addr(sV[buf]) + swz(r, c), p.v_cache + off, ok);
            }
        };
        if (n_tiles > 0) load_kv(0, 0);
        cp_async_commit();

        // ---- per-warp state: 16 rows; lane holds rows g and g+8 ----
        const int g = lane >> 2, t4 = lane & 3;
        const int row_a = i0 + warp * 16 + g;  // query index within the sequence
        const int row_b = row_a + 8;
        float o[16][4];
#pragma unroll
        for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
        uint32_t qa[8][4];

        for (int t = 0; t < n_tiles; ++t) {
            const int buf = t & 1;
            if (t + 1 < n_tiles) load_kv(t + 1, buf ^ 1);
            cp_async_commit();
            cp_async_wait<1>();
            __syncthreads();
            if (t == 0) {
                // Q fragments for this warp's 16 rows, all 8 k-steps
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const int mi = lane >> 3, r = warp * 16 + (lane & 7) + (mi & 1) * 8;
                    ldsm_x4(qa[kk], smem_addr(sQ) + swz(r, kk * 2 + (mi >> 1)));
                }
            }
            // ---- S = Q K^T (16 x 64 per warp) ----
            float s[8][4];
#pragma unroll
            for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
                for (int np = 0; np < 4; ++np) {  // pairs of 8-key blocks
                    uint32_t kb[4];
                    const int mi = lane >> 3;
                    const int key = np * 16 + (lane & 7) + (mi >> 1) * 8;
                    ldsm_x4(kb, smem_addr(sK[buf]) + swz(key, kk * 2 + (mi & 1)));
                    mma16816<DT>(s[2 * np], qa[kk], kb[0], kb[1]);
                    mma16816<DT>(s[2 * np + 1], qa[kk], kb[2], kb[3]);
                }
            }
            // ---- mask + online softmax ----
            const int key0 = t * kBN;
            float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int key = key0 + n * 8 + t4 * 2 + e;
                    const bool va = key < lk && (!p.causal || key <= shift + row_a);
                    const bool vb = key < lk && (!p.causal || key <= shift + row_b);
                    s[n][e] = va ? s[n][e] * p.scale_log2 : -INFINITY;
                    s[n][2 + e] = vb ? s[n][2 + e] * p.scale_log2 : -INFINITY;
                    mx_a = fmaxf(mx_a, s[n][e]);
                    mx_b = fmaxf(mx_b, s[n][2 + e]);
                }
            }
#pragma unroll
            for (int off = 1; off < 4; off <<= 1) {
                mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, off));
                mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, off));
            }
            const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
            const float base_a = mn_a == -INFINITY ? 0.f : mn_a;
            const float base_b = mn_b == -INFINITY ? 0.f : mn_b;
            const float al_a = ex2(m_a - base_a), al_b = ex2(m_b - base_b);
            m_a = mn_a;
            m_b = mn_b;
            float rs_a = 0.f, rs_b = 0.f;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                s[n][0] = ex2(s[n][0] - base_a);
                s[n][1] = ex2(s[n][1] - base_a);
                s[n][2] = ex2(s[n][2] - base_b);
                s[n][3] = ex2(s[n][3] - base_b);
                rs_a += s[n][0] + s[n][1];
                rs_b += s[n][2] + s[n][3];
            }
            l_a = l_a * al_a + rs_a;
            l_b = l_b * al_b + rs_b;
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                o[n][0] *= al_a;
                o[n][1] *= al_a;
                o[n][2] *= al_b;
                o[n][3] *= al_b;
            }
            // ---- O += P V ----
            // P goes to the tensor cores in V's 16-bit type.  fp16 keeps 11
            // significant bits of each weight; bf16 keeps only 8, so for bf16
            // P is carried as hi + lo (two bf16 terms, ~16 bits) and the
            // product is taken twice.
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {  // 16 keys per k-step
                uint32_t pa[4], pl[4];
                split_pair<DT>(s[2 * kk][0], s[2 * kk][1], pa[0], pl[0]);
                split_pair<DT>(s[2 * kk][2], s[2 * kk][3], pa[1], pl[1]);
                split_pair<DT>(s[2 * kk + 1][0], s[2 * kk + 1][1], pa[2], pl[2]);
                split_pair<DT>(s[2 * kk + 1][2], s[2 * kk + 1][3], pa[3], pl[3]);
#pragma unroll
                for (int np = 0; np < 8; ++np) {  // pairs of 8-column blocks of D
                    uint32_t vb[4];
                    const int mi = lane >> 3;
                    const int key = kk * 16 + (lane & 7) + (mi & 1) * 8;
                    ldsm_x4_t(vb, smem_addr(sV[buf]) + swz(key, np * 2 + (mi >> 1)));
                    mma16816<DT>(o[2 * np], pa, vb[0], vb[1]);
                    mma16816<DT>(o[2 * np + 1], pa, vb[2], vb[3]);
                    if constexpr (DT == PA_BF16) {
                        mma16816<DT>(o[2 * np], pl, vb[0], vb[1]);
                        mma16816<DT>(o[2 * np + 1], pl, vb[2], vb[3]);
                    }
                }
            }
            __syncthreads();  // the buffer is refilled next iteration
        }
        cp_async_wait<0>();
        __syncthreads();

        // ---- finish rows: O / l (rows without keys stay 0) ----
        float la = l_a, lb = l_b;  // per-lane partial sums -> row sums
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
            la += __shfl_xor_sync(0xffffffffu, la, off);
            lb += __shfl_xor_sync(0xffffffffu, lb, off);
        }
        const float inv_a = la > 0.f ? 1.f / la : 0.f;
        const float inv_b = lb > 0.f ? 1.f / lb : 0.f;
        uint16_t* out = static_cast<uint16_t*>(p.out);
        if (row_a < lq) {
            uint16_t* dst = out + static_cast<int64_t>(__ldg(p.cu_q + b) + row_a) * hstride + h * kD;
#pragma unroll
            for (int n = 0; n < 16; ++n)
                *reinterpret_cast<uint32_t*>(dst + n * 8 + t4 * 2) = pack2<DT>(o[n][0] * inv_a, o[n][1] * inv_a);
        }
        if (row_b < lq) {
            uint16_t* dst = out + static_cast<int64_t>(__ldg(p.cu_q + b) + row_b) * hstride + h * kD;
#pragma unroll
            for (int n = 0; n < 16; ++n)
                *reinterpret_cast<uint32_t*>(dst + n * 8 + t4 * 2) = pack2<DT>(o[n][2] * inv_b, o[n][3] * inv_b);
        }
    }
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
    if (cache->head_size != kD) return PA_ERR_UNSUPPORTED;
    if (q_dtype != PA_F16 && q_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (cache->kv_dtype != q_dtype) return PA_ERR_UNSUPPORTED;
    const int bs = cache->block_size;
    if (bs != 16 && bs != 32 && bs != 64) return PA_ERR_UNSUPPORTED;
    if (num_seqs > 16384) return PA_ERR_UNSUPPORTED;

    PrefillParams p{};
    p.out = out;
    p.q = static_cast<const uint16_t*>(q);
    p.k_cache = static_cast<const uint16_t*>(cache->k_cache);
    p.v_cache = static_cast<const uint16_t*>(cache->v_cache);
    p.block_table = block_table;
    p.cu_q = cu_seq_lens_q;
    p.cu_k = cu_seq_lens_k;
    p.status = dev_status;
    p.num_blocks = cache->num_blocks;
    p.block_size = bs;
    p.num_kv_heads = cache->num_kv_heads;
    p.num_heads = num_heads;
    p.num_seqs = num_seqs;
    p.max_blocks = max_blocks_per_seq;
    p.max_q = max_seqlen_q;
    p.max_k = max_seqlen_k;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = scale * 1.4426950408889634f;

    const int smem = kQBytes + 4 * kTileBytes + (num_seqs + 1) * 4;
    if (smem > device_max_smem_optin()) return PA_ERR_UNSUPPORTED;
    static LaunchCache cache_bf16, cache_f16;
    auto kern = q_dtype == PA_BF16 ? paged_prefill_mma_kernel<PA_BF16> : paged_prefill_mma_kernel<PA_F16>;
    const int per_sm = blocks_per_sm(kern, kThreads, smem, q_dtype == PA_BF16 ? cache_bf16 : cache_f16);
    if (per_sm <= 0) return PA_ERR_CUDA;
    const int64_t max_items = static_cast<int64_t>(num_seqs) * ((max_seqlen_q + kBM - 1) / kBM) * num_heads;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * per_sm;
    const int grid = static_cast<int>(max_items < cap ? max_items : cap);
    if (grid <= 0) return PA_OK;
    kern<<<grid, kThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(p);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
