// Tree attention (generation phase) and causal prefill (context phase):
// split-KV flash-decode with GQA head stacking, warp-level mma.sync tensor cores.
//
// A single kernel with a topology-aware mask verifies every candidate path at
// once (speculative-decoding survey page, SpecInfer "Token Tree Verifier");
// TensorRT-LLM's attention plugin splits the batch into context and generation
// requests (NVIDIA blog "ReDrafter in TensorRT-LLM", section
// "Inflight-batching Compatible Engine").
//
// Work unit = (request b, kv head h, 64-row query tile, KV split).  The G query
// heads that share kv head h are stacked as rows (row r -> node p = r / G,
// head h*G + r % G), so every K/V byte is read by exactly one CTA per tile.
// Each unit walks its KV positions in chunks of 64: positions [0, C_b) come from
// the KV cache (all visible), positions [C_b, C_b + P_b) are the packed drafts
// (visible iff the node's ancestor-mask bit is set).  Chunks are double-
// buffered in shared memory with cp.async; S = Q K^T and O += P V run on
// mma.sync.m16n8k16 (bf16 in, fp32 accumulate) with an online softmax in exp2
// form.  A unit whose KV is split writes fp32 partials (O, m, l); the CTA that
// takes the last ticket of its (b, h, tile) merges them.  No CTA waits.
#include <cuda_bf16.h>

#include "rd_internal.cuh"

namespace {

constexpr int kChunk = 64;            // KV positions per stage
constexpr int kWarps = 4;             // 16 query rows per warp
constexpr int kRows = 16 * kWarps;    // query rows per tile
constexpr int kThreads = 32 * kWarps;
constexpr float kLog2e = 1.4426950408889634f;

struct AttnArgs {
    bool causal;
    int P_max, Hq, Hkv, G, tiles, splits, split_len, mask_words;
    float scale_log2;
    const uint16_t* q;
    const uint16_t* k_new;
    const uint16_t* v_new;
    const uint16_t* k_cache;
    const uint16_t* v_cache;
    const int64_t* ctx_offsets;
    int64_t total_kv;
    int max_kv;
    const int32_t* lens;       // packed_len [B] (tree) or cu_seqlens [B+1] (causal)
    const uint32_t* mask;
    uint16_t* o;
    float* o_part;             // [units_rows, splits, D]
    float2* ml_part;           // [units_rows, splits]  (m, l)
    unsigned int* tickets;     // [B * Hkv * tiles]
    int32_t* status;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid)
{
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
        "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// byte offset of 16-byte chunk c of row r in a [kChunk][D] bf16 tile, XOR-swizzled
template <int D>
__device__ __forceinline__ uint32_t tile_off(int r, int c)
{
    return (uint32_t)(r * (D * 2) + ((c ^ (r & 7)) << 4));
}

// Row geometry of one unit.
struct Unit {
    int b, h, tile, split;
    int n_rows;        // valid rows in the whole (b, h): P_b*G (tree) or T_b*G (causal)
    int64_t kv_base;   // first cache row of this request (tree) / sequence (causal)
    int C;             // context length (tree); 0 (causal)
    int Pb;            // packed length (tree); sequence length (causal)
    int n_pos;         // KV positions of the unit's (b, h): C + Pb (tree) or Tb (causal)
};

// Source row of KV position j of a unit, or nullptr if j is beyond the sequence.
template <int D>
__device__ __forceinline__ const uint16_t* kv_row(const AttnArgs& a, const Unit& u, int j,
                                                  bool is_v)
{
    if (a.causal) {
        if (j >= u.Pb) return nullptr;
        const uint16_t* base = is_v ? a.v_new : a.k_new;
        return base + ((size_t)(u.kv_base + j) * a.Hkv + u.h) * D;
    }
    if (j < u.C) {
        const uint16_t* base = is_v ? a.v_cache : a.k_cache;
        return base + ((size_t)(u.kv_base + j) * a.Hkv + u.h) * D;
    }
    if (j < u.C + u.Pb) {
        const uint16_t* base = is_v ? a.v_new : a.k_new;
        return base + (((size_t)u.b * a.P_max + (j - u.C)) * a.Hkv + u.h) * D;
    }
    return nullptr;
}

template <int D>
__device__ __forceinline__ void load_chunk(const AttnArgs& a, const Unit& u, int pos0,
                                           uint16_t* sk, uint16_t* sv, int tid)
{
    constexpr int kPieces = D / 8;     // 16-byte pieces per row
    const uint32_t k_s = smem_u32(sk), v_s = smem_u32(sv);
    for (int idx = tid; idx < kChunk * kPieces; idx += kThreads) {
        const int r = idx / kPieces, c = idx % kPieces;
        const uint16_t* ks = kv_row<D>(a, u, pos0 + r, false);
        const uint16_t* vs = kv_row<D>(a, u, pos0 + r, true);
        const bool ok = ks != nullptr;
        cp_async16(k_s + tile_off<D>(r, c), ok ? ks + c * 8 : a.q, ok);
        cp_async16(v_s + tile_off<D>(r, c), ok ? vs + c * 8 : a.q, ok);
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads)
attention_kernel(const AttnArgs a)
{
    constexpr int KS = D / 16;         // k-steps of QK^T
    constexpr int NT = D / 8;          // n-tiles of PV
    extern __shared__ __align__(128) unsigned char smem[];
    uint16_t* sk[2] = {reinterpret_cast<uint16_t*>(smem),
                       reinterpret_cast<uint16_t*>(smem + kChunk * D * 2)};
    uint16_t* sv[2] = {reinterpret_cast<uint16_t*>(smem + 2 * kChunk * D * 2),
                       reinterpret_cast<uint16_t*>(smem + 3 * kChunk * D * 2)};
    __shared__ int s_last;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;

    Unit u;
    u.b = blockIdx.z;
    u.h = blockIdx.y;
    u.tile = blockIdx.x / a.splits;
    u.split = blockIdx.x % a.splits;
    bool bad = false;
    if (a.causal) {
        const int s0 = a.lens[u.b], s1 = a.lens[u.b + 1];
        u.kv_base = s0;
        u.C = 0;
        u.Pb = s1 - s0;
        bad = u.Pb < 0 || u.Pb > a.max_kv || s1 > a.total_kv;
        u.n_pos = u.Pb;
    } else {
        const int64_t c0 = a.ctx_offsets[u.b], c1 = a.ctx_offsets[u.b + 1];
        u.kv_base = c0;
        u.C = (int)(c1 - c0);
        u.Pb = a.lens[u.b];
        bad = c1 < c0 || c1 - c0 > a.max_kv || c1 > a.total_kv || u.Pb < 0 || u.Pb > a.P_max;
        u.n_pos = u.C + u.Pb;
    }
    if (bad) {
        if (tid == 0 && u.tile == 0 && u.split == 0 && u.h == 0) rd_flag(a.status, RD_DEV_BAD_LENGTH);
        u.Pb = 0;
        u.C = 0;
        u.n_pos = 0;
    }
    u.n_rows = u.Pb * a.G;
    const int row0 = u.tile * kRows;                       // first row of the tile
    const int hq0 = u.h * a.G;

    // ---- tiles without valid rows: padded tree rows are written as zeros --------
    if (row0 >= u.n_rows) {
        if (!a.causal && u.split == 0) {
            for (int idx = tid; idx < kRows * (D / 8); idx += kThreads) {
                const int r = row0 + idx / (D / 8), c = idx % (D / 8);
                const int p = r / a.G;
                if (p < a.P_max)
                    reinterpret_cast<uint4*>(a.o + (((size_t)u.b * a.P_max + p) * a.Hq + hq0 +
                                                    r % a.G) * D)[c] = make_uint4(0, 0, 0, 0);
            }
        }
        return;
    }

    // ---- KV range of this unit ------------------------------------------------------
    int pos_begin, pos_end, n_splits;
    if (a.causal) {
        const int last_row = min(u.n_rows, row0 + kRows) - 1;
        pos_begin = 0;
        pos_end = last_row / a.G + 1;                      // keys 0..t_max
        n_splits = 1;
    } else {
        n_splits = (u.n_pos + a.split_len - 1) / a.split_len;
        pos_begin = u.split * a.split_len;
        pos_end = min(u.n_pos, pos_begin + a.split_len);
    }
    if (u.split >= n_splits) return;

    // ---- query fragments (rows g and g+8 of this warp's 16) ------------------------
    const int wr0 = row0 + warp * 16;
    const int rA = wr0 + g, rB = wr0 + g + 8;
    const bool vA = rA < u.n_rows, vB = rB < u.n_rows;
    const bool warp_live = wr0 < u.n_rows;
    auto q_ptr = [&](int r) -> const uint16_t* {
        const int p = r / a.G, hq = hq0 + r % a.G;
        if (a.causal) return a.q + ((size_t)(u.kv_base + p) * a.Hq + hq) * D;
        return a.q + (((size_t)u.b * a.P_max + p) * a.Hq + hq) * D;
    };
    uint32_t qf[KS][4];
    {
        const uint32_t* qa = vA ? reinterpret_cast<const uint32_t*>(q_ptr(rA)) : nullptr;
        const uint32_t* qb = vB ? reinterpret_cast<const uint32_t*>(q_ptr(rB)) : nullptr;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int c0 = ks * 8 + t4;                    // 32-bit word index (2 bf16)
            qf[ks][0] = qa ? __ldg(qa + c0) : 0u;
            qf[ks][1] = qb ? __ldg(qb + c0) : 0u;
            qf[ks][2] = qa ? __ldg(qa + c0 + 4) : 0u;
            qf[ks][3] = qb ? __ldg(qb + c0 + 4) : 0u;
        }
    }
    // query position (for masks): tree -> packed node p; causal -> token t
    const int pA = rA / a.G, pB = rB / a.G;

    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;

    const int n_chunks = (pos_end - pos_begin + kChunk - 1) / kChunk;
    if (n_chunks > 0) load_chunk<D>(a, u, pos_begin, sk[0], sv[0], tid);
    cp_async_commit();

    for (int ci = 0; ci < n_chunks; ++ci) {
        const int st = ci & 1;
        const int pos0 = pos_begin + ci * kChunk;
        cp_async_wait_all();
        __syncthreads();
        if (ci + 1 < n_chunks) load_chunk<D>(a, u, pos0 + kChunk, sk[st ^ 1], sv[st ^ 1], tid);
        cp_async_commit();
        if (!warp_live) continue;

        // S = Q K^T for 64 positions
        float s[kChunk / 8][4];
#pragma unroll
        for (int n = 0; n < kChunk / 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
        const uint32_t kbase = smem_u32(sk[st]);
#pragma unroll
        for (int n = 0; n < kChunk / 8; ++n) {
#pragma unroll
            for (int ks = 0; ks < KS; ks += 2) {
                uint32_t b0, b1, b2, b3;
                const int r = n * 8 + (lane & 7);
                const int c = ks * 2 + (lane >> 3);
                ldsm_x4(kbase + tile_off<D>(r, c), b0, b1, b2, b3);
                mma16816(s[n], qf[ks], b0, b1);
                mma16816(s[n], qf[ks + 1], b2, b3);
            }
        }
        // scale (log2 domain) and mask
        // chunks entirely visible to both rows of this thread skip the mask
        const bool full = a.causal ? (pos0 + kChunk - 1 <= min(pA, pB) && pos0 + kChunk <= pos_end)
                                   : (pos0 + kChunk <= min(u.C, pos_end));
#pragma unroll
        for (int n = 0; n < kChunk / 8; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float x = s[n][e] * a.scale_log2;
                if (!full) {
                    const int j = pos0 + n * 8 + 2 * t4 + (e & 1);
                    const int qp = (e < 2) ? pA : pB;
                    const bool live = (e < 2) ? vA : vB;
                    bool vis;
                    if (j >= pos_end || !live) vis = false;
                    else if (a.causal) vis = j <= qp;
                    else if (j < u.C) vis = true;
                    else {
                        const int k = j - u.C;
                        const uint32_t w = __ldg(a.mask + ((size_t)u.b * a.P_max + qp) *
                                                              a.mask_words + (k >> 5));
                        vis = (w >> (k & 31)) & 1u;
                    }
                    if (!vis) x = -INFINITY;
                }
                s[n][e] = x;
            }
        }
        // online softmax (rows A = g, B = g + 8)
        float cA = -INFINITY, cB = -INFINITY;
#pragma unroll
        for (int n = 0; n < kChunk / 8; ++n) {
            cA = fmaxf(cA, fmaxf(s[n][0], s[n][1]));
            cB = fmaxf(cB, fmaxf(s[n][2], s[n][3]));
        }
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
            cA = fmaxf(cA, __shfl_xor_sync(0xffffffffu, cA, off));
            cB = fmaxf(cB, __shfl_xor_sync(0xffffffffu, cB, off));
        }
        const float nA = fmaxf(mA, cA), nB = fmaxf(mB, cB);
        const float baseA = (nA == -INFINITY) ? 0.f : nA;
        const float baseB = (nB == -INFINITY) ? 0.f : nB;
        const float alA = exp2f(mA - baseA), alB = exp2f(mB - baseB);
        mA = nA;
        mB = nB;
        lA *= alA;
        lB *= alB;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            acc[n][0] *= alA; acc[n][1] *= alA;
            acc[n][2] *= alB; acc[n][3] *= alB;
        }
        uint32_t pf[kChunk / 16][4];
#pragma unroll
        for (int n = 0; n < kChunk / 8; ++n) {
            const float p0 = exp2f(s[n][0] - baseA), p1 = exp2f(s[n][1] - baseA);
            const float p2 = exp2f(s[n][2] - baseB), p3 = exp2f(s[n][3] - baseB);
            lA += p0 + p1;
            lB += p2 + p3;
            const int kk = n >> 1;
            if ((n & 1) == 0) {
                pf[kk][0] = pack_bf16(p0, p1);
                pf[kk][1] = pack_bf16(p2, p3);
            } else {
                pf[kk][2] = pack_bf16(p0, p1);
                pf[kk][3] = pack_bf16(p2, p3);
            }
        }
        // O += P V
        const uint32_t vbase = smem_u32(sv[st]);
#pragma unroll
        for (int kk = 0; kk < kChunk / 16; ++kk) {
#pragma unroll
            for (int n = 0; n < NT; n += 2) {
                uint32_t b0, b1, b2, b3;
                const int r = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = n + (lane >> 4);
                ldsm_x4_t(vbase + tile_off<D>(r, c), b0, b1, b2, b3);
                mma16816(acc[n], pf[kk], b0, b1);
                mma16816(acc[n + 1], pf[kk], b2, b3);
            }
        }
    }
    cp_async_wait_all();

    // row sums across the quad
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
        lA += __shfl_xor_sync(0xffffffffu, lA, off);
        lB += __shfl_xor_sync(0xffffffffu, lB, off);
    }

    auto out_ptr = [&](int r) -> uint16_t* {
        const int p = r / a.G, hq = hq0 + r % a.G;
        if (a.causal) return a.o + ((size_t)(u.kv_base + p) * a.Hq + hq) * D;
        return a.o + (((size_t)u.b * a.P_max + p) * a.Hq + hq) * D;
    };

    if (n_splits == 1) {
        // rows of this tile beyond n_rows (tree): zero them
        if (warp_live || !a.causal) {
            const float iA = (vA && lA > 0.f) ? 1.f / lA : 0.f;
            const float iB = (vB && lB > 0.f) ? 1.f / lB : 0.f;
            const bool wA = vA || (!a.causal && rA / a.G < a.P_max);
            const bool wB = vB || (!a.causal && rB / a.G < a.P_max);
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const int d = n * 8 + 2 * t4;
                if (wA) *reinterpret_cast<uint32_t*>(out_ptr(rA) + d) =
                        pack_bf16(acc[n][0] * iA, acc[n][1] * iA);
                if (wB) *reinterpret_cast<uint32_t*>(out_ptr(rB) + d) =
                        pack_bf16(acc[n][2] * iB, acc[n][3] * iB);
            }
        }
        return;
    }

    // ---- split-KV: write fp32 partials, last CTA of (b, h, tile) merges ----------
    const size_t unit_id = ((size_t)u.b * a.Hkv + u.h) * a.tiles + u.tile;
    const size_t prow0 = unit_id * kRows;
    {
        const int lrA = warp * 16 + g, lrB = lrA + 8;
        float* oA = a.o_part + ((prow0 + lrA) * a.splits + u.split) * D;
        float* oB = a.o_part + ((prow0 + lrB) * a.splits + u.split) * D;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const int d = n * 8 + 2 * t4;
            *reinterpret_cast<float2*>(oA + d) = make_float2(acc[n][0], acc[n][1]);
            *reinterpret_cast<float2*>(oB + d) = make_float2(acc[n][2], acc[n][3]);
        }
        if (t4 == 0) {
            a.ml_part[(prow0 + lrA) * a.splits + u.split] = make_float2(mA, lA);
            a.ml_part[(prow0 + lrB) * a.splits + u.split] = make_float2(mB, lB);
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned t = atomicAdd(a.tickets + unit_id, 1u);
        s_last = (t == (unsigned)n_splits - 1u);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int idx = tid; idx < kRows * D; idx += kThreads) {
        const int lr = idx / D, d = idx % D;
        const int r = row0 + lr;
        if (r / a.G >= a.P_max) continue;
        float M = -INFINITY;
        for (int sp = 0; sp < n_splits; ++sp) M = fmaxf(M, __ldcg(&a.ml_part[(prow0 + lr) * a.splits + sp].x));
        float Lsum = 0.f, O = 0.f;
        if (r < u.n_rows && M != -INFINITY) {
            for (int sp = 0; sp < n_splits; ++sp) {
                const float2 ml = __ldcg(&a.ml_part[(prow0 + lr) * a.splits + sp]);
                if (ml.x == -INFINITY) continue;
                const float w = exp2f(ml.x - M);
                Lsum += ml.y * w;
                O += __ldcg(&a.o_part[((prow0 + lr) * a.splits + sp) * D + d]) * w;
            }
        }
        const float val = (r < u.n_rows && Lsum > 0.f) ? O / Lsum : 0.f;
        if (r < u.n_rows || !a.causal) {
            __nv_bfloat16 hv = __float2bfloat16_rn(val);
            out_ptr(r)[d] = *reinterpret_cast<uint16_t*>(&hv);
        }
    }
    if (tid == 0) a.tickets[unit_id] = 0u;
}

}  // namespace

rd_attn_plan rd_attn_make_plan(bool causal, int B, int P_max, int Hq, int Hkv, int D,
                               int max_kv)
{
    (void)D;
    rd_attn_plan plan;
    const int G = Hq / Hkv;
    const long rows = causal ? (long)max_kv * G : (long)P_max * G;
    plan.tiles = (int)((rows + kRows - 1) / kRows);
    if (plan.tiles < 1) plan.tiles = 1;
    const long span = causal ? (long)max_kv : (long)max_kv + P_max;
    const long base_units = (long)B * Hkv * plan.tiles;
    const long target = 4L * 152;
    int splits = 1;
    long split_len = ((span + kChunk - 1) / kChunk) * kChunk;
    if (!causal && base_units < target) {
        long want = (target + base_units - 1) / base_units;
        long len = (span + want - 1) / want;
        if (len < 256) len = 256;
        len = ((len + kChunk - 1) / kChunk) * kChunk;
        split_len = len;
        splits = (int)((span + len - 1) / len);
    }
    if (split_len < kChunk) split_len = kChunk;
    plan.splits = splits < 1 ? 1 : splits;
    plan.split_len = (int)split_len;
    if (plan.splits > 1) {
        const size_t unit_rows = (size_t)B * Hkv * plan.tiles * kRows;
        plan.ws_bytes = unit_rows * plan.splits * (size_t)D * sizeof(float) +
                        unit_rows * plan.splits * sizeof(float2) +
                        (size_t)B * Hkv * plan.tiles * sizeof(unsigned int);
    } else {
        plan.ws_bytes = 0;
    }
    return plan;
}

cudaError_t rd_launch_attention(bool causal, const rd_attn_plan& plan, int B, int P_max,
                                int Hq, int Hkv, int D, float scale, const void* q,
                                const void* k_new, const void* v_new,
                                const void* k_cache, const void* v_cache,
                                const int64_t* ctx_offsets, int64_t total_kv, int max_kv,
                                const int32_t* lens, const uint32_t* mask, int mask_words,
                                void* o, void* workspace, int32_t* dev_status,
                                cudaStream_t stream)
{
    AttnArgs a;
    a.causal = causal;
    a.P_max = P_max;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.tiles = plan.tiles;
    a.splits = plan.splits;
    a.split_len = plan.split_len;
    a.mask_words = mask_words;
    a.scale_log2 = scale * kLog2e;
    a.q = static_cast<const uint16_t*>(q);
    a.k_new = static_cast<const uint16_t*>(k_new);
    a.v_new = static_cast<const uint16_t*>(v_new);
    a.k_cache = static_cast<const uint16_t*>(k_cache);
    a.v_cache = static_cast<const uint16_t*>(v_cache);
    a.ctx_offsets = ctx_offsets;
    a.total_kv = total_kv;
    a.max_kv = max_kv;
    a.lens = lens;
    a.mask = mask;
    a.o = static_cast<uint16_t*>(o);
    a.status = dev_status;
    a.o_part = nullptr;
    a.ml_part = nullptr;
    a.tickets = nullptr;
    if (plan.splits > 1) {
        const size_t unit_rows = (size_t)B * Hkv * plan.tiles * kRows;
        a.o_part = static_cast<float*>(workspace);
        a.ml_part = reinterpret_cast<float2*>(a.o_part + unit_rows * plan.splits * D);
        a.tickets = reinterpret_cast<unsigned int*>(a.ml_part + unit_rows * plan.splits);
    }
    dim3 grid((unsigned)(plan.tiles * plan.splits), (unsigned)Hkv, (unsigned)B);
    const size_t smem = 4 * (size_t)kChunk * D * 2;
    if (D == 128) {
        cudaError_t e = cudaFuncSetAttribute(attention_kernel<128>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        attention_kernel<128><<<grid, kThreads, smem, stream>>>(a);
    } else {
        attention_kernel<64><<<grid, kThreads, smem, stream>>>(a);
    }
    return cudaGetLastError();
}
