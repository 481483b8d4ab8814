// Tree attention (generation phase) on the 5th-generation tensor cores: TMA-fed,
// tcgen05 MMA with TMEM accumulators, persistent.
//
// A single kernel with a topology-aware mask verifies every candidate path at once
// (speculative-decoding survey page, SpecInfer "Token Tree Verifier").  The context
// phase of an in-flight batch (NVIDIA blog "ReDrafter in TensorRT-LLM", section
// "Inflight-batching Compatible Engine") runs in the paired-tile causal kernel.
//
// Work unit = (request b, kv head h, 128-row query tile, KV split).  The G query
// heads that share kv head h are stacked as rows (row r -> node p = r / G, head
// h*G + r % G), so each K/V byte is read once per tile.
// A unit walks its KV chunks (64 positions): the context (all visible, the last
// chunk ragged), then the packed drafts (visible iff the node's ancestor-mask
// bit is set).  Persistent CTAs, two per SM, take units round-robin in
// tile-major order.
//
// Warp roles (256 threads; warpgroup 1 gives registers to warpgroup 0):
//   warps 0-3  softmax: row r is TMEM lane r (a tile of <= 64 valid rows puts a
//              row in two lanes, each taking half of a chunk's columns).  Turn S
//              into 16-bit P written over S in TMEM (online softmax in exp2
//              form, O rescaled only when a row maximum grows by more than 2^8),
//              and write the output rows.
//   warp 4     producer: TMA loads (128-byte swizzle) of K and V chunks.
//   warp 5     MMA issuer and TMEM owner: S = Q K^T (M=128, N=64, K=D) and
//              O += P V (M=128, N=D, K=64; A = P in TMEM).
//   warps 6-7  FP8: widen e4m3 chunks into the 16-bit ring; 16-bit paths:
//              warp 6 loads the query tiles into shared memory (TMA).
// The 16-bit path (template flag PIPE) keeps two S tiles in TMEM and issues S of
// chunk j+1 before PV of chunk j, so the tensor core computes the next scores
// while the softmax warps work; its queries sit in shared memory and K and V
// have separate rings (a K stage frees as soon as S has read it).  The FP8 path
// keeps one S tile with the queries in TMEM (written by its softmax warps) and
// issues S of a chunk right behind PV of the one before.
// FP8 variant (template flag F8; context K/V stored as e4m3 with per-tensor
// scales): the producer TMA-loads e4m3 context chunks into an 8-bit ring; warps
// 6-7 widen them (exactly) into the 16-bit ring the MMA reads, and convert the
// bf16 draft chunks, divided by the scales, the same way.  The MMA runs kind::f16
// with f16 operands (e4m3 widens to f16 exactly; both operands of one MMA share
// a type); the K scale is folded into the softmax scale, the V scale into the
// output normalisation.
// Every wait is bounded by a clock budget; on expiry the CTA records RD_DEV_TIMEOUT,
// drains its in-flight copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "attn_common.cuh"
#include "rd_internal.cuh"
#include "tc_ptx.cuh"

namespace {
using namespace rdtc;
using namespace rdattn;

constexpr int kM = 128;                    // query rows per tile = TMEM lanes
constexpr int kN = 64;                     // KV positions per chunk
constexpr int kCtasPerSm = 2;              // two independent pipelines per SM
constexpr int kSoftmaxWarps = 4;           // warpgroup 0
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
// Warpgroup 1: producer, MMA issuer (S and PV), two FP8 converter warps (idle in bf16).
constexpr int kThreads = kSoftmaxThreads + 128;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;                // S and PV issuer and TMEM owner
constexpr int kConvWarp0 = 6;              // FP8: converter warps 6 and 7; else warp 6 writes queries
// Register split (setmaxnreg): two CTAs of 256 threads share an SM, so each CTA
// launches with 128 registers per thread, 32,768 in all; warpgroup 1 gives back
// down to kRegsOther and the softmax warpgroup takes kRegsSoftmax:
// 128 x (192 + 64) = 32,768, and two CTAs' (192 + 64) registers x 32 lanes fit
// one SM sub-partition's 16,384.
constexpr int kRegsLaunch = 128;
constexpr int kRegsSoftmax = 192;
constexpr int kRegsOther = 64;
static_assert(128 * (kRegsSoftmax + kRegsOther) <= kThreads * kRegsLaunch, "register split");
static_assert(32 * kCtasPerSm * (kRegsSoftmax + kRegsOther) <= 16384, "register split per sub-partition");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when a max grows by > 2^8
constexpr long long kWaitBudget = 4000000000LL;   // ~2 s of SM clock per wait
constexpr int kSkMaxB = 480;               // chunk-range division up to this many requests
constexpr uint32_t kSkMinChunks = 8;       // chunks per CTA at least (chunk-range division)

template <int D, bool F8 = false, bool PIPE = false> struct Cfg {
    // PIPE (the 16-bit path) pipelines S: two S tiles in tensor memory, so that S
    // of the next chunk is computed while the softmax warps work on this one,
    // with the queries in shared memory.  FP8 (whose shared memory holds the
    // 8-bit ring): one S tile and the queries in tensor memory.
    static_assert(F8 != PIPE, "every instantiation is the 16-bit pipelined path or the FP8 path");
    static constexpr bool kPipe = PIPE;
    static constexpr bool kMaySk = PIPE || F8;          // tree attention (chunk ranges possible)
    static constexpr int kNc = kN;                      // KV positions per chunk
    static constexpr int kDB = D / 64;                  // 64-element (128-byte) column blocks
    static constexpr int kKBytes = kNc * D * 2;         // one K (or V) chunk
    // PIPE: separate K and V rings (a K stage is free once S has read it, so K
    // loads run ahead of the V loads) and the query tile.  Otherwise one ring of
    // K + V stages (16-bit), and for FP8 the 8-bit ring of context chunks.
    // The 16-bit path takes its query tiles by TMA into shared memory (warp 6).
    static constexpr bool kQTma = PIPE;
    static constexpr int kStages = F8 ? 2 : (D == 128 ? 2 : 4);
    static constexpr int kF8Stages = F8 ? 2 : 0;
    static constexpr int kF8Ring = kF8Stages > 0 ? kF8Stages : 1;   // ring index modulus
    static constexpr int kStageBytes = PIPE ? kKBytes : 2 * kKBytes;
    static constexpr int kF8Bytes = 2 * kNc * D;        // one 8-bit K + V chunk
    static constexpr int kStageOff = 0;                 // FP8: K + V stages; else K stages
    static constexpr int kVOff = kStageOff + kStages * kStageBytes;    // V stages (16-bit path)
    static constexpr int kF8Off = kVOff + (PIPE ? kStages * kKBytes : 0);
    static constexpr int kQOff = kF8Off + kF8Stages * kF8Bytes;
    static constexpr int kQBytes = kQTma ? kM * D * 2 : 0;             // [D / 64][128 rows][128 B]
    static constexpr int kBarOff = kQOff + kQBytes;
    // chunk-range table: per request the prefix of live chunks and chunks per unit
    static constexpr int kSkOff = kBarOff + 512;
    static constexpr int kSkBytes = (2 * kSkMaxB + 1) * 4;
    static constexpr int kSmemBytes = kSkOff + kSkBytes + 1024;   // + alignment slack
    static_assert(kSmemBytes <= 113 * 1024, "two CTAs per SM");
    // Tensor memory (32-bit columns x 128 lanes), a quarter of the SM's per CTA:
    // S tiles, with P (16-bit pairs, the A operand of PV) written over the first
    // half of its tile once S is in registers; the O accumulator; (FP8) the
    // tile's queries (16-bit pairs, the A operand of S).
    static constexpr uint32_t kTmemCols = 256;
    static constexpr uint32_t kSCol = 0;                // S tile b at kSCol + b * kNc
    static constexpr uint32_t kOCol = kPipe ? 2 * kNc : kNc;   // D (<= 128) columns
    static constexpr uint32_t kQCol = kOCol + 128;      // FP8: D / 2 (<= 64) columns
    static_assert(kPipe ? kOCol + 128 <= kTmemCols : kQCol + 64 <= kTmemCols, "tensor memory layout");
};

struct TcArgs {
    int B, P_max, Hq, Hkv, G, tiles, mask_words, n_units;   // n_units = B * Hkv * tiles
    // Work division.  Chunk ranges (tree attention, B <= kSkMaxB): the live units'
    // chunks, in request / tile / kv-head order, are one sequence of W chunks,
    // and CTA c takes chunks [c W / grid, (c + 1) W / grid); a unit cut by such a
    // boundary is computed in pieces whose fp32 partials the last piece to finish
    // merges.  Otherwise whole units, round-robin in tile-major order.
    bool sk;
    float scale_log2;
    const uint16_t* q;
    const int64_t* ctx_offsets;
    int64_t total_kv;
    int max_kv;
    const int32_t* lens;
    const uint32_t* mask;
    uint16_t* o;
    float* o_part;
    float2* ml_part;
    int4* sk_desc;           // chunk ranges: per CTA, the cut unit its range starts inside (merge)
    int32_t* status;
    // paged context (block_table != nullptr): position j of request b is row
    // j % page_size of page block_table[b * max_pages + j / page_size]
    const int32_t* block_table;
    const int32_t* ctx_lens;
    int max_pages, page_size, num_pages;
    // FP8 variant: draft K/V (bf16, converted by the converter warps), the
    // reciprocal scales applied to them, and the V scale of the output
    const uint16_t* k_new;
    const uint16_t* v_new;
    float k_inv, v_inv, out_scale;
    // failure-detection test hook: > 0 makes the MMA issuer first wait, with
    // this clock budget, on a barrier that nothing completes
    long long stall_budget;
    // 16-bit path: the query tiles come by TMA (G a power of two <= 16) through
    // map_q128 (boxes of 128 / G rows x G heads x 64 columns) and map_q16 (16 / G
    // rows), else by plain loads of warp 6
    bool q_tma;
};

struct Barriers {
    uint64_t kv_full[8];     // FP8: K + V stages; 16-bit path: K stages
    uint64_t kv_empty[8];
    uint64_t v_full[4];      // 16-bit path: V stages
    uint64_t v_empty[4];
    uint64_t s_full[2];      // S of a chunk is in its tensor-memory tile (FP8: tile 0 only)
    uint64_t pv_done[2];     // 16-bit path: PV of a chunk of that S tile has completed
    uint64_t p_full[2];      // P of a chunk is written over its S tile (softmax warps)
    uint64_t o_final;        // PV of the unit's last chunk has completed
    uint64_t o_free;         // the epilogue has read O (softmax warps)
    uint64_t q_full;         // the unit's queries are written (FP8: softmax warps; else loader warps)
    uint64_t q_free;         // every S MMA of the unit has completed
    uint64_t drain;
    uint64_t f8_full[4];
    uint64_t f8_empty[4];
    uint64_t never;          // completed by nobody (failure-detection test hook)
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Barriers) <= 512, "barrier block");

// Geometry of one work item (a whole unit, or the piece of a unit that one CTA
// takes), computed identically by every role.
struct UnitGeo {
    int b, h, tile;
    bool live;            // has chunks to process
    bool zero_tile;       // tree tile without valid rows: write zeros
    int n_rows;           // valid rows of (b, h)
    int64_t kv_base;      // first row of this request / sequence in the K/V map
    int C;                // context length
    int Pb;               // packed length
    int c_first, n_ctx;   // first context chunk and number of context chunks
    int d_first, n_draft; // first draft chunk and number of draft chunks
    // a piece of a cut unit and its partial slot (2 blockIdx.x, or 2 blockIdx.x
    // + 1 when the unit starts inside this CTA's range and runs past its end)
    bool cut;
    int split;
};

// Lengths of request b; false (and zero lengths) if they are invalid.
__device__ __forceinline__ bool req_geo(const TcArgs& a, int b, UnitGeo& g)
{
    bool bad;
    g.Pb = a.lens[b];
    if (a.block_table != nullptr) {
        const int c = a.ctx_lens[b];
        g.kv_base = 0;
        g.C = c;
        bad = c < 0 || c > a.max_kv || (long long)c > (long long)a.max_pages * a.page_size ||
              g.Pb < 0 || g.Pb > a.P_max;
    } else {
        const int64_t c0 = a.ctx_offsets[b], c1 = a.ctx_offsets[b + 1];
        g.kv_base = c0;
        g.C = (int)(c1 - c0);
        bad = c0 < 0 || c1 < c0 || c1 - c0 > a.max_kv || c1 > a.total_kv || g.Pb < 0 ||
              g.Pb > a.P_max;
    }
    if (bad) { g.C = 0; g.Pb = 0; }
    g.n_rows = g.Pb * a.G;
    return !bad;
}

// Whole unit u (round-robin division).  Units run tile-major, then request and
// kv head: the CTAs take units round-robin, and this order puts the tiles past
// the valid rows of a tree batch (mostly padding) last instead of interleaving
// them with the live units.
template <int NC>
__device__ __forceinline__ UnitGeo unit_geo(const TcArgs& a, int u)
{
    UnitGeo g;
    const int bh = a.B * a.Hkv;
    g.tile = u / bh;
    g.b = (u % bh) / a.Hkv;
    g.h = u % a.Hkv;
    g.live = false;
    g.zero_tile = false;
    g.c_first = g.n_ctx = g.d_first = g.n_draft = 0;
    g.cut = false;
    g.split = 0;
    const bool ok = req_geo(a, g.b, g);
    const int row0 = g.tile * kM;
    if (row0 >= g.n_rows) {
        g.zero_tile = row0 < a.P_max * a.G;
    } else {
        g.live = true;
        g.n_ctx = (g.C + NC - 1) / NC;
        g.n_draft = (g.Pb + NC - 1) / NC;
    }
    if (!ok && g.h == 0 && g.tile == 0 && threadIdx.x == 0) rd_flag(a.status, RD_DEV_BAD_LENGTH);
    return g;
}

// Chunk-range division over n = min(grid, W / kSkMinChunks) CTAs (at least one;
// no range is empty, and none is so short that its pieces' partials and merge
// cost more than the chunks): CTA c < n starts at chunk floor(c W / n).
__device__ __forceinline__ uint32_t sk_ctas(uint32_t W)
{
    return max(1u, min((uint32_t)gridDim.x, W / kSkMinChunks));
}
__device__ __forceinline__ uint32_t sk_start(uint32_t W, int c)
{
    return (uint32_t)(((uint64_t)c * W) / sk_ctas(W));
}

// The table: pre[b] = live chunks of requests before b (pre[B] = W), nb[b] =
// chunks of one unit of request b (its context and draft chunks; zero without
// valid rows), tiles of request b = (pre[b + 1] - pre[b]) / (Hkv nb[b]).  Built by
// one warp before the roles start.
template <int NC>
__device__ void sk_build(const TcArgs& a, uint32_t* pre, uint32_t* nb, int lane)
{
    uint32_t carry = 0;
    for (int b0 = 0; b0 < a.B; b0 += 32) {
        const int b = b0 + lane;
        uint32_t w = 0;
        if (b < a.B) {
            UnitGeo g;
            if (!req_geo(a, b, g)) rd_flag(a.status, RD_DEV_BAD_LENGTH);
            const int tiles = (g.n_rows + kM - 1) / kM;
            const uint32_t n = tiles > 0 ? (uint32_t)((g.C + NC - 1) / NC + (g.Pb + NC - 1) / NC) : 0u;
            nb[b] = n;
            w = (uint32_t)(a.Hkv * tiles) * n;
        }
        uint32_t incl = w;                                   // inclusive warp scan
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += y;
        }
        if (b < a.B) pre[b + 1] = carry + incl;
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) pre[0] = 0;
    __syncwarp();
    // This CTA's merge descriptor: when its range starts inside a unit that began
    // in the previous CTA's range, that unit is cut and this CTA names it for the
    // merge kernel (unit id in tile-major order, its first CTA c0, its number of
    // pieces, whether it starts inside c0's range, its request's packed length).
    if (lane == 0) {
        int4 d = make_int4(-1, 0, 0, 0);
        const uint32_t W = carry;
        const uint32_t n = W > 0 ? sk_ctas(W) : 0u;
        const int c = blockIdx.x;
        if (c >= 1 && (uint32_t)c < n) {
            const uint32_t x = sk_start(W, c);
            int lo = 0, hi = a.B - 1;                       // last b with pre[b] <= x
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (pre[mid] <= x) lo = mid; else hi = mid - 1;
            }
            const uint32_t n_b = nb[lo];
            const uint32_t k = (x - pre[lo]) / n_b;
            const uint32_t U0 = pre[lo] + k * n_b;
            const uint32_t prev = sk_start(W, c - 1);
            if (U0 < x && U0 >= prev) {
                const int tile = (int)(k / a.Hkv), h = (int)(k % a.Hkv);
                const uint32_t last = U0 + n_b - 1;
                const int c1 = (int)((((uint64_t)last + 1) * n - 1) / W);
                d.x = (tile * a.B + lo) * a.Hkv + h;
                d.y = c - 1;
                d.z = (c1 - (c - 1) + 1) | (U0 > prev ? (1 << 30) : 0);
                d.w = a.lens[lo];
            }
        }
        a.sk_desc[c] = d;
    }
}

// Cursor over this CTA's work: a unit index (round-robin) or a chunk position.
struct Work {
    int u;
    uint32_t x;
};
template <bool MAYSK>
__device__ __forceinline__ Work work_begin(const TcArgs& a, const uint32_t* pre)
{
    Work w;
    w.u = blockIdx.x;
    w.x = 0u;
    if (MAYSK && a.sk) {
        const uint32_t W = pre[a.B];
        w.x = blockIdx.x < sk_ctas(W) ? sk_start(W, blockIdx.x) : W;   // W: no work
    }
    return w;
}

// The CTA's next work item into g (round-robin: every unit, live or not; chunk
// ranges: pieces of live units only); false when the CTA's work is done.
template <int NC, bool MAYSK>
__device__ __forceinline__ bool work_next(const TcArgs& a, const uint32_t* pre, const uint32_t* nb,
                                          Work& w, UnitGeo& g)
{
    if (!(MAYSK && a.sk)) {
        if (w.u >= a.n_units) return false;
        g = unit_geo<NC>(a, w.u);
        w.u += gridDim.x;
        return true;
    }
    const uint32_t W = pre[a.B];
    if (blockIdx.x >= sk_ctas(W)) return false;
    const uint32_t end = sk_start(W, blockIdx.x + 1);
    if (w.x >= end) return false;
    int lo = 0, hi = a.B - 1;                               // last b with pre[b] <= x
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= w.x) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const uint32_t n_b = nb[b];
    const uint32_t k = (w.x - pre[b]) / n_b;                // unit of request b: (tile, kv head)
    const uint32_t U0 = pre[b] + k * n_b;
    const int cb = (int)(w.x - U0);
    const int ce = (int)min(n_b, end - U0);
    g.b = b;
    g.tile = (int)(k / a.Hkv);
    g.h = (int)(k % a.Hkv);
    req_geo(a, b, g);
    g.live = true;
    g.zero_tile = false;
    const int n_cc = (g.C + NC - 1) / NC;
    g.c_first = min(cb, n_cc);
    g.n_ctx = max(0, min(ce, n_cc) - cb);
    g.d_first = max(cb, n_cc) - n_cc;
    g.n_draft = max(0, ce - max(cb, n_cc));
    g.cut = !(cb == 0 && ce == (int)n_b);
    // the unit starts inside this CTA's range (not at its start) and is cut: the
    // range's last piece, slot 2 c + 1; otherwise slot 2 c
    g.split = 2 * (int)blockIdx.x + ((g.cut && cb == 0 && U0 > sk_start(W, blockIdx.x)) ? 1 : 0);
    w.x = U0 + ce;
    return true;
}

// Prefetch into L1 the per-request words that unit_geo will read for unit u, so
// that computing that unit's geometry later costs an L1 hit.
__device__ __forceinline__ void prefetch_geo(const TcArgs& a, int u)
{
    const int b = (u % (a.B * a.Hkv)) / a.Hkv;
    const void* p0 = a.lens + b;
    const void* p1 = a.block_table != nullptr ? (const void*)(a.ctx_lens + b) : (const void*)(a.ctx_offsets + b);
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p0));
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p1));
}

template <bool F8>
__device__ __forceinline__ uint32_t pack16(float lo, float hi)
{
    if constexpr (F8) {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        return pack_bf16(lo, hi);
    }
}

// two bf16 (one 32-bit word) times a scale, as two f16
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w, float scale)
{
    return pack16<true>(__uint_as_float(w << 16) * scale, __uint_as_float(w & 0xffff0000u) * scale);
}

// two e4m3 values (one 16-bit word) to two f16, exactly
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w16)
{
    uint32_t r;
    asm("{\n\t.reg .b16 t;\n\tmov.b16 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
        : "=r"(r) : "h"((unsigned short)w16));
    return r;
}

// The same wait with the waiting loop out of line: for a wait on the softmax
// warps' hot path that rarely has to wait, so that the loop's registers are not
// reserved there.
__device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, volatile int* abort)
{
    return mbar_wait(bar, parity, abort, kWaitBudget);
}
__device__ __forceinline__ bool warp_wait_lean(uint64_t* bar, uint32_t parity, volatile int* abort)
{
    const bool ok = mbar_try_wait(bar, parity) || mbar_wait_slow(bar, parity, abort);
    return __all_sync(0xffffffffu, ok);
}

template <int D, bool F8, bool PIPE>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
tree_attention_tc_kernel(const TcArgs a, const __grid_constant__ CUtensorMap map_kc,
                         const __grid_constant__ CUtensorMap map_vc,
                         const __grid_constant__ CUtensorMap map_kd,
                         const __grid_constant__ CUtensorMap map_vd,
                         const __grid_constant__ CUtensorMap map_q128,
                         const __grid_constant__ CUtensorMap map_q16)
{
    using C = Cfg<D, F8, PIPE>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Barriers& bar = *reinterpret_cast<Barriers*>(smem + C::kBarOff);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    volatile int* abort = &bar.abort;
    volatile int no_abort = 0;
    // the merge launch that follows a chunk-range launch may start now: its CTAs
    // wait (griddepcontrol.wait) until this grid has completed and its writes are
    // visible, so only their launch overlaps this kernel's tail
    if (C::kMaySk && a.sk) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (tid == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(&bar.kv_full[i], F8 ? 2 : 1);        // FP8: the two converter warps
            mbar_init(&bar.kv_empty[i], 1);                // FP8: PV (after S); else S has read K
            if (C::kPipe) {
                mbar_init(&bar.v_full[i], 1);
                mbar_init(&bar.v_empty[i], 1);             // PV has read V
            }
        }
        for (int i = 0; i < C::kF8Stages; ++i) {
            mbar_init(&bar.f8_full[i], 1);
            mbar_init(&bar.f8_empty[i], 2);
        }
        mbar_init(&bar.s_full[0], 1);
        mbar_init(&bar.s_full[1], 1);
        mbar_init(&bar.pv_done[0], 1);
        mbar_init(&bar.pv_done[1], 1);
        mbar_init(&bar.p_full[0], kSoftmaxWarps);
        mbar_init(&bar.p_full[1], kSoftmaxWarps);
        mbar_init(&bar.o_final, 1);
        mbar_init(&bar.o_free, kSoftmaxWarps);
        mbar_init(&bar.q_full, C::kQTma ? 1 : kSoftmaxWarps);
        mbar_init(&bar.q_free, 1);
        mbar_init(&bar.drain, 1);
        mbar_init(&bar.never, 1);
        bar.abort = 0;
        mbar_fence_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&bar.tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    uint32_t* sk_pre = reinterpret_cast<uint32_t*>(smem + C::kSkOff);
    uint32_t* sk_nb = sk_pre + kSkMaxB + 1;
    if constexpr (C::kMaySk) {
        if (a.sk && warp == 0) sk_build<C::kNc>(a, sk_pre, sk_nb, lane);
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_desc(&map_kc);
        tma_prefetch_desc(&map_vc);
        tma_prefetch_desc(&map_kd);
        tma_prefetch_desc(&map_vd);
        if (C::kQTma && a.q_tma) {
            tma_prefetch_desc(&map_q128);
            tma_prefetch_desc(&map_q16);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bar.tmem_base;

    auto fail = [&]() {
        *abort = 1;
        rd_flag(a.status, RD_DEV_TIMEOUT);
    };

    if (warp >= kSoftmaxWarps) {
    // Warpgroup 1 gives registers back first (all four warps, unconditionally),
    // then splits into its roles.
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
    if (F8 && warp == kProducerWarp) {
        // ------------------------------------------------- producer (8-bit context)
        if (lane == 0) {
            uint32_t g8 = 0;                              // context chunks only
            Work wk = work_begin<C::kMaySk>(a, sk_pre);
            UnitGeo geo;
            while (!*abort && work_next<C::kNc, C::kMaySk>(a, sk_pre, sk_nb, wk, geo)) {
                if (!geo.live) continue;
                bool ok = true;
                for (int j = 0; j < geo.n_ctx; ++j, ++g8) {
                    const int st = g8 % C::kF8Ring;
                    if (g8 >= (uint32_t)C::kF8Ring &&
                        !mbar_wait(&bar.f8_empty[st], ((g8 / C::kF8Ring) - 1) & 1, abort, kWaitBudget)) {
                        ok = false;
                        break;
                    }
                    unsigned char* dst = smem + C::kF8Off + st * C::kF8Bytes;
                    mbar_arrive_expect_tx(&bar.f8_full[st], C::kF8Bytes);
                    const int z = (int)(geo.kv_base + (int64_t)(geo.c_first + j) * C::kNc);
                    tma_load_3d(dst, &map_kc, &bar.f8_full[st], 0, geo.h, z);
                    tma_load_3d(dst + C::kNc * D, &map_vc, &bar.f8_full[st], 0, geo.h, z);
                }
                if (!ok) { fail(); break; }
            }
            const uint32_t first = g8 > (uint32_t)C::kF8Ring ? g8 - C::kF8Ring : 0u;
            for (uint32_t k = first; k < g8; ++k)
                mbar_wait(&bar.f8_full[k % C::kF8Ring], (k / C::kF8Ring) & 1, &no_abort, kWaitBudget);
        }
    } else if (F8 && warp >= kConvWarp0) {
        // ------------------------------------------------------------ converters
        // Thread row (0-63) writes K row `row` and V row `row` of a 16-bit stage;
        // the stage is released as one once PV has read it.
        const int row = tid - kConvWarp0 * 32;
        uint32_t g = 0, g8 = 0;
        // one 128-byte e4m3 row (swizzled) -> one 256-byte f16 row in two 128-byte blocks
        auto widen_row = [&](const unsigned char* src, unsigned char* dst) {
#pragma unroll
            for (int c = 0; c < D / 16; ++c) {
                const uint4 x = *reinterpret_cast<const uint4*>(src + sw128(row, c));
                uint4 lo, hi;
                lo.x = e4m3x2_to_f16x2(x.x & 0xffffu); lo.y = e4m3x2_to_f16x2(x.x >> 16);
                lo.z = e4m3x2_to_f16x2(x.y & 0xffffu); lo.w = e4m3x2_to_f16x2(x.y >> 16);
                hi.x = e4m3x2_to_f16x2(x.z & 0xffffu); hi.y = e4m3x2_to_f16x2(x.z >> 16);
                hi.z = e4m3x2_to_f16x2(x.w & 0xffffu); hi.w = e4m3x2_to_f16x2(x.w >> 16);
                const int c16 = 2 * c;              // two 16-bit chunks of 8 values
                *reinterpret_cast<uint4*>(dst + (c16 >> 3) * (C::kNc * 128) + sw128(row, c16 & 7)) = lo;
                *reinterpret_cast<uint4*>(dst + ((c16 + 1) >> 3) * (C::kNc * 128) +
                                          sw128(row, (c16 + 1) & 7)) = hi;
            }
        };
        // one bf16 draft row times a scale -> f16
        auto draft_row = [&](const uint16_t* base, const UnitGeo& geo, int d, float sc,
                             unsigned char* dst) {
            const uint4* src = d < geo.Pb
                ? reinterpret_cast<const uint4*>(base + (((size_t)geo.b * a.P_max + d) * a.Hkv + geo.h) * D)
                : nullptr;
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {
                uint4 y = make_uint4(0, 0, 0, 0);
                if (src) {
                    const uint4 x = __ldg(src + c);
                    y.x = bf16x2_to_f16x2(x.x, sc); y.y = bf16x2_to_f16x2(x.y, sc);
                    y.z = bf16x2_to_f16x2(x.z, sc); y.w = bf16x2_to_f16x2(x.w, sc);
                }
                *reinterpret_cast<uint4*>(dst + (c >> 3) * (C::kNc * 128) + sw128(row, c & 7)) = y;
            }
        };
        Work wk = work_begin<C::kMaySk>(a, sk_pre);
        UnitGeo geo;
        while (!*abort && work_next<C::kNc, C::kMaySk>(a, sk_pre, sk_nb, wk, geo)) {
            if (!geo.live) continue;
            const int n = geo.n_ctx + geo.n_draft;
            bool ok = true;
            for (int j = 0; j < n; ++j, ++g) {
                const int st = g % C::kStages;
                const uint32_t prev = ((g / C::kStages) - 1) & 1;
                unsigned char* kdst = smem + C::kStageOff + st * C::kStageBytes;
                unsigned char* vdst = kdst + C::kKBytes;
                const bool ctx = j < geo.n_ctx;
                const int s8 = g8 % C::kF8Ring;
                const unsigned char* src = smem + C::kF8Off + s8 * C::kF8Bytes;
                if (ctx && !warp_wait(&bar.f8_full[s8], (g8 / C::kF8Ring) & 1, abort, kWaitBudget)) {
                    ok = false;
                    break;
                }
                if (g >= (uint32_t)C::kStages && !warp_wait(&bar.kv_empty[st], prev, abort, kWaitBudget)) {
                    ok = false;
                    break;
                }
                const int d = (geo.d_first + j - geo.n_ctx) * C::kNc + row;   // draft row (drafts only)
                if (ctx) {
                    widen_row(src, kdst);
                    widen_row(src + C::kNc * D, vdst);
                } else {
                    draft_row(a.k_new, geo, d, a.k_inv, kdst);
                    draft_row(a.v_new, geo, d, a.v_inv, vdst);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.kv_full[st]);
                if (ctx && lane == 0) mbar_arrive(&bar.f8_empty[s8]);
                if (ctx) ++g8;
            }
            if (!ok) { fail(); break; }
        }
    } else if (PIPE && warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        // K and V of the chunk sequence (every live unit's chunks in order) into
        // their own rings.  K of chunk t is issued before V of chunk t - 1: a K
        // stage comes free once S has read it, a V stage only once PV has, and S
        // of a chunk runs ahead of PV of the chunk before.
        if (lane == 0) {
            struct Cursor {
                Work w;
                bool more;                                // positioned on a live item
                int j, n, n_ctx, c_first, d_first, b, h;
                int64_t kv_base;
            };
            auto seek = [&](Cursor& c) {                  // the next live item from c.w on
                UnitGeo geo;
                while ((c.more = work_next<C::kNc, C::kMaySk>(a, sk_pre, sk_nb, c.w, geo))) {
                    if (!geo.live) continue;
                    c.j = 0;
                    c.n = geo.n_ctx + geo.n_draft;
                    c.n_ctx = geo.n_ctx;
                    c.c_first = geo.c_first;
                    c.d_first = geo.d_first;
                    c.b = geo.b;
                    c.h = geo.h;
                    c.kv_base = geo.kv_base;
                    return;
                }
            };
            auto advance = [&](Cursor& c) {
                if (++c.j == c.n) seek(c);
            };
            const bool paged = a.block_table != nullptr;
            // tensor map and first row of chunk c.j: context (contiguous, or the page
            // holding it), or the packed drafts
            auto locate = [&](const Cursor& c, bool is_v, const CUtensorMap*& map) -> int {
                if (c.j < c.n_ctx) {
                    map = is_v ? &map_vc : &map_kc;
                    const int pos0 = (c.c_first + c.j) * kN;
                    if (!paged) return (int)(c.kv_base + pos0);
                    int pg = __ldg(a.block_table + (size_t)c.b * a.max_pages + pos0 / a.page_size);
                    if (pg < 0 || pg >= a.num_pages) {
                        rd_flag(a.status, RD_DEV_BAD_INDEX);
                        pg = 0;
                    }
                    return pg * a.page_size + pos0 % a.page_size;
                }
                map = is_v ? &map_vd : &map_kd;
                return c.b * a.P_max + (c.d_first + c.j - c.n_ctx) * kN;
            };
            auto issue = [&](const Cursor& c, uint32_t g, bool is_v) -> bool {
                const int st = g % C::kStages;
                uint64_t* full = is_v ? &bar.v_full[st] : &bar.kv_full[st];
                uint64_t* empty = is_v ? &bar.v_empty[st] : &bar.kv_empty[st];
                if (g >= (uint32_t)C::kStages &&
                    !mbar_wait(empty, ((g / C::kStages) - 1) & 1, abort, kWaitBudget))
                    return false;
                const CUtensorMap* map;
                const int z = locate(c, is_v, map);
                unsigned char* dst = smem + (is_v ? C::kVOff : C::kStageOff) + st * C::kKBytes;
                mbar_arrive_expect_tx(full, C::kKBytes);
#pragma unroll
                for (int db = 0; db < C::kDB; ++db)
                    tma_load_3d(dst + db * (kN * 128), map, full, db * 64, c.h, z);
                return true;
            };
            Cursor ck;
            ck.w = work_begin<C::kMaySk>(a, sk_pre);
            seek(ck);
            Cursor cv = ck;
            uint32_t gk = 0, gv = 0;                      // K and V chunks issued
            while (!*abort) {
                const bool k_more = ck.more;
                const bool v_more = cv.more;
                if (!k_more && !v_more) break;
                if (k_more) {
                    if (!issue(ck, gk, false)) { fail(); break; }
                    advance(ck);
                    ++gk;
                }
                if (v_more && (gv + 1 < gk || !k_more)) {
                    if (!issue(cv, gv, true)) { fail(); break; }
                    advance(cv);
                    ++gv;
                }
            }
            // drain: every issued copy must land before the CTA may exit
            for (uint32_t k = gk > (uint32_t)C::kStages ? gk - C::kStages : 0u; k < gk; ++k)
                mbar_wait(&bar.kv_full[k % C::kStages], (k / C::kStages) & 1, &no_abort, kWaitBudget);
            for (uint32_t k = gv > (uint32_t)C::kStages ? gv - C::kStages : 0u; k < gv; ++k)
                mbar_wait(&bar.v_full[k % C::kStages], (k / C::kStages) & 1, &no_abort, kWaitBudget);
        }
    } else if (!F8 && warp == kConvWarp0) {
        // ------------------------------------------------------- query writer
        // Each live unit's query tile into shared memory (the A operand of S,
        // 128-byte swizzle), once every S MMA of the unit before has completed.
        // Row m holds query row tile * 128 + m, or in a tile with at most 64 valid
        // rows (paired lanes) row tile * 128 + 16 (m / 32) + m % 16, so that TMEM
        // lanes m and m ^ 16 get the same scores.  With G a power of two <= 16 the
        // tile is one TMA box per 64 columns (rows r = p G + g are G heads of
        // consecutive positions), or eight 16-row boxes when paired; rows past the
        // valid ones then hold whatever the tensor holds there (their scores are
        // masked).  Otherwise the warp loads the rows (zeros past the valid ones).
        // The next unit's boxes are prefetched into L2 when this unit's are issued.
        auto q_row0 = [&](const UnitGeo& ug) -> int {   // tensor row of the tile's first position
            const int p0 = ug.tile * (kM / a.G);
            return ug.b * a.P_max + p0;
        };
        auto paired_of = [&](const UnitGeo& ug) { return ug.n_rows - ug.tile * kM <= 64; };
        // TMA boxes of unit ug: fn(map, smem byte offset, x, y, z)
        auto for_boxes = [&](const UnitGeo& ug, auto&& fn) {
            const int z0 = q_row0(ug), y = ug.h * a.G;
            if (!paired_of(ug)) {
#pragma unroll
                for (int db = 0; db < C::kDB; ++db) fn(&map_q128, db * (kM * 128), db * 64, y, z0);
            } else {
#pragma unroll 1
                for (int k = 0; k < 8; ++k)                 // smem rows 16k.., query rows 16 (k / 2)..
#pragma unroll
                    for (int db = 0; db < C::kDB; ++db)
                        fn(&map_q16, db * (kM * 128) + k * 16 * 128, db * 64, y, z0 + 16 * (k >> 1) / a.G);
            }
        };
        auto q_src = [&](const UnitGeo& ug, int m) -> const uint4* {
            const int qr = ug.tile * kM + (paired_of(ug) ? 16 * (m >> 5) + (m & 15) : m);
            if (qr >= ug.n_rows) return nullptr;
            const int qp = qr / a.G;
            const size_t qrow = (size_t)ug.b * a.P_max + qp;
            return reinterpret_cast<const uint4*>(a.q + (qrow * a.Hq + ug.h * a.G + qr % a.G) * D);
        };
        uint32_t it = 0;
        Work wk = work_begin<C::kMaySk>(a, sk_pre);
        UnitGeo geo;
        while (!*abort && work_next<C::kNc, C::kMaySk>(a, sk_pre, sk_nb, wk, geo)) {
            if (!geo.live) continue;
            if (it > 0 && !warp_wait(&bar.q_free, (it - 1) & 1, abort, kWaitBudget)) { fail(); break; }
            if (a.q_tma) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bar.q_full, kM * D * 2);
                    for_boxes(geo, [&](const CUtensorMap* map, int off, int x, int y, int z) {
                        tma_load_3d(smem + C::kQOff + off, map, &bar.q_full, x, y, z);
                    });
                    Work w2 = wk;
                    UnitGeo nx;
                    if (work_next<C::kNc, C::kMaySk>(a, sk_pre, sk_nb, w2, nx) && nx.live)
                        for_boxes(nx, [&](const CUtensorMap* map, int, int x, int y, int z) {
                            tma_prefetch_3d(map, x, y, z);
                        });
                }
            } else {
#pragma unroll 1
                for (int m = lane; m < kM; m += 32) {
                    const uint4* src = q_src(geo, m);
#pragma unroll
                    for (int db = 0; db < C::kDB; ++db) {
                        uint4 v[8];
#pragma unroll
                        for (int c = 0; c < 8; ++c) v[c] = src ? __ldg(src + db * 8 + c) : make_uint4(0, 0, 0, 0);
                        unsigned char* dst = smem + C::kQOff + db * (kM * 128);
#pragma unroll
                        for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(dst + sw128(m, c)) = v[c];
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.q_full);
            }
            ++it;
        }
        // drain: the last tile's copies must land before the CTA may exit
        if (a.q_tma && lane == 0 && it > 0)
            mbar_wait(&bar.q_full, (it - 1) & 1, &no_abort, kWaitBudget);
    } else if (!F8 && !PIPE && warp == kProducerWarp) {
        // ------------------------------------------------ producer (one K + V ring)
        if (lane == 0) {
            uint32_t g = 0;                               // global chunk counter
            Work wk = work_begin<C::kMaySk>(a, sk_pre);
            UnitGeo geo;
            while (!*abort && work_next<C::kNc, C::kMaySk>(a, sk_pre, sk_nb, wk, geo)) {
                if (!geo.live) continue;
                const int n = geo.n_ctx + geo.n_draft;
                // first cache row of context chunk j (paged: looked up one chunk ahead,
                // so the block-table read overlaps the wait for a free stage)
                auto page_row = [&](int j) -> int {
                    const int pos0 = (geo.c_first + j) * kN;
                    int pg = __ldg(a.block_table + (size_t)geo.b * a.max_pages + pos0 / a.page_size);
                    if (pg < 0 || pg >= a.num_pages) {
                        rd_flag(a.status, RD_DEV_BAD_INDEX);
                        pg = 0;
                    }
                    return pg * a.page_size + pos0 % a.page_size;
                };
                const bool paged = a.block_table != nullptr;
                int next_row = (paged && geo.n_ctx > 0) ? page_row(0) : 0;
                for (int j = 0; j < n; ++j, ++g) {
                    const int st = g % C::kStages;
                    const int this_row = next_row;
                    if (paged && j + 1 < geo.n_ctx) next_row = page_row(j + 1);
                    if (g >= (uint32_t)C::kStages &&
                        !mbar_wait(&bar.kv_empty[st], ((g / C::kStages) - 1) & 1, abort,
                                   kWaitBudget)) { fail(); break; }
                    unsigned char* ks = smem + C::kStageOff + st * C::kStageBytes;
                    unsigned char* vs = ks + C::kKBytes;
                    mbar_arrive_expect_tx(&bar.kv_full[st], C::kStageBytes);
                    const CUtensorMap* mk;
                    const CUtensorMap* mv;
                    int z;
                    if (j < geo.n_ctx) {
                        mk = &map_kc; mv = &map_vc;
                        z = paged ? this_row : (int)(geo.kv_base + (int64_t)(geo.c_first + j) * kN);
                    } else {
                        mk = &map_kd; mv = &map_vd;
                        z = geo.b * a.P_max + (geo.d_first + j - geo.n_ctx) * kN;
                    }
#pragma unroll
                    for (int db = 0; db < C::kDB; ++db) {
                        tma_load_3d(ks + db * (kN * 128), mk, &bar.kv_full[st], db * 64, geo.h, z);
                        tma_load_3d(vs + db * (kN * 128), mv, &bar.kv_full[st], db * 64, geo.h, z);
                    }
                }
            }
            // drain: every issued copy must land before the CTA may exit
            const uint32_t first = g > (uint32_t)C::kStages ? g - C::kStages : 0u;
            for (uint32_t k = first; k < g; ++k)
                mbar_wait(&bar.kv_full[k % C::kStages], (k / C::kStages) & 1, &no_abort, kWaitBudget);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------- MMA issuer
        // 16-bit path, per unit: S_0, then for each chunk j: S_{j+1} into the
        // other S tile (behind PV_{j-1}, whose A operand, P, lives there: the MMAs
        // of one thread run in issue order, so S writes the tile after PV has read
        // it), then, once the softmax warps have written P_j, O += P_j V_j.  So
        // the tensor core computes the next scores while the softmax warps work.
        // FP8 path, per chunk: S_j right behind PV_{j-1} into the one S tile,
        // then PV_j once P_j is written.
        // After the last S of a unit, q_free tells the query writers that the
        // queries may be overwritten; before the first PV of a unit (which
        // restarts O), o_free that the epilogue of the unit before has read O.
        if (lane == 0) {
            constexpr uint32_t idS = F8 ? idesc_f16(kM, C::kNc, false, false) : idesc_bf16(kM, C::kNc, false, false);
            constexpr uint32_t idPV = F8 ? idesc_f16(kM, D, false, true) : idesc_bf16(kM, D, false, true);
            uint32_t g = 0, unit_iter = 0;
            // Shared-memory descriptors differ only in their start-address field
            // (bits 0-13, address >> 4): build the base once and add offsets,
            // which keeps the issuing thread's work per MMA to two additions.
            const uint64_t k_desc = smem_desc(smem_addr(smem + C::kStageOff), 16, 1024, kSwizzle128B);
            const uint64_t v_desc = smem_desc(smem_addr(smem + (C::kPipe ? C::kVOff : C::kStageOff + C::kKBytes)),
                                              C::kNc * 128, 1024, kSwizzle128B);
            const uint64_t q_desc = smem_desc(smem_addr(smem + C::kQOff), 16, 1024, kSwizzle128B);
            if (a.stall_budget > 0 && !mbar_wait(&bar.never, 0, abort, a.stall_budget)) fail();
            Work wk = work_begin<C::kMaySk>(a, sk_pre);
            UnitGeo geo;
            while (!*abort && work_next<C::kNc, C::kMaySk>(a, sk_pre, sk_nb, wk, geo)) {
                if (!geo.live) continue;
                const int n = geo.n_ctx + geo.n_draft;
                if (!mbar_wait(&bar.q_full, unit_iter & 1, abort, kWaitBudget)) { fail(); break; }
                bool ok = true;
                if constexpr (C::kPipe) {
                    // S_j: K-major Q (shared memory) times the K stage, D/16 K-steps
                    auto issue_s = [&](int j) -> bool {
                        const uint32_t gg = g + j;
                        const int st = (int)(gg % C::kStages);
                        if (!mbar_wait(&bar.kv_full[st], (gg / C::kStages) & 1, abort, kWaitBudget))
                            return false;
                        tc_fence_after();
                        const uint64_t kd = k_desc + (uint64_t)((st * C::kKBytes) >> 4);
                        const uint32_t sd = tmem + C::kSCol + (gg & 1) * C::kNc;
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks) {
                            const uint32_t a_off = ((ks >> 2) * (kM * 128) + (ks & 3) * 32) >> 4;
                            const uint32_t b_off = ((ks >> 2) * (C::kNc * 128) + (ks & 3) * 32) >> 4;
                            mma_smem_a(sd, q_desc + a_off, kd + b_off, idS, ks > 0);
                        }
                        mma_commit(&bar.kv_empty[st]);          // the K stage has been read
                        mma_commit(&bar.s_full[gg & 1]);
                        if (j == n - 1) mma_commit(&bar.q_free);
                        return true;
                    };
                    ok = issue_s(0);
                    for (int j = 0; ok && j < n; ++j) {
                        if (j + 1 < n && !issue_s(j + 1)) { ok = false; break; }
                        const uint32_t gg = g + j;
                        const int st = (int)(gg % C::kStages);
                        if (j == 0 && unit_iter > 0 &&
                            !mbar_wait(&bar.o_free, (unit_iter - 1) & 1, abort, kWaitBudget)) {
                            ok = false;
                            break;
                        }
                        // one P barrier per S tile: the softmax warps may finish chunk
                        // j + 1 (whose S is already issued) before this wait for P_j
                        if (!mbar_wait(&bar.p_full[gg & 1], (gg >> 1) & 1, abort, kWaitBudget) ||
                            !mbar_wait(&bar.v_full[st], (gg / C::kStages) & 1, abort, kWaitBudget)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        // O += P V: K-steps of 16 positions, A = P over S tile gg & 1
                        const uint64_t vd = v_desc + (uint64_t)((st * C::kKBytes) >> 4);
                        const uint32_t pa = tmem + C::kSCol + (gg & 1) * C::kNc;
#pragma unroll
                        for (int kk = 0; kk < C::kNc / 16; ++kk)
                            mma_tmem_a(tmem + C::kOCol, pa + kk * 8, vd + (uint64_t)((kk * 2048) >> 4), idPV,
                                       j > 0 || kk > 0);
                        mma_commit(&bar.v_empty[st]);
                        mma_commit(&bar.pv_done[gg & 1]);
                    }
                } else {
                    for (int j = 0; j < n; ++j) {
                        const uint32_t gg = g + j;
                        const int st = (int)(gg % C::kStages);
                        if (!mbar_wait(&bar.kv_full[st], (gg / C::kStages) & 1, abort, kWaitBudget)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        // D/16 K-steps into the S columns
                        const uint64_t kd = k_desc + (uint64_t)((st * C::kStageBytes) >> 4);
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks) {
                            const uint32_t off = ((ks >> 2) * (C::kNc * 128) + (ks & 3) * 32) >> 4;
                            mma_tmem_a(tmem + C::kSCol, tmem + C::kQCol + ks * 8, kd + off, idS, ks > 0);
                        }
                        mma_commit(&bar.s_full[0]);
                        if (j == n - 1) mma_commit(&bar.q_free);
                        if (j == 0 && unit_iter > 0 &&
                            !mbar_wait(&bar.o_free, (unit_iter - 1) & 1, abort, kWaitBudget)) {
                            ok = false;
                            break;
                        }
                        if (!mbar_wait(&bar.p_full[0], gg & 1, abort, kWaitBudget)) { ok = false; break; }
                        tc_fence_after();
                        // O += P V: K-steps of 16 positions, A = P over the S columns
                        const uint64_t vd = v_desc + (uint64_t)((st * C::kStageBytes) >> 4);
#pragma unroll
                        for (int kk = 0; kk < C::kNc / 16; ++kk)
                            mma_tmem_a(tmem + C::kOCol, tmem + C::kSCol + kk * 8,
                                       vd + (uint64_t)((kk * 2048) >> 4), idPV, j > 0 || kk > 0);
                        mma_commit(&bar.kv_empty[st]);
                    }
                }
                if (!ok) { fail(); break; }
                mma_commit(&bar.o_final);
                g += n;
                ++unit_iter;
            }
            // drain: every issued MMA must finish before TMEM is freed
            mma_commit(&bar.drain);
            mbar_wait(&bar.drain, 0, &no_abort, kWaitBudget);
        }
    }
    } else {
        // ------------------------------------------------------------ softmax
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        // Thread tid owns TMEM lane tid.  A tile with more than 64 valid rows
        // keeps row r in lane r, and a thread takes all 64 columns of a chunk.
        // A tile with at most 64 valid rows is paired: row r = 16 w + (lane & 15)
        // of warp w sits in lanes lane and lane ^ 16 of that warp (both hold its
        // query, hence the same scores), and each lane takes 32 of the chunk's
        // columns.  A lane's P row is zero outside its own columns, so its O is
        // the partial sum over them; the two lanes share one running maximum
        // (exchanged every chunk), so their rescales agree and their O and l add
        // up in the epilogue.
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const uint32_t s_col = tmem + lane_base + C::kSCol;
        const uint32_t o_col = tmem + lane_base + C::kOCol;
        auto is_paired = [&](const UnitGeo& ug) { return ug.n_rows - ug.tile * kM <= 64; };
        // the queries of unit ug -> the Q columns of this thread's lane
        auto load_q = [&](const UnitGeo& ug) {
            const bool pr = is_paired(ug);
            const int qr = ug.tile * kM + (pr ? warp * 16 + (lane & 15) : tid);
            const bool qv_ok = qr < ug.n_rows;
            const uint4* src = nullptr;
            if (qv_ok) {
                const int qp = qr / a.G;
                const size_t qrow = (size_t)ug.b * a.P_max + qp;
                src = reinterpret_cast<const uint4*>(a.q + (qrow * a.Hq + ug.h * a.G + qr % a.G) * D);
            }
#pragma unroll
            for (int half = 0; half < D / 64; ++half) {
                uint32_t qv[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 v = qv_ok ? __ldg(src + half * 8 + c) : make_uint4(0, 0, 0, 0);
                    if constexpr (F8) {
                        v.x = bf16x2_to_f16x2(v.x, 1.f); v.y = bf16x2_to_f16x2(v.y, 1.f);
                        v.z = bf16x2_to_f16x2(v.z, 1.f); v.w = bf16x2_to_f16x2(v.w, 1.f);
                    }
                    qv[c * 4 + 0] = v.x; qv[c * 4 + 1] = v.y;
                    qv[c * 4 + 2] = v.z; qv[c * 4 + 3] = v.w;
                }
                tmem_st32(tmem + lane_base + C::kQCol + half * 32, qv);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.q_full);
        };
        // zero output rows of tile `tile` of (b, h): a tree tile without valid rows
        auto zero_tile = [&](int b, int h, int tile) {
            const int row = tile * kM + tid;
            const int p = row / a.G;
            if (p < a.P_max) {
                uint4* dst = reinterpret_cast<uint4*>(
                    a.o + (((size_t)b * a.P_max + p) * a.Hq + h * a.G + row % a.G) * D);
#pragma unroll
                for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
            }
        };
        uint32_t g = 0, unit_iter = 0;
        bool q_ready = false;                              // (not PIPE) the next item's queries are written
        Work wk = work_begin<C::kMaySk>(a, sk_pre);
        UnitGeo geo;
        bool have_next = false;                            // (not PIPE) the next item, looked up ahead
        Work next_w;
        UnitGeo next_geo;
        while (!*abort) {
            if (have_next) {
                geo = next_geo;
                wk = next_w;
                have_next = false;
            } else if (!work_next<C::kNc, C::kMaySk>(a, sk_pre, sk_nb, wk, geo)) {
                break;
            }
            // the words the next unit's geometry needs, into L1 now (its loads then
            // overlap this unit's chunks)
            if (!(C::kMaySk && a.sk) && wk.u < a.n_units) prefetch_geo(a, wk.u);
            const int hq0 = geo.h * a.G;
            if (geo.zero_tile) {                           // padded rows of a tree tile
                zero_tile(geo.b, geo.h, geo.tile);
                continue;
            }
            if (!geo.live) continue;
            const int n = geo.n_ctx + geo.n_draft;
            const bool paired = is_paired(geo);
            const int hf = paired ? lane >> 4 : 0;         // column half of a paired lane
            const int r = paired ? warp * 16 + (lane & 15) : tid;   // row within the tile
            const int row = geo.tile * kM + r;
            const bool valid = row < geo.n_rows;
            const int qpos = row / a.G;                    // node p
            // queries not written ahead (the first live unit, or one after a unit
            // that was not live): the S MMAs of the last live unit have completed,
            // as this warp waited for them at that unit's end
            if constexpr (!C::kQTma) {
                if (!q_ready) load_q(geo);
                q_ready = false;
            }
            float m = -INFINITY, l = 0.f;
            // a warp whose rows are all padding reads no scores; it writes zero P
            // rows (the S columns hold scores again every chunk)
            const bool dead = __all_sync(0xffffffffu, !valid);
            const uint32_t* mrow = valid
                ? a.mask + ((size_t)geo.b * a.P_max + qpos) * a.mask_words : nullptr;
            // One chunk (global index gg, S in the columns at sc): NCOL = 64 columns
            // per lane, or 32 for a paired lane.  FP8: the commit that completed S_j
            // also tracked PV_{j-1}, so O is stable here; 16-bit path: PV_{j-1} may
            // still run, and a rescale of O first waits for it.
            auto chunk = [&](auto ncol, int j, uint32_t gg, uint32_t sc) -> bool {
                constexpr int NCOL = decltype(ncol)::value;
                const int c0 = NCOL == 32 ? 32 * hf : 0;  // first column of this lane
                float s[NCOL];
                {
                    // the load is warp-collective (one address for all lanes): read
                    // all 64 columns; a paired lane keeps its 32
                    uint32_t sr[64];
                    tmem_ld32(sc, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
                    tmem_ld32(sc + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < NCOL; ++c)
                        s[c] = __uint_as_float(NCOL == 64 ? sr[c] : (hf ? sr[32 + c] : sr[c]));
                }
                // ---- visibility ---------------------------------------------------
                if (!valid) {
#pragma unroll
                    for (int c = 0; c < NCOL; ++c) s[c] = -INFINITY;
                } else if (j < geo.n_ctx) {
                    const int pos0 = (geo.c_first + j) * C::kNc + c0;
                    if (pos0 + NCOL > geo.C) {             // the ragged last context chunk
#pragma unroll
                        for (int c = 0; c < NCOL; ++c)
                            if (pos0 + c >= geo.C) s[c] = -INFINITY;
                    }
                } else {
                    const int d0 = (geo.d_first + j - geo.n_ctx) * C::kNc + c0;   // a multiple of 32
                    const uint32_t w0 = (d0 >> 5) < a.mask_words ? __ldg(mrow + (d0 >> 5)) : 0u;
                    const uint32_t w1 = (NCOL == 64 && (d0 >> 5) + 1 < a.mask_words)
                        ? __ldg(mrow + (d0 >> 5) + 1) : 0u;
#pragma unroll
                    for (int c = 0; c < NCOL; ++c) {
                        const uint32_t w = c < 32 ? w0 : w1;
                        const bool vis = (d0 + c < geo.Pb) && ((w >> (c & 31)) & 1u);
                        if (!vis) s[c] = -INFINITY;
                    }
                }
                // ---- online softmax (log2 domain) --------------------------------
                float mx8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) mx8[e] = s[e];
#pragma unroll
                for (int c = 8; c < NCOL; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], s[c]);
                float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                 fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
                if constexpr (NCOL == 32) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float ms = mx * a.scale_log2;
                const bool need = ms > m + kRescaleThreshold;
                const float m_new = need ? ms : m;
                if (__any_sync(0xffffffffu, need) && j > 0) {
                    if constexpr (C::kPipe) {
                        // PV_{j-1} has completed: phase (gg - 1) / 2 of the barrier of
                        // its S tile.  That barrier is at most one phase past it (PV_{j+1}
                        // waits for P_{j+1}) and PV_{j-3} completed before S_j (issued
                        // after it) did, so the parity names the phase.
                        if (!warp_wait_lean(&bar.pv_done[(gg - 1) & 1], ((gg - 1) >> 1) & 1, abort))
                            return false;
                        tc_fence_after();
                    }
                    const float alpha = need ? fast_exp2(m - m_new) : 1.f;
#pragma unroll
                    for (int cb = 0; cb < D / 32; ++cb) {
                        uint32_t o[32];
                        tmem_ld32(o_col + cb * 32, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                        tmem_st32(o_col + cb * 32, o);
                    }
                }
                if (need) {
                    l *= fast_exp2(m - m_new);             // 0 while m is -inf
                    m = m_new;
                }
                const float base = (m == -INFINITY) ? 0.f : m;
                float lsum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                uint32_t pv[NCOL / 2];
#pragma unroll
                for (int c8 = 0; c8 < NCOL / 8; ++c8) {
                    float p[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        p[e] = fast_exp2(fmaf(s[c8 * 8 + e], a.scale_log2, -base));
                        lsum[e] += p[e];
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) pv[c8 * 4 + e] = pack16<F8>(p[2 * e], p[2 * e + 1]);
                }
                // P (16-bit) over the first half of this lane's S columns, PV's A
                // operand; a paired lane writes zeros over the other lane's columns
                if constexpr (NCOL == 64) {
                    tmem_st32(sc, pv);
                } else {
                    uint32_t pw[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) pw[c] = ((c >> 4) == hf) ? pv[c & 15] : 0u;
                    tmem_st32(sc, pw);
                }
                l += ((lsum[0] + lsum[1]) + (lsum[2] + lsum[3])) +
                     ((lsum[4] + lsum[5]) + (lsum[6] + lsum[7]));
                return true;
            };
            bool ok = true;
            for (int j = 0; j < n; ++j) {
                const uint32_t gg = g + j;
                const int sb = C::kPipe ? (int)(gg & 1) : 0;            // S tile
                const uint32_t sph = C::kPipe ? (gg >> 1) & 1 : gg & 1;  // its phase parity
                const uint32_t sc = s_col + sb * C::kNc;
                if (!warp_wait(&bar.s_full[sb], sph, abort, kWaitBudget)) { ok = false; break; }
                tc_fence_after();
                if (dead) {
                    uint32_t zero[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) zero[c] = 0u;
                    tmem_st32(sc, zero);
                } else if (paired) {
                    if (!chunk(std::integral_constant<int, 32>{}, j, gg, sc)) { ok = false; break; }
                } else {
                    if (!chunk(std::integral_constant<int, 64>{}, j, gg, sc)) { ok = false; break; }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.p_full[sb]);
            }
            // every S MMA of this unit has completed once q_free does; then the next
            // unit's queries (if it is live) go into the Q columns, so that its first
            // S MMA overlaps this unit's PV drain and epilogue
            if constexpr (!C::kQTma) {
                if (ok && !warp_wait(&bar.q_free, unit_iter & 1, abort, kWaitBudget)) ok = false;
                next_w = wk;
                if (ok && work_next<C::kNc, C::kMaySk>(a, sk_pre, sk_nb, next_w, next_geo)) {
                    have_next = true;
                    if (next_geo.live) {
                        tc_fence_after();
                        load_q(next_geo);
                        q_ready = true;
                    }
                }
            }
            if (!ok || !warp_wait(&bar.o_final, unit_iter & 1, abort, kWaitBudget)) { fail(); break; }
            tc_fence_after();
            // ---- epilogue ----------------------------------------------------------
            // A paired row's O and l are the sums over its two lanes; lane half hf
            // then writes output columns [hf D/2, (hf + 1) D/2).
            const float l_row = paired ? l + __shfl_xor_sync(0xffffffffu, l, 16) : l;
            // O in registers (all blocks behind one wait); once read, the next
            // unit's first PV may start
            uint32_t ob[D / 32][32];
#pragma unroll
            for (int cb = 0; cb < D / 32; ++cb) tmem_ld32(o_col + cb * 32, ob[cb]);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.o_free);
            if (paired) {
#pragma unroll
                for (int cb = 0; cb < D / 32; ++cb)
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        ob[cb][c] = __float_as_uint(__uint_as_float(ob[cb][c]) +
                                                    __shfl_xor_sync(0xffffffffu, __uint_as_float(ob[cb][c]), 16));
            }
            auto mine = [&](int cb) { return !paired || (cb >= D / 64) == (hf == 1); };
            const bool split_mode = geo.cut;
            if (!split_mode) {
                const float inv = (valid && l_row > 0.f) ? a.out_scale / l_row : 0.f;
                const bool write = qpos < a.P_max;         // valid rows, and padded rows as zeros
                uint16_t* dst = nullptr;
                if (write) {
                    const size_t orow = (size_t)geo.b * a.P_max + qpos;
                    dst = a.o + (orow * a.Hq + hq0 + row % a.G) * D;
                }
                // bf16 rows, 32 columns (64 bytes) at a time, each lane its own row
#pragma unroll
                for (int cb = 0; cb < D / 32; ++cb) {
                    const uint32_t (&o)[32] = ob[cb];
                    uint4 v[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int c = 8 * i;
                        v[i].x = pack_bf16(__uint_as_float(o[c + 0]) * inv, __uint_as_float(o[c + 1]) * inv);
                        v[i].y = pack_bf16(__uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv);
                        v[i].z = pack_bf16(__uint_as_float(o[c + 4]) * inv, __uint_as_float(o[c + 5]) * inv);
                        v[i].w = pack_bf16(__uint_as_float(o[c + 6]) * inv, __uint_as_float(o[c + 7]) * inv);
                    }
                    if (write && mine(cb)) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) reinterpret_cast<uint4*>(dst + cb * 32)[i] = v[i];
                    }
                }
                // paired: rows 64-127 of the tile hold no valid row; their padded
                // outputs are zero (half a row per lane)
                if (paired) {
                    const int row2 = geo.tile * kM + 64 + r;
                    if (row2 / a.G < a.P_max) {
                        uint4* dst2 = reinterpret_cast<uint4*>(
                            a.o + (((size_t)geo.b * a.P_max + row2 / a.G) * a.Hq + hq0 + row2 % a.G) * D +
                            hf * (D / 2));
#pragma unroll
                        for (int c = 0; c < D / 16; ++c) dst2[c] = make_uint4(0, 0, 0, 0);
                    }
                }
            } else {
                // fp32 partials of this piece of a cut unit, in slot 2 blockIdx.x (or
                // 2 blockIdx.x + 1 for a piece that ends the CTA's range after an
                // earlier piece): O as float4 [slot][D / 4][128 rows], so that a
                // warp's store covers consecutive rows, and (m, l) as [slot][128
                // rows].  The merge kernel launched after this one combines them.
                float4* op = reinterpret_cast<float4*>(a.o_part) + (size_t)geo.split * (D / 4) * kM + r;
#pragma unroll
                for (int cb = 0; cb < D / 32; ++cb) {
                    if (mine(cb)) {
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            op[(size_t)(cb * 8 + q) * kM] =
                                make_float4(__uint_as_float(ob[cb][4 * q]), __uint_as_float(ob[cb][4 * q + 1]),
                                            __uint_as_float(ob[cb][4 * q + 2]), __uint_as_float(ob[cb][4 * q + 3]));
                    }
                }
                if (hf == 0) a.ml_part[(size_t)geo.split * kM + r] = make_float2(m, l_row);
            }
            g += n;
            ++unit_iter;
        }
        // chunk-range division: the tiles past each request's valid rows (the
        // chunk ranges hold live units only), round-robin
        if (C::kMaySk && a.sk && !*abort) {
            const int bh = a.B * a.Hkv;
            for (int idx = blockIdx.x; idx < a.n_units; idx += gridDim.x) {
                const int tile = idx / bh, b = (idx % bh) / a.Hkv, h = idx % a.Hkv;
                const uint32_t n_b = sk_nb[b];
                const int tiles_b = n_b > 0 ? (int)((sk_pre[b + 1] - sk_pre[b]) / ((uint32_t)a.Hkv * n_b)) : 0;
                if (tile >= tiles_b && tile * kM < a.P_max * a.G) zero_tile(b, h, tile);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// Merge of the cut units (chunk-range division): CTA c merges the unit named by
// attention CTA c's descriptor (a unit cut by the start of c's range that began
// in c - 1's range; none: return).  512 threads: thread t takes tile row t % 128
// and columns [D/4 (t / 128), +D/4).  The unit's pieces are those of CTAs
// c0 .. c0 + n_seg - 1, piece s in slot 2 (c0 + s), except 2 c0 + 1 when the unit
// starts inside c0's range; out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s
// (M the largest m_s: a first pass over the pieces' m, then the sums, four
// pieces' loads at a time).
constexpr int kMergeThreads = 512;
template <int D>
__global__ void __launch_bounds__(kMergeThreads)
merge_pieces_kernel(const TcArgs a)
{
    constexpr int QC = D / 4;                           // columns per thread (D = 128: 32)
    constexpr int NQ = QC / 4;                          // float4 per thread
    // launched as a programmatic dependent of the attention grid: wait for it to
    // complete (and its partials and descriptors to be visible)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int4 dsc = a.sk_desc[blockIdx.x];
    if (dsc.x < 0) return;
    const int bh = a.B * a.Hkv;
    const int tile = dsc.x / bh, b = (dsc.x % bh) / a.Hkv, h = dsc.x % a.Hkv;
    const int c0 = dsc.y, n_seg = dsc.z & 0xffff;
    const bool c0_last = (dsc.z >> 30) & 1;
    const int r = threadIdx.x % kM, qc = threadIdx.x / kM;
    const int row = tile * kM + r;
    const int p = row / a.G;
    if (p >= a.P_max) return;
    uint16_t* dst = a.o + (((size_t)b * a.P_max + p) * a.Hq + h * a.G + row % a.G) * D + qc * QC;
    const bool valid = row < dsc.w * a.G;
    auto slot = [&](int sp) { return (sp == 0 && c0_last) ? 2 * c0 + 1 : 2 * (c0 + sp); };
    float acc[QC];
#pragma unroll
    for (int c = 0; c < QC; ++c) acc[c] = 0.f;
    float inv = 0.f;
    if (valid) {
        float M = -INFINITY;
        for (int s0 = 0; s0 < n_seg; s0 += 8) {
            float m8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                m8[i] = s0 + i < n_seg ? __ldcg(&a.ml_part[(size_t)slot(s0 + i) * kM + r].x) : -INFINITY;
#pragma unroll
            for (int i = 0; i < 8; ++i) M = fmaxf(M, m8[i]);
        }
        float L = 0.f;
        for (int s0 = 0; s0 < n_seg; s0 += 4) {
            float2 ml[4];
            float4 x[4][NQ];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const bool in = s0 + i < n_seg;
                const size_t sl = in ? (size_t)slot(s0 + i) : 0;
                ml[i] = in ? __ldcg(&a.ml_part[sl * kM + r]) : make_float2(-INFINITY, 0.f);
                const float4* src = reinterpret_cast<const float4*>(a.o_part) + (sl * (D / 4) + qc * NQ) * kM + r;
#pragma unroll
                for (int q = 0; q < NQ; ++q)
                    x[i][q] = in ? __ldcg(src + (size_t)q * kM) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float w = ml[i].x == -INFINITY ? 0.f : exp2f(ml[i].x - M);
                L += ml[i].y * w;
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    acc[4 * q + 0] += x[i][q].x * w;
                    acc[4 * q + 1] += x[i][q].y * w;
                    acc[4 * q + 2] += x[i][q].z * w;
                    acc[4 * q + 3] += x[i][q].w * w;
                }
            }
        }
        inv = (M != -INFINITY && L > 0.f) ? a.out_scale / L : 0.f;
    }
#pragma unroll
    for (int c = 0; c < QC; c += 8) {
        uint4 v;
        v.x = pack_bf16(acc[c + 0] * inv, acc[c + 1] * inv);
        v.y = pack_bf16(acc[c + 2] * inv, acc[c + 3] * inv);
        v.z = pack_bf16(acc[c + 4] * inv, acc[c + 5] * inv);
        v.w = pack_bf16(acc[c + 6] * inv, acc[c + 7] * inv);
        *reinterpret_cast<uint4*>(dst + c) = v;
    }
}

// ------------------------------------------------------------------ host side
// [rows, heads, D] e4m3 -> boxes of kNc (64) positions x 1 head x D bytes, 128-byte swizzle
bool make_fp8_map(CUtensorMap* map, const void* base, int64_t rows, int heads, int D)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)D, (cuuint64_t)heads * D};
    cuuint32_t box[3] = {(cuuint32_t)D, 1, (cuuint32_t)kN};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// One launch of an instantiation (dynamic shared memory set per call: cheap, and
// the attribute must be set on every device the library runs on).
template <int D, bool F8, bool PIPE>
cudaError_t launch(int grid, cudaStream_t stream, const TcArgs& a, const CUtensorMap& m0,
                   const CUtensorMap& m1, const CUtensorMap& m2, const CUtensorMap& m3,
                   const CUtensorMap& m4, const CUtensorMap& m5)
{
    using Cf = Cfg<D, F8, PIPE>;
    cudaError_t e = cudaFuncSetAttribute(tree_attention_tc_kernel<D, F8, PIPE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::kSmemBytes);
    if (e != cudaSuccess) return e;
    tree_attention_tc_kernel<D, F8, PIPE><<<grid, kThreads, Cf::kSmemBytes, stream>>>(a, m0, m1, m2, m3, m4, m5);
    e = cudaGetLastError();
    if (e != cudaSuccess || !a.sk) return e;
    // chunk-range division: merge the units that CTA boundaries cut, launched as a
    // programmatic dependent (its launch overlaps the attention kernel's tail)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, merge_pieces_kernel<D>, a);
}

}  // namespace

rd_attn_plan rd_attn_make_plan(int B, int P_max, int Hq, int Hkv, int D, int max_kv)
{
    rd_attn_plan plan;
    const int G = Hq / Hkv;
    const long rows = (long)P_max * G;
    plan.tiles = (int)((rows + kM - 1) / kM);
    if (plan.tiles < 1) plan.tiles = 1;
    const long units = (long)B * Hkv * plan.tiles;
    const long ctas = (long)kCtasPerSm * rd_device_sm_count();
    // chunk ranges with fewer units than two per CTA (whole
    // units round-robin leave most CTAs idle or hold the launch on the longest
    // unit), while the request table fits in shared memory and the chunk count
    // in 32 bits; a batch with more units balances well enough whole, and needs
    // no partials, merge or workspace
    const long unit_chunks = ((long)max_kv + kN - 1) / kN + ((long)P_max + kN - 1) / kN;
    plan.stream_k = units < 2 * ctas && B <= kSkMaxB && units * unit_chunks < (1L << 31);
    plan.grid = (int)(plan.stream_k ? ctas : std::min(units, ctas));
    if (plan.grid < 1) plan.grid = 1;
    // pieces of cut units: two 128-row fp32 slots (O and (m, l)) per CTA, then
    // one merge descriptor per CTA
    plan.ws_bytes = plan.stream_k
        ? (size_t)2 * plan.grid * kM * ((size_t)D * sizeof(float) + sizeof(float2)) +
              (size_t)plan.grid * sizeof(int4)
        : 0;
    return plan;
}

cudaError_t rd_launch_attention(const rd_attn_plan& plan, int B, int P_max,
                                int Hq, int Hkv, int D, float scale, const void* q,
                                const void* k_new, const void* v_new,
                                const void* k_cache, const void* v_cache,
                                const int64_t* ctx_offsets, int64_t total_kv, int max_kv,
                                const int32_t* lens, const uint32_t* mask, int mask_words,
                                void* o, void* workspace, int32_t* dev_status,
                                cudaStream_t stream, const rd_paged_kv* paged,
                                const rd_fp8_kv* fp8)
{
    TcArgs a;
    a.block_table = paged ? paged->block_table : nullptr;
    a.ctx_lens = paged ? paged->ctx_lens : nullptr;
    a.max_pages = paged ? paged->max_pages : 0;
    a.page_size = paged ? paged->page_size : 1;
    a.num_pages = paged ? paged->num_pages : 0;
    a.B = B;
    a.P_max = P_max;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.tiles = plan.tiles;
    a.sk = plan.stream_k;
    a.mask_words = mask_words;
    a.n_units = B * Hkv * plan.tiles;
    a.scale_log2 = scale * kLog2e;
    a.q = static_cast<const uint16_t*>(q);
    a.ctx_offsets = ctx_offsets;
    a.total_kv = total_kv;
    a.max_kv = max_kv;
    a.lens = lens;
    a.mask = mask;
    a.o = static_cast<uint16_t*>(o);
    a.status = dev_status;
    a.o_part = nullptr;
    a.ml_part = nullptr;
    a.sk_desc = nullptr;
    a.k_new = static_cast<const uint16_t*>(k_new);
    a.v_new = static_cast<const uint16_t*>(v_new);
    a.k_inv = a.v_inv = a.out_scale = 1.f;
    if (fp8 != nullptr) {
        a.k_inv = 1.f / fp8->k_scale;
        a.v_inv = 1.f / fp8->v_scale;
        a.out_scale = fp8->v_scale;
        a.scale_log2 *= fp8->k_scale;
    }
    if (plan.stream_k) {
        const size_t slot_rows = (size_t)2 * plan.grid * kM;
        a.o_part = static_cast<float*>(workspace);
        a.ml_part = reinterpret_cast<float2*>(a.o_part + slot_rows * D);
        a.sk_desc = reinterpret_cast<int4*>(a.ml_part + slot_rows);
    }
    CUtensorMap mkc, mvc, mkd, mvd;
    const void* kc = k_cache;
    const void* vc = v_cache;
    const int64_t kc_rows = paged ? (int64_t)paged->num_pages * paged->page_size : total_kv;
    const int64_t kd_rows = (int64_t)B * P_max;
    const void* kd = k_new;
    const void* vd = v_new;
    if (kc == nullptr || kc_rows == 0) { kc = kd; vc = vd; }
    const int grid = plan.grid;
    a.stall_budget = rd_attention_stall_budget();
    if (fp8 != nullptr) {
        // 8-bit context maps (the drafts are read by the converter warps)
        if (D != 128 || paged || total_kv < 1 ||
            !make_fp8_map(&mkc, fp8->k_cache, total_kv, Hkv, D) ||
            !make_fp8_map(&mvc, fp8->v_cache, total_kv, Hkv, D))
            return cudaErrorInvalidValue;
        a.q_tma = false;
        return launch<128, true, false>(grid, stream, a, mkc, mvc, mkc, mvc, mkc, mvc);
    }
    if (!make_kv_map(&mkc, kc, kc_rows > 0 ? kc_rows : kd_rows, Hkv, D) ||
        !make_kv_map(&mvc, vc, kc_rows > 0 ? kc_rows : kd_rows, Hkv, D) ||
        !make_kv_map(&mkd, kd, kd_rows, Hkv, D) || !make_kv_map(&mvd, vd, kd_rows, Hkv, D))
        return cudaErrorInvalidValue;
    // query tiles by TMA when a tile is whole boxes: G a power of two <= 16 (it
    // divides the 16 rows of a paired box and the 128 of a tile)
    CUtensorMap mq128, mq16;
    const int64_t q_rows = (int64_t)B * P_max;
    a.q_tma = a.G <= 16 && (a.G & (a.G - 1)) == 0 && (reinterpret_cast<uintptr_t>(q) & 15) == 0 &&
              make_q_map(&mq128, q, q_rows, Hq, D, a.G, kM / a.G) &&
              make_q_map(&mq16, q, q_rows, Hq, D, a.G, 16 / a.G);
    if (!a.q_tma) { mq128 = mkc; mq16 = mkc; }
    return D == 128 ? launch<128, false, true>(grid, stream, a, mkc, mvc, mkd, mvd, mq128, mq16)
                    : launch<64, false, true>(grid, stream, a, mkc, mvc, mkd, mvd, mq128, mq16);
}
