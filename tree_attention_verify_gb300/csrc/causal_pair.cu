// Causal prefill (the context half of an in-flight batch) with paired tiles:
// one CTA per SM, two 128-row query tiles per work unit, 512 TMEM columns.
//
// TensorRT-LLM's attention plugin splits context and generation requests (NVIDIA
// blog "ReDrafter in TensorRT-LLM", section "Inflight-batching Compatible
// Engine"); the context requests need ordinary causal attention over their
// prefill chunk.
//
// Unit = (sequence b, kv head h, pair p): the G query heads of kv head h are
// stacked as rows (row r -> token r / G, head h G + r % G) and the unit takes
// rows [256 p, 256 p + 256) as tile A (the first 128) and tile B (the next 128).
// Tile t reads the 64-position KV chunks its last token can see; with G = 4 both
// tiles of a pair (tokens 64 p .. 64 p + 63) read the same chunks, each K/V
// chunk is loaded once for both.  Units go round-robin over the CTAs, pair-major
// and the last pairs (the longest) first.
//
// Warp roles (384 threads; setmaxnreg gives warpgroup 2's registers to the two
// softmax warpgroups):
//   warps 0-3  softmax of tile A, warps 4-7 softmax of tile B: row r of a tile
//              is TMEM lane r.  Per chunk: S from TMEM, causal mask, online
//              softmax in exp2 form (O rescaled when a row maximum grows by more
//              than 2^8), 16-bit P written over the tile's S columns; at the end
//              of the unit, O normalised to bf16 and stored: a tile whose 128
//              rows all belong to the sequence goes through a shared-memory
//              staging tile and one TMA store per 64 columns (the stores leave
//              the load/store pipe free for the next unit's loads), other tiles
//              by direct 16-byte row stores.
//   warp 8     producer: TMA loads of K and V chunks into a ring of stages.
//   warp 9     MMA issuer, TMEM owner: copies the unit's two query tiles from
//              shared memory into TMEM (tcgen05.cp), then per chunk j issues
//              PV_A(j), S_A(j+1), PV_B(j), S_B(j+1) as each tile's P is ready, so
//              the tensor core works on one tile while the other's softmax runs.
//   warp 10    query loader: the next unit's two query tiles into shared memory
//              (TMA boxes of 128 / G positions x G heads x 64 columns when G is a
//              power of two <= 128, else plain loads).
// Every wait is bounded by a clock budget; on expiry the CTA records
// RD_DEV_TIMEOUT, drains its in-flight copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "attn_common.cuh"
#include "rd_internal.cuh"
#include "tc_ptx.cuh"

namespace {
using namespace rdtc;
using namespace rdattn;

constexpr int kM = 128;                    // rows per tile = TMEM lanes
constexpr int kN = kChunk;                 // KV positions per chunk
constexpr int kThreads = 384;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kQWarp = 10;
// Register split: 384 threads launch with 168 registers each (64,512 in all);
// the two softmax warpgroups take 192, warpgroup 2 keeps 120:
// 128 x (192 + 192 + 120) = 64,512, and per sub-partition 32 x 504 = 16,128.
constexpr int kRegsLaunch = 168;
constexpr int kRegsSoftmax = 192;
constexpr int kRegsOther = 120;
static_assert(128 * (2 * kRegsSoftmax + kRegsOther) <= kThreads * kRegsLaunch, "register split");
static_assert(32 * (2 * kRegsSoftmax + kRegsOther) <= 16384, "register split per sub-partition");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr long long kWaitBudget = 4000000000LL;   // ~2 s of SM clock per wait

template <int D> struct PCfg {
    static constexpr int kDB = D / 64;                  // 128-byte column blocks
    static constexpr int kKBytes = kN * D * 2;          // one K (or V) chunk
    static constexpr int kStageBytes = 2 * kKBytes;     // K + V
    static constexpr int kStages = D == 128 ? 3 : 8;
    static constexpr int kQBytes = kM * D * 2;          // one tile's queries (or outputs)
    static constexpr int kStageOff = 0;
    static constexpr int kQOff = kStages * kStageBytes;           // query tiles A, B
    static constexpr int kOStageOff = kQOff + 2 * kQBytes;        // output staging tiles A, B
    static constexpr int kBarOff = kOStageOff + 2 * kQBytes;
    static constexpr int kSmemBytes = kBarOff + 512 + 1024;       // + barriers + alignment slack
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
    // TMEM (512 columns): per tile t, S/P at 64 t, O at 128 + 128 t, Q at 384 + 64 t
    static constexpr uint32_t kTmemCols = 512;
    __host__ __device__ static constexpr uint32_t s_col(int t) { return 64u * t; }
    __host__ __device__ static constexpr uint32_t o_col(int t) { return 128u + 128u * t; }
    __host__ __device__ static constexpr uint32_t q_col(int t) { return 384u + 64u * t; }
};

struct PArgs {
    int B, Hq, Hkv, G, pairs, n_units;
    float scale_log2;
    const uint16_t* q;
    const int32_t* cu;        // cu_seqlens [B + 1]
    int64_t total;            // rows of q / k / v
    int max_len;
    uint16_t* o;
    int32_t* status;
    long long stall_budget;   // failure-detection test hook (> 0: the issuer stalls first)
    bool q_tma;
};

struct PBar {
    uint64_t kv_full[8];
    uint64_t kv_empty[8];
    uint64_t q_full;          // the unit's query tiles landed in shared memory
    uint64_t q_free;          // copied into TMEM: the shared tiles may be overwritten
    uint64_t s_full[2];       // S of a tile's chunk is in TMEM
    uint64_t p_full[2];       // P of a tile's chunk is written (its softmax warps)
    uint64_t o_final[2];      // the tile's last PV of the unit has completed
    uint64_t o_free[2];       // the tile's epilogue has read O
    uint64_t stg_free[2];     // the tile's last output store has read its staging tile
    uint64_t stg_full[2];     // the tile's four softmax warps have written the staging tile
    uint64_t drain;
    uint64_t never;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(PBar) <= 512, "barrier block");

// Geometry of unit u, identical in every role.  nt[t] = chunks of tile t (0: the
// tile has no valid rows); n = chunks of the unit = max(nt).
struct PGeo {
    int b, h, pair;
    int64_t kv_base;
    int C, n_rows, n;
    int nt[2];
    bool live;
};

// cu_seqlens[b], cu_seqlens[b + 1] of unit u's sequence: every role loads them one
// unit ahead, so that the load does not wait behind the unit's output stores
__device__ __forceinline__ int2 cu_load(const PArgs& a, int u)
{
    const int b = (u % (a.B * a.Hkv)) / a.Hkv;
    return make_int2(a.cu[b], a.cu[b + 1]);
}

__device__ __forceinline__ PGeo pair_geo(const PArgs& a, int u, int2 cu)
{
    PGeo g;
    const int bh = a.B * a.Hkv;
    g.pair = a.pairs - 1 - u / bh;                // the longest pairs first
    g.b = (u % bh) / a.Hkv;
    g.h = u % a.Hkv;
    const int s0 = cu.x, s1 = cu.y;
    g.kv_base = s0;
    g.C = s1 - s0;
    const bool bad = s0 < 0 || g.C < 0 || g.C > a.max_len || s1 > a.total;
    if (bad) g.C = 0;
    if (bad && g.h == 0 && g.pair == 0 && threadIdx.x == 0) rd_flag(a.status, RD_DEV_BAD_LENGTH);
    g.n_rows = g.C * a.G;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int r0 = g.pair * 2 * kM + t * kM;
        g.nt[t] = r0 < g.n_rows ? ((min(g.n_rows, r0 + kM) - 1) / a.G) / kN + 1 : 0;
    }
    g.n = max(g.nt[0], g.nt[1]);
    g.live = g.nt[0] > 0;
    return g;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
causal_pair_kernel(const PArgs a, const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_v,
                   const __grid_constant__ CUtensorMap map_q,
                   const __grid_constant__ CUtensorMap map_o)
{
    using C = PCfg<D>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    PBar& bar = *reinterpret_cast<PBar*>(smem + C::kBarOff);
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    volatile int* abort = &bar.abort;
    volatile int no_abort = 0;

    if (tid == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(&bar.kv_full[i], 1);
            mbar_init(&bar.kv_empty[i], 1);
        }
        mbar_init(&bar.q_full, 1);
        mbar_init(&bar.q_free, 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bar.s_full[t], 1);
            mbar_init(&bar.p_full[t], 4);
            mbar_init(&bar.o_final[t], 1);
            mbar_init(&bar.o_free[t], 4);
            mbar_init(&bar.stg_free[t], 1);
            mbar_init(&bar.stg_full[t], 4);
        }
        mbar_init(&bar.drain, 1);
        mbar_init(&bar.never, 1);
        bar.abort = 0;
        mbar_fence_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&bar.tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_desc(&map_k);
        tma_prefetch_desc(&map_v);
        if (a.q_tma) {
            tma_prefetch_desc(&map_q);
            tma_prefetch_desc(&map_o);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bar.tmem_base;
    const int2 first_cu = blockIdx.x < a.n_units ? cu_load(a, blockIdx.x) : make_int2(0, 0);
    auto fail = [&]() {
        *abort = 1;
        rd_flag(a.status, RD_DEV_TIMEOUT);
    };

    if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t g = 0;                               // chunks issued
            int2 cu_next = first_cu;
            for (int u = blockIdx.x; u < a.n_units && !*abort; u += gridDim.x) {
                const PGeo geo = pair_geo(a, u, cu_next);
                if ((long)u + gridDim.x < a.n_units) cu_next = cu_load(a, u + gridDim.x);
                if (!geo.live) continue;
                bool ok = true;
                for (int j = 0; j < geo.n; ++j, ++g) {
                    const int st = (int)(g % C::kStages);
                    if (g >= (uint32_t)C::kStages &&
                        !mbar_wait(&bar.kv_empty[st], ((g / C::kStages) - 1) & 1, abort, kWaitBudget)) {
                        ok = false;
                        break;
                    }
                    unsigned char* ks = smem + C::kStageOff + st * C::kStageBytes;
                    unsigned char* vs = ks + C::kKBytes;
                    mbar_arrive_expect_tx(&bar.kv_full[st], C::kStageBytes);
                    const int z = (int)(geo.kv_base + (int64_t)j * kN);
#pragma unroll
                    for (int db = 0; db < C::kDB; ++db) {
                        tma_load_3d(ks + db * (kN * 128), &map_k, &bar.kv_full[st], db * 64, geo.h, z);
                        tma_load_3d(vs + db * (kN * 128), &map_v, &bar.kv_full[st], db * 64, geo.h, z);
                    }
                }
                if (!ok) { fail(); break; }
            }
            // drain: every issued copy must land before the CTA may exit
            for (uint32_t k = g > (uint32_t)C::kStages ? g - C::kStages : 0u; k < g; ++k)
                mbar_wait(&bar.kv_full[k % C::kStages], (k / C::kStages) & 1, &no_abort, kWaitBudget);
        }
    } else if (warp == kQWarp) {
        // ------------------------------------------------------- query loader
        // Tile t of unit u: rows [256 p + 128 t, +128); row m of the shared tile
        // = query row 256 p + 128 t + m (rows past the valid ones: whatever the
        // tensor holds there, or zero with plain loads; their scores are masked).
        uint32_t it = 0;
        int2 cu_next = first_cu;
        for (int u = blockIdx.x; u < a.n_units && !*abort; u += gridDim.x) {
            const PGeo geo = pair_geo(a, u, cu_next);
            if ((long)u + gridDim.x < a.n_units) cu_next = cu_load(a, u + gridDim.x);
            if (!geo.live) continue;
            if (it > 0 && !warp_wait(&bar.q_free, (it - 1) & 1, abort, kWaitBudget)) { fail(); break; }
            if (a.q_tma) {
                if (lane == 0) {
                    uint32_t bytes = 0;
                    for (int t = 0; t < 2; ++t)
                        if (geo.nt[t] > 0) bytes += C::kQBytes;
                    mbar_arrive_expect_tx(&bar.q_full, bytes);
                    for (int t = 0; t < 2; ++t) {
                        if (geo.nt[t] == 0) continue;
                        const int z = (int)(geo.kv_base + (geo.pair * 2 * kM + t * kM) / a.G);
#pragma unroll
                        for (int db = 0; db < C::kDB; ++db)
                            tma_load_3d(smem + C::kQOff + t * C::kQBytes + db * (kM * 128), &map_q, &bar.q_full,
                                        db * 64, geo.h * a.G, z);
                    }
                }
            } else {
                for (int t = 0; t < 2; ++t) {
                    if (geo.nt[t] == 0) continue;
#pragma unroll 1
                    for (int m = lane; m < kM; m += 32) {
                        const int row = geo.pair * 2 * kM + t * kM + m;
                        const uint4* src = row < geo.n_rows
                            ? reinterpret_cast<const uint4*>(
                                  a.q + (((size_t)geo.kv_base + row / a.G) * a.Hq + geo.h * a.G + row % a.G) * D)
                            : nullptr;
#pragma unroll
                        for (int db = 0; db < C::kDB; ++db) {
                            uint4 v[8];
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                v[c] = src ? __ldg(src + db * 8 + c) : make_uint4(0, 0, 0, 0);
                            unsigned char* dst = smem + C::kQOff + t * C::kQBytes + db * (kM * 128);
#pragma unroll
                            for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(dst + sw128(m, c)) = v[c];
                        }
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.q_full);
            }
            ++it;
        }
        if (a.q_tma && lane == 0 && it > 0)
            mbar_wait(&bar.q_full, (it - 1) & 1, &no_abort, kWaitBudget);
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // Per unit: wait for its query tiles, copy them into the Q columns
        // (tcgen05.cp, in issue order after the S MMAs of the unit before, which
        // read those columns), free the shared tiles, issue S_t(0) for each
        // active tile, then per chunk j and tile t (while j < nt[t]): wait for
        // P_t(j), O_t += P_t(j) V_j, then S_t(j + 1) into the same S columns (it
        // runs after PV_t(j) has read P there: the MMAs of one thread run in issue
        // order).  The commit that completes S_t(j + 1) therefore also covers
        // PV_t(j), so softmax t finds O_t stable when it rescales.  The stage of
        // chunk j is released after its last reader, and a tile's first PV of a
        // unit (which restarts O_t) waits until the epilogue of the unit before
        // has read O_t.
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16(kM, kN, false, false);
            constexpr uint32_t idPV = idesc_bf16(kM, D, false, true);
            const uint64_t k_desc = smem_desc(smem_addr(smem + C::kStageOff), 16, 1024, kSwizzle128B);
            const uint64_t v_desc = smem_desc(smem_addr(smem + C::kStageOff + C::kKBytes), kN * 128, 1024,
                                              kSwizzle128B);
            const uint64_t q_desc = smem_desc(smem_addr(smem + C::kQOff), 16, 1024, kSwizzle128B);
            if (a.stall_budget > 0 && !mbar_wait(&bar.never, 0, abort, a.stall_budget)) fail();
            uint32_t g = 0, it = 0;
            uint32_t ct[2] = {0u, 0u};    // chunks of tile t so far (s_full / p_full phases)
            uint32_t ut[2] = {0u, 0u};    // units in which tile t was active (o_final / o_free)
            int2 cu_next = first_cu;
            for (int u = blockIdx.x; u < a.n_units && !*abort; u += gridDim.x) {
                const PGeo geo = pair_geo(a, u, cu_next);
                if ((long)u + gridDim.x < a.n_units) cu_next = cu_load(a, u + gridDim.x);
                if (!geo.live) continue;
                const int nb = geo.nt[1] > 0 ? 2 : 1;                     // active tiles
                if (!mbar_wait(&bar.q_full, it & 1, abort, kWaitBudget)) { fail(); break; }
                tc_fence_after();
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (t >= nb) break;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t a_off = (t * C::kQBytes + (ks >> 2) * (kM * 128) + (ks & 3) * 32) >> 4;
                        tmem_cp_128x256b(tmem + C::q_col(t) + ks * 8, q_desc + a_off);
                    }
                }
                mma_commit(&bar.q_free);
                // S_t(j) of global chunk gg: D/16 K-steps, A = Q_t (TMEM), B = the K stage
                auto issue_s = [&](int t, uint32_t gg) {
                    const int st = (int)(gg % C::kStages);
                    const uint64_t kd = k_desc + (uint64_t)((st * C::kStageBytes) >> 4);
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t off = ((ks >> 2) * (kN * 128) + (ks & 3) * 32) >> 4;
                        mma_tmem_a(tmem + C::s_col(t), tmem + C::q_col(t) + ks * 8, kd + off, idS, ks > 0);
                    }
                    mma_commit(&bar.s_full[t]);
                };
                auto kv_wait = [&](uint32_t gg) {
                    const int st = (int)(gg % C::kStages);
                    return mbar_wait(&bar.kv_full[st], (gg / C::kStages) & 1, abort, kWaitBudget);
                };
                bool ok = kv_wait(g);
                if (ok) {
                    tc_fence_after();
                    issue_s(0, g);
                    if (nb > 1) issue_s(1, g);
                }
                for (int j = 0; ok && j < geo.n; ++j) {
                    const uint32_t gg = g + j;
                    const int st = (int)(gg % C::kStages);
                    bool next_ready = false;                  // kv_full of chunk j + 1 waited for
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        if (j >= geo.nt[t]) continue;
                        if (j == 0 && ut[t] > 0 &&
                            !mbar_wait(&bar.o_free[t], (ut[t] - 1) & 1, abort, kWaitBudget)) {
                            ok = false;
                            break;
                        }
                        if (!mbar_wait(&bar.p_full[t], ct[t] & 1, abort, kWaitBudget)) { ok = false; break; }
                        tc_fence_after();
                        // O_t += P_t V_j: K-steps of 16 positions, A = P over the S columns
                        const uint64_t vd = v_desc + (uint64_t)((st * C::kStageBytes) >> 4);
#pragma unroll
                        for (int kk = 0; kk < kN / 16; ++kk)
                            mma_tmem_a(tmem + C::o_col(t), tmem + C::s_col(t) + kk * 8,
                                       vd + (uint64_t)((kk * 2048) >> 4), idPV, j > 0 || kk > 0);
                        ++ct[t];
                        if (j + 1 < geo.nt[t]) {
                            if (!next_ready) {
                                if (!kv_wait(gg + 1)) { ok = false; break; }
                                tc_fence_after();
                                next_ready = true;
                            }
                            issue_s(t, gg + 1);
                        } else {
                            mma_commit(&bar.o_final[t]);
                            ++ut[t];
                        }
                    }
                    if (!ok) break;
                    mma_commit(&bar.kv_empty[st]);            // both tiles have read chunk j
                }
                if (!ok) { fail(); break; }
                g += geo.n;
                ++it;
            }
            // drain: every issued MMA must finish before TMEM is freed
            mma_commit(&bar.drain);
            mbar_wait(&bar.drain, 0, &no_abort, kWaitBudget);
        }
    }
    } else {
        // ------------------------------------------------------------ softmax
        // Warpgroup t owns tile t; thread (warp w, lane) owns TMEM lane 32 (w % 4)
        // + lane, row r of the tile, and all 64 columns of a chunk.
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        const int t = warp >> 2;
        const int r = (warp & 3) * 32 + lane;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t sc = tmem + lane_base + C::s_col(t);
        const uint32_t oc = tmem + lane_base + C::o_col(t);
        uint32_t cs = 0, us = 0;          // chunks and units of tile t so far
        uint32_t su = 0;                  // staged output tiles so far
        int2 cu_next = first_cu;
        for (int u = blockIdx.x; u < a.n_units && !*abort; u += gridDim.x) {
            const PGeo geo = pair_geo(a, u, cu_next);
            if ((long)u + gridDim.x < a.n_units) cu_next = cu_load(a, u + gridDim.x);
            if (!geo.live || geo.nt[t] == 0) continue;
            const int row = geo.pair * 2 * kM + t * kM + r;
            const bool valid = row < geo.n_rows;
            const int qpos = row / a.G;                    // token of this row
            const int lim = valid ? min(geo.C, qpos + 1) : 0;   // visible positions: pos < lim
            // a warp whose rows are all past the sequence reads no scores and
            // writes zero P rows
            const bool dead = __all_sync(0xffffffffu, !valid);
            float m = -INFINITY, l = 0.f;
            bool ok = true;
            for (int j = 0; j < geo.nt[t]; ++j, ++cs) {
                if (!warp_wait(&bar.s_full[t], cs & 1, abort, kWaitBudget)) { ok = false; break; }
                tc_fence_after();
                if (dead) {
                    uint32_t zero[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) zero[c] = 0u;
                    tmem_st32(sc, zero);
                } else {
                    float s[kN];
                    {
                        uint32_t sr[kN];
                        tmem_ld32(sc, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
                        tmem_ld32(sc + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
                        tmem_ld_wait();
#pragma unroll
                        for (int c = 0; c < kN; ++c) s[c] = __uint_as_float(sr[c]);
                    }
                    const int pos0 = j * kN;
                    if (pos0 + kN > lim) {
#pragma unroll
                        for (int c = 0; c < kN; ++c)
                            if (pos0 + c >= lim) s[c] = -INFINITY;
                    }
                    // online softmax in the log2 domain: the row maximum m (of the
                    // scaled scores) moves only when it grows by more than 2^8,
                    // and O and l are rescaled then
                    float mx8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) mx8[e] = s[e];
#pragma unroll
                    for (int c = 8; c < kN; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], s[c]);
                    const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                           fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
                    const float ms = mx * a.scale_log2;
                    const bool need = ms > m + kRescaleThreshold;
                    const float m_new = need ? ms : m;
                    if (__any_sync(0xffffffffu, need) && j > 0) {
                        // PV_t(j - 1) completed with S_t(j) (issued after it)
                        const float alpha = need ? fast_exp2(m - m_new) : 1.f;
#pragma unroll 1
                        for (int cb = 0; cb < D / 32; ++cb) {
                            uint32_t o[32];
                            tmem_ld32(oc + cb * 32, o);
                            tmem_ld_wait();
#pragma unroll
                            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                            tmem_st32(oc + cb * 32, o);
                        }
                    }
                    if (need) {
                        l *= fast_exp2(m - m_new);         // 0 while m is -inf
                        m = m_new;
                    }
                    const float base = (m == -INFINITY) ? 0.f : m;
                    float lsum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                    uint32_t pv[kN / 2];
#pragma unroll
                    for (int c8 = 0; c8 < kN / 8; ++c8) {
                        float p[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            p[e] = fast_exp2(fmaf(s[c8 * 8 + e], a.scale_log2, -base));
                            lsum[e] += p[e];
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e) pv[c8 * 4 + e] = pack_bf16(p[2 * e], p[2 * e + 1]);
                    }
                    // P (bf16) over the first 32 of the tile's S columns: PV's A operand
                    tmem_st32(sc, pv);
                    l += ((lsum[0] + lsum[1]) + (lsum[2] + lsum[3])) +
                         ((lsum[4] + lsum[5]) + (lsum[6] + lsum[7]));
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.p_full[t]);
            }
            if (!ok || !warp_wait(&bar.o_final[t], us & 1, abort, kWaitBudget)) { fail(); break; }
            tc_fence_after();
            // ---- epilogue: O to registers (normalised and packed to bf16 32
            // columns at a time), release O_t, store the row
            const float inv = (valid && l > 0.f) ? 1.f / l : 0.f;
            uint4 ob[D / 8];
#pragma unroll
            for (int cb = 0; cb < D / 32; ++cb) {
                uint32_t o[32];
                tmem_ld32(oc + cb * 32, o);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = 8 * i;
                    ob[cb * 4 + i] = make_uint4(
                        pack_bf16(__uint_as_float(o[c + 0]) * inv, __uint_as_float(o[c + 1]) * inv),
                        pack_bf16(__uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv),
                        pack_bf16(__uint_as_float(o[c + 4]) * inv, __uint_as_float(o[c + 5]) * inv),
                        pack_bf16(__uint_as_float(o[c + 6]) * inv, __uint_as_float(o[c + 7]) * inv));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.o_free[t]);
            ++us;
            const int row0 = geo.pair * 2 * kM + t * kM;
            if (a.q_tma && row0 + kM <= geo.n_rows) {
                // whole tile: staging tile (rows of 128 bytes per 64 columns, the
                // TMA box layout), then the TMA stores by thread 0 of the group.
                // The staging tile is free once the group's previous stores have
                // read it; all waits are bounded.
                unsigned char* stg = smem + C::kOStageOff + t * C::kQBytes;
                const bool issuer = (tid & 127) == 0;
                if (issuer) {
                    tma_store_wait_read();
                    mbar_arrive(&bar.stg_free[t]);
                }
                if (!warp_wait(&bar.stg_free[t], su & 1, abort, kWaitBudget)) { fail(); break; }
#pragma unroll
                for (int db = 0; db < C::kDB; ++db)
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4*>(stg + db * (kM * 128) + sw128(r, c)) = ob[db * 8 + c];
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.stg_full[t]);
                // the issuer's wait decides for its whole warp (a lane that left the
                // loop alone would strand the others in the next warp-wide wait)
                bool st_ok = true;
                if (issuer) st_ok = mbar_wait(&bar.stg_full[t], su & 1, abort, kWaitBudget);
                if (!__all_sync(0xffffffffu, st_ok)) { fail(); break; }
                if (issuer) {
                    const int z = (int)(geo.kv_base + row0 / a.G);
#pragma unroll
                    for (int db = 0; db < C::kDB; ++db)
                        tma_store_3d(&map_o, stg + db * (kM * 128), db * 64, geo.h * a.G, z);
                    tma_store_commit();
                }
                ++su;
            } else if (valid) {
                uint4* dst = reinterpret_cast<uint4*>(
                    a.o + (((size_t)geo.kv_base + qpos) * a.Hq + geo.h * a.G + row % a.G) * D);
#pragma unroll
                for (int i = 0; i < D / 8; ++i) dst[i] = ob[i];
            }
        }
        // the output stores must have completed before the CTA exits
        if ((tid & 127) == 0) tma_store_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D>
cudaError_t launch_pair(int grid, cudaStream_t stream, const PArgs& a, const CUtensorMap& mk,
                        const CUtensorMap& mv, const CUtensorMap& mq, const CUtensorMap& mo)
{
    using C = PCfg<D>;
    // the register split assumes the launch allocation: refuse to launch a build
    // whose kernel was given fewer registers per thread
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, causal_pair_kernel<D>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kRegsLaunch) return cudaErrorInvalidDeviceFunction;
    e = cudaFuncSetAttribute(causal_pair_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
    if (e != cudaSuccess) return e;
    causal_pair_kernel<D><<<grid, kThreads, C::kSmemBytes, stream>>>(a, mk, mv, mq, mo);
    return cudaGetLastError();
}

}  // namespace

cudaError_t rd_launch_causal_pair(int B, int Hq, int Hkv, int D, float scale, const void* q,
                                  const void* k, const void* v, const int32_t* cu_seqlens,
                                  int64_t total, int max_len, void* o, int32_t* dev_status,
                                  cudaStream_t stream)
{
    PArgs a;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    const long rows = (long)max_len * a.G;
    a.pairs = (int)((rows + 2 * kM - 1) / (2 * kM));
    if (a.pairs < 1) a.pairs = 1;
    const long units = (long)B * Hkv * a.pairs;
    if (units > 0x7fffffffL) return cudaErrorInvalidValue;
    a.n_units = (int)units;
    a.scale_log2 = scale * kLog2e;
    a.q = static_cast<const uint16_t*>(q);
    a.cu = cu_seqlens;
    a.total = total;
    a.max_len = max_len;
    a.o = static_cast<uint16_t*>(o);
    a.status = dev_status;
    a.stall_budget = rd_attention_stall_budget();
    CUtensorMap mk, mv, mq, mo;
    if (!make_kv_map(&mk, k, total, Hkv, D) || !make_kv_map(&mv, v, total, Hkv, D))
        return cudaErrorInvalidValue;
    // query tiles by TMA, and whole output tiles by TMA stores, when G is a power
    // of two <= 128 (a tile is one box of 128 / G positions x G heads per 64
    // columns; the output has the queries' layout)
    a.q_tma = a.G <= kM && (a.G & (a.G - 1)) == 0 && make_q_map(&mq, q, total, Hq, D, a.G, kM / a.G) &&
              make_q_map(&mo, o, total, Hq, D, a.G, kM / a.G);
    if (!a.q_tma) { mq = mk; mo = mk; }
    const int grid = (int)std::min<long>(units, rd_device_sm_count());
    return D == 128 ? launch_pair<128>(grid, stream, a, mk, mv, mq, mo)
                    : launch_pair<64>(grid, stream, a, mk, mv, mq, mo);
}
