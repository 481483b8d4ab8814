// rd_beam_search_step kernel: one step of the drafter's beam search.
//
// The RNN drafter runs a beam search from the initial token and the LLM's last
// hidden state and so produces several candidate sequences (Apple x NVIDIA news
// page, paragraph on the RNN draft model; "Recurrent Drafter for Fast
// Speculative Decoding in LLMs", abstract).  One step: every candidate (beam w,
// token v) scores scores_in[w] + log softmax(logits[w])[v]; the W best
// candidates (best first; equal scores go to the lower w*V + v) become the new
// beams.  A beam whose score is -inf (not live yet) contributes no candidate.
//
// One thread-block cluster of C CTAs per request; CTA r takes beam rows r,
// r + C, ....  C = min(W, 8) while the grid fits one wave of two CTAs per SM,
// else min(W, 4) (measured at W = 8: one row per CTA is faster while every CTA
// has its own slot; at 64 requests, two rows per CTA in one wave beat two
// waves of one).  For each of its rows a CTA finds the row's
// log-sum-exp and its W best tokens (higher value first, lower token on ties),
// which are also its best candidates since the row's score offset
// scores_in[w] - lse[w] is common to them.  A row of up to kRegQ x 8 x kThreads
// tokens is read once, with 16-byte loads, into registers: its maximum by packed
// bf16 max, then the sum of exponentials without rescaling, then the tokens at
// or above a threshold (below) from the same registers.  Longer or unaligned
// rows are streamed twice with a running (max, sum).  Selections are by place:
// a candidate's place is the number of candidates ordered before it, counted by
// its own thread, so every candidate is placed at once with no rounds of
// reductions.  Every CTA writes its rows' log-sum-exp and W best into rank 0's
// shared memory and leaves after one cluster barrier; rank 0 places the W x W
// candidates and writes the new beams, whose prefixes and scores it staged at
// start.  No CTA waits for another outside its cluster.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "rd_internal.cuh"

namespace cg = cooperative_groups;

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kNoIndex = 0x7fffffff;
constexpr int kMaxCluster = 8;           // CTAs per request, at most
constexpr int kCtasPerSm = 2;            // resident CTAs per SM (64 registers x 512 threads)
constexpr int kCap = 1024;                 // candidate slots per row (and W x W merge slots)
constexpr int kRegQ = 8;                   // 16-byte words per thread held in registers
constexpr uint32_t kNegInf2 = 0xff80ff80u; // two bf16 -inf
constexpr int kPrefixCap = 512;            // beam prefixes staged in shared memory up to W t
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// candidate order: higher score first, then lower index
__device__ __forceinline__ bool before(float s1, int i1, float s2, int i2)
{
    return s1 > s2 || (s1 == s2 && i1 < i2);
}

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b)   // per-half bf16 max
{
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float ex2(float x)      // 2^x; x <= 0 here, -inf gives 0
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// the larger of the two bf16 values of every word of a 16-byte group, as fp32
__device__ __forceinline__ float group_max(const uint4& x)
{
    const uint32_t m = bmax2(bmax2(x.x, x.y), bmax2(x.z, x.w));
    return fmaxf(lo_bf16(m), hi_bf16(m));
}

template <int W>
struct RowOut {
    float lse;           // natural-log log-sum-exp of the row (-inf: row not live)
    float val[W];        // the row's W best logits, best first
    int tok[W];
};

template <int W>
__global__ void __launch_bounds__(kThreads, 2)
beam_step_kernel(const uint16_t* __restrict__ logits, const float* __restrict__ scores_in,
                 const int32_t* __restrict__ beams_in, int V, int t,
                 int32_t* __restrict__ beams_out, float* __restrict__ scores_out,
                 int32_t* __restrict__ parent, int32_t* dev_status)
{
    __shared__ RowOut<W> s_row[W];            // this CTA's rows (ceil(W / C) of them)
    __shared__ RowOut<W> s_all[W];            // rank 0: every row of the request
    __shared__ float s_sc[W];                 // rank 0: scores_in of the request
    __shared__ int s_bin[kPrefixCap];         // rank 0: beams_in of the request (W t <= cap)
    __shared__ float2 s_red[kWarps];
    __shared__ float s_rs[kWarps];
    __shared__ int s_ri[kWarps];
    __shared__ float s_win[W];
    __shared__ int s_wi[W];
    __shared__ float s_cv[kCap];          // candidates of a row: logit and token
    __shared__ int s_ci[kCap];
    __shared__ int s_cnt;

    const cg::cluster_group cl = cg::this_cluster();
    const int C = (int)cl.num_blocks();
    const int rank = (int)cl.block_rank();
    const int b = blockIdx.x / C;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    static_assert(W * W <= kCap, "merge slots");

    // The CTAs write their rows into rank 0's shared memory once every CTA of the
    // cluster has started: arrive now, wait just before those writes.
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    const bool stage_prefix = W * t <= kPrefixCap;
    if (rank == 0) {                           // what the merge reads, early
        if (tid < W) s_sc[tid] = scores_in[(size_t)b * W + tid];
        if (stage_prefix)
            for (int e = tid; e < W * t; e += kThreads) s_bin[e] = beams_in[(size_t)b * W * t + e];
    }

    // W rounds of a CTA-wide (best score, lowest index) selection over the
    // threads' sorted lists ls/li; the winners land in s_win / s_wi
    auto select = [&](float (&ls)[W], int (&li)[W]) {
        int head = 0;
        for (int r = 0; r < W; ++r) {
            float bs = -INFINITY;
            int bi = kNoIndex;
#pragma unroll
            for (int k = 0; k < W; ++k)
                if (k == head) { bs = ls[k]; bi = li[k]; }
            float ws = bs;
            int wi = bi;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float os = __shfl_xor_sync(0xffffffffu, ws, o);
                const int oi = __shfl_xor_sync(0xffffffffu, wi, o);
                if (before(os, oi, ws, wi)) { ws = os; wi = oi; }
            }
            if (lane == 0) { s_rs[warp] = ws; s_ri[warp] = wi; }
            __syncthreads();
            if (warp == 0) {                     // the warps' winners, by shuffles
                float fs = lane < kWarps ? s_rs[lane] : -INFINITY;
                int fi = lane < kWarps ? s_ri[lane] : kNoIndex;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float os = __shfl_xor_sync(0xffffffffu, fs, o);
                    const int oi = __shfl_xor_sync(0xffffffffu, fi, o);
                    if (before(os, oi, fs, fi)) { fs = os; fi = oi; }
                }
                if (lane == 0) { s_win[r] = fs; s_wi[r] = fi; }
            }
            __syncthreads();
            if (bi != kNoIndex && bi == s_wi[r]) ++head;   // the owner of the winner advances
        }
        __syncthreads();
    };

    // ---- this CTA's rows: one pass each --------------------------------------
    const int rows = (W + C - 1) / C;
    const int n4 = V / 8;
    for (int k = 0; k < rows; ++k) {
        const int w = rank + k * C;
        RowOut<W>& out = s_row[k];
        if (w >= W || scores_in[(size_t)b * W + w] == -INFINITY) {   // no candidates
            if (tid == 0) out.lse = -INFINITY;
            continue;
        }
        const uint16_t* row = logits + ((size_t)b * W + w) * V;
        const bool vec = (V % 8 == 0) && (reinterpret_cast<uintptr_t>(row) % 16 == 0);
        const uint4* r4 = reinterpret_cast<const uint4*>(row);
        const bool in_regs = vec && n4 <= kRegQ * kThreads;
        // visit every token of the row: f(logit, token), four 16-byte loads in
        // flight per thread before any of them is used
        auto for_row = [&](auto&& f) {
            if (vec) {
                for (int base = tid; base < n4; base += 4 * kThreads) {
                    uint4 x[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int i = base + q * kThreads;
                        x[q] = i < n4 ? __ldg(r4 + i) : make_uint4(0, 0, 0, 0);
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int i = base + q * kThreads;
                        if (i >= n4) break;
                        const uint32_t xw[4] = {x[q].x, x[q].y, x[q].z, x[q].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            f(lo_bf16(xw[e]), i * 8 + 2 * e);
                            f(hi_bf16(xw[e]), i * 8 + 2 * e + 1);
                        }
                    }
                }
            } else {
                for (int v = tid; v < V; v += kThreads)
                    f(__uint_as_float((uint32_t)__ldg(row + v) << 16), v);
            }
        };
        // ---- pass 1: this thread's maximum and sum of exponentials (log2 units)
        float m = -INFINITY, sum = 0.f, tmax = -INFINITY;
        uint4 x[kRegQ];                            // the held row (in_regs)
        if (in_regs) {
#pragma unroll
            for (int q = 0; q < kRegQ; ++q) {
                const int i = tid + q * kThreads;
                x[q] = i < n4 ? __ldg(r4 + i) : make_uint4(kNegInf2, kNegInf2, kNegInf2, kNegInf2);
            }
#pragma unroll
            for (int q = 0; q < kRegQ; ++q) tmax = fmaxf(tmax, group_max(x[q]));
            if (tmax != -INFINITY) {
                m = tmax * kLog2e;
#pragma unroll
                for (int q = 0; q < kRegQ; ++q) {
                    if (tid + q * kThreads < n4) {
                        const uint32_t xw[4] = {x[q].x, x[q].y, x[q].z, x[q].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            sum += ex2(fmaf(lo_bf16(xw[e]), kLog2e, -m)) +
                                   ex2(fmaf(hi_bf16(xw[e]), kLog2e, -m));
                    }
                }
            }
        } else {
            for_row([&](float xv, int) {
                const float y = xv * kLog2e;
                if (y > m) { sum = (m == -INFINITY) ? 0.f : sum * ex2(m - y); m = y; }
                if (y != -INFINITY) sum += ex2(y - m);
                tmax = fmaxf(tmax, xv);
            });
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float om = __shfl_xor_sync(0xffffffffu, m, o);
            const float os = __shfl_xor_sync(0xffffffffu, sum, o);
            const float nm = fmaxf(m, om);
            sum = (nm == -INFINITY) ? 0.f : sum * ex2(m - nm) + os * ex2(om - nm);
            m = nm;
        }
        // a threshold: the W-th largest of a warp's 32 thread maxima.  At least W
        // tokens of the row reach it, so every token of the row's top W does too
        float tw = -INFINITY;
        {
            float cv = tmax;
            for (int r = 0; r < W; ++r) {
                float wm = cv;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
                tw = wm;
                const unsigned owner = __ballot_sync(0xffffffffu, cv == wm);
                if (lane == __ffs(owner) - 1) cv = -INFINITY;   // one maximum leaves per round
            }
        }
        if (lane == 0) { s_red[warp] = make_float2(m, sum); s_rs[warp] = tw; }
        if (tid == 0) s_cnt = 0;
        __syncthreads();
        float thr = -INFINITY;
        for (int q = 0; q < kWarps; ++q) thr = fmaxf(thr, s_rs[q]);
        if (warp == 0) {                           // the row's log-sum-exp, by shuffles
            float M = lane < kWarps ? s_red[lane].x : -INFINITY;
            float S = lane < kWarps ? s_red[lane].y : 0.f;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float om = __shfl_xor_sync(0xffffffffu, M, o);
                const float os = __shfl_xor_sync(0xffffffffu, S, o);
                const float nm = fmaxf(M, om);
                S = (nm == -INFINITY) ? 0.f : S * ex2(M - nm) + os * ex2(om - nm);
                M = nm;
            }
            if (lane == 0) out.lse = (M + log2f(S)) * kLn2;
        }
        // ---- pass 2: the tokens that reach the threshold -------------------------
        auto keep = [&](float xv, int v) {
            if (xv >= thr) {
                const int slot = atomicAdd(&s_cnt, 1);
                if (slot < kCap) { s_cv[slot] = xv; s_ci[slot] = v; }
            }
        };
        if (in_regs) {
#pragma unroll
            for (int q = 0; q < kRegQ; ++q) {
                const int i = tid + q * kThreads;
                if (i < n4 && group_max(x[q]) >= thr) {   // most groups hold no candidate
                    const uint32_t xw[4] = {x[q].x, x[q].y, x[q].z, x[q].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        keep(lo_bf16(xw[e]), i * 8 + 2 * e);
                        keep(hi_bf16(xw[e]), i * 8 + 2 * e + 1);
                    }
                }
            }
        } else {
            for_row(keep);                         // a second read, from L1/L2
        }
        __syncthreads();
        const int cnt = s_cnt;
        if (cnt <= kCap) {
            // the row's W best among the candidates: a candidate's place is the
            // number of candidates before it (tokens differ, so the order is strict)
            if (tid < W && tid >= cnt) { out.val[tid] = -INFINITY; out.tok[tid] = kNoIndex; }
            for (int c = tid; c < cnt; c += kThreads) {
                const float cv = s_cv[c];
                const int ci = s_ci[c];
                int place = 0;
                for (int d = 0; d < cnt; ++d) place += before(s_cv[d], s_ci[d], cv, ci) ? 1 : 0;
                if (place < W) { out.val[place] = cv; out.tok[place] = ci; }
            }
        } else {
            // more candidates than room (ties or -inf rows): every thread's best W,
            // then W CTA-wide rounds
            float ls[W];
            int li[W];
#pragma unroll
            for (int q = 0; q < W; ++q) { ls[q] = -INFINITY; li[q] = kNoIndex; }
            for_row([&](float xv, int v) {
                if (!before(xv, v, ls[W - 1], li[W - 1])) return;
                float cs = xv;
                int ci = v;
#pragma unroll
                for (int q = 0; q < W; ++q) {    // insert into the sorted list
                    if (before(cs, ci, ls[q], li[q])) {
                        const float ts = ls[q];
                        const int ti = li[q];
                        ls[q] = cs; li[q] = ci;
                        cs = ts; ci = ti;
                    }
                }
            });
            select(ls, li);
            if (tid < W) {
                out.val[tid] = s_win[tid];
                out.tok[tid] = s_wi[tid];
            }
        }
        __syncthreads();
    }
    // ---- every row into rank 0's shared memory ---------------------------------
    __syncthreads();                             // s_row complete
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");   // every CTA has started
    {
        constexpr int kWords = (int)(sizeof(RowOut<W>) / 4);
        uint32_t* dst = reinterpret_cast<uint32_t*>(cl.map_shared_rank(&s_all[0], 0));
        const uint32_t* src = reinterpret_cast<const uint32_t*>(&s_row[0]);
        for (int e = tid; e < rows * kWords; e += kThreads) {
            const int w = rank + (e / kWords) * C;
            if (w < W) dst[w * kWords + e % kWords] = src[e];
        }
    }
    cl.sync();                                   // rows published to rank 0
    if (rank != 0) return;                       // no shared memory of a peer is read after this

    // ---- rank 0: the request's W best candidates ---------------------------------
    // candidate (row w, its q-th best) in slot w W + q; its place among the W x W
    // is the number of candidates before it (equal pairs: the lower slot first)
    for (int c = tid; c < W * W; c += kThreads) {
        const int w = c / W, q = c % W;
        const RowOut<W>& ro = s_all[w];
        float cs = -INFINITY;
        int ci = kNoIndex;
        if (ro.lse != -INFINITY && ro.tok[q] != kNoIndex) {
            cs = s_sc[w] + (ro.val[q] - ro.lse);
            ci = w * V + ro.tok[q];
        }
        s_cv[c] = cs;
        s_ci[c] = ci;
    }
    __syncthreads();
    for (int c = tid; c < W * W; c += kThreads) {
        const float cs = s_cv[c];
        const int ci = s_ci[c];
        int place = 0;
        for (int d = 0; d < W * W; ++d) {
            const float ds = s_cv[d];
            const int di = s_ci[d];
            place += (before(ds, di, cs, ci) || (ds == cs && di == ci && d < c)) ? 1 : 0;
        }
        if (place < W) { s_win[place] = cs; s_wi[place] = ci; }
    }
    __syncthreads();
    for (int k = tid; k < W * (t + 1); k += kThreads) {
        const int r = k / (t + 1), pos = k % (t + 1);
        const int fi = s_wi[r];
        const bool ok = fi != kNoIndex && s_win[r] != -INFINITY;
        const int pw = ok ? fi / V : 0, tok = ok ? fi % V : -1;
        beams_out[((size_t)b * W + r) * (t + 1) + pos] =
            pos < t ? (ok ? (stage_prefix ? s_bin[pw * t + pos]
                                          : beams_in[((size_t)b * W + pw) * t + pos]) : -1) : tok;
        if (pos == 0) {
            scores_out[(size_t)b * W + r] = ok ? s_win[r] : -INFINITY;
            parent[(size_t)b * W + r] = ok ? pw : -1;
            if (!ok) rd_flag(dev_status, RD_DEV_BAD_LENGTH);
        }
    }
}

}  // namespace

cudaError_t rd_launch_beam_step(const void* logits, const float* scores_in,
                                const int32_t* beams_in, int B, int W, int V, int t,
                                int32_t* beams_out, float* scores_out, int32_t* parent,
                                int32_t* dev_status, cudaStream_t stream)
{
    const uint16_t* lg = static_cast<const uint16_t*>(logits);
    int C = W < kMaxCluster ? W : kMaxCluster;
    if ((long)B * C > (long)kCtasPerSm * rd_device_sm_count()) C = W < 4 ? W : 4;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(B * C));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
#define RD_BEAM_CASE(WW)                                                                     \
    case WW:                                                                                 \
        return cudaLaunchKernelEx(&cfg, beam_step_kernel<WW>, lg, scores_in, beams_in, V, t, \
                                  beams_out, scores_out, parent, dev_status);
    switch (W) {
        RD_BEAM_CASE(1) RD_BEAM_CASE(2) RD_BEAM_CASE(3) RD_BEAM_CASE(4) RD_BEAM_CASE(5)
        RD_BEAM_CASE(6) RD_BEAM_CASE(7) RD_BEAM_CASE(8) RD_BEAM_CASE(9) RD_BEAM_CASE(10)
        RD_BEAM_CASE(11) RD_BEAM_CASE(12) RD_BEAM_CASE(13) RD_BEAM_CASE(14) RD_BEAM_CASE(15)
        RD_BEAM_CASE(16)
    default: return cudaErrorInvalidValue;
    }
#undef RD_BEAM_CASE
}
