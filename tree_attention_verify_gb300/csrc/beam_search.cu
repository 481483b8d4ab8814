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
// One thread-block cluster of up to four CTAs per request; CTA r takes beam
// rows r, r + 4, ... (clusters of four with two rows per CTA measured faster
// than one CTA per row at W = 8).  For each of its rows a CTA streams the row
// with 16-byte loads for the running (max, sum of exponentials) and the
// candidates, and selects the row's W best tokens (higher value first, lower
// token on ties), which are also its best candidates since the row's score
// offset scores_in[w] - lse[w] is common to them.  Rank 0 of the cluster reads
// every row's log-sum-exp and W candidates from distributed shared memory and
// picks the request's W best.  No CTA waits for another outside its cluster.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "rd_internal.cuh"

namespace cg = cooperative_groups;

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kNoIndex = 0x7fffffff;
constexpr int kMaxCluster = 4;           // CTAs per request
constexpr int kCap = 1024;                 // candidate slots per row
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// candidate order: higher score first, then lower index
__device__ __forceinline__ bool before(float s1, int i1, float s2, int i2)
{
    return s1 > s2 || (s1 == s2 && i1 < i2);
}

template <int W>
struct RowOut {
    float lse;           // natural-log log-sum-exp of the row (-inf: row not live)
    float val[W];        // the row's W best logits, best first
    int tok[W];
};

template <int W>
__global__ void __launch_bounds__(kThreads)
beam_step_kernel(const uint16_t* __restrict__ logits, const float* __restrict__ scores_in,
                 const int32_t* __restrict__ beams_in, int V, int t,
                 int32_t* __restrict__ beams_out, float* __restrict__ scores_out,
                 int32_t* __restrict__ parent, int32_t* dev_status)
{
    constexpr int kRowsPerCta = (W + kMaxCluster - 1) / kMaxCluster;
    __shared__ RowOut<W> s_row[kRowsPerCta];
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
    for (int k = 0; k < kRowsPerCta; ++k) {
        const int w = rank + k * C;
        RowOut<W>& out = s_row[k];
        const bool live = w < W && scores_in[(size_t)b * W + w] != -INFINITY;
        if (!live) {
            if (tid == 0) out.lse = -INFINITY;
            continue;
        }
        const uint16_t* row = logits + ((size_t)b * W + w) * V;
        const bool vec = (V % 8 == 0) && (reinterpret_cast<uintptr_t>(row) % 16 == 0);
        // visit every token of the row: f(logit, token), four 16-byte loads in
        // flight per thread before any of them is used
        auto for_row = [&](auto&& f) {
            if (vec) {
                const uint4* r4 = reinterpret_cast<const uint4*>(row);
                const int n4 = V / 8;
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
                            f(__uint_as_float(xw[e] << 16), i * 8 + 2 * e);
                            f(__uint_as_float(xw[e] & 0xffff0000u), i * 8 + 2 * e + 1);
                        }
                    }
                }
            } else {
                for (int v = tid; v < V; v += kThreads)
                    f(__uint_as_float((uint32_t)__ldg(row + v) << 16), v);
            }
        };
        // ---- pass 1: log-sum-exp and every thread's best token ----------------
        float m = -INFINITY, sum = 0.f;          // log2 units
        float bv = -INFINITY;
        int bi = kNoIndex;
        for_row([&](float x, int v) {
            const float y = x * kLog2e;
            if (y > m) { sum = (m == -INFINITY) ? 0.f : sum * exp2f(m - y); m = y; }
            if (y != -INFINITY) sum += exp2f(y - m);
            if (before(x, v, bv, bi)) { bv = x; bi = v; }
        });
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float om = __shfl_xor_sync(0xffffffffu, m, o);
            const float os = __shfl_xor_sync(0xffffffffu, sum, o);
            const float nm = fmaxf(m, om);
            sum = (nm == -INFINITY) ? 0.f : sum * exp2f(m - nm) + os * exp2f(om - nm);
            m = nm;
        }
        // a threshold: the W-th best of a warp's 32 thread maxima.  At least W
        // tokens of the row reach it, so every token of the row's top W does too
        float tw = -INFINITY;
        {
            float cv = bv;
            int ci = bi;
            for (int r = 0; r < W; ++r) {
                float ws = cv;
                int wi = ci;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float os = __shfl_xor_sync(0xffffffffu, ws, o);
                    const int oi = __shfl_xor_sync(0xffffffffu, wi, o);
                    if (before(os, oi, ws, wi)) { ws = os; wi = oi; }
                }
                if (r == W - 1) tw = (wi == kNoIndex) ? -INFINITY : ws;
                if (ci != kNoIndex && ci == wi) { cv = -INFINITY; ci = kNoIndex; }
            }
        }
        if (lane == 0) { s_red[warp] = make_float2(m, sum); s_rs[warp] = tw; }
        if (tid == 0) s_cnt = 0;
        __syncthreads();
        float thr = -INFINITY;
        for (int q = 0; q < kWarps; ++q) thr = fmaxf(thr, s_rs[q]);
        if (tid == 0) {
            float M = -INFINITY, S = 0.f;
            for (int q = 0; q < kWarps; ++q) {
                const float nm = fmaxf(M, s_red[q].x);
                S = (nm == -INFINITY) ? 0.f : S * exp2f(M - nm) + s_red[q].y * exp2f(s_red[q].x - nm);
                M = nm;
            }
            out.lse = (M + log2f(S)) * kLn2;
        }
        // ---- pass 2: the tokens that reach the threshold (from L1/L2) -----------
        for_row([&](float x, int v) {
            if (x >= thr) {
                const int k = atomicAdd(&s_cnt, 1);
                if (k < kCap) { s_cv[k] = x; s_ci[k] = v; }
            }
        });
        __syncthreads();
        const int cnt = s_cnt;
        if (cnt <= kCap) {
            // the row's W best among the candidates, by one warp
            if (warp == 0) {
                for (int r = 0; r < W; ++r) {
                    float ws = -INFINITY;
                    int wi = kNoIndex, wk = -1;
                    for (int q = lane; q < cnt; q += 32)
                        if (s_ci[q] != kNoIndex && before(s_cv[q], s_ci[q], ws, wi)) {
                            ws = s_cv[q]; wi = s_ci[q]; wk = q;
                        }
                    const int mine = wi;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        const float os = __shfl_xor_sync(0xffffffffu, ws, o);
                        const int oi = __shfl_xor_sync(0xffffffffu, wi, o);
                        if (before(os, oi, ws, wi)) { ws = os; wi = oi; }
                    }
                    if (lane == 0) { out.val[r] = ws; out.tok[r] = wi; }
                    if (mine != kNoIndex && mine == wi) s_ci[wk] = kNoIndex;   // taken
                    __syncwarp();
                }
            }
        } else {
            // more candidates than room (ties or -inf rows): every thread's best W,
            // then W CTA-wide rounds
            float ls[W];
            int li[W];
#pragma unroll
            for (int q = 0; q < W; ++q) { ls[q] = -INFINITY; li[q] = kNoIndex; }
            for_row([&](float x, int v) {
                if (!before(x, v, ls[W - 1], li[W - 1])) return;
                float cs = x;
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
    cl.sync();                                   // every row published

    // ---- rank 0: the request's W best candidates -------------------------------
    if (rank == 0) {
        float ls[W];
        int li[W];
#pragma unroll
        for (int q = 0; q < W; ++q) { ls[q] = -INFINITY; li[q] = kNoIndex; }
        if (tid < W * W) {                           // candidate (row w, its q-th best)
            const int w = tid / W, q = tid % W;
            const RowOut<W>* ro = cl.map_shared_rank(&s_row[w / C], w % C);
            const float lse = ro->lse;
            const int tok = ro->tok[q];
            if (lse != -INFINITY && tok != kNoIndex) {
                ls[0] = scores_in[(size_t)b * W + w] + (ro->val[q] - lse);
                li[0] = w * V + tok;
            }
        }
        select(ls, li);
        for (int k = tid; k < W * (t + 1); k += kThreads) {
            const int r = k / (t + 1), pos = k % (t + 1);
            const int fi = s_wi[r];
            const bool ok = fi != kNoIndex && s_win[r] != -INFINITY;
            const int pw = ok ? fi / V : 0, tok = ok ? fi % V : -1;
            beams_out[((size_t)b * W + r) * (t + 1) + pos] =
                pos < t ? (ok ? beams_in[((size_t)b * W + pw) * t + pos] : -1) : tok;
            if (pos == 0) {
                scores_out[(size_t)b * W + r] = ok ? s_win[r] : -INFINITY;
                parent[(size_t)b * W + r] = ok ? pw : -1;
                if (!ok) rd_flag(dev_status, RD_DEV_BAD_LENGTH);
            }
        }
    }
    cl.sync();                                   // rank 0 is done reading its peers
}

}  // namespace

cudaError_t rd_launch_beam_step(const void* logits, const float* scores_in,
                                const int32_t* beams_in, int B, int W, int V, int t,
                                int32_t* beams_out, float* scores_out, int32_t* parent,
                                int32_t* dev_status, cudaStream_t stream)
{
    const uint16_t* lg = static_cast<const uint16_t*>(logits);
    const int C = W < kMaxCluster ? W : kMaxCluster;
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
