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
// One CTA per request.  Pass 1: log-sum-exp of every beam row (fp32).  Pass 2:
// every thread keeps its best W candidates in registers (insertion), then W
// rounds of a CTA-wide (max score, min index) reduction pick the winners in
// order.  No CTA waits for another.
#include <cuda_bf16.h>

#include "rd_internal.cuh"

namespace {

constexpr int kThreads = 512;
constexpr int kNoIndex = 0x7fffffff;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float bf16_at(const uint16_t* row, int v)
{
    return __uint_as_float((uint32_t)row[v] << 16);
}

// candidate order: higher score first, then lower flat index
__device__ __forceinline__ bool before(float s1, int i1, float s2, int i2)
{
    return s1 > s2 || (s1 == s2 && i1 < i2);
}

template <int W>
__global__ void __launch_bounds__(kThreads)
beam_step_kernel(const uint16_t* __restrict__ logits, const float* __restrict__ scores_in,
                 const int32_t* __restrict__ beams_in, int V, int t,
                 int32_t* __restrict__ beams_out, float* __restrict__ scores_out,
                 int32_t* __restrict__ parent, int32_t* dev_status)
{
    __shared__ float s_red[kThreads / 32];
    __shared__ float s_bias[W];       // scores_in[w] - lse[w]
    __shared__ float s_win[W];
    __shared__ int s_wi[W];
    __shared__ float s_rs[kThreads / 32];
    __shared__ int s_ri[kThreads / 32];
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint16_t* lg = logits + (size_t)b * W * V;

    // ---- pass 1: log-sum-exp per beam row --------------------------------------
    for (int w = 0; w < W; ++w) {
        const uint16_t* row = lg + (size_t)w * V;
        float mx = -INFINITY;
        for (int v = tid; v < V; v += kThreads) mx = fmaxf(mx, bf16_at(row, v));
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) s_red[warp] = mx;
        __syncthreads();
        mx = s_red[0];
        for (int k = 1; k < kThreads / 32; ++k) mx = fmaxf(mx, s_red[k]);
        __syncthreads();
        const float base = mx * kLog2e;
        float sum = 0.f;
        for (int v = tid; v < V; v += kThreads) sum += exp2f(fmaf(bf16_at(row, v), kLog2e, -base));
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) s_red[warp] = sum;
        __syncthreads();
        if (tid == 0) {
            float tot = 0.f;
            for (int k = 0; k < kThreads / 32; ++k) tot += s_red[k];
            const float lse = mx + log2f(tot) * kLn2;
            const float si = scores_in[(size_t)b * W + w];
            s_bias[w] = (si == -INFINITY) ? -INFINITY : si - lse;
        }
        __syncthreads();
    }

    // ---- pass 2: per-thread best W, then W CTA-wide selection rounds ------------
    float ls[W];
    int li[W];
#pragma unroll
    for (int k = 0; k < W; ++k) { ls[k] = -INFINITY; li[k] = kNoIndex; }
    for (int w = 0; w < W; ++w) {
        const float bias = s_bias[w];
        if (bias == -INFINITY) continue;
        const uint16_t* row = lg + (size_t)w * V;
        for (int v = tid; v < V; v += kThreads) {
            float cs = bias + bf16_at(row, v);
            int ci = w * V + v;
            if (!before(cs, ci, ls[W - 1], li[W - 1])) continue;
#pragma unroll
            for (int k = 0; k < W; ++k) {        // insert into the sorted list
                if (before(cs, ci, ls[k], li[k])) {
                    const float ts = ls[k];
                    const int ti = li[k];
                    ls[k] = cs; li[k] = ci;
                    cs = ts; ci = ti;
                }
            }
        }
    }
    int head = 0;
    for (int r = 0; r < W; ++r) {
        float bs = -INFINITY;
        int bi = kNoIndex;
#pragma unroll
        for (int k = 0; k < W; ++k)
            if (k == head) { bs = ls[k]; bi = li[k]; }
        float ws = bs;
        int wi = bi;
        for (int o = 16; o > 0; o >>= 1) {
            const float os = __shfl_xor_sync(0xffffffffu, ws, o);
            const int oi = __shfl_xor_sync(0xffffffffu, wi, o);
            if (before(os, oi, ws, wi)) { ws = os; wi = oi; }
        }
        if (lane == 0) { s_rs[warp] = ws; s_ri[warp] = wi; }
        __syncthreads();
        if (tid == 0) {
            float fs = s_rs[0];
            int fi = s_ri[0];
            for (int k = 1; k < kThreads / 32; ++k)
                if (before(s_rs[k], s_ri[k], fs, fi)) { fs = s_rs[k]; fi = s_ri[k]; }
            s_win[r] = fs;
            s_wi[r] = fi;
        }
        __syncthreads();
        if (bi != kNoIndex && bi == s_wi[r]) ++head;   // the owner of the winner advances
        __syncthreads();
    }
    // ---- outputs ------------------------------------------------------------
    for (int k = tid; k < W * (t + 1); k += kThreads) {
        const int r = k / (t + 1), pos = k % (t + 1);
        const int fi = s_wi[r];
        const bool ok = fi != kNoIndex;
        const int pw = ok ? fi / V : 0, tok = ok ? fi % V : -1;
        beams_out[((size_t)b * W + r) * (t + 1) + pos] =
            pos < t ? (ok ? beams_in[((size_t)b * W + pw) * t + pos] : -1) : tok;
        if (pos == 0) {
            scores_out[(size_t)b * W + r] = s_win[r];
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
#define RD_BEAM_CASE(WW)                                                                     \
    case WW:                                                                                 \
        beam_step_kernel<WW><<<B, kThreads, 0, stream>>>(lg, scores_in, beams_in, V, t,      \
                                                         beams_out, scores_out, parent,      \
                                                         dev_status);                        \
        break;
    switch (W) {
        RD_BEAM_CASE(1) RD_BEAM_CASE(2) RD_BEAM_CASE(3) RD_BEAM_CASE(4) RD_BEAM_CASE(5)
        RD_BEAM_CASE(6) RD_BEAM_CASE(7) RD_BEAM_CASE(8) RD_BEAM_CASE(9) RD_BEAM_CASE(10)
        RD_BEAM_CASE(11) RD_BEAM_CASE(12) RD_BEAM_CASE(13) RD_BEAM_CASE(14) RD_BEAM_CASE(15)
        RD_BEAM_CASE(16)
    default: return cudaErrorInvalidValue;
    }
#undef RD_BEAM_CASE
    return cudaGetLastError();
}
