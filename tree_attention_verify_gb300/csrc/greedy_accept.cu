// rd_greedy_accept kernel: vocab argmax at every packed node, then per-request
// acceptance of the longest draft prefix that greedy decoding reproduces.
//
// Greedy verification picks the best beam before the next drafting step (NVIDIA
// blog "ReDrafter in TensorRT-LLM", introduction; greedy decoding: Apple x
// NVIDIA news page, benchmark paragraph).  The argmax is taken once per PACKED
// row, so deduplicated positions are read once and [B, W, L, V] logits are never
// formed.
//
// Two launches.  Argmax grid: CTA (x = p*splits + s, y = b) scans vocab chunk s
// of row (b, p) with 16-byte streaming loads, reduces (max value, lowest index)
// in the CTA, folds it into a 64-bit key with atomicMax (high word =
// order-preserving bits of the fp32 value, low word = ~index, so the maximum key
// is the maximum value with the lowest index) and exits: no fence, no ticket, so
// a CTA holds its slot only while it streams.  Acceptance grid, one CTA per
// request: a programmatic-dependent launch, scheduled while the argmax grid
// runs, that waits until that grid has completed and its keys are visible,
// then decodes and resets the keys and runs the acceptance.  No CTA spins on
// another.
#include <cuda_bf16.h>

#include "rd_internal.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kVecPerIter = 4;          // 16-byte loads in flight per thread
constexpr int kStage = 512;             // beams / unpacker entries staged for the acceptance walk
constexpr int kNoIndex = 0x7fffffff;

__device__ __forceinline__ uint4 ld_stream(const uint4* p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float max8(const uint4& x)
{
    __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&x.x),
                               *reinterpret_cast<const __nv_bfloat162*>(&x.y));
    __nv_bfloat162 c = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&x.z),
                               *reinterpret_cast<const __nv_bfloat162*>(&x.w));
    __nv_bfloat162 m = __hmax2(a, c);
    uint32_t u = *reinterpret_cast<uint32_t*>(&m);
    return fmaxf(bf16_lo(u), bf16_hi(u));
}

__device__ __forceinline__ float elem8(const uint4& x, int e)
{
    uint32_t w = (e < 2) ? x.x : (e < 4) ? x.y : (e < 6) ? x.z : x.w;
    return (e & 1) ? bf16_hi(w) : bf16_lo(w);
}

// Larger key <=> larger value, then lower index.  -0 is folded into +0 so the
// two zeros tie, as they compare equal.
__device__ __forceinline__ unsigned long long make_key(float v, int idx)
{
    uint32_t u = __float_as_uint(__fadd_rn(v, 0.0f));
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)u << 32) | (unsigned long long)(0xffffffffu - (uint32_t)idx);
}

__device__ __forceinline__ void better(float& best, int& bidx, float v, int i)
{
    if (v > best || (v == best && i < bidx)) { best = v; bidx = i; }
}

// Acceptance of request b (its CTA of the acceptance grid): decode and reset
// the argmax keys, then walk every beam.  The request's beams and unpacker rows
// are staged in shared memory with one coalesced load when they fit, so a beam's
// walk costs no dependent global round trips.
__device__ __noinline__ void accept_request(int b, int P_max, int V, int Pb, bool bad_len,
                                            const int32_t* __restrict__ beams,
                                            const int32_t* __restrict__ unpacker, int W, int L,
                                            int32_t* __restrict__ argmax_out,
                                            int32_t* __restrict__ accept_len,
                                            int32_t* __restrict__ best_beam,
                                            int32_t* __restrict__ n_accepted,
                                            int32_t* __restrict__ out_tokens,
                                            unsigned long long* keys,
                                            int32_t* dev_status, int* s_g, int* s_acc,
                                            int* s_bb, int* s_up)
{
    const int tid = threadIdx.x;
    const int32_t* bb = beams + (size_t)b * W * L;
    const int32_t* up = unpacker + (size_t)b * W * L;
    const bool staged = W * L <= kStage;
    for (int q = tid; q < P_max; q += kThreads) {
        const unsigned long long k = atomicExch(keys + (size_t)b * P_max + q, 0ull);
        const int g = (bad_len || q >= Pb) ? -1 : (int)(0xffffffffu - (uint32_t)k);
        s_g[q] = g;
        argmax_out[(size_t)b * P_max + q] = g;
    }
    if (staged) {
        for (int i = tid; i < W * L; i += kThreads) {
            s_bb[i] = __ldg(bb + i);
            s_up[i] = __ldg(up + i);
        }
    }
    __syncthreads();
    const int32_t* wb = staged ? s_bb : bb;
    const int32_t* wu = staged ? s_up : up;
    if (tid < W) {
        int a = 0;
        if (!bad_len) {
            for (int j = 1; j < L; ++j) {
                const int prev = wu[tid * L + j - 1];
                const int tok = wb[tid * L + j];
                if (prev < 0 || prev >= Pb) { rd_flag(dev_status, RD_DEV_BAD_INDEX); break; }
                if (tok < 0 || tok >= V) rd_flag(dev_status, RD_DEV_BAD_TOKEN);
                if (tok != s_g[prev]) break;
                a = j;
            }
        }
        s_acc[tid] = a;
        accept_len[(size_t)b * W + tid] = a;
    }
    __syncthreads();
    if (tid == 0) {
        if (bad_len) rd_flag(dev_status, RD_DEV_BAD_LENGTH);
        int best = 0;
        for (int w = 1; w < W; ++w)
            if (s_acc[w] > s_acc[best]) best = w;
        const int a = s_acc[best];
        best_beam[b] = best;
        n_accepted[b] = a;
        int32_t* ot = out_tokens + (size_t)b * L;
        for (int j = 0; j < L; ++j) ot[j] = -1;
        for (int j = 1; j <= a; ++j) ot[j - 1] = wb[best * L + j];
        const int last = wu[best * L + a];
        if (!bad_len) {
            if (last >= 0 && last < Pb) ot[a] = s_g[last];
            else rd_flag(dev_status, RD_DEV_BAD_INDEX);
        }
    }
}

template <bool kVec>
__global__ void __launch_bounds__(kThreads)
argmax_kernel(const uint16_t* __restrict__ logits, int P_max, int V, int splits, int chunk,
              const int32_t* __restrict__ packed_len, unsigned long long* keys)
{
    // the acceptance grid may launch now: it waits for this grid to complete
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ float s_best[kThreads / RD_WARP];
    __shared__ int s_idx[kThreads / RD_WARP];

    const int b = blockIdx.y;
    const int p = blockIdx.x / splits;
    const int s = blockIdx.x % splits;
    const int tid = threadIdx.x;
    const int Pb = __ldg(packed_len + b);
    const bool bad_len = Pb < 0 || Pb > P_max;

    if (!bad_len && p < Pb) {
        const int v0 = s * chunk;
        const int v1 = min(V, v0 + chunk);
        const uint16_t* row = logits + ((size_t)b * P_max + p) * (size_t)V;
        float best = -INFINITY;
        int bidx = kNoIndex, first = kNoIndex;
        if (kVec) {
            const uint4* rv = reinterpret_cast<const uint4*>(row);
            const int q0 = v0 >> 3, q1 = v1 >> 3;
            for (int base = q0; base < q1; base += kThreads * kVecPerIter) {
                uint4 x[kVecPerIter];
#pragma unroll
                for (int k = 0; k < kVecPerIter; ++k) {
                    const int qi = base + k * kThreads + tid;
                    if (qi < q1) x[k] = ld_stream(rv + qi);
                }
#pragma unroll
                for (int k = 0; k < kVecPerIter; ++k) {
                    const int qi = base + k * kThreads + tid;
                    if (qi < q1) {
                        if (first == kNoIndex) first = qi * 8;
                        const float m = max8(x[k]);
                        if (m > best) {                  // first element equal to m
                            int e = 0;
                            while (e < 7 && elem8(x[k], e) != m) ++e;
                            best = m;
                            bidx = qi * 8 + e;
                        }
                    }
                }
            }
        } else {
            for (int v = v0 + tid; v < v1; v += kThreads) {
                const float x = __uint_as_float(((uint32_t)__ldg(row + v)) << 16);
                if (first == kNoIndex) first = v;
                if (x > best) { best = x; bidx = v; }
            }
        }
        if (bidx == kNoIndex && first != kNoIndex) bidx = first;   // every value -inf
        // CTA reduction: max value, lowest index
#pragma unroll
        for (int off = RD_WARP / 2; off > 0; off >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bidx, off);
            better(best, bidx, ob, oi);
        }
        if ((tid & 31) == 0) { s_best[tid >> 5] = best; s_idx[tid >> 5] = bidx; }
        __syncthreads();
        if (tid == 0) {
            for (int w = 1; w < kThreads / RD_WARP; ++w) better(best, bidx, s_best[w], s_idx[w]);
            if (bidx != kNoIndex) atomicMax(keys + (size_t)b * P_max + p, make_key(best, bidx));
        }
    }
}

// Acceptance of request b, once every argmax key of the launch before is final
// (a programmatic-dependent launch: griddepcontrol.wait returns when that grid
// has completed and its writes are visible).
__global__ void __launch_bounds__(kThreads)
accept_kernel(int P_max, int V, const int32_t* __restrict__ beams,
              const int32_t* __restrict__ unpacker, const int32_t* __restrict__ packed_len,
              int W, int L, int32_t* __restrict__ argmax_out, int32_t* __restrict__ accept_len,
              int32_t* __restrict__ best_beam, int32_t* __restrict__ n_accepted,
              int32_t* __restrict__ out_tokens, unsigned long long* keys, int32_t* dev_status)
{
    __shared__ int s_g[RD_MAX_PACKED];
    __shared__ int s_acc[RD_MAX_BEAMS];
    __shared__ int s_bb[kStage];
    __shared__ int s_up[kStage];
    const int b = blockIdx.x;
    const int Pb = __ldg(packed_len + b);
    const bool bad_len = Pb < 0 || Pb > P_max;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    accept_request(b, P_max, V, Pb, bad_len, beams, unpacker, W, L, argmax_out, accept_len,
                   best_beam, n_accepted, out_tokens, keys, dev_status, s_g, s_acc,
                   s_bb, s_up);
}

}  // namespace

// keys [B*P_max] (64-bit), then one reserved 32-bit word per request (part of
// the size rd.h states; never written, so the workspace stays zero)
size_t rd_accept_workspace_bytes(int B, int P_max)
{
    return (size_t)B * P_max * sizeof(unsigned long long) + (size_t)B * sizeof(unsigned int);
}

rd_accept_plan rd_accept_make_plan(int B, int P_max, int V)
{
    // enough CTAs to cover the SMs several times, but at least ~16 KB per CTA
    const long rows = (long)B * P_max;
    const long target_ctas = 8L * rd_device_sm_count();
    long splits = (target_ctas + rows - 1) / rows;
    long max_splits = ((long)V * 2 + 16383) / 16384;
    if (splits > max_splits) splits = max_splits;
    if (splits < 1) splits = 1;
    long chunk = ((V + splits - 1) / splits + 7) & ~7L;
    splits = (V + chunk - 1) / chunk;
    rd_accept_plan plan;
    plan.splits = (int)splits;
    plan.chunk = (int)chunk;
    return plan;
}

cudaError_t rd_launch_greedy_accept(const void* logits, int B, int P_max, int V,
                                    const int32_t* beams, const int32_t* unpacker,
                                    const int32_t* packed_len, int W, int L,
                                    int32_t* argmax, int32_t* accept_len,
                                    int32_t* best_beam, int32_t* n_accepted,
                                    int32_t* out_tokens, void* workspace,
                                    int32_t* dev_status, cudaStream_t stream)
{
    const rd_accept_plan plan = rd_accept_make_plan(B, P_max, V);
    auto* keys = static_cast<unsigned long long*>(workspace);
    const bool vec = (V % 8 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
    dim3 grid((unsigned)(P_max * plan.splits), (unsigned)B);
    const uint16_t* lg = static_cast<const uint16_t*>(logits);
    if (vec)
        argmax_kernel<true><<<grid, kThreads, 0, stream>>>(lg, P_max, V, plan.splits, plan.chunk,
                                                           packed_len, keys);
    else
        argmax_kernel<false><<<grid, kThreads, 0, stream>>>(lg, P_max, V, plan.splits, plan.chunk,
                                                            packed_len, keys);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)B);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, accept_kernel, P_max, V, beams, unpacker, packed_len, W, L,
                              argmax, accept_len, best_beam, n_accepted, out_tokens, keys,
                              dev_status);
}
