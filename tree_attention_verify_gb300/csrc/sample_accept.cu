// rd_sample_accept kernel: stochastic verification of the draft tree by
// multi-step speculative sampling.
//
// Rejection sampling (speculative-decoding survey page, rejection-sampling
// paragraph) keeps a drafted token x when u < p(x) / q(x); SpecInfer's
// multi-step speculative sampling (same page, "Token Tree Verifier") tests the
// children of the current node in turn and replaces the target by the
// normalised residual max(0, p - q) after every rejection; when no child is
// kept, one token is drawn from the current target.
//
// One thread-block cluster per request walks its tree; the CTAs of the cluster
// split the vocabulary and combine their partial results through distributed
// shared memory, so every CTA takes the same decisions.  Only the nodes on the
// walk are read: for each visited node one pass over its target and draft rows
// gives the softmax maxima and sums (p and q are then known per element), each
// rejection costs one more pass (the residual's mass), and the final draw one
// pass (the exponential race argmin_y -ln(u_y) / R(y), lowest y on ties).
// Repeated passes over the same rows are served from L2.  Sums run in fp32;
// the ratio test runs on log2 values so that probabilities below the fp32
// range (low temperatures) still compare correctly.
#include <cooperative_groups.h>

#include "rd_internal.cuh"

namespace cg = cooperative_groups;

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / RD_WARP;
constexpr int kMaxCluster = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Bring [p, p + bytes) into L2 ahead of use (16-byte aligned start and size).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ float bf16_at(const uint16_t* row, int v)
{
    return __uint_as_float(((uint32_t)__ldg(row + v)) << 16);
}

// Running (max, sum of 2^(x - max)) pair, log2 units.
struct MaxSum {
    float m, s;
};

__device__ __forceinline__ MaxSum ms_merge(MaxSum a, MaxSum b)
{
    if (a.m == -INFINITY) return b;
    if (b.m == -INFINITY) return a;
    const float m = fmaxf(a.m, b.m);
    return {m, a.s * ex2(a.m - m) + b.s * ex2(b.m - m)};
}

// Fold eight values (already in log2 units) into a running pair.
__device__ __forceinline__ void ms_add8(MaxSum& ms, const float (&x)[8])
{
    float lm = x[0];
#pragma unroll
    for (int e = 1; e < 8; ++e) lm = fmaxf(lm, x[e]);
    if (lm == -INFINITY) return;
    if (lm > ms.m) {
        ms.s = (ms.m == -INFINITY) ? 0.f : ms.s * ex2(ms.m - lm);
        ms.m = lm;
    }
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc += ex2(x[e] - ms.m);
    ms.s += acc;
}

struct KeyIdx {
    float key;
    int idx;
};

__device__ __forceinline__ KeyIdx ki_min(KeyIdx a, KeyIdx b)
{
    return (b.key < a.key || (b.key == a.key && b.idx < a.idx)) ? b : a;
}

// Per-CTA scratch of the cluster reductions: partials published for the peers
// (two slots, alternating, so a slot is rewritten only after every peer has
// passed the next cluster barrier) and the warp partials.
struct Scratch {
    float4 pub[2][kMaxCluster];    // [slot][rank of the writer]
    float4 warp[kWarps];
};

// Reduce one float4 per thread over the CTA, then over the cluster, with `op`
// applied in a fixed order (warp lanes, warps, cluster ranks) so that every
// thread of every CTA obtains the identical value.
template <typename Op>
__device__ float4 cluster_reduce(float4 x, Scratch& sc, int& slot, const cg::cluster_group& cl,
                                 Op op)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        float4 o;
        o.x = __shfl_xor_sync(0xffffffffu, x.x, off);
        o.y = __shfl_xor_sync(0xffffffffu, x.y, off);
        o.z = __shfl_xor_sync(0xffffffffu, x.z, off);
        o.w = __shfl_xor_sync(0xffffffffu, x.w, off);
        x = op(x, o);
    }
    __syncthreads();                        // the previous reduction's readers are done
    if ((threadIdx.x & 31) == 0) sc.warp[threadIdx.x >> 5] = x;
    __syncthreads();
    const int n = (int)cl.num_blocks();
    if (threadIdx.x < 32) {
        // every lane folds the warp partials; lane i < n stores the result into
        // CTA i of the cluster (a remote store, so the barrier below is the only
        // wait and every CTA then reads its own shared memory)
        float4 r = sc.warp[0];
        for (int i = 1; i < kWarps; ++i) r = op(r, sc.warp[i]);
        if ((int)threadIdx.x < n) *cl.map_shared_rank(&sc.pub[slot][cl.block_rank()], threadIdx.x) = r;
    }
    cl.sync();
    float4 r = sc.pub[slot][0];
    for (int i = 1; i < n; ++i) r = op(r, sc.pub[slot][i]);
    slot ^= 1;
    return r;
}

__device__ __forceinline__ float4 op_maxsum2(float4 a, float4 b)
{
    const MaxSum t = ms_merge(MaxSum{a.x, a.y}, MaxSum{b.x, b.y});
    const MaxSum d = ms_merge(MaxSum{a.z, a.w}, MaxSum{b.z, b.w});
    return make_float4(t.m, t.s, d.m, d.s);
}

__device__ __forceinline__ float4 op_sum(float4 a, float4 b)
{
    return make_float4(a.x + b.x, 0.f, 0.f, 0.f);
}

__device__ __forceinline__ float4 op_keymin(float4 a, float4 b)
{
    const KeyIdx r = ki_min(KeyIdx{a.x, __float_as_int(a.y)}, KeyIdx{b.x, __float_as_int(b.y)});
    return make_float4(r.key, __int_as_float(r.idx), 0.f, 0.f);
}

// Visit the elements [v0, v1) of both rows: f(v, target_x, draft_x).
template <typename F>
__device__ __forceinline__ void for_each_pair(const uint16_t* tr, const uint16_t* dr, int v0,
                                              int v1, bool vec, F&& f)
{
    if (vec) {
        // two 16-byte loads per row in flight per thread before any is used
        const uint4* t4 = reinterpret_cast<const uint4*>(tr);
        const uint4* d4 = reinterpret_cast<const uint4*>(dr);
        const int i1 = v1 >> 3;
        for (int base = (v0 >> 3) + (int)threadIdx.x; base < i1; base += 2 * kThreads) {
            uint4 a[2], c[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int i = base + q * kThreads;
                a[q] = i < i1 ? __ldg(t4 + i) : make_uint4(0, 0, 0, 0);
                c[q] = i < i1 ? __ldg(d4 + i) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int i = base + q * kThreads;
                if (i >= i1) break;
                const uint32_t aw[4] = {a[q].x, a[q].y, a[q].z, a[q].w};
                const uint32_t cw[4] = {c[q].x, c[q].y, c[q].z, c[q].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    f(i * 8 + 2 * e, __uint_as_float(aw[e] << 16), __uint_as_float(cw[e] << 16));
                    f(i * 8 + 2 * e + 1, __uint_as_float(aw[e] & 0xffff0000u),
                      __uint_as_float(cw[e] & 0xffff0000u));
                }
            }
        }
    } else {
        for (int v = v0 + (int)threadIdx.x; v < v1; v += kThreads)
            f(v, bf16_at(tr, v), bf16_at(dr, v));
    }
}

__global__ void __launch_bounds__(kThreads)
sample_accept_kernel(const uint16_t* __restrict__ target, const uint16_t* __restrict__ draft,
                     int P_max, int V, float c2, const int32_t* __restrict__ beams,
                     const int32_t* __restrict__ packer, const int32_t* __restrict__ unpacker,
                     const int32_t* __restrict__ packed_len, int W, int L,
                     const float* __restrict__ u_accept, const float* __restrict__ u_sample,
                     int32_t* __restrict__ accept_len, int32_t* __restrict__ best_beam,
                     int32_t* __restrict__ n_accepted, int32_t* __restrict__ out_tokens,
                     int32_t* dev_status)
{
    __shared__ int s_parent[RD_MAX_PACKED];
    __shared__ int s_token[RD_MAX_PACKED];
    __shared__ int s_walk[RD_MAX_PACKED + 1];
    __shared__ int s_out[RD_MAX_PACKED + 1];
    __shared__ float s_invz[RD_MAX_BEAMS + 1];
    __shared__ float s_lz[RD_MAX_BEAMS + 1];
    __shared__ int s_kid[RD_MAX_PACKED];         // children of the current node, in order
    __shared__ float s_kt[RD_MAX_PACKED], s_kd[RD_MAX_PACKED], s_ku[RD_MAX_PACKED];
    __shared__ int s_nkid;
    __shared__ Scratch sc;
    __shared__ int s_best;

    const cg::cluster_group cl = cg::this_cluster();
    const int C = (int)cl.num_blocks();
    const int rank = (int)cl.block_rank();
    const int b = blockIdx.x / C;
    const int tid = threadIdx.x;
    const bool lead = rank == 0;
    // this CTA's slice of the vocabulary (multiples of 8 except the end)
    const int span = (((V + 7) / 8 + C - 1) / C) * 8;
    const int v0 = min(V, rank * span), v1 = min(V, v0 + span);

    const int Pb = __ldg(packed_len + b);
    const int32_t* bb = beams + (size_t)b * W * L;
    const int32_t* up = unpacker + (size_t)b * W * L;
    if (Pb < 1 || Pb > P_max) {
        if (lead) {
            if (tid == 0) {
                rd_flag(dev_status, RD_DEV_BAD_LENGTH);
                n_accepted[b] = 0;
                best_beam[b] = 0;
            }
            for (int j = tid; j < L; j += kThreads) out_tokens[(size_t)b * L + j] = -1;
            for (int w = tid; w < W; w += kThreads) accept_len[(size_t)b * W + w] = 0;
        }
        return;                                 // every CTA of the cluster returns here
    }
    // parent and token of every packed node (a node's parent precedes it)
    for (int c = tid; c < Pb; c += kThreads) {
        const int f = __ldg(packer + (size_t)b * P_max + c);
        int par = -1, tok = -1;
        if (f < 0 || f >= W * L) {
            if (lead) rd_flag(dev_status, RD_DEV_BAD_INDEX);
        } else {
            tok = __ldg(bb + f);
            if (f % L > 0) {
                par = __ldg(up + f - 1);
                if (par < 0 || par >= c) {
                    if (lead) rd_flag(dev_status, RD_DEV_BAD_INDEX);
                    par = -1;
                }
            }
            if (tok < 0 || tok >= V) {
                if (lead) rd_flag(dev_status, RD_DEV_BAD_TOKEN);
                tok = -1;
            }
        }
        s_parent[c] = par;
        s_token[c] = tok;
    }
    __syncthreads();
    // a peer stores into this CTA's shared memory only once every CTA of the
    // cluster has started: arrive now, wait before the walk (whose cluster
    // reductions do the remote stores); every CTA of the cluster gets here
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    const float* ua = u_accept + (size_t)b * P_max;
    const float* us = u_sample + (size_t)b * V;
    // the walk most often follows beam 0 (its nodes come first among every
    // node's children): bring that path's rows of this CTA's slice into L2
    {
        const uint32_t bytes = (uint32_t)((v1 - v0) & ~7) * 2u;
        const bool aligned = V % 8 == 0 && reinterpret_cast<uintptr_t>(target) % 16 == 0 &&
                             reinterpret_cast<uintptr_t>(draft) % 16 == 0;
        if (tid < L && aligned && bytes >= 16) {
            const int nd = __ldg(up + tid);
            if (nd >= 0 && nd < Pb) {
                const size_t off = ((size_t)b * P_max + nd) * V + v0;
                prefetch_l2(target + off, bytes);
                prefetch_l2(draft + off, bytes);
            }
        }
    }
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    int slot = 0;
    int node = 0, a = 0;
    if (tid == 0) s_walk[0] = 0;
    for (;;) {
        const uint16_t* tr = target + ((size_t)b * P_max + node) * V;
        const uint16_t* dr = draft + ((size_t)b * P_max + node) * V;
        const bool vec = (V % 8 == 0) && (reinterpret_cast<uintptr_t>(tr) % 16 == 0) &&
                         (reinterpret_cast<uintptr_t>(dr) % 16 == 0);
        // ---- children of this node: their tokens' logits and uniforms, read now
        // so that their latency overlaps pass 1; the first child's rows (the
        // likeliest next node) are prefetched into L2 --------------------------
        __syncthreads();                      // the previous node's reads are done
        if (tid < 32) {                       // children in packed order, by ballot
            int nk = 0;
            for (int c0 = node + 1; c0 < Pb; c0 += 32) {
                const int c = c0 + (int)tid;
                const bool kid = c < Pb && s_parent[c] == node && s_token[c] >= 0;
                const unsigned m = __ballot_sync(0xffffffffu, kid);
                if (kid) s_kid[nk + __popc(m & ((1u << tid) - 1u))] = c;
                nk += __popc(m);
            }
            if (tid == 0) {
                s_nkid = nk;
                const uint32_t bytes = (uint32_t)((v1 - v0) & ~7) * 2u;
                if (nk > 0 && vec && bytes >= 16) {
                    const size_t off = ((size_t)b * P_max + s_kid[0]) * V + v0;
                    prefetch_l2(target + off, bytes);
                    prefetch_l2(draft + off, bytes);
                }
            }
        }
        __syncthreads();
        const int nkid = s_nkid;
        for (int i = tid; i < nkid; i += kThreads) {
            const int c = s_kid[i], x = s_token[c];
            s_kt[i] = bf16_at(tr, x);
            s_kd[i] = bf16_at(dr, x);
            s_ku[i] = __ldg(ua + c);
        }
        // ---- pass 1: softmax maxima and sums of both rows (log2 units) --------
        MaxSum mt{-INFINITY, 0.f}, md{-INFINITY, 0.f};
        if (vec) {
            const uint4* t4 = reinterpret_cast<const uint4*>(tr);
            const uint4* d4 = reinterpret_cast<const uint4*>(dr);
            auto fold = [&](const uint4& ta, const uint4& da) {
                const uint32_t tw[4] = {ta.x, ta.y, ta.z, ta.w}, dw[4] = {da.x, da.y, da.z, da.w};
                float xt[8], xd[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    xt[2 * e] = __uint_as_float(tw[e] << 16) * c2;
                    xt[2 * e + 1] = __uint_as_float(tw[e] & 0xffff0000u) * c2;
                    xd[2 * e] = __uint_as_float(dw[e] << 16) * c2;
                    xd[2 * e + 1] = __uint_as_float(dw[e] & 0xffff0000u) * c2;
                }
                ms_add8(mt, xt);
                ms_add8(md, xd);
            };
            const int i1 = v1 >> 3;
            for (int i = (v0 >> 3) + tid; i < i1; i += 2 * kThreads) {
                const bool two = i + kThreads < i1;      // both loads issued before use
                const uint4 ta = __ldg(t4 + i), da = __ldg(d4 + i);
                uint4 tb = make_uint4(0, 0, 0, 0), db = tb;
                if (two) { tb = __ldg(t4 + i + kThreads); db = __ldg(d4 + i + kThreads); }
                fold(ta, da);
                if (two) fold(tb, db);
            }
        } else {
            for_each_pair(tr, dr, v0, v1, false, [&](int, float t, float d) {
                mt = ms_merge(mt, MaxSum{t * c2, 1.f});
                md = ms_merge(md, MaxSum{d * c2, 1.f});
            });
        }
        const float4 st = cluster_reduce(make_float4(mt.m, mt.s, md.m, md.s), sc, slot, cl,
                                         op_maxsum2);
        mt = MaxSum{st.x, st.y};
        md = MaxSum{st.z, st.w};
        const float it = 1.f / mt.s, id = 1.f / md.s;
        const float lst = __log2f(mt.s), lsd = __log2f(md.s);
        // residual after k rejections: R_0 = p, R_{j+1} = max(0, R_j - q) / Z_j
        auto resid = [&](float p, float q, int k) {
            for (int j = 0; j < k; ++j)
                if (s_invz[j] > 0.f) p = fmaxf(p - q, 0.f) * s_invz[j];
            return p;
        };
        // ---- children in packed order -----------------------------------------
        int k = 0, accepted = -1;
        for (int i = 0; i < nkid; ++i) {
            const int c = s_kid[i];
            // u q(x) < R_k(x), on log2 values
            const float lq = s_kd[i] * c2 - md.m - lsd;
            float lr = s_kt[i] * c2 - mt.m - lst;
            for (int j = 0; j < k; ++j) {
                if (s_invz[j] > 0.f)
                    lr = (lr > lq) ? lr + __log2f(-expm1f((lq - lr) * kLn2)) - s_lz[j] : -INFINITY;
            }
            const float u = s_ku[i];
            const float lu = u > 0.f ? __log2f(u) : -INFINITY;
            if (lu + lq < lr) { accepted = c; break; }
            // rejected: mass of the next residual
            float z = 0.f;
            for_each_pair(tr, dr, v0, v1, vec, [&](int, float t, float d) {
                const float p = ex2(t * c2 - mt.m) * it, q = ex2(d * c2 - md.m) * id;
                z += fmaxf(resid(p, q, k) - q, 0.f);
            });
            z = cluster_reduce(make_float4(z, 0.f, 0.f, 0.f), sc, slot, cl, op_sum).x;
            if (tid == 0) {
                s_invz[k] = z > 0.f ? 1.f / z : 0.f;
                s_lz[k] = z > 0.f ? __log2f(z) : 0.f;
            }
            __syncthreads();
            ++k;
        }
        if (accepted >= 0) {
            if (tid == 0) {
                s_out[a] = s_token[accepted];
                s_walk[a + 1] = accepted;
            }
            ++a;
            node = accepted;
            continue;
        }
        // ---- the draw: exponential race over the current target ---------------
        KeyIdx best{INFINITY, 0x7fffffff};
        for_each_pair(tr, dr, v0, v1, vec, [&](int v, float t, float d) {
            const float p = ex2(t * c2 - mt.m) * it, q = ex2(d * c2 - md.m) * id;
            const float r = resid(p, q, k);
            if (r > 0.f) best = ki_min(best, KeyIdx{-__log2f(__ldg(us + v)) / r, v});
        });
        const float4 bk = cluster_reduce(make_float4(best.key, __int_as_float(best.idx), 0.f, 0.f),
                                         sc, slot, cl, op_keymin);
        const int y = __float_as_int(bk.y);
        if (tid == 0) s_out[a] = y < V ? y : -1;
        break;
    }
    __syncthreads();
    if (lead) {
        for (int j = tid; j < L; j += kThreads)
            out_tokens[(size_t)b * L + j] = j <= a ? s_out[j] : -1;
        if (tid == 0) {
            n_accepted[b] = a;
            s_best = W;
        }
        __syncthreads();
        for (int w = tid; w < W; w += kThreads) {
            // leading positions of beam w on the walk (loads issued independently)
            int n = -1;
            bool on = true;
            for (int j = 0; j <= a && j < L; ++j) {
                on = on && __ldg(up + w * L + j) == s_walk[j];
                if (on) n = j;
            }
            accept_len[(size_t)b * W + w] = n < 0 ? 0 : n;
            if (n == a) atomicMin(&s_best, w);
        }
        __syncthreads();
        if (tid == 0) best_beam[b] = s_best < W ? s_best : 0;
    }
    cl.sync();                 // no CTA leaves while a peer may still read its partials
}

}  // namespace

int rd_sample_cluster_size(int B)
{
    // enough CTAs to cover the SMs once, at most kMaxCluster per request (a
    // sweep at B = 64 / 16 / 1 found 4 / 8 / 4-8 CTAs per request fastest:
    // more CTAs add cluster-barrier cost to every pass, fewer add pass length)
    const long sms = rd_device_sm_count();
    int c = 1;
    while (c < kMaxCluster && (long)B * c < sms) c *= 2;
    return c;
}

cudaError_t rd_launch_sample_accept(const void* target, const void* draft, int B, int P_max,
                                    int V, float temperature, const int32_t* beams,
                                    const int32_t* packer, const int32_t* unpacker,
                                    const int32_t* packed_len, int W, int L,
                                    const float* u_accept, const float* u_sample,
                                    int32_t* accept_len, int32_t* best_beam,
                                    int32_t* n_accepted, int32_t* out_tokens,
                                    int32_t* dev_status, cudaStream_t stream)
{
    const int C = rd_sample_cluster_size(B);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(B * C));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, sample_accept_kernel, static_cast<const uint16_t*>(target),
                              static_cast<const uint16_t*>(draft), P_max, V,
                              kLog2e / temperature, beams, packer, unpacker, packed_len, W, L,
                              u_accept, u_sample, accept_len, best_beam, n_accepted, out_tokens,
                              dev_status);
}
