// rd_pack_beams kernel: prefix dedup of beam-search drafts into a trie.
//
// Dynamic tree attention removes the prefixes that several beams share from the
// tokens the LLM verifies ("Recurrent Drafter for Fast Speculative Decoding in
// LLMs", abstract, point (2)).  Packed order: the flattened beams (w*L + i) with
// every repeated prefix deleted, order kept.
//
// One warp per request, lane = beam.  Two prefixes of length i+1 are equal iff
// their last tokens are equal and their prefixes of length i are equal, so the
// warp walks depth by depth and keeps, per beam, the lowest beam that shares its
// prefix ("canonical beam").  A position whose canonical beam is itself is a new
// trie node; a warp scan over the per-beam new-node counts gives packed indices.
#include "rd_internal.cuh"

namespace {

constexpr int kMaxMaskWords = RD_MAX_PACKED / 32;

__global__ void __launch_bounds__(RD_WARP)
pack_beams_kernel(const int32_t* __restrict__ beams, int W, int L, int P_cap,
                  int32_t* __restrict__ tokens, int32_t* __restrict__ packer,
                  int32_t* __restrict__ unpacker, uint32_t* __restrict__ mask,
                  int32_t* __restrict__ depth, int32_t* __restrict__ packed_len,
                  int32_t* dev_status)
{
    extern __shared__ unsigned char smem[];
    // canon[w*L + i]: lowest beam sharing prefix (w, 0..i)   (uint8, W <= 32)
    // pidx [w*L + i]: packed index of node (w, i)             (int16)
    unsigned char* canon = smem;
    int16_t* pidx = reinterpret_cast<int16_t*>(smem + ((W * L + 15) & ~15));

    const int b = blockIdx.x;
    const int lane = threadIdx.x;
    const bool active = lane < W;
    const int32_t* bb = beams + (size_t)b * W * L;
    const int NW = (P_cap + 31) / 32;

    // --- canonical beam per depth -------------------------------------------------
    int prev = 0;                                      // canonical beam at depth i-1
    int n_new = 0;                                     // new nodes on this beam
    for (int i = 0; i < L; ++i) {
        int tok = active ? bb[lane * L + i] : 0;
        int c = lane;
        for (int w2 = 0; w2 < W; ++w2) {               // first beam with equal prefix
            int t2 = __shfl_sync(0xffffffffu, tok, w2);
            int p2 = __shfl_sync(0xffffffffu, prev, w2);
            if (w2 < c && t2 == tok && p2 == prev) c = w2;
        }
        if (active) {
            canon[lane * L + i] = (unsigned char)c;
            n_new += (c == lane);
        }
        prev = c;
    }
    // --- packed index of new nodes: exclusive scan of new-node counts over beams --
    int incl = n_new;
    for (int off = 1; off < RD_WARP; off <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    const int P = __shfl_sync(0xffffffffu, incl, RD_WARP - 1);
    int next = incl - n_new;
    __syncwarp();
    if (active) {
        for (int i = 0; i < L; ++i)
            if (canon[lane * L + i] == lane) pidx[lane * L + i] = (int16_t)next++;
    }
    __syncwarp();
    if (P > P_cap && lane == 0) rd_flag(dev_status, RD_DEV_OVERFLOW);

    // --- unpacker, node rows, ancestor masks --------------------------------------
    int32_t* up = unpacker + (size_t)b * W * L;
    int32_t* tk = tokens + (size_t)b * P_cap;
    int32_t* pk = packer + (size_t)b * P_cap;
    int32_t* dp = depth ? depth + (size_t)b * P_cap : nullptr;
    uint32_t* mk = mask + (size_t)b * P_cap * NW;
    if (active) {
        uint32_t run[kMaxMaskWords];
#pragma unroll
        for (int k = 0; k < kMaxMaskWords; ++k) run[k] = 0u;
        for (int i = 0; i < L; ++i) {
            const int c = canon[lane * L + i];
            const int p = pidx[c * L + i];
            up[lane * L + i] = p;
            if (p < P_cap) {
#pragma unroll
                for (int k = 0; k < kMaxMaskWords; ++k)
                    if (k == (p >> 5)) run[k] |= 1u << (p & 31);
            }
            if (c == lane && p < P_cap) {              // first occurrence: write the row
                tk[p] = bb[lane * L + i];
                pk[p] = lane * L + i;
                if (dp) dp[p] = i;
#pragma unroll
                for (int k = 0; k < kMaxMaskWords; ++k)
                    if (k < NW) mk[(size_t)p * NW + k] = run[k];
            }
        }
    }
    // padded rows
    for (int p = P + lane; p < P_cap; p += RD_WARP) {
        tk[p] = 0;
        pk[p] = -1;
        if (dp) dp[p] = 0;
        for (int k = 0; k < NW; ++k) mk[(size_t)p * NW + k] = 0u;
    }
    if (lane == 0) packed_len[b] = P;
}

}  // namespace

cudaError_t rd_launch_pack(const int32_t* beams, int B, int W, int L, int P_cap,
                           int32_t* tokens, int32_t* packer, int32_t* unpacker,
                           uint32_t* mask, int32_t* depth, int32_t* packed_len,
                           int32_t* dev_status, cudaStream_t stream)
{
    size_t smem = (size_t)((W * L + 15) & ~15) + sizeof(int16_t) * (size_t)W * L;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(pack_beams_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    pack_beams_kernel<<<B, RD_WARP, smem, stream>>>(beams, W, L, P_cap, tokens, packer,
                                                    unpacker, mask, depth, packed_len,
                                                    dev_status);
    return cudaGetLastError();
}
