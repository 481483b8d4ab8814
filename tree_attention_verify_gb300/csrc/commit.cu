// rd_commit_accepted kernel: append the K/V of each request's accepted path to
// its paged KV cache.
//
// Verification accepts the best path before the next drafting step (NVIDIA
// blog "ReDrafter in TensorRT-LLM", introduction).  The tokens it confirms are
// the best beam's anchor and accepted drafts, nodes (w*, 0..a); their keys and
// values were computed for the packed drafts in this step and become context
// positions C_b .. C_b + a of the request's paged cache (TensorRT-LLM's paged KV
// caching, same blog, introduction).  The greedy token after the last accepted
// node has no K/V yet: it is the next step's anchor.
//
// One CTA per (path position i, request b) copies one [Hkv, D] row of K and of
// V with 16-byte accesses.
#include "rd_internal.cuh"

namespace {

__global__ void __launch_bounds__(128)
commit_kernel(int W, int L, int P_max, int row_vecs, const uint4* __restrict__ k_new,
              const uint4* __restrict__ v_new, const int32_t* __restrict__ unpacker,
              const int32_t* __restrict__ best_beam, const int32_t* __restrict__ n_accepted,
              uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, int num_pages,
              int page_size, const int32_t* __restrict__ block_table, int max_pages,
              const int32_t* __restrict__ ctx_lens, int32_t* __restrict__ new_ctx_lens,
              int32_t* dev_status)
{
    const int i = blockIdx.x;
    const int b = blockIdx.y;
    const int w = best_beam[b], a = n_accepted[b], C = ctx_lens[b];
    const bool bad = w < 0 || w >= W || a < 0 || a >= L || C < 0;
    if (i == 0 && threadIdx.x == 0) {
        if (bad) rd_flag(dev_status, RD_DEV_BAD_INDEX);
        new_ctx_lens[b] = bad ? C : C + a + 1;
    }
    if (bad || i > a) return;
    const int pos = C + i;
    const int slot = pos / page_size;
    if (slot >= max_pages) {
        if (threadIdx.x == 0) rd_flag(dev_status, RD_DEV_BAD_LENGTH);
        return;
    }
    const int page = block_table[(size_t)b * max_pages + slot];
    const int node = unpacker[((size_t)b * W + w) * L + i];
    if (page < 0 || page >= num_pages || node < 0 || node >= P_max) {
        if (threadIdx.x == 0) rd_flag(dev_status, RD_DEV_BAD_INDEX);
        return;
    }
    const size_t src = ((size_t)b * P_max + node) * row_vecs;
    const size_t dst = ((size_t)page * page_size + pos % page_size) * row_vecs;
    for (int k = threadIdx.x; k < row_vecs; k += blockDim.x) {
        k_pool[dst + k] = __ldg(k_new + src + k);
        v_pool[dst + k] = __ldg(v_new + src + k);
    }
}

}  // namespace

cudaError_t rd_launch_commit(int B, int W, int L, int P_max, int Hkv, int D, const void* k_new,
                             const void* v_new, const int32_t* unpacker,
                             const int32_t* best_beam, const int32_t* n_accepted, void* k_pool,
                             void* v_pool, int num_pages, int page_size,
                             const int32_t* block_table, int max_pages, const int32_t* ctx_lens,
                             int32_t* new_ctx_lens, int32_t* dev_status, cudaStream_t stream)
{
    const int row_vecs = Hkv * D * 2 / 16;
    commit_kernel<<<dim3((unsigned)L, (unsigned)B), 128, 0, stream>>>(
        W, L, P_max, row_vecs, static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
        unpacker, best_beam, n_accepted, static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool),
        num_pages, page_size, block_table, max_pages, ctx_lens, new_ctx_lens, dev_status);
    return cudaGetLastError();
}
