// Internal helpers shared by the librd kernels (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "rd.h"

#define RD_WARP 32

// OR error bits into the caller's device status word; never traps.
__device__ __forceinline__ void rd_flag(int32_t* status, unsigned bits)
{
    if (status != nullptr) atomicOr(reinterpret_cast<int*>(status), static_cast<int>(bits));
}

// Number of SMs of the current device (looked up once per device); the grid
// and split plans are sized from it.  Without a visible device (a host-only
// workspace query) it returns kRdFallbackSms, the count of a GB300.
constexpr int kRdFallbackSms = 152;
int rd_device_sm_count();

// Clock budget of the planted wait armed by rd_debug_stall_attention (0 = off).
long long rd_attention_stall_budget();

// Launchers (one per kernel family), called by the C entry points in rd_api.cu
// after host-side validation.  Each returns the cudaGetLastError() of its launches.
cudaError_t rd_launch_pack(const int32_t* beams, int B, int W, int L, int P_cap,
                           int32_t* tokens, int32_t* packer, int32_t* unpacker,
                           uint32_t* mask, int32_t* depth, int32_t* packed_len,
                           int32_t* dev_status, cudaStream_t stream);

cudaError_t rd_launch_unpack(const void* packed, int esize, int B, int P_max, int Dh,
                             const int32_t* unpacker, int W, int L, void* out,
                             int32_t* dev_status, cudaStream_t stream);

struct rd_accept_plan {
    int splits;        // vocab chunks per packed row
    int chunk;         // elements per chunk (multiple of 8)
};
rd_accept_plan rd_accept_make_plan(int B, int P_max, int V);
size_t rd_accept_workspace_bytes(int B, int P_max);
cudaError_t rd_launch_greedy_accept(const void* logits, int B, int P_max, int V,
                                    const int32_t* beams, const int32_t* unpacker,
                                    const int32_t* packed_len, int W, int L,
                                    int32_t* argmax, int32_t* accept_len,
                                    int32_t* best_beam, int32_t* n_accepted,
                                    int32_t* out_tokens, void* workspace,
                                    int32_t* dev_status, cudaStream_t stream);

cudaError_t rd_launch_sample_accept(const void* target, const void* draft, int B, int P_max,
                                    int V, float temperature, const int32_t* beams,
                                    const int32_t* packer, const int32_t* unpacker,
                                    const int32_t* packed_len, int W, int L,
                                    const float* u_accept, const float* u_sample,
                                    int32_t* accept_len, int32_t* best_beam,
                                    int32_t* n_accepted, int32_t* out_tokens,
                                    int32_t* dev_status, cudaStream_t stream);

// Tree attention (attention_tc.cu): the 16-bit, paged and FP8 variants.
struct rd_attn_plan {
    int tiles;         // row tiles per (request, kv head)
    bool stream_k;     // chunk-range division (tree attention), else whole units round-robin
    int grid;          // CTAs of the launch
    size_t ws_bytes;   // workspace bytes needed (chunk ranges: partials of cut units)
};
struct rd_paged_kv {
    const int32_t* block_table;   // [B, max_pages]
    const int32_t* ctx_lens;      // [B]
    int max_pages, page_size, num_pages;
};
struct rd_fp8_kv {
    const void* k_cache;          // e4m3 [total_ctx, Hkv, D]
    const void* v_cache;
    float k_scale, v_scale;
};
rd_attn_plan rd_attn_make_plan(int B, int P_max, int Hq, int Hkv, int D, int max_kv);
cudaError_t rd_launch_attention(const rd_attn_plan& plan, int B, int P_max,
                                int Hq, int Hkv, int D, float scale, const void* q,
                                const void* k_new, const void* v_new,
                                const void* k_cache, const void* v_cache,
                                const int64_t* ctx_offsets, int64_t total_kv, int max_kv,
                                const int32_t* lens, const uint32_t* mask, int mask_words,
                                void* o, void* workspace, int32_t* dev_status,
                                cudaStream_t stream, const rd_paged_kv* paged = nullptr,
                                const rd_fp8_kv* fp8 = nullptr);

// Causal prefill with paired 128-row query tiles, one CTA per SM (causal_pair.cu).
cudaError_t rd_launch_causal_pair(int B, int Hq, int Hkv, int D, float scale, const void* q,
                                  const void* k, const void* v, const int32_t* cu_seqlens,
                                  int64_t total, int max_len, void* o, int32_t* dev_status,
                                  cudaStream_t stream);

cudaError_t rd_launch_commit(int B, int W, int L, int P_max, int Hkv, int D, const void* k_new,
                             const void* v_new, const int32_t* unpacker,
                             const int32_t* best_beam, const int32_t* n_accepted, void* k_pool,
                             void* v_pool, int num_pages, int page_size,
                             const int32_t* block_table, int max_pages, const int32_t* ctx_lens,
                             int32_t* new_ctx_lens, int32_t* dev_status, cudaStream_t stream);

cudaError_t rd_launch_beam_step(const void* logits, const float* scores_in,
                                const int32_t* beams_in, int B, int W, int V, int t,
                                int32_t* beams_out, float* scores_out, int32_t* parent,
                                int32_t* dev_status, cudaStream_t stream);
