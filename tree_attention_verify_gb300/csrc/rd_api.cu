// C entry points of librd: host-side validation, then one launch per call on the
// caller's stream.  See include/rd.h for the contract of every function.
#include <atomic>

#include "rd_internal.cuh"

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<long long> g_stall_budget{0};

rd_status from_cuda(cudaError_t e) { return e == cudaSuccess ? RD_OK : RD_ERR_CUDA; }

bool attn_shape_ok(int Hq, int Hkv, int D)
{
    return Hq > 0 && Hkv > 0 && Hq % Hkv == 0;
}

// TMA tensor maps and 16-byte vector accesses need 16-byte aligned bases.
bool aligned16(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

int rd_device_sm_count()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        cudaGetLastError();                       // do not leave the error for a later call
        return kRdFallbackSms;
    }
    if (dev >= kMaxDevices) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return kRdFallbackSms;
        return n;
    }
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            return kRdFallbackSms;
        }
        g_sm_count[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

long long rd_attention_stall_budget() { return g_stall_budget.load(std::memory_order_relaxed); }

extern "C" {

void rd_debug_stall_attention(long long budget_cycles)
{
    g_stall_budget.store(budget_cycles > 0 ? budget_cycles : 0, std::memory_order_relaxed);
}

const char* rd_status_string(rd_status s)
{
    switch (s) {
    case RD_OK: return "ok";
    case RD_ERR_INVALID_ARG: return "invalid argument";
    case RD_ERR_UNSUPPORTED: return "unsupported configuration";
    case RD_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

rd_status rd_pack_beams(const int32_t* beams, int B, int W, int L, int P_cap,
                        int32_t* tokens, int32_t* packer, int32_t* unpacker,
                        uint32_t* mask, int32_t* depth, int32_t* packed_len,
                        int32_t* dev_status, rd_stream_t stream)
{
    if (B < 0 || W < 1 || L < 1 || P_cap < 1) return RD_ERR_INVALID_ARG;
    if (W > RD_MAX_BEAMS || P_cap > RD_MAX_PACKED || (long)W * L > 4096)
        return RD_ERR_UNSUPPORTED;
    if (B == 0) return RD_OK;
    if (!beams || !tokens || !packer || !unpacker || !mask || !packed_len)
        return RD_ERR_INVALID_ARG;
    return from_cuda(rd_launch_pack(beams, B, W, L, P_cap, tokens, packer, unpacker, mask,
                                    depth, packed_len, dev_status, (cudaStream_t)stream));
}

size_t rd_tree_attention_workspace_size(int B, int P_max, int Hq, int Hkv, int D,
                                        int max_ctx)
{
    if (B <= 0 || P_max < 1 || !attn_shape_ok(Hq, Hkv, D) || max_ctx < 0) return 0;
    return rd_attn_make_plan(B, P_max, Hq, Hkv, D, max_ctx).ws_bytes;
}

rd_status rd_tree_attention(int B, int P_max, int Hq, int Hkv, int D, float scale,
                            const void* q, const void* k_new, const void* v_new,
                            const void* k_cache, const void* v_cache,
                            const int64_t* ctx_offsets, int64_t total_ctx, int max_ctx,
                            const int32_t* packed_len, const uint32_t* mask,
                            int mask_words, void* o, void* workspace, size_t ws_bytes,
                            int32_t* dev_status, rd_stream_t stream)
{
    if (B < 0 || P_max < 1 || !attn_shape_ok(Hq, Hkv, D) || total_ctx < 0 || max_ctx < 0)
        return RD_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return RD_ERR_UNSUPPORTED;
    if (P_max > RD_MAX_PACKED || B > 65535 || Hkv > 65535) return RD_ERR_UNSUPPORTED;
    if (mask_words != (P_max + 31) / 32) return RD_ERR_INVALID_ARG;
    if (B == 0) return RD_OK;
    if (!q || !k_new || !v_new || !ctx_offsets || !packed_len || !mask || !o)
        return RD_ERR_INVALID_ARG;
    if (total_ctx > 0 && (!k_cache || !v_cache)) return RD_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) ||
        !aligned16(v_cache) || !aligned16(o) || !aligned16(workspace))
        return RD_ERR_INVALID_ARG;
    const rd_attn_plan plan = rd_attn_make_plan(B, P_max, Hq, Hkv, D, max_ctx);
    if (plan.ws_bytes > 0 && (!workspace || ws_bytes < plan.ws_bytes))
        return RD_ERR_INVALID_ARG;
    if (scale <= 0.f) scale = 1.0f / sqrtf((float)D);
    return from_cuda(rd_launch_attention(plan, B, P_max, Hq, Hkv, D, scale, q, k_new,
                                         v_new, k_cache, v_cache, ctx_offsets, total_ctx,
                                         max_ctx, packed_len, mask, mask_words, o, workspace,
                                         dev_status, (cudaStream_t)stream));
}

rd_status rd_tree_attention_fp8(int B, int P_max, int Hq, int Hkv, int D, float scale,
                                const void* q, const void* k_new, const void* v_new,
                                const void* k_cache, const void* v_cache, float k_scale,
                                float v_scale, const int64_t* ctx_offsets, int64_t total_ctx,
                                int max_ctx, const int32_t* packed_len, const uint32_t* mask,
                                int mask_words, void* o, void* workspace, size_t ws_bytes,
                                int32_t* dev_status, rd_stream_t stream)
{
    if (B < 0 || P_max < 1 || !attn_shape_ok(Hq, Hkv, D) || total_ctx < 0 || max_ctx < 0)
        return RD_ERR_INVALID_ARG;
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || !isfinite(k_scale) || !isfinite(v_scale))
        return RD_ERR_INVALID_ARG;
    if (D != 128) return RD_ERR_UNSUPPORTED;
    if (P_max > RD_MAX_PACKED || B > 65535 || Hkv > 65535) return RD_ERR_UNSUPPORTED;
    if (mask_words != (P_max + 31) / 32) return RD_ERR_INVALID_ARG;
    if (B == 0) return RD_OK;
    if (total_ctx < 1) return RD_ERR_UNSUPPORTED;   /* no context: use rd_tree_attention */
    if (!q || !k_new || !v_new || !k_cache || !v_cache || !ctx_offsets || !packed_len || !mask ||
        !o)
        return RD_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) ||
        !aligned16(v_cache) || !aligned16(o) || !aligned16(workspace))
        return RD_ERR_INVALID_ARG;
    const rd_attn_plan plan = rd_attn_make_plan(B, P_max, Hq, Hkv, D, max_ctx);
    if (plan.ws_bytes > 0 && (!workspace || ws_bytes < plan.ws_bytes))
        return RD_ERR_INVALID_ARG;
    if (scale <= 0.f) scale = 1.0f / sqrtf((float)D);
    rd_fp8_kv f8;
    f8.k_cache = k_cache;
    f8.v_cache = v_cache;
    f8.k_scale = k_scale;
    f8.v_scale = v_scale;
    return from_cuda(rd_launch_attention(plan, B, P_max, Hq, Hkv, D, scale, q, k_new,
                                         v_new, nullptr, nullptr, ctx_offsets, total_ctx,
                                         max_ctx, packed_len, mask, mask_words, o, workspace,
                                         dev_status, (cudaStream_t)stream, nullptr, &f8));
}

rd_status rd_tree_attention_paged(int B, int P_max, int Hq, int Hkv, int D, float scale,
                                  const void* q, const void* k_new, const void* v_new,
                                  const void* k_pool, const void* v_pool, int num_pages,
                                  int page_size, const int32_t* block_table, int max_pages,
                                  const int32_t* ctx_lens, int max_ctx,
                                  const int32_t* packed_len, const uint32_t* mask,
                                  int mask_words, void* o, void* workspace, size_t ws_bytes,
                                  int32_t* dev_status, rd_stream_t stream)
{
    if (B < 0 || P_max < 1 || !attn_shape_ok(Hq, Hkv, D) || num_pages < 0 || max_pages < 0 ||
        max_ctx < 0 || page_size < 1)
        return RD_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return RD_ERR_UNSUPPORTED;
    if (page_size % 64 != 0) return RD_ERR_UNSUPPORTED;
    if (P_max > RD_MAX_PACKED || B > 65535 || Hkv > 65535) return RD_ERR_UNSUPPORTED;
    if ((long long)num_pages * page_size > 0x7fffffffLL) return RD_ERR_UNSUPPORTED;
    if (mask_words != (P_max + 31) / 32) return RD_ERR_INVALID_ARG;
    if (B == 0) return RD_OK;
    if (!q || !k_new || !v_new || !block_table || !ctx_lens || !packed_len || !mask || !o)
        return RD_ERR_INVALID_ARG;
    if (num_pages > 0 && (!k_pool || !v_pool)) return RD_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) ||
        !aligned16(v_pool) || !aligned16(o) || !aligned16(workspace))
        return RD_ERR_INVALID_ARG;
    const rd_attn_plan plan = rd_attn_make_plan(B, P_max, Hq, Hkv, D, max_ctx);
    if (plan.ws_bytes > 0 && (!workspace || ws_bytes < plan.ws_bytes))
        return RD_ERR_INVALID_ARG;
    if (scale <= 0.f) scale = 1.0f / sqrtf((float)D);
    rd_paged_kv pg;
    pg.block_table = block_table;
    pg.ctx_lens = ctx_lens;
    pg.max_pages = max_pages;
    pg.page_size = page_size;
    pg.num_pages = num_pages;
    return from_cuda(rd_launch_attention(plan, B, P_max, Hq, Hkv, D, scale, q, k_new,
                                         v_new, num_pages > 0 ? k_pool : nullptr,
                                         num_pages > 0 ? v_pool : nullptr, nullptr, 0, max_ctx,
                                         packed_len, mask, mask_words, o, workspace,
                                         dev_status, (cudaStream_t)stream, &pg));
}

rd_status rd_commit_accepted(int B, int W, int L, int P_max, int Hkv, int D,
                             const void* k_new, const void* v_new, const int32_t* unpacker,
                             const int32_t* best_beam, const int32_t* n_accepted,
                             void* k_pool, void* v_pool, int num_pages, int page_size,
                             const int32_t* block_table, int max_pages,
                             const int32_t* ctx_lens, int32_t* new_ctx_lens,
                             int32_t* dev_status, rd_stream_t stream)
{
    if (B < 0 || W < 1 || L < 1 || P_max < 1 || Hkv < 1 || num_pages < 0 || page_size < 1 ||
        max_pages < 0)
        return RD_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return RD_ERR_UNSUPPORTED;
    if (B > 65535 || L > 65535) return RD_ERR_UNSUPPORTED;
    if (B == 0) return RD_OK;
    if (!k_new || !v_new || !unpacker || !best_beam || !n_accepted || !k_pool || !v_pool ||
        !block_table || !ctx_lens || !new_ctx_lens || ctx_lens == new_ctx_lens)
        return RD_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool))
        return RD_ERR_INVALID_ARG;
    return from_cuda(rd_launch_commit(B, W, L, P_max, Hkv, D, k_new, v_new, unpacker, best_beam,
                                      n_accepted, k_pool, v_pool, num_pages, page_size,
                                      block_table, max_pages, ctx_lens, new_ctx_lens, dev_status,
                                      (cudaStream_t)stream));
}

rd_status rd_causal_attention(int B, int Hq, int Hkv, int D, float scale,
                              const void* q, const void* k, const void* v,
                              const int32_t* cu_seqlens, int64_t total_tokens,
                              int max_seqlen, void* o, int32_t* dev_status,
                              rd_stream_t stream)
{
    if (B < 0 || !attn_shape_ok(Hq, Hkv, D) || total_tokens < 0 || max_seqlen < 0)
        return RD_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return RD_ERR_UNSUPPORTED;
    if (B > 65535 || Hkv > 65535) return RD_ERR_UNSUPPORTED;
    if (B == 0 || max_seqlen == 0 || total_tokens == 0) return RD_OK;
    if (!q || !k || !v || !cu_seqlens || !o) return RD_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return RD_ERR_INVALID_ARG;
    if (scale <= 0.f) scale = 1.0f / sqrtf((float)D);
    return from_cuda(rd_launch_causal_pair(B, Hq, Hkv, D, scale, q, k, v, cu_seqlens,
                                           total_tokens, max_seqlen, o, dev_status,
                                           (cudaStream_t)stream));
}

rd_status rd_unpack(const void* packed, rd_dtype dt, int B, int P_max, int Dh,
                    const int32_t* unpacker, int W, int L, void* out,
                    int32_t* dev_status, rd_stream_t stream)
{
    int esize;
    switch (dt) {
    case RD_BF16: case RD_F16: esize = 2; break;
    case RD_F32: case RD_I32: esize = 4; break;
    default: return RD_ERR_INVALID_ARG;
    }
    if (B < 0 || P_max < 1 || Dh < 0 || W < 1 || L < 1) return RD_ERR_INVALID_ARG;
    if ((long)B * W * L > 0x7fffffffL) return RD_ERR_UNSUPPORTED;
    if (B == 0 || Dh == 0) return RD_OK;
    if (!packed || !unpacker || !out) return RD_ERR_INVALID_ARG;
    return from_cuda(rd_launch_unpack(packed, esize, B, P_max, Dh, unpacker, W, L, out,
                                      dev_status, (cudaStream_t)stream));
}

size_t rd_greedy_accept_workspace_size(int B, int P_max, int V)
{
    if (B <= 0 || P_max < 1 || V < 1) return 0;
    return rd_accept_workspace_bytes(B, P_max);
}

rd_status rd_greedy_accept(const void* logits, int B, int P_max, int V,
                           const int32_t* beams, const int32_t* unpacker,
                           const int32_t* packed_len, int W, int L,
                           int32_t* argmax, int32_t* accept_len, int32_t* best_beam,
                           int32_t* n_accepted, int32_t* out_tokens,
                           void* workspace, size_t ws_bytes,
                           int32_t* dev_status, rd_stream_t stream)
{
    if (B < 0 || P_max < 1 || V < 1 || W < 1 || L < 1) return RD_ERR_INVALID_ARG;
    if (W > RD_MAX_BEAMS || P_max > RD_MAX_PACKED || B > 65535) return RD_ERR_UNSUPPORTED;
    if (B == 0) return RD_OK;
    if (!logits || !beams || !unpacker || !packed_len || !argmax || !accept_len ||
        !best_beam || !n_accepted || !out_tokens || !workspace)
        return RD_ERR_INVALID_ARG;
    if (ws_bytes < rd_accept_workspace_bytes(B, P_max)) return RD_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 8 != 0) return RD_ERR_INVALID_ARG;
    return from_cuda(rd_launch_greedy_accept(logits, B, P_max, V, beams, unpacker, packed_len,
                                             W, L, argmax, accept_len, best_beam, n_accepted,
                                             out_tokens, workspace, dev_status,
                                             (cudaStream_t)stream));
}

rd_status rd_sample_accept(const void* target_logits, const void* draft_logits, int B, int P_max,
                           int V, float temperature, const int32_t* beams,
                           const int32_t* packer, const int32_t* unpacker,
                           const int32_t* packed_len, int W, int L, const float* u_accept,
                           const float* u_sample, int32_t* accept_len, int32_t* best_beam,
                           int32_t* n_accepted, int32_t* out_tokens, int32_t* dev_status,
                           rd_stream_t stream)
{
    if (B < 0 || P_max < 1 || V < 1 || W < 1 || L < 1) return RD_ERR_INVALID_ARG;
    if (!(temperature > 0.f) || !isfinite(temperature)) return RD_ERR_INVALID_ARG;
    if (W > RD_MAX_BEAMS || P_max > RD_MAX_PACKED || L > RD_MAX_PACKED || B > 0x7fffffff)
        return RD_ERR_UNSUPPORTED;
    if (B == 0) return RD_OK;
    if (!target_logits || !draft_logits || !beams || !packer || !unpacker || !packed_len ||
        !u_accept || !u_sample || !accept_len || !best_beam || !n_accepted || !out_tokens)
        return RD_ERR_INVALID_ARG;
    return from_cuda(rd_launch_sample_accept(target_logits, draft_logits, B, P_max, V,
                                             temperature, beams, packer, unpacker, packed_len,
                                             W, L, u_accept, u_sample, accept_len, best_beam,
                                             n_accepted, out_tokens, dev_status,
                                             (cudaStream_t)stream));
}

rd_status rd_beam_search_step(const void* logits, const float* scores_in,
                              const int32_t* beams_in, int B, int W, int V, int t,
                              int32_t* beams_out, float* scores_out, int32_t* parent,
                              int32_t* dev_status, rd_stream_t stream)
{
    if (B < 0 || W < 1 || V < 1 || t < 0 || V < W) return RD_ERR_INVALID_ARG;
    if (W > 16 || (long long)W * V > 0x7fffffffLL) return RD_ERR_UNSUPPORTED;
    if (B == 0) return RD_OK;
    if (!logits || !scores_in || (t > 0 && !beams_in) || !beams_out || !scores_out || !parent)
        return RD_ERR_INVALID_ARG;
    return from_cuda(rd_launch_beam_step(logits, scores_in, beams_in, B, W, V, t, beams_out,
                                         scores_out, parent, dev_status, (cudaStream_t)stream));
}

}  // extern "C"
