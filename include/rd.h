/*
 * rd.h -- C ABI of librd, the GB300 (sm_103a) verification step of
 * ReDrafter-style recurrent-drafter speculative decoding.
 *
 * One verification step of a generation sub-batch is
 *
 *   rd_pack_beams      dedup the W beams x L tokens of each request into a
 *                      prefix trie ("dynamic tree attention")
 *   rd_tree_attention  attention of the packed draft queries over the request's
 *                      KV cache plus their own trie ancestors
 *   rd_greedy_accept   greedy verification: best beam and accepted length
 *   rd_unpack          gather a packed [B, P, D] tensor back to [B, W, L, D]
 *
 * and a context-phase (prefill) sub-batch of an in-flight batch uses
 * rd_causal_attention.  Sources of each definition are cited per function.
 *
 * Conventions shared by every entry point
 *  - All tensor arguments are DEVICE pointers to contiguous row-major arrays
 *    on the current CUDA device, laid out as stated per argument.  The caller
 *    owns every buffer.  The library never allocates, frees or synchronises.
 *  - Each call validates its host-side arguments, enqueues its kernel(s) on
 *    `stream` (0 = the legacy default stream) and returns at once.
 *  - Host-detectable errors return a status without launching anything.
 *    A launch failure returns RD_ERR_CUDA.
 *  - Data-dependent errors cannot be seen on the host: kernels OR bits into
 *    *dev_status (an int32 in device memory, which the caller zeroes and
 *    reads when it likes) and skip the offending access.  Kernels never trap.
 *  - A batch with no requests (B == 0) returns RD_OK and launches nothing:
 *    the context or generation half of an in-flight batch may be empty
 *    (NVIDIA blog "ReDrafter in TensorRT-LLM", section "Inflight-batching
 *    Compatible Engine": every operator on either path must accept empty
 *    tensors).
 *  - bf16 tensors are passed as raw 16-bit storage.
 */
#ifndef RD_H
#define RD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle as cudaStream_t / CUstream. */
typedef struct CUstream_st* rd_stream_t;

typedef enum {
    RD_OK = 0,
    RD_ERR_INVALID_ARG = 1,  /* null pointer, bad shape, workspace too small  */
    RD_ERR_UNSUPPORTED = 2,  /* valid but outside what the kernels implement  */
    RD_ERR_CUDA = 3          /* the CUDA runtime reported an error            */
} rd_status;

typedef enum { RD_BF16 = 0, RD_F16 = 1, RD_F32 = 2, RD_I32 = 3 } rd_dtype;

/* bits OR-ed into *dev_status by the kernels */
#define RD_DEV_BAD_INDEX   1u   /* an unpacker index outside [0, P_max) or [0, packed_len) */
#define RD_DEV_BAD_TOKEN   2u   /* a draft token outside [0, V)                           */
#define RD_DEV_OVERFLOW    4u   /* a request packed to more nodes than P_cap              */
#define RD_DEV_BAD_LENGTH  8u   /* packed_len / context / sequence length beyond its bound */
#define RD_DEV_TIMEOUT    16u   /* a bounded wait inside a kernel ran out                 */

/* Limits of this implementation (RD_ERR_UNSUPPORTED beyond them). */
#define RD_MAX_BEAMS      32    /* W                                   */
#define RD_MAX_PACKED    256    /* P_cap / P_max                       */

const char* rd_status_string(rd_status s);

/*
 * rd_pack_beams -- prefix dedup of beam-search drafts.
 *
 * Source: "Recurrent Drafter for Fast Speculative Decoding in LLMs", abstract
 * point (2): dynamic tree attention over the beam search results removes
 * duplicated prefixes from the candidates; Apple x NVIDIA news page, paragraph
 * on dynamic tree attention: shared prefixes are found and removed from the
 * tokens the LLM has to verify.
 *
 * beams      int32 [B, W, L]. Position 0 of every beam is the anchor (the token
 *            the LLM already emitted); positions 1..L-1 are drafts.
 * P_cap      row stride of every packed output, 1..RD_MAX_PACKED.  W*L always
 *            suffices.  A request with more than P_cap distinct prefixes sets
 *            RD_DEV_OVERFLOW; its rows beyond P_cap are not written.
 * Outputs, per request b (node = a distinct prefix beams[b, w, 0..i]):
 *   tokens     int32 [B, P_cap]   token of packed node p (0 on padded rows)
 *   packer     int32 [B, P_cap]   flat beam position w*L+i of the node's first
 *                                 occurrence (-1 on padded rows); strictly
 *                                 increasing: packed order = flattened beams
 *                                 with every repeated prefix deleted
 *   unpacker   int32 [B, W, L]    packed index of node (w, i)
 *   mask       uint32 [B, P_cap, ceil(P_cap/32)]  bit k of row p (LSB-first
 *                                 within each word) is set iff node k is on
 *                                 the path root..p (itself included)
 *   depth      int32 [B, P_cap]   i of the node (its position offset); may be NULL
 *   packed_len int32 [B]          number of nodes P_b
 * dev_status int32 device word (see above).
 * Errors: RD_ERR_INVALID_ARG for null pointers with B > 0 or W, L < 1 or
 * P_cap < 1; RD_ERR_UNSUPPORTED for W > RD_MAX_BEAMS or P_cap > RD_MAX_PACKED.
 */
rd_status rd_pack_beams(const int32_t* beams, int B, int W, int L, int P_cap,
                        int32_t* tokens, int32_t* packer, int32_t* unpacker,
                        uint32_t* mask, int32_t* depth, int32_t* packed_len,
                        int32_t* dev_status, rd_stream_t stream);

/*
 * rd_tree_attention -- attention of the packed drafts, generation phase.
 *
 * Source: NVIDIA blog "ReDrafter in TensorRT-LLM" (custom attention kernel in
 * TensorRT-LLM; the attention plugin splits context and generation requests);
 * speculative-decoding survey page, SpecInfer "Token Tree Verifier": a single
 * kernel with a topology-aware causal mask verifies every candidate sequence.
 *
 * For request b, query head hq (kv head h = hq / (Hq/Hkv)) and packed node
 * p < packed_len[b]:
 *   o[b,p,hq,:] = sum_k softmax_k(scale * q[b,p,hq,:] . key_k) * value_k
 * over the keys k of the context (k_cache rows ctx_offsets[b] ..
 * ctx_offsets[b+1]-1, all visible) and the packed drafts k_new[b,k,h,:]
 * whose bit k is set in mask row p (its ancestors and itself).
 * Rows p >= packed_len[b] are written as 0.
 *
 * q          bf16 [B, P_max, Hq, D]     (post-RoPE)
 * k_new,v_new bf16 [B, P_max, Hkv, D]   K/V of the packed draft tokens
 * k_cache,v_cache bf16 [total_ctx, Hkv, D]  contiguous ragged KV cache
 * ctx_offsets int64 [B+1]               prefix sums of context lengths
 * total_ctx  rows of k_cache / v_cache (host-known; ctx_offsets[B] must not
 *            exceed it, else RD_DEV_BAD_LENGTH and that request is skipped)
 * max_ctx    bound on every context length (sizes the workspace; a longer
 *            context sets RD_DEV_BAD_LENGTH and is skipped)
 * packed_len int32 [B]; mask uint32 [B, P_max, mask_words] as rd_pack_beams
 *            writes it (mask_words = ceil(P_max/32))
 * o          bf16 [B, P_max, Hq, D]
 * scale      softmax scale; <= 0 selects 1/sqrt(D)
 * workspace  device scratch of rd_tree_attention_workspace_size() bytes: the
 *            CTAs split the batch's KV chunks into equal ranges, and the fp32
 *            partials of the units that a range boundary cuts go here, with one
 *            descriptor per CTA naming the unit it merges (a second kernel,
 *            launched on the same stream, merges them).  No initial contents are needed; every
 *            call writes what it reads.  Calls that share a workspace must not
 *            overlap in time.  The size depends on the SM count of the current
 *            device: query it with the device current that the call will run
 *            on.  A batch of at least two units (request, kv head, 128-row
 *            tile) per CTA, or of B > 480, runs whole units round-robin and
 *            needs none.
 * Supported: D in {64, 128}; Hq % Hkv == 0; 1 <= P_max <= RD_MAX_PACKED.
 */
size_t rd_tree_attention_workspace_size(int B, int P_max, int Hq, int Hkv, int D,
                                        int max_ctx);
rd_status rd_tree_attention(int B, int P_max, int Hq, int Hkv, int D, float scale,
                            const void* q, const void* k_new, const void* v_new,
                            const void* k_cache, const void* v_cache,
                            const int64_t* ctx_offsets, int64_t total_ctx, int max_ctx,
                            const int32_t* packed_len, const uint32_t* mask,
                            int mask_words, void* o, void* workspace, size_t ws_bytes,
                            int32_t* dev_status, rd_stream_t stream);

/*
 * rd_tree_attention_fp8 -- rd_tree_attention with the context K/V cache stored
 * in FP8 (e4m3) with one scale per tensor (TensorRT-LLM's FP8 quantisation:
 * NVIDIA blog "ReDrafter in TensorRT-LLM", introduction).  Context key j is
 * k_scale * e4m3(k_cache[j]) and likewise for values; the packed drafts stay
 * bf16.  Same computation, outputs and workspace as rd_tree_attention.
 *
 * k_cache,v_cache uint8 e4m3 bit patterns [total_ctx, Hkv, D]
 * k_scale,v_scale finite, > 0
 * Supported: D = 128, total_ctx >= 1 (RD_ERR_UNSUPPORTED otherwise).
 * The contraction runs in f16 (every e4m3 value and every bf16 query is
 * exact in f16 within f16's range; draft K/V are divided by the scales and
 * rounded to f16).
 */
rd_status rd_tree_attention_fp8(int B, int P_max, int Hq, int Hkv, int D, float scale,
                                const void* q, const void* k_new, const void* v_new,
                                const void* k_cache, const void* v_cache, float k_scale,
                                float v_scale, const int64_t* ctx_offsets, int64_t total_ctx,
                                int max_ctx, const int32_t* packed_len, const uint32_t* mask,
                                int mask_words, void* o, void* workspace, size_t ws_bytes,
                                int32_t* dev_status, rd_stream_t stream);

/*
 * rd_tree_attention_paged -- rd_tree_attention with the context in a paged KV
 * cache (TensorRT-LLM's paged KV caching: NVIDIA blog "ReDrafter in
 * TensorRT-LLM", introduction).  Same computation, outputs and workspace as
 * rd_tree_attention (size the workspace with rd_tree_attention_workspace_size
 * and the same max_ctx); only the context rows are found through a block table:
 *
 * k_pool,v_pool bf16 [num_pages, page_size, Hkv, D]
 * block_table  int32 [B, max_pages]: context position j of request b is row
 *              j % page_size of page block_table[b, j / page_size]
 * ctx_lens     int32 [B] context lengths (<= max_ctx and <= max_pages*page_size,
 *              else RD_DEV_BAD_LENGTH and the request is skipped)
 * page_size    a multiple of 64 (RD_ERR_UNSUPPORTED otherwise); num_pages *
 *              page_size < 2^31.  A page id outside [0, num_pages) sets
 *              RD_DEV_BAD_INDEX (page 0 is read in its place).
 */
rd_status rd_tree_attention_paged(int B, int P_max, int Hq, int Hkv, int D, float scale,
                                  const void* q, const void* k_new, const void* v_new,
                                  const void* k_pool, const void* v_pool, int num_pages,
                                  int page_size, const int32_t* block_table, int max_pages,
                                  const int32_t* ctx_lens, int max_ctx,
                                  const int32_t* packed_len, const uint32_t* mask,
                                  int mask_words, void* o, void* workspace, size_t ws_bytes,
                                  int32_t* dev_status, rd_stream_t stream);

/*
 * rd_commit_accepted -- append the K/V of each request's accepted path to its
 * paged cache, after rd_greedy_accept.
 *
 * Source: NVIDIA blog "ReDrafter in TensorRT-LLM", introduction (verify the
 * drafts and accept the best path before drafting the next tokens; paged KV
 * caching).  The confirmed tokens of request b are the best beam's anchor and
 * accepted drafts, nodes (w*, i) for i = 0..a with w* = best_beam[b] and
 * a = n_accepted[b]; their rows k_new[b, unpacker[b, w*, i], :, :] (and v_new)
 * are written at context position ctx_lens[b] + i (page
 * block_table[b, pos / page_size], row pos % page_size), and
 * new_ctx_lens[b] = ctx_lens[b] + a + 1.  The greedy token after the last
 * accepted node has no K/V yet (it is the next step's anchor).
 *
 * k_new,v_new bf16 [B, P_max, Hkv, D]; unpacker int32 [B, W, L]; best_beam,
 * n_accepted int32 [B]; k_pool,v_pool bf16 [num_pages, page_size, Hkv, D]
 * (modified); block_table int32 [B, max_pages]; ctx_lens int32 [B] (read);
 * new_ctx_lens int32 [B] (written; must not alias ctx_lens).
 * A best beam, accepted length, unpacker index or page id out of range sets
 * RD_DEV_BAD_INDEX; a position beyond max_pages*page_size sets
 * RD_DEV_BAD_LENGTH; the offending row is skipped.
 */
rd_status rd_commit_accepted(int B, int W, int L, int P_max, int Hkv, int D,
                             const void* k_new, const void* v_new, const int32_t* unpacker,
                             const int32_t* best_beam, const int32_t* n_accepted,
                             void* k_pool, void* v_pool, int num_pages, int page_size,
                             const int32_t* block_table, int max_pages,
                             const int32_t* ctx_lens, int32_t* new_ctx_lens,
                             int32_t* dev_status, rd_stream_t stream);

/*
 * rd_causal_attention -- causal prefill of the context-phase requests of an
 * in-flight batch (NVIDIA blog "ReDrafter in TensorRT-LLM", section
 * "Inflight-batching Compatible Engine": the batch splits into a context and a
 * generation sub-batch).  Token t of sequence b attends to tokens 0..t of the
 * same sequence; there is no earlier context.
 *
 * q, o       bf16 [total_tokens, Hq, D];  k, v bf16 [total_tokens, Hkv, D]
 * cu_seqlens int32 [B+1] prefix sums of sequence lengths (cu_seqlens[B] must
 *            not exceed total_tokens)
 * max_seqlen bound on every sequence length (RD_DEV_BAD_LENGTH beyond it)
 * Supported: D in {64, 128}; Hq % Hkv == 0.
 */
rd_status rd_causal_attention(int B, int Hq, int Hkv, int D, float scale,
                              const void* q, const void* k, const void* v,
                              const int32_t* cu_seqlens, int64_t total_tokens,
                              int max_seqlen, void* o, int32_t* dev_status,
                              rd_stream_t stream);

/*
 * rd_unpack -- out[b, w, i, :] = packed[b, unpacker[b, w, i], :].
 *
 * Source: NVIDIA blog "ReDrafter in TensorRT-LLM", section "Implementing
 * in-Engine Validation and Drafting" (the PyTorch unpack: a gather along the
 * packed dimension reshaped to [B, W, L, D]).  An exact copy of the bits.
 *
 * packed   [B, P_max, Dh] of dtype dt (2- or 4-byte elements)
 * unpacker int32 [B, W, L]; an index outside [0, P_max) sets RD_DEV_BAD_INDEX
 *          and writes zeros for that row
 * out      [B, W, L, Dh] of dtype dt
 */
rd_status rd_unpack(const void* packed, rd_dtype dt, int B, int P_max, int Dh,
                    const int32_t* unpacker, int W, int L, void* out,
                    int32_t* dev_status, rd_stream_t stream);

/*
 * rd_beam_search_step -- one step of the drafter's beam search (the step that
 * produces the beams rd_pack_beams consumes).
 *
 * Source: Apple x NVIDIA news page, paragraph on the RNN draft model (from the
 * initial token and the LLM's last hidden state the drafter runs a beam search
 * that yields several candidate token sequences); "Recurrent Drafter for Fast
 * Speculative Decoding in LLMs", abstract.  The drafter network itself is out
 * of scope: its logits are an input.
 *
 * Candidate (w, v) of request b scores
 *   scores_in[b, w] + logits[b, w, v] - log sum_u exp(logits[b, w, u]);
 * a beam whose score is -inf (not live yet) has no candidates.  The W best
 * candidates, best first (equal scores: the lower flat index w*V + v first),
 * become the new beams: beams_out[b, r] = beams_in[b, parent[b, r]] followed
 * by token v_r, scores_out[b, r] = its score.  Scores are computed in fp32;
 * candidates whose scores differ by less than their fp32 rounding may be
 * ordered either way.
 *
 * logits bf16 [B, W, V]; scores_in fp32 [B, W]; beams_in int32 [B, W, t]
 * (t >= 0; may be NULL when t == 0); beams_out int32 [B, W, t+1];
 * scores_out fp32 [B, W]; parent int32 [B, W].  1 <= W <= 16, V >= W.
 * Fewer than W live candidates set RD_DEV_BAD_LENGTH (parent -1, token -1).
 */
rd_status rd_beam_search_step(const void* logits, const float* scores_in,
                              const int32_t* beams_in, int B, int W, int V, int t,
                              int32_t* beams_out, float* scores_out, int32_t* parent,
                              int32_t* dev_status, rd_stream_t stream);

/*
 * rd_greedy_accept -- greedy verification of the drafts.
 *
 * Source: NVIDIA blog "ReDrafter in TensorRT-LLM", introduction (verify the
 * drafts and accept the best path before drafting the next tokens; accept more
 * than one token per decoder iteration); Apple x NVIDIA news page, benchmark
 * paragraph (greedy decoding).
 *
 *  (i)   argmax[b,p] = argmax_v logits[b,p,v] for p < packed_len[b], the
 *        lowest index on ties; -1 on padded rows.
 *  (ii)  accept_len[b,w] = the largest n <= L-1 such that
 *        beams[b,w,j] == argmax[b, unpacker[b,w,j-1]] for every j = 1..n.
 *  (iii) best_beam[b] = argmax_w accept_len[b,w], the lowest w on ties;
 *        n_accepted[b] = accept_len[b, best_beam[b]] = a.
 *  (iv)  out_tokens[b, 0..a-1] = beams[b, best, 1..a];
 *        out_tokens[b, a] = argmax[b, unpacker[b, best, a]] (the greedy token
 *        after the last accepted node); the rest -1.
 *
 * logits     bf16 [B, P_max, V] (rows p >= packed_len[b] are not read)
 * beams, unpacker int32 [B, W, L]; packed_len int32 [B]
 * Outputs: argmax int32 [B, P_max], accept_len int32 [B, W], best_beam,
 *          n_accepted int32 [B], out_tokens int32 [B, L].
 * workspace  device scratch of rd_greedy_accept_workspace_size() bytes.  It
 *            must be zero-filled before its first use; every call leaves it
 *            zeroed.  Calls that share a workspace must not overlap in time.
 * A context-phase request is the case W = L = 1 (its one row is the last
 * prompt position): out_tokens[b, 0] is its greedy next token.
 */
size_t rd_greedy_accept_workspace_size(int B, int P_max, int V);
rd_status rd_greedy_accept(const void* logits, int B, int P_max, int V,
                           const int32_t* beams, const int32_t* unpacker,
                           const int32_t* packed_len, int W, int L,
                           int32_t* argmax, int32_t* accept_len, int32_t* best_beam,
                           int32_t* n_accepted, int32_t* out_tokens,
                           void* workspace, size_t ws_bytes,
                           int32_t* dev_status, rd_stream_t stream);

/*
 * rd_debug_stall_attention -- failure-detection test hook.  The pages have no
 * counterpart: it exists to test the kernels' bounded waits without a GPU fault.
 *
 * budget_cycles > 0 arms it for every later rd_tree_attention,
 * rd_tree_attention_paged, rd_tree_attention_fp8 and rd_causal_attention
 * launch of this process: before its first MMA, each CTA's MMA-issuing thread
 * waits on a barrier that nothing completes, for at most budget_cycles SM
 * clock cycles.  That wait runs out, the CTA records RD_DEV_TIMEOUT, its other
 * roles stop at their next wait, it waits (with the normal budget) for the
 * copies and MMAs it has issued, frees its tensor memory and returns.  The
 * outputs of such a launch are undefined; the next call needs nothing reset.
 * budget_cycles <= 0 disarms it (the default).  Process-wide;
 * do not arm it while other threads launch attention they rely on.
 */
void rd_debug_stall_attention(long long budget_cycles);

/*
 * rd_greedy_accept_noalloc -- rd_greedy_accept for callers that cannot
 * allocate device memory.  The pages have no counterpart: this is a library
 * convenience, not part of the method.
 *
 * Same arguments and results as rd_greedy_accept, without the workspace.  Some
 * callers cannot call cudaMalloc on the serving path (a plugin inside a host
 * framework that owns all device memory, a runtime that must not allocate after
 * start-up because an allocation can synchronise the device or fail under
 * memory pressure).  This entry point takes its scratch from a fixed array in
 * device global memory that the library owns: about 768 KB, held on every GPU
 * that loads librd until the process exits.
 *  - Limits: B * P_max <= 65536 and B <= 65535; beyond them it returns
 *    RD_ERR_UNSUPPORTED without launching.
 *  - It allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 *    routine.  It clears the part of the array it uses with cudaMemsetAsync on
 *    `stream` before its kernel.
 *  - Every call on a device shares the one array: calls whose work overlaps on
 *    the GPU (different streams or host threads without ordering) race and
 *    give wrong results.  Order them on one stream.
 *  - The first call on a device looks the array's device address up with that
 *    device current (cudaGetSymbolAddress); make that first call before any
 *    stream capture begins.  The address is kept for the life of the process:
 *    after a cudaDeviceReset of that device it is stale, so do not call this
 *    entry point on a device that has been reset.
 *  - All tensors must be on the current device.
 */
rd_status rd_greedy_accept_noalloc(const void* logits, int B, int P_max, int V,
                                   const int32_t* beams, const int32_t* unpacker,
                                   const int32_t* packed_len, int W, int L,
                                   int32_t* argmax, int32_t* accept_len,
                                   int32_t* best_beam, int32_t* n_accepted,
                                   int32_t* out_tokens, int32_t* dev_status,
                                   rd_stream_t stream);

/*
 * rd_sample_accept -- stochastic verification of the draft tree by multi-step
 * speculative sampling: rejection sampling (speculative-decoding survey page,
 * rejection-sampling paragraph: keep a proposal x when u < p(x) / q(x)) applied
 * child by child over the tree as in SpecInfer's multi-step speculative
 * sampling (same page, "Token Tree Verifier").
 *
 * For request b the walk starts at packed node 0 (beam 0's anchor).  At node n,
 * with p = softmax(target_logits[b, n] / temperature) and
 * q = softmax(draft_logits[b, n] / temperature), the children of n (the packed
 * nodes whose parent is n) are tested in increasing packed index: child c with
 * token x is accepted when u_accept[b, c] * q(x) < p(x) and becomes the current
 * node; after a rejection p is replaced by max(0, p - q) / sum(max(0, p - q))
 * (left unchanged when that sum is 0).  When every child is rejected, or n has
 * none, one token is drawn from p by the exponential race
 * argmin_y -ln(u_sample[b, y]) / p(y) (lowest y on ties) and the walk ends.
 *
 * target_logits, draft_logits  bf16 [B, P_max, V]: the LLM's and the drafter's
 *                 next-token logits at every packed node
 * beams, unpacker int32 [B, W, L]; packer int32 [B, P_max]; packed_len int32 [B]
 *                 (as produced by rd_pack_beams)
 * temperature     finite, > 0
 * u_accept        float32 [B, P_max] uniforms in [0, 1), one per packed node
 * u_sample        float32 [B, V] uniforms in [0, 1), one per vocabulary entry
 * accept_len      int32 [B, W] out: leading drafts of beam w on the accepted walk
 * best_beam       int32 [B] out: lowest beam whose prefix is the accepted walk
 * n_accepted      int32 [B] out: accepted drafts a
 * out_tokens      int32 [B, L] out: the a accepted drafts, the drawn token, then -1
 * Computes in fp32 (decisions closer than fp32 rounding may differ from exact
 * arithmetic).  Supported: W <= 32, P_max <= 256 (RD_ERR_UNSUPPORTED).  Device
 * errors: packed_len outside [1, P_max] sets RD_DEV_BAD_LENGTH (outputs 0 / -1);
 * a packer or parent index out of range RD_DEV_BAD_INDEX and a token outside
 * [0, V) RD_DEV_BAD_TOKEN (that node is never accepted).  No workspace.
 */
rd_status rd_sample_accept(const void* target_logits, const void* draft_logits, int B, int P_max,
                           int V, float temperature, const int32_t* beams,
                           const int32_t* packer, const int32_t* unpacker,
                           const int32_t* packed_len, int W, int L, const float* u_accept,
                           const float* u_sample, int32_t* accept_len, int32_t* best_beam,
                           int32_t* n_accepted, int32_t* out_tokens, int32_t* dev_status,
                           rd_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* RD_H */
