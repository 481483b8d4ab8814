// rd_greedy_accept_noalloc: greedy verification for callers that cannot
// allocate device memory.
//
// rd_greedy_accept needs a small scratch area (one 64-bit argmax key per packed
// row and one reserved word per request).  Its caller normally allocates it.  Some
// callers cannot: code that runs inside a memory pool they do not own, plugins
// whose host framework forbids cudaMalloc on the serving path, or runtimes that
// must not allocate after start-up because an allocation can synchronise the
// device or fail under memory pressure.  This entry point takes the scratch from
// a fixed array in device global memory instead, owned by the library.
//
// Limits and sharing:
//  - the array holds kMaxRows argmax keys and kMaxRequests reserved words
//    (B * P_max <= 65536 and B <= 65535, else RD_ERR_UNSUPPORTED);
//    every GPU that loads librd holds it (about 768 KB) until the process exits;
//  - every call on a device uses the same array: calls whose kernels overlap on
//    the GPU (two streams, or two threads) race and give wrong results;
//  - each call clears the part it uses (cudaMemsetAsync on the caller's stream)
//    before its kernel, so a previous call's leftovers never leak into it;
//  - the first call on a device looks up the array's device address
//    (cudaGetSymbolAddress) with that device current; make that first call
//    before any stream capture begins.  The address is cached for the life of
//    the process, so it is stale after a cudaDeviceReset of that device.
#include <mutex>

#include "rd_internal.cuh"

namespace {

constexpr size_t kMaxRows = 65536;         // B * P_max
constexpr size_t kMaxRequests = 65535;     // B
constexpr size_t kKeyBytes = kMaxRows * sizeof(unsigned long long);
constexpr size_t kScratchBytes = kKeyBytes + kMaxRequests * sizeof(unsigned int);

// Device-resident scratch.  In host code this name is only a stand-in for the
// symbol, never a device address: the address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_accept_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_ptr(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_accept_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" rd_status rd_greedy_accept_noalloc(const void* logits, int B, int P_max, int V,
                                              const int32_t* beams, const int32_t* unpacker,
                                              const int32_t* packed_len, int W, int L,
                                              int32_t* argmax, int32_t* accept_len,
                                              int32_t* best_beam, int32_t* n_accepted,
                                              int32_t* out_tokens, int32_t* dev_status,
                                              rd_stream_t stream)
{
    if (B < 0 || P_max < 1 || V < 1 || W < 1 || L < 1) return RD_ERR_INVALID_ARG;
    if (W > RD_MAX_BEAMS || P_max > RD_MAX_PACKED || B > 65535) return RD_ERR_UNSUPPORTED;
    if ((size_t)B * P_max > kMaxRows || (size_t)B > kMaxRequests) return RD_ERR_UNSUPPORTED;
    if (B == 0) return RD_OK;
    if (!logits || !beams || !unpacker || !packed_len || !argmax || !accept_len ||
        !best_beam || !n_accepted || !out_tokens)
        return RD_ERR_INVALID_ARG;
    void* scratch = nullptr;
    if (scratch_ptr(&scratch) != cudaSuccess) return RD_ERR_CUDA;
    // the kernels expect keys [B*P_max] (64-bit) followed by B reserved 32-bit words, all zero
    cudaStream_t s = (cudaStream_t)stream;
    const size_t used = (size_t)B * P_max * sizeof(unsigned long long) + (size_t)B * sizeof(unsigned int);
    if (cudaMemsetAsync(scratch, 0, used, s) != cudaSuccess) return RD_ERR_CUDA;
    return rd_launch_greedy_accept(logits, B, P_max, V, beams, unpacker, packed_len, W, L,
                                   argmax, accept_len, best_beam, n_accepted, out_tokens,
                                   scratch, dev_status, s) == cudaSuccess
               ? RD_OK
               : RD_ERR_CUDA;
}
