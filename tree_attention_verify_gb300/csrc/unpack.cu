// rd_unpack kernel: out[b, w, i, :] = packed[b, unpacker[b, w, i], :].
//
// The gather of the PyTorch unpack in the NVIDIA blog "ReDrafter in
// TensorRT-LLM" (section "Implementing in-Engine Validation and Drafting"),
// as a bit-exact row copy.  One CTA per output row; 16-byte vector copies when
// the row pitch and both base pointers allow it, 4- or 2-byte words otherwise.
#include "rd_internal.cuh"

namespace {

template <typename T>
__global__ void __launch_bounds__(128)
unpack_kernel(const T* __restrict__ packed, int P_max, size_t row_words,
              const int32_t* __restrict__ unpacker, int WL, T* __restrict__ out,
              int32_t* dev_status)
{
    const int r = blockIdx.x;                  // output row = b*W*L + w*L + i
    const int b = r / WL;
    const int p = __ldg(unpacker + r);
    T* dst = out + (size_t)r * row_words;
    if (p < 0 || p >= P_max) {
        if (threadIdx.x == 0) rd_flag(dev_status, RD_DEV_BAD_INDEX);
        for (size_t k = threadIdx.x; k < row_words; k += blockDim.x) dst[k] = T{};
        return;
    }
    const T* src = packed + ((size_t)b * P_max + p) * row_words;
    for (size_t k = threadIdx.x; k < row_words; k += blockDim.x) dst[k] = __ldg(src + k);
}

}  // namespace

cudaError_t rd_launch_unpack(const void* packed, int esize, int B, int P_max, int Dh,
                             const int32_t* unpacker, int W, int L, void* out,
                             int32_t* dev_status, cudaStream_t stream)
{
    const size_t row_bytes = (size_t)Dh * esize;
    const int rows = B * W * L;
    const int WL = W * L;
    const bool v16 = row_bytes % 16 == 0 && (reinterpret_cast<uintptr_t>(packed) % 16) == 0 &&
                     (reinterpret_cast<uintptr_t>(out) % 16) == 0;
    const bool v4 = row_bytes % 4 == 0 && (reinterpret_cast<uintptr_t>(packed) % 4) == 0 &&
                    (reinterpret_cast<uintptr_t>(out) % 4) == 0;
    if (v16)
        unpack_kernel<uint4><<<rows, 128, 0, stream>>>(
            static_cast<const uint4*>(packed), P_max, row_bytes / 16, unpacker, WL,
            static_cast<uint4*>(out), dev_status);
    else if (v4)
        unpack_kernel<uint32_t><<<rows, 128, 0, stream>>>(
            static_cast<const uint32_t*>(packed), P_max, row_bytes / 4, unpacker, WL,
            static_cast<uint32_t*>(out), dev_status);
    else
        unpack_kernel<uint16_t><<<rows, 128, 0, stream>>>(
            static_cast<const uint16_t*>(packed), P_max, row_bytes / 2, unpacker, WL,
            static_cast<uint16_t*>(out), dev_status);
    return cudaGetLastError();
}
