// Helpers shared by the attention kernels (tree attention and the paired-tile
// causal kernel): 128-byte-swizzle addressing, bf16 packing, exp2, a bounded
// warp-wide barrier wait, and the TMA tensor maps of the K/V cache and queries.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "tc_ptx.cuh"

namespace rdattn {

constexpr int kChunk = 64;                 // KV positions per chunk (one TMA box)

// 16-byte chunk c of row r in a [rows][128 B] tile with the 128-byte swizzle
__device__ __forceinline__ uint32_t sw128(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// 2^x with the hardware approximation (ex2.approx; 2^-inf = 0)
__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Warp-uniform bounded wait: every lane waits, and the warp fails as one if any
// lane ran out of budget or saw the abort flag.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          long long budget)
{
    const bool ok = rdtc::mbar_wait(bar, parity, abort, budget);
    return __all_sync(0xffffffffu, ok);
}

// ------------------------------------------------------------------ host side
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, []() {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [rows, heads, D] bf16 -> boxes of 64 positions x 1 head x 64 columns, 128-byte swizzle
inline bool make_kv_map(CUtensorMap* map, const void* base, int64_t rows, int heads, int D)
{
    auto fn = encode_fn();
    if (!fn) return false;
    if (rows < 1) rows = 1;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)heads * D * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)kChunk};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// queries [rows, Hq, D] bf16 -> boxes of box_rows positions x G heads x 64 columns,
// 128-byte swizzle: a box lands as box_rows * G rows of 128 bytes, row p G + g
inline bool make_q_map(CUtensorMap* map, const void* base, int64_t rows, int heads, int D, int G,
                       int box_rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    if (rows < 1) rows = 1;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)heads * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace rdattn
