// Internal helpers shared by libpagedkv's CUDA translation units.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "paged_kv.h"

namespace pkv {

constexpr int kHeadDim = 128;   // the only head_dim the decode kernels are built for
constexpr int kMaxGroup = 8;    // query heads per KV head (one 8-wide MMA column tile)

__device__ __forceinline__ void flag_error(int32_t* dev_err, int bit) {
    if (dev_err) atomicOr(reinterpret_cast<int*>(dev_err), bit);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int launch_status() {
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Bytes at the start of a decode workspace that must be zero before a call.
size_t decode_workspace_zero_bytes(int rows);

}  // namespace pkv
