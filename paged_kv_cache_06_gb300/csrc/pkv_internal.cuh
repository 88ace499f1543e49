// Internal helpers shared by libpagedkv's CUDA translation units.
#pragma once

#include <cuda.h>
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
size_t decode_workspace_zero_bytes(int rows, int q_heads, int kv_heads, int head_dim,
                                   int max_seq_len, int block_size);

// TMA / tensor-core decode kernel (decode_tma.cu).
bool tma_decode_supported(int rows, int q_heads, int kv_heads, int head_dim, int block_size);
size_t tma_workspace_bytes(int rows, int q_heads, int kv_heads, int max_seq_len);
size_t tma_workspace_zero_bytes(int rows, int kv_heads, int max_seq_len);
// Per-step decode plan (decode_tma.cu): bytes for these sizes, and its launch.
size_t tma_plan_bytes(int rows, int kv_heads, int max_seq_len);
int tma_plan_launch(void* plan, size_t plan_bytes, const int32_t* tables, const int32_t* seq_lens,
                    const int32_t* positions, int rows, int q_heads, int kv_heads, int block_size,
                    int mbpr, int num_blocks, int max_seq_len, int32_t* dev_err,
                    cudaStream_t stream);
// New-token append fused into the decode launch (positions / k_new / v_new as
// in paged_kv_append).
struct AppendArgs {
    const int32_t* positions;
    const void* k_new;
    const void* v_new;
};
// Cached tiled tensor map (128-byte swizzle) over a 3-D array: dims and box
// innermost first, strides in bytes of dims 1 and 2.
int tiled_map_3d(const void* base, CUtensorMapDataType dtype, const int64_t dims[3],
                 const int64_t strides[2], const int box[3], CUtensorMap* out);

// The tcgen05 chunked-prefill kernel (arguments validated by the caller).
// workspace: prefill_workspace_bytes() of caller memory (arrival words, zero
// between calls, then partials), or null for the library-owned scratch.
size_t prefill_workspace_bytes();
size_t prefill_count_bytes();
int prefill_tc_launch(void* out, const void* q, const void* k_pool, const void* v_pool,
                      const int32_t* block_tables, const int32_t* seq_lens,
                      const int32_t* q_start, int rows, int total_q, int q_heads, int kv_heads,
                      int block_size, float scale, int max_blocks_per_row, int num_blocks,
                      int max_seq_len, void* workspace, int32_t* dev_err, cudaStream_t stream);

int tma_decode_launch(void* out, const void* q, const void* k_base, const void* v_base,
                      const int32_t* tables, const int32_t* seq_lens, int rows, int q_heads,
                      int kv_heads, int block_size, float scale, int mbpr, int num_blocks,
                      int max_seq_len, int width, void* workspace, int32_t* dev_err,
                      cudaStream_t stream, const AppendArgs* append = nullptr, bool pdl = false,
                      const float* k_scale = nullptr, const float* v_scale = nullptr,
                      const void* plan = nullptr);

}  // namespace pkv
