// FP8 (E4M3) KV pools: append with quantisation, and decode.
//
// "PagedAttention" (deepconcepts.dev), section "Checking it on a real
// system", names FP8 KV as a way to change the bytes per token, the term
// paging itself never touches.  The pages fix no format; the one used here is
// E4M3 with one float scale per KV head: a stored code c stands for
// e4m3(c) * scale[head].  A new element x is stored as the nearest E4M3 value
// (ties to even, saturating at 448) of the binary32 quotient x / scale.
#include "pkv_internal.cuh"
#include "fp8_codec.cuh"

namespace pkv {

// grid: rows; threads: (K or V, head, 8-dim chunk).
__global__ void append_fp8_kernel(uint8_t* __restrict__ k_pool, uint8_t* __restrict__ v_pool,
                                  const float* __restrict__ k_scale,
                                  const float* __restrict__ v_scale,
                                  const int32_t* __restrict__ tables,
                                  const int32_t* __restrict__ positions,
                                  const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                  int kv_heads, int head_dim, int block_size, int mbpr,
                                  int num_blocks, int32_t* dev_err) {
    const int r = blockIdx.x;
    const int pos = positions[r];
    if (pos < 0) return;
    const int lb = pos / block_size;
    if (lb >= mbpr) {
        if (threadIdx.x == 0) flag_error(dev_err, PKV_DEV_ERR_POSITION);
        return;
    }
    const int pb = tables[(int64_t)r * mbpr + lb];
    if (pb < 0 || pb >= num_blocks) {
        if (threadIdx.x == 0) flag_error(dev_err, PKV_DEV_ERR_BLOCK_ID);
        return;
    }
    const int chunks = head_dim / 8;
    const int per = kv_heads * chunks;  // 16-byte input vectors per token and pool
    const int64_t slot = ((int64_t)pb * block_size + pos % block_size) * kv_heads * head_dim;
    for (int i = threadIdx.x; i < 2 * per; i += blockDim.x) {
        const bool is_v = i >= per;
        const int j = is_v ? i - per : i;
        const int h = j / chunks;
        const uint4 x = (is_v ? v_new : k_new)[(int64_t)r * per + j];
        const uint2 q = quantize8(x, is_v ? v_scale[h] : k_scale[h]);
        *reinterpret_cast<uint2*>((is_v ? v_pool : k_pool) + slot + (int64_t)j * 8) = q;
    }
}

}  // namespace pkv

extern "C" int paged_kv_append_fp8(void* k_pool, void* v_pool, const float* k_scale,
                                   const float* v_scale, const int32_t* block_tables,
                                   const int32_t* positions, const void* k_new, const void* v_new,
                                   int rows, int kv_heads, int head_dim, int block_size,
                                   int max_blocks_per_row, int num_blocks, int32_t* dev_err,
                                   cudaStream_t stream) {
    using namespace pkv;
    if (rows < 0 || kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || max_blocks_per_row <= 0 ||
        num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (head_dim % 8) return PKV_ERR_UNSUPPORTED;
    if (rows == 0) return PKV_OK;
    if (rows > 2147483647) return PKV_ERR_UNSUPPORTED;
    if (!k_pool || !v_pool || !k_scale || !v_scale || !block_tables || !positions || !k_new || !v_new)
        return PKV_ERR_INVALID_ARG;
    if (((uintptr_t)k_pool | (uintptr_t)v_pool) % 8 || !aligned16(k_new) || !aligned16(v_new))
        return PKV_ERR_INVALID_ARG;
    append_fp8_kernel<<<rows, 64, 0, stream>>>(
        static_cast<uint8_t*>(k_pool), static_cast<uint8_t*>(v_pool), k_scale, v_scale, block_tables,
        positions, static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), kv_heads,
        head_dim, block_size, max_blocks_per_row, num_blocks, dev_err);
    return launch_status();
}

extern "C" int paged_attention_decode_fp8(void* out, const void* q, const void* k_pool,
                                          const void* v_pool, const float* k_scale,
                                          const float* v_scale, const int32_t* block_tables,
                                          const int32_t* seq_lens, int rows, int q_heads,
                                          int kv_heads, int head_dim, int block_size, float scale,
                                          int max_blocks_per_row, int num_blocks, int max_seq_len,
                                          void* workspace, size_t workspace_bytes,
                                          int32_t* dev_err, cudaStream_t stream) {
    using namespace pkv;
    if (q_heads <= 0 || kv_heads <= 0 || head_dim <= 0 || q_heads % kv_heads) return PKV_ERR_INVALID_ARG;
    if (rows < 0 || block_size <= 0 || block_size > 1024 || max_blocks_per_row <= 0 ||
        num_blocks <= 0 || max_seq_len < 0 || !isfinite(scale))
        return PKV_ERR_INVALID_ARG;
    if ((int64_t)max_seq_len > (int64_t)max_blocks_per_row * block_size) return PKV_ERR_INVALID_ARG;
    if (!tma_decode_supported(rows, q_heads, kv_heads, head_dim, block_size) || kv_heads > 16)
        return PKV_ERR_UNSUPPORTED;
    if (rows == 0) return PKV_OK;
    if (!out || !q || !k_pool || !v_pool || !k_scale || !v_scale || !block_tables || !seq_lens)
        return PKV_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
        return PKV_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < tma_workspace_bytes(rows, q_heads, kv_heads, max_seq_len))
        return PKV_ERR_WORKSPACE;
    return tma_decode_launch(out, q, k_pool, v_pool, block_tables, seq_lens, rows, q_heads, kv_heads,
                             block_size, scale, max_blocks_per_row, num_blocks, max_seq_len, 0,
                             workspace, dev_err, stream, nullptr, false, k_scale, v_scale);
}

extern "C" int paged_attention_append_decode_fp8(
    void* out, const void* q, void* k_pool, void* v_pool, const float* k_scale, const float* v_scale,
    const int32_t* block_tables, const int32_t* seq_lens, const int32_t* positions, const void* k_new,
    const void* v_new, int rows, int q_heads, int kv_heads, int head_dim, int block_size, float scale,
    int max_blocks_per_row, int num_blocks, int max_seq_len, void* workspace, size_t workspace_bytes,
    unsigned flags, int32_t* dev_err, cudaStream_t stream) {
    using namespace pkv;
    if (q_heads <= 0 || kv_heads <= 0 || head_dim <= 0 || q_heads % kv_heads) return PKV_ERR_INVALID_ARG;
    if (rows < 0 || block_size <= 0 || block_size > 1024 || max_blocks_per_row <= 0 ||
        num_blocks <= 0 || max_seq_len < 0 || !isfinite(scale) || (flags & ~PKV_FLAG_PDL))
        return PKV_ERR_INVALID_ARG;
    if ((int64_t)max_seq_len > (int64_t)max_blocks_per_row * block_size) return PKV_ERR_INVALID_ARG;
    if (!tma_decode_supported(rows, q_heads, kv_heads, head_dim, block_size) || kv_heads > 16)
        return PKV_ERR_UNSUPPORTED;
    if (rows == 0) return PKV_OK;
    if (!out || !q || !k_pool || !v_pool || !k_scale || !v_scale || !block_tables || !seq_lens ||
        !positions || !k_new || !v_new)
        return PKV_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) ||
        !aligned16(k_new) || !aligned16(v_new))
        return PKV_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < tma_workspace_bytes(rows, q_heads, kv_heads, max_seq_len))
        return PKV_ERR_WORKSPACE;
    const AppendArgs app{positions, k_new, v_new};
    return tma_decode_launch(out, q, k_pool, v_pool, block_tables, seq_lens, rows, q_heads, kv_heads,
                             block_size, scale, max_blocks_per_row, num_blocks, max_seq_len, 0,
                             workspace, dev_err, stream, &app, (flags & PKV_FLAG_PDL) != 0, k_scale,
                             v_scale);
}
