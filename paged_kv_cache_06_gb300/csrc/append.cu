// paged_kv_append: write each row's new K/V token into its slot.
//
// "SLM paged attention" (aicassindra.com), section "The architecture": a
// row's table turns the logical block index (position / block_size) into a
// physical block id, and the final block takes one slot after another.
//
// One thread block per row; each thread moves 16-byte vectors.  Per layer at
// 32 rows this is 32 KB of traffic, so the kernel is launch-latency bound.
#include "pkv_internal.cuh"

namespace pkv {

__global__ void __launch_bounds__(128) append_kernel(
    uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, const int32_t* __restrict__ tables,
    const int32_t* __restrict__ positions, const uint4* __restrict__ k_new,
    const uint4* __restrict__ v_new, int kv_heads, int head_dim, int block_size, int mbpr,
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
    // One token of one row = kv_heads * head_dim halves = vecs 16-byte vectors,
    // contiguous both in k_new and in the pool slot.
    const int vecs = kv_heads * head_dim / 8;
    const int64_t dst = ((int64_t)pb * block_size + pos % block_size) * vecs;
    const int64_t src = (int64_t)r * vecs;
    for (int i = threadIdx.x; i < 2 * vecs; i += blockDim.x) {
        if (i < vecs)
            k_pool[dst + i] = k_new[src + i];
        else
            v_pool[dst + i - vecs] = v_new[src + i - vecs];
    }
}

}  // namespace pkv

extern "C" int paged_kv_append(void* k_pool, void* v_pool, const int32_t* block_tables,
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
    if (!k_pool || !v_pool || !block_tables || !positions || !k_new || !v_new)
        return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_new) || !aligned16(v_new))
        return PKV_ERR_INVALID_ARG;
    const int vecs2 = 2 * kv_heads * head_dim / 8;
    const int threads = vecs2 >= 128 ? 128 : ((vecs2 + 31) / 32) * 32;
    append_kernel<<<rows, threads, 0, stream>>>(
        static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), block_tables, positions,
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), kv_heads, head_dim,
        block_size, max_blocks_per_row, num_blocks, dev_err);
    return launch_status();
}
