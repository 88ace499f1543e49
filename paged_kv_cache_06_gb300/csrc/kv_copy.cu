// Block copies for copy-on-write, and the prefill scatter into blocks.
//
// "SLM paged attention" (aicassindra.com), sections "The architecture" and
// "End-to-end flow": a sequence about to write into a block it shares gets a
// private copy of that one block, and its table entry is switched to the
// copy.  "Paged attention" (danielfleming.xyz), section "What changed": a
// batched prefill pads its rows on the left to the batch's longest prompt,
// and each row's K/V then moves into the row's blocks without the padding.
//
// Both are pure data movement: 16-byte vectors, consecutive threads on
// consecutive addresses, grids sized in whole blocks of work.
#include "pkv_internal.cuh"

namespace pkv {

constexpr int kCopyThreads = 256;
constexpr int kVecsPerThread = 4;

// grid (pair, pool, chunk): block dst_ids[pair] of pool (K or V) := block src_ids[pair].
__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(
    uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, const int32_t* __restrict__ src_ids,
    const int32_t* __restrict__ dst_ids, int64_t block_vecs, int num_blocks, int32_t* dev_err) {
    const int i = blockIdx.x;
    const int src = src_ids[i], dst = dst_ids[i];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
            flag_error(dev_err, PKV_DEV_ERR_BLOCK_ID);
        return;
    }
    if (src == dst) return;
    uint4* pool = blockIdx.y == 0 ? k_pool : v_pool;
    const uint4* s = pool + (int64_t)src * block_vecs;
    uint4* d = pool + (int64_t)dst * block_vecs;
    const int64_t base = (int64_t)blockIdx.z * kCopyThreads * kVecsPerThread + threadIdx.x;
    uint4 tmp[kVecsPerThread];
#pragma unroll
    for (int k = 0; k < kVecsPerThread; ++k) {
        const int64_t j = base + (int64_t)k * kCopyThreads;
        if (j < block_vecs) tmp[k] = s[j];
    }
#pragma unroll
    for (int k = 0; k < kVecsPerThread; ++k) {
        const int64_t j = base + (int64_t)k * kCopyThreads;
        if (j < block_vecs) d[j] = tmp[k];
    }
}

constexpr int kScatterTokens = 16;  // tokens per thread block

// grid (row, token chunk): tokens [chunk * 16, chunk * 16 + 16) of the row.
__global__ void __launch_bounds__(kCopyThreads) prefill_scatter_kernel(
    uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, const int32_t* __restrict__ tables,
    const int32_t* __restrict__ src_start, const int32_t* __restrict__ dst_start,
    const int32_t* __restrict__ lengths, const uint4* __restrict__ k_src,
    const uint4* __restrict__ v_src, int width, int tok_vecs, int block_size, int mbpr,
    int num_blocks, int32_t* dev_err) {
    const int r = blockIdx.x;
    const int len = lengths[r];
    const int t0 = blockIdx.y * kScatterTokens;
    if (len <= 0 || t0 >= len) return;
    const int s0 = src_start[r], d0 = dst_start[r];
    if (s0 < 0 || d0 < 0 || (int64_t)s0 + len > width) {
        if (threadIdx.x == 0 && blockIdx.y == 0) flag_error(dev_err, PKV_DEV_ERR_POSITION);
        return;
    }
    const int ntok = min(kScatterTokens, len - t0);
    // Each thread copies 16-byte vectors of the chunk's tokens, K then V.
    const int total = 2 * ntok * tok_vecs;
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const bool is_v = i >= ntok * tok_vecs;
        const int j = is_v ? i - ntok * tok_vecs : i;
        const int t = t0 + j / tok_vecs;
        const int c = j % tok_vecs;
        const int pos = d0 + t;
        const int lb = pos / block_size;
        if (lb >= mbpr) {
            if (c == 0) flag_error(dev_err, PKV_DEV_ERR_POSITION);
            continue;
        }
        const int pb = tables[(int64_t)r * mbpr + lb];
        if (pb < 0 || pb >= num_blocks) {
            if (c == 0) flag_error(dev_err, PKV_DEV_ERR_BLOCK_ID);
            continue;
        }
        const int64_t dst = ((int64_t)pb * block_size + pos % block_size) * tok_vecs + c;
        const int64_t src = ((int64_t)r * width + s0 + t) * tok_vecs + c;
        if (is_v)
            v_pool[dst] = v_src[src];
        else
            k_pool[dst] = k_src[src];
    }
}

}  // namespace pkv

extern "C" int paged_kv_copy_blocks(void* k_pool, void* v_pool, const int32_t* src_ids,
                                    const int32_t* dst_ids, int n, int block_size, int kv_heads,
                                    int head_dim, int num_blocks, int32_t* dev_err,
                                    cudaStream_t stream) {
    using namespace pkv;
    if (n < 0 || block_size <= 0 || kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (head_dim % 8) return PKV_ERR_UNSUPPORTED;
    if (n == 0) return PKV_OK;
    if (!k_pool || !v_pool || !src_ids || !dst_ids) return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(v_pool)) return PKV_ERR_INVALID_ARG;
    const int64_t block_vecs = (int64_t)block_size * kv_heads * head_dim / 8;
    const int64_t chunks = (block_vecs + kCopyThreads * kVecsPerThread - 1) / (kCopyThreads * kVecsPerThread);
    if (chunks > 65535) return PKV_ERR_UNSUPPORTED;
    // grid.x is the pair index (up to 2^31 - 1), y the pool, z the chunk
    copy_blocks_kernel<<<dim3((unsigned)n, 2, (unsigned)chunks), kCopyThreads, 0, stream>>>(
        static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), src_ids, dst_ids, block_vecs,
        num_blocks, dev_err);
    return launch_status();
}

extern "C" int paged_kv_prefill_scatter(void* k_pool, void* v_pool, const int32_t* block_tables,
                                        const int32_t* src_start, const int32_t* dst_start,
                                        const int32_t* lengths, const void* k_src,
                                        const void* v_src, int rows, int width, int kv_heads,
                                        int head_dim, int block_size, int max_blocks_per_row,
                                        int num_blocks, int32_t* dev_err, cudaStream_t stream) {
    using namespace pkv;
    if (rows < 0 || width < 0 || kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        max_blocks_per_row <= 0 || num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (head_dim % 8) return PKV_ERR_UNSUPPORTED;
    if (rows == 0 || width == 0) return PKV_OK;
    if (rows > 2147483647 / 2) return PKV_ERR_UNSUPPORTED;
    if (!k_pool || !v_pool || !block_tables || !src_start || !dst_start || !lengths || !k_src ||
        !v_src)
        return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_src) || !aligned16(v_src))
        return PKV_ERR_INVALID_ARG;
    const int chunks = (width + kScatterTokens - 1) / kScatterTokens;
    if (chunks > 65535) return PKV_ERR_UNSUPPORTED;
    prefill_scatter_kernel<<<dim3((unsigned)rows, (unsigned)chunks), kCopyThreads, 0, stream>>>(
        static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), block_tables, src_start,
        dst_start, lengths, static_cast<const uint4*>(k_src), static_cast<const uint4*>(v_src),
        width, kv_heads * head_dim / 8, block_size, max_blocks_per_row, num_blocks, dev_err);
    return launch_status();
}
