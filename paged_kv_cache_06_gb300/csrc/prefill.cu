// Chunked-prefill paged attention: argument checks of the C entry point.
// The kernel (tcgen05 tensor cores, accumulators in tensor memory) is in
// prefill_tc.cu.
//
// "Paged attention" (danielfleming.xyz), closing sections: the following
// engine breaks long prompts into pieces of a fixed size (512 tokens) and runs
// decode steps in between; "Continuous batching", closing section: chunking
// long prefills is named as the next step.  Row r's chunk is its newest
// C_r = q_start[r+1] - q_start[r] tokens, already written to the row's blocks;
// query i sits at position p_r + i (p_r = seq_lens[r] - C_r) and attends to
// the row's tokens 0 .. p_r + i.
#include "pkv_internal.cuh"

extern "C" size_t paged_attention_prefill_workspace_size(int rows, int q_heads, int kv_heads,
                                                        int head_dim, int block_size) {
    if (rows < 0 || q_heads <= 0 || kv_heads <= 0 || q_heads % kv_heads || head_dim <= 0 ||
        block_size <= 0)
        return 0;
    return pkv::prefill_workspace_bytes();
}

extern "C" int paged_attention_prefill(void* out, const void* q, const void* k_pool,
                                       const void* v_pool, const int32_t* block_tables,
                                       const int32_t* seq_lens, const int32_t* q_start, int rows,
                                       int total_q, int q_heads, int kv_heads, int head_dim,
                                       int block_size, float scale, int max_blocks_per_row,
                                       int num_blocks, int max_seq_len, void* workspace,
                                       size_t workspace_bytes, int32_t* dev_err,
                                       cudaStream_t stream) {
    using namespace pkv;
    if (rows < 0 || total_q < 0 || q_heads <= 0 || kv_heads <= 0 || q_heads % kv_heads ||
        block_size <= 0 || max_blocks_per_row <= 0 || num_blocks <= 0 || max_seq_len < 0 ||
        !isfinite(scale))
        return PKV_ERR_INVALID_ARG;
    if ((int64_t)max_seq_len > (int64_t)max_blocks_per_row * block_size) return PKV_ERR_INVALID_ARG;
    if (head_dim != kHeadDim || block_size % 16 || rows > 1024 || q_heads > 65535)
        return PKV_ERR_UNSUPPORTED;
    if (rows == 0 || total_q == 0) return PKV_OK;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !seq_lens || !q_start)
        return PKV_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
        return PKV_ERR_INVALID_ARG;
    if (workspace && ((reinterpret_cast<uintptr_t>(workspace) & 255) ||
                      workspace_bytes < prefill_workspace_bytes()))
        return PKV_ERR_WORKSPACE;
    return prefill_tc_launch(out, q, k_pool, v_pool, block_tables, seq_lens, q_start, rows, total_q,
                             q_heads, kv_heads, block_size, scale, max_blocks_per_row, num_blocks,
                             max_seq_len, workspace, dev_err, stream);
}
