// paged_attention_decode_noalloc: the decode kernel with library-owned scratch.
//
// For callers that cannot hand the library a device workspace: for example a
// host framework that owns all device memory through its own pool and gives
// plug-ins no buffers of their own, or a serving loop that forbids cudaMalloc
// after start-up because cudaMalloc / cudaFree can synchronise the device and
// stall every other stream.  Those callers still pass their inputs and
// outputs; the split-K scratch lives in one static device array instead.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds PKV_NOALLOC_WORKSPACE_BYTES for it until the process exits.
// In host code its name is only a host-side stand-in, so the device address
// is looked up once per device (cudaGetSymbolAddress, with that device
// current) on the first call made on that device, and cached.
#include <mutex>

#include "pkv_internal.cuh"

namespace {

constexpr size_t kScratchBytes = PKV_NOALLOC_WORKSPACE_BYTES;

// Split-K records of the decode kernel, shared by every
// paged_attention_decode_noalloc call on a device.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_address[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (looked up once).
int scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_address[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
            return PKV_ERR_CUDA;
        g_scratch_address[dev] = p;
    }
    *out = g_scratch_address[dev];
    return PKV_OK;
}

}  // namespace

extern "C" int paged_attention_decode_noalloc(void* out, const void* q, const void* k_pool,
                                              const void* v_pool, const int32_t* block_tables,
                                              const int32_t* seq_lens, int rows, int q_heads,
                                              int kv_heads, int head_dim, int block_size,
                                              float scale, int max_blocks_per_row, int num_blocks,
                                              int max_seq_len, int32_t* dev_err,
                                              cudaStream_t stream) {
    const size_t need = paged_attention_workspace_size(rows, q_heads, kv_heads, head_dim,
                                                       max_seq_len, block_size);
    if (need == 0) {
        // Sizes the decode entry point rejects: let it name the problem.
        return paged_attention_decode(out, q, k_pool, v_pool, block_tables, seq_lens, rows,
                                      q_heads, kv_heads, head_dim, block_size, scale,
                                      max_blocks_per_row, num_blocks, max_seq_len, nullptr, 0,
                                      dev_err, stream);
    }
    if (need > kScratchBytes) return PKV_ERR_WORKSPACE;  // beyond the static scratch
    if (rows == 0) return PKV_OK;
    void* scratch = nullptr;
    const int st = scratch_for_current_device(&scratch);
    if (st != PKV_OK) return st;
    // The array keeps the previous call's contents (words left set by a call
    // that timed out, or by a call of another shape); the record words must
    // start at zero.
    const size_t zero = pkv::decode_workspace_zero_bytes(rows, q_heads, kv_heads, head_dim,
                                                         max_seq_len, block_size);
    if (cudaMemsetAsync(scratch, 0, zero, stream) != cudaSuccess) return PKV_ERR_CUDA;
    return paged_attention_decode(out, q, k_pool, v_pool, block_tables, seq_lens, rows, q_heads,
                                  kv_heads, head_dim, block_size, scale, max_blocks_per_row,
                                  num_blocks, max_seq_len, scratch, kScratchBytes, dev_err, stream);
}
