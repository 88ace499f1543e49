// Chunked-prefill paged attention for sm_103a: several query tokens per row,
// causal within the row's chunk.
//
// "Paged attention" (danielfleming.xyz), closing sections: the next engine
// splits long prompts into fixed chunks (512 tokens) so decode steps run
// between them; "Continuous batching", closing section: a long prefill split
// into fixed size chunks.  Row r's chunk is its newest
// C_r = q_start[r+1] - q_start[r] tokens, already written to the row's blocks;
// query i sits at position p_r + i (p_r = seq_lens[r] - C_r) and attends to
// the row's tokens 0 .. p_r + i ("PagedAttention", deepconcepts.dev, section
// "PagedAttention": the keys are gathered through the row's block table).
//
// Work split.  A block takes 64 queries of one row and one query head
// (grid.y), as four warps of 16.  The producer warp stages the queries with
// two TMA boxes, then streams the row's keys and values through a 2-stage
// ring, 64 tokens (four 16-token granules, each inside one physical block)
// per stage, up to the last position the block's queries may see.  Per stage
// every consumer warp computes, with mma.sync m16n8k16 (fp16 in, fp32
// accumulate):
//   S[16 q][64 tok] = Q[16][128] . K^T          (causal mask, scale, base-2)
//   online softmax per query in fp32
//   O[16 q][128]   += P[16][64] . V[64][128]
// A block's causal mask only bites in the stages that reach past its first
// query's position.  Every wait is bounded; table entries are range-checked
// before a copy is issued.
#include "pkv_internal.cuh"
#include "ptx.cuh"

namespace pkv {
namespace prefill {

using namespace ptx;

constexpr int kQTile = 64;                  // queries per block
constexpr int kKTile = 64;                  // key tokens per stage
constexpr int kGranule = 16;
constexpr int kStages = 2;
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32 + 32;  // consumers + producer
constexpr int kMaxRows = 1024;
constexpr uint32_t kBox = 16 * 128;         // 16 rows x 128 B
constexpr uint32_t kSlot = 4 * kBox;        // granule: K 0-63, K 64-127, V 0-63, V 64-127
constexpr uint32_t kSlotV = 2 * kBox;
constexpr uint32_t kStageBytes = 4 * kSlot; // 64 tokens
constexpr uint32_t kQHalf = kQTile * 128;   // 64 queries x 64 dims
constexpr float kLog2e = 1.4426950408889634f;

struct Params {
    __half* out;
    const int32_t* tables;
    const int32_t* seq_lens;
    const int32_t* q_start;
    int rows, hq, group, bs, mbpr, nb, limit;
    float scale_log2;
    int32_t* dev_err;
};

struct Smem {
    static constexpr uint32_t q = 0;                                  // [2 halves] queries
    static constexpr uint32_t kv = q + 2 * kQHalf;                    // [stages] granule slots
    static constexpr uint32_t bars = kv + kStages * kStageBytes;      // q, full[2], empty[2]
    static constexpr uint32_t valid = bars + 64;                      // [stages][4] tokens
    static constexpr uint32_t part = valid + kStages * 4 * 4;         // scan partials [threads]
    static constexpr uint32_t pre = part + kThreads * 4;              // tile prefix [rows + 1]
    __host__ __device__ static constexpr uint32_t total(int rows) {
        return pre + (uint32_t)(rows + 1) * 4 + 1024;
    }
};
static_assert(Smem::kv % 1024 == 0, "128B-swizzled stages need 1024-byte alignment");

__global__ void __launch_bounds__(kThreads, 2)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const Params p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_q = sbase + Smem::bars;
    const uint32_t bar_full = bar_q + 8;
    const uint32_t bar_empty = bar_full + kStages * 8;
    int* sm_valid = reinterpret_cast<int*>(smem + Smem::valid);
    int* sm_part = reinterpret_cast<int*>(smem + Smem::part);
    int* sm_pre = reinterpret_cast<int*>(smem + Smem::pre);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rows = p.rows;
    const int h = blockIdx.y, kvh = h / p.group;

    // ---- tiles per row, their prefix, and this block's (row, tile) ----
    const int per = (rows + kThreads - 1) / kThreads;
    int sum = 0;
    for (int i = 0; i < per; ++i) {
        const int r = tid * per + i;
        if (r < rows) {
            const int C = p.q_start[r + 1] - p.q_start[r];
            const int L = p.seq_lens[r];
            int t = (C + kQTile - 1) / kQTile;
            if (C < 0 || L < C || L > p.limit) {
                if (blockIdx.x == 0 && h == 0) flag_error(p.dev_err, PKV_DEV_ERR_SEQ_LEN);
                t = 0;
            }
            sm_pre[r] = t;
            sum += t;
        }
    }
    sm_part[tid] = sum;
    if (tid == 0) {
        mbar_init(bar_q, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (warp == 0) {
        constexpr int kPer = (kThreads + 31) / 32;
        int v[kPer], acc = 0;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int idx = lane * kPer + j;
            v[j] = idx < kThreads ? sm_part[idx] : 0;
            acc += v[j];
        }
        int incl = acc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        int run = incl - acc;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int idx = lane * kPer + j;
            if (idx < kThreads) sm_part[idx] = run;
            run += v[j];
        }
    }
    __syncthreads();
    {
        int run = sm_part[tid];
        for (int i = 0; i < per; ++i) {
            const int r = tid * per + i;
            if (r < rows) {
                const int c = sm_pre[r];
                sm_pre[r] = run;
                run += c;
            }
        }
        if (tid == kThreads - 1) sm_pre[rows] = run;
    }
    __syncthreads();
    const int b = blockIdx.x;
    if (b >= sm_pre[rows]) return;  // the grid is an upper bound on the tiles
    int lo = 0, hi = rows - 1;
    while (lo < hi) {  // largest row whose first tile is <= b
        const int mid = (lo + hi + 1) >> 1;
        if (sm_pre[mid] <= b) lo = mid; else hi = mid - 1;
    }
    const int r = lo;
    const int tile = b - sm_pre[r];
    const int C = p.q_start[r + 1] - p.q_start[r];
    const int L = p.seq_lens[r];
    const int pos0 = L - C;                       // position of the chunk's first query
    const int i_first = tile * kQTile;            // chunk-local index of the block's first query
    const int nq = min(kQTile, C - i_first);
    const int kend = pos0 + i_first + nq;         // keys 0 .. kend-1 are visible to someone
    const int nkt = (kend + kKTile - 1) / kKTile;
    const int qrow0 = p.q_start[r] + i_first;     // packed index of the block's first query

    if (warp == kWarps) {
        // ============================ producer ============================
        if (lane == 0) {
            mbar_arrive_expect_tx(bar_q, 2 * kQHalf);
            tma_load_3d(sbase + Smem::q, &qmap, 0, h, qrow0, bar_q);
            tma_load_3d(sbase + Smem::q + kQHalf, &qmap, 64, h, qrow0, bar_q);
        }
        for (int kt = 0; kt < nkt; ++kt) {
            const int s = kt % kStages;
            const uint32_t round = (uint32_t)kt / kStages;
            if (!mbar_wait(bar_empty + 8 * s, (round & 1) ^ 1)) {
                if (lane == 0) flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
                break;
            }
            int valid = 0, zrow = 0;
            bool issue = false;
            if (lane < 4) {
                const int tok0 = kt * kKTile + lane * kGranule;
                valid = max(0, min(kGranule, kend - tok0));
                if (valid > 0) {
                    const int pb = p.tables[(int64_t)r * p.mbpr + tok0 / p.bs];
                    if (pb < 0 || pb >= p.nb) {
                        flag_error(p.dev_err, PKV_DEV_ERR_BLOCK_ID);
                        valid = 0;
                    } else {
                        zrow = pb * p.bs + tok0 % p.bs;
                        issue = true;
                    }
                }
                sm_valid[s * 4 + lane] = valid;
            }
            const uint32_t nissue = __popc(__ballot_sync(0xffffffffu, issue));
            __syncwarp();
            const uint32_t fb = bar_full + 8 * s;
            if (lane == 0) mbar_arrive_expect_tx(fb, nissue * kSlot);
            __syncwarp();
            if (issue) {
                const uint32_t dst = sbase + Smem::kv + s * kStageBytes + lane * kSlot;
                tma_load_3d(dst, &kmap, 0, kvh, zrow, fb);
                tma_load_3d(dst + kBox, &kmap, 64, kvh, zrow, fb);
                tma_load_3d(dst + kSlotV, &vmap, 0, kvh, zrow, fb);
                tma_load_3d(dst + kSlotV + kBox, &vmap, 64, kvh, zrow, fb);
            }
        }
        // Drain: every armed stage's copies land before the block exits.
        for (int kt = max(0, nkt - kStages); kt < nkt; ++kt)
            if (!mbar_wait(bar_full + 8 * (kt % kStages), ((uint32_t)kt / kStages) & 1) && lane == 0)
                flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
        if (!mbar_wait(bar_q, 0) && lane == 0) flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
        return;
    }

    // ============================== consumers ==============================
    const int gq = lane >> 2, tq = lane & 3;
    if (!mbar_wait(bar_q, 0)) {
        if (lane == 0) flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
        return;
    }
    // A fragments of Q (16 queries of this warp x 128 dims), eight k-steps.
    uint32_t qa[8][4];
    {
        const int row = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int chunk = (ks & 3) * 2 + (lane >> 4);
            ldsm_x4(sbase + Smem::q + (ks >> 2) * kQHalf + row * 128 + ((chunk ^ (row & 7)) << 4),
                    qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
        }
    }
    // Last visible key of this lane's two queries (rows gq and gq + 8).
    const int ia = i_first + warp * 16 + gq, ib = ia + 8;
    const int vis_a = min(pos0 + ia, kend - 1), vis_b = min(pos0 + ib, kend - 1);
    const int warp_first = pos0 + i_first + warp * 16;  // smallest position among the warp's queries

    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
    float o[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

    for (int kt = 0; kt < nkt; ++kt) {
        const int s = kt % kStages;
        if (!mbar_wait(bar_full + 8 * s, ((uint32_t)kt / kStages) & 1)) {
            if (lane == 0) flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
            return;
        }
        const uint32_t stage = sbase + Smem::kv + s * kStageBytes;
        unsigned char* stage_ptr = smem + Smem::kv + s * kStageBytes;
        // V rows past a granule's valid tokens may hold anything: zero them
        // (every warp writes the same zeros before reading).
        bool wrote = false;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int v = sm_valid[s * 4 + g];
            if (v < kGranule) {
                uint4* v0 = reinterpret_cast<uint4*>(stage_ptr + g * kSlot + kSlotV);
                for (int i = lane; i < (kGranule - v) * 8; i += 32) {
                    const int row = v + (i >> 3);
                    v0[row * 8 + (i & 7)] = make_uint4(0, 0, 0, 0);
                    v0[kBox / 16 + row * 8 + (i & 7)] = make_uint4(0, 0, 0, 0);
                }
                wrote = true;
            }
        }
        if (wrote) __syncwarp();

        // ---- S = Q K^T over the stage's 64 tokens: n-tiles of 8 tokens ----
        float sc[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
        {
            const int row = (lane & 7) + ((lane >> 4) << 3);  // token within the granule
#pragma unroll
            for (int g = 0; g < 4; ++g) {
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const int chunk = (ks & 3) * 2 + ((lane >> 3) & 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(stage + g * kSlot + (ks >> 2) * kBox + row * 128 + ((chunk ^ (row & 7)) << 4),
                            b0, b1, b2, b3);
                    mma16816(sc[2 * g], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
                    mma16816(sc[2 * g + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
                }
            }
        }
        // ---- scale, causal mask, online softmax ----
        const bool full_tile = kt * kKTile + kKTile - 1 <= warp_first;
        float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const int t = kt * kKTile + n * 8 + 2 * tq;
            sc[n][0] = (full_tile || t <= vis_a) ? sc[n][0] * p.scale_log2 : -INFINITY;
            sc[n][1] = (full_tile || t + 1 <= vis_a) ? sc[n][1] * p.scale_log2 : -INFINITY;
            sc[n][2] = (full_tile || t <= vis_b) ? sc[n][2] * p.scale_log2 : -INFINITY;
            sc[n][3] = (full_tile || t + 1 <= vis_b) ? sc[n][3] * p.scale_log2 : -INFINITY;
            mx_a = fmaxf(mx_a, fmaxf(sc[n][0], sc[n][1]));
            mx_b = fmaxf(mx_b, fmaxf(sc[n][2], sc[n][3]));
        }
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
            mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, off));
            mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, off));
        }
        const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
        const float mu_a = mn_a == -INFINITY ? 0.f : mn_a;
        const float mu_b = mn_b == -INFINITY ? 0.f : mn_b;
        const float al_a = fast_exp2(m_a - mu_a), al_b = fast_exp2(m_b - mu_b);
        m_a = mn_a;
        m_b = mn_b;
        uint32_t pa[8][2];  // P as packed fp16: [n-tile][row gq / gq + 8]
        float rs_a = 0.f, rs_b = 0.f;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            pa[n][0] = pack_half2(fast_exp2(sc[n][0] - mu_a), fast_exp2(sc[n][1] - mu_a));
            pa[n][1] = pack_half2(fast_exp2(sc[n][2] - mu_b), fast_exp2(sc[n][3] - mu_b));
            // the sums take the fp16 weights the MMA multiplies by
            const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&pa[n][0]));
            const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&pa[n][1]));
            rs_a += fa.x + fa.y;
            rs_b += fb.x + fb.y;
        }
        l_a = l_a * al_a + rs_a;
        l_b = l_b * al_b + rs_b;
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            o[n][0] *= al_a;
            o[n][1] *= al_a;
            o[n][2] *= al_b;
            o[n][3] *= al_b;
        }
        // ---- O += P V: k-steps of 16 tokens (one granule), n-tiles of 8 dims ----
        {
            const int row = (lane & 7) + ((lane >> 3) & 1) * 8;  // token within the granule
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const uint32_t a0 = pa[2 * g][0], a1 = pa[2 * g][1];
                const uint32_t a2 = pa[2 * g + 1][0], a3 = pa[2 * g + 1][1];
#pragma unroll
                for (int dp = 0; dp < 8; ++dp) {
                    const int chunk = 2 * dp + (lane >> 4);  // 16-byte chunk of the 128 dims
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(stage + g * kSlot + kSlotV + (chunk >> 3) * kBox + row * 128 +
                                  (((chunk & 7) ^ (row & 7)) << 4),
                              b0, b1, b2, b3);
                    mma16816(o[2 * dp], a0, a1, a2, a3, b0, b1);
                    mma16816(o[2 * dp + 1], a0, a1, a2, a3, b2, b3);
                }
            }
        }
        __syncwarp();
        // Generic-proxy writes are ordered before TMA refills the stage.
        if (wrote) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (lane == 0) mbar_arrive(bar_empty + 8 * s);
    }

    // ---- normalise and store this lane's two queries ----
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
        l_a += __shfl_xor_sync(0xffffffffu, l_a, off);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, off);
    }
    const float inv_a = l_a > 0.f ? __fdividef(1.f, l_a) : 0.f;
    const float inv_b = l_b > 0.f ? __fdividef(1.f, l_b) : 0.f;
    const int local_a = warp * 16 + gq, local_b = local_a + 8;
    __half* out_a = p.out + ((int64_t)(qrow0 + local_a) * p.hq + h) * kHeadDim;
    __half* out_b = p.out + ((int64_t)(qrow0 + local_b) * p.hq + h) * kHeadDim;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
        const int d = n * 8 + 2 * tq;
        if (local_a < nq)
            *reinterpret_cast<uint32_t*>(out_a + d) = pack_half2(o[n][0] * inv_a, o[n][1] * inv_a);
        if (local_b < nq)
            *reinterpret_cast<uint32_t*>(out_b + d) = pack_half2(o[n][2] * inv_b, o[n][3] * inv_b);
    }
}

}  // namespace prefill
}  // namespace pkv

extern "C" int paged_attention_prefill(void* out, const void* q, const void* k_pool,
                                       const void* v_pool, const int32_t* block_tables,
                                       const int32_t* seq_lens, const int32_t* q_start, int rows,
                                       int total_q, int q_heads, int kv_heads, int head_dim,
                                       int block_size, float scale, int max_blocks_per_row,
                                       int num_blocks, int max_seq_len, int32_t* dev_err,
                                       cudaStream_t stream) {
    using namespace pkv;
    using namespace pkv::prefill;
    if (rows < 0 || total_q < 0 || q_heads <= 0 || kv_heads <= 0 || q_heads % kv_heads ||
        block_size <= 0 || max_blocks_per_row <= 0 || num_blocks <= 0 || max_seq_len < 0 ||
        !isfinite(scale))
        return PKV_ERR_INVALID_ARG;
    if ((int64_t)max_seq_len > (int64_t)max_blocks_per_row * block_size) return PKV_ERR_INVALID_ARG;
    if (head_dim != kHeadDim || block_size % kGranule || rows > kMaxRows || q_heads > 65535)
        return PKV_ERR_UNSUPPORTED;
    if (rows == 0 || total_q == 0) return PKV_OK;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !seq_lens || !q_start)
        return PKV_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
        return PKV_ERR_INVALID_ARG;
    const int64_t pool_rows = (int64_t)num_blocks * block_size;
    if (pool_rows >= (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;
    const int64_t grid_x = ((int64_t)total_q + kQTile - 1) / kQTile + rows;
    if (grid_x >= (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;

    CUtensorMap qm, km, vm;
    int st;
    {
        const int64_t dims[3] = {kHeadDim, q_heads, total_q};
        const int64_t strides[2] = {kHeadDim * 2, (int64_t)q_heads * kHeadDim * 2};
        const int box[3] = {64, 1, kQTile};
        if ((st = tiled_map_3d(q, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, dims, strides, box, &qm)) != PKV_OK)
            return st;
    }
    {
        const int64_t dims[3] = {kHeadDim, kv_heads, pool_rows};
        const int64_t strides[2] = {kHeadDim * 2, (int64_t)kv_heads * kHeadDim * 2};
        const int box[3] = {64, 1, kGranule};
        if ((st = tiled_map_3d(k_pool, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, dims, strides, box, &km)) != PKV_OK)
            return st;
        if ((st = tiled_map_3d(v_pool, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, dims, strides, box, &vm)) != PKV_OK)
            return st;
    }
    Params prm{};
    prm.out = static_cast<__half*>(out);
    prm.tables = block_tables;
    prm.seq_lens = seq_lens;
    prm.q_start = q_start;
    prm.rows = rows;
    prm.hq = q_heads;
    prm.group = q_heads / kv_heads;
    prm.bs = block_size;
    prm.mbpr = max_blocks_per_row;
    prm.nb = num_blocks;
    prm.limit = max_seq_len;
    prm.scale_log2 = scale * kLog2e;
    prm.dev_err = dev_err;

    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Smem::total(kMaxRows)) != cudaSuccess)
            return PKV_ERR_CUDA;
        attr_set = true;
    }
    prefill_kernel<<<dim3((unsigned)grid_x, (unsigned)q_heads), kThreads, Smem::total(rows), stream>>>(
        qm, km, vm, prm);
    return launch_status();
}
