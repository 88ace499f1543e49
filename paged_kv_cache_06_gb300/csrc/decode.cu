// paged_attention_decode and the padded comparator.
//
// "PagedAttention" (deepconcepts.dev), sections "PagedAttention" and "What
// the block table costs": the kernel walks each sequence's block table and
// gathers the listed blocks; its closing note on FlashAttention: the softmax
// sum split over blocks and recombined through running maxima is exact.
// "Paged attention" (danielfleming.xyz), section "What changed": each row is
// read at its own true length.
//
// Work split: grid (split, row).  A thread block takes one row's tokens
// [split * kSplit, (split + 1) * kSplit) for every KV head and its group of
// query heads; its 8 warps stride over those tokens, each keeping a running
// max / sum / accumulator (online softmax, base-2 exponent).  Warps combine
// in shared memory.  A row covered by one split writes its output directly;
// otherwise each split stores (max, sum, accumulator) to the workspace and
// the last split to arrive (per-row atomic counter) merges them with
// log-sum-exp weights, writes the output and re-arms the counter.
#include <math.h>

#include "pkv_internal.cuh"

namespace pkv {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSplit = 256;  // tokens per thread block
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeParams {
    __half* out;
    const __half* q;
    const __half* k;
    const __half* v;
    const int32_t* tables;
    const int32_t* seq_lens;
    int rows, hq, hk, group, bs, mbpr, nb;
    int limit;       // largest valid seq_len
    int width;       // padded comparator: columns per row
    int nsplit_max;
    float scale_log2;
    int* counters;   // [rows]
    float* ws_m;     // [rows][nsplit_max][hq]
    float* ws_l;     // [rows][nsplit_max][hq]
    float* ws_acc;   // [rows][nsplit_max][hq][128]
    int32_t* dev_err;
};

struct WorkspaceLayout {
    size_t counters, m, l, acc, total;
};

inline WorkspaceLayout workspace_layout(int rows, int hq, int nsplit_max) {
    WorkspaceLayout w;
    const size_t parts = (size_t)rows * nsplit_max * hq;
    w.counters = 0;
    w.m = align_up(sizeof(int) * (size_t)rows, 256);
    w.l = w.m + align_up(sizeof(float) * parts, 256);
    w.acc = w.l + align_up(sizeof(float) * parts, 256);
    w.total = w.acc + align_up(sizeof(float) * parts * kHeadDim, 256);
    return w;
}

inline int splits_for(int max_seq_len) { return max_seq_len <= 0 ? 1 : (max_seq_len + kSplit - 1) / kSplit; }

template <bool kPaged>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(const DecodeParams p) {
    __shared__ float sm_m[kWarps][kMaxGroup];
    __shared__ float sm_l[kWarps][kMaxGroup];
    __shared__ float sm_acc[kWarps][kMaxGroup][kHeadDim];
    __shared__ int sm_last;

    const int s = blockIdx.x;
    const int r = blockIdx.y;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    int L = p.seq_lens[r];
    if (L < 0 || L > p.limit) {
        if (s == 0 && tid == 0) flag_error(p.dev_err, PKV_DEV_ERR_SEQ_LEN);
        L = L < 0 ? 0 : p.limit;
    }
    const int span = kPaged ? L : p.width;  // columns this row reads
    const int nsplit = span <= 0 ? 1 : (span + kSplit - 1) / kSplit;
    if (s >= nsplit) return;
    const int t0 = s * kSplit;
    const int t1 = min(span, t0 + kSplit);
    const bool direct = nsplit == 1;

    for (int kvh = 0; kvh < p.hk; ++kvh) {
        float qf[kMaxGroup][4], acc[kMaxGroup][4], m[kMaxGroup], l[kMaxGroup];
#pragma unroll
        for (int g = 0; g < kMaxGroup; ++g) {
            m[g] = -INFINITY;
            l[g] = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[g][j] = 0.f, qf[g][j] = 0.f;
            if (g < p.group) {
                const __half* qp = p.q + ((int64_t)r * p.hq + kvh * p.group + g) * kHeadDim + 4 * lane;
                const uint2 raw = *reinterpret_cast<const uint2*>(qp);
                const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
                const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
                qf[g][0] = a.x * p.scale_log2;
                qf[g][1] = a.y * p.scale_log2;
                qf[g][2] = b.x * p.scale_log2;
                qf[g][3] = b.y * p.scale_log2;
            }
        }
        for (int t = t0 + warp; t < t1; t += kWarps) {
            int64_t off;
            if (kPaged) {
                const int pb = p.tables[(int64_t)r * p.mbpr + t / p.bs];
                if (pb < 0 || pb >= p.nb) {
                    if (lane == 0) flag_error(p.dev_err, PKV_DEV_ERR_BLOCK_ID);
                    continue;
                }
                off = (((int64_t)pb * p.bs + t % p.bs) * p.hk + kvh) * kHeadDim + 4 * lane;
            } else {
                off = (((int64_t)r * p.width + t) * p.hk + kvh) * kHeadDim + 4 * lane;
            }
            const bool valid = t < L;
            const uint2 kr = __ldg(reinterpret_cast<const uint2*>(p.k + off));
            const uint2 vr = __ldg(reinterpret_cast<const uint2*>(p.v + off));
            const float2 k01 = __half22float2(*reinterpret_cast<const __half2*>(&kr.x));
            const float2 k23 = __half22float2(*reinterpret_cast<const __half2*>(&kr.y));
            const float2 v01 = __half22float2(*reinterpret_cast<const __half2*>(&vr.x));
            const float2 v23 = __half22float2(*reinterpret_cast<const __half2*>(&vr.y));
#pragma unroll
            for (int g = 0; g < kMaxGroup; ++g) {
                if (g < p.group) {
                    float part = qf[g][0] * k01.x + qf[g][1] * k01.y + qf[g][2] * k23.x + qf[g][3] * k23.y;
                    const float sc = warp_sum(part);
                    if (valid) {
                        const float mn = fmaxf(m[g], sc);
                        const float alpha = exp2f(m[g] - mn);
                        const float pr = exp2f(sc - mn);
                        l[g] = l[g] * alpha + pr;
                        acc[g][0] = acc[g][0] * alpha + pr * v01.x;
                        acc[g][1] = acc[g][1] * alpha + pr * v01.y;
                        acc[g][2] = acc[g][2] * alpha + pr * v23.x;
                        acc[g][3] = acc[g][3] * alpha + pr * v23.y;
                        m[g] = mn;
                    }
                }
            }
        }
        // Combine the warps of this block.
#pragma unroll
        for (int g = 0; g < kMaxGroup; ++g) {
            if (lane == 0) {
                sm_m[warp][g] = m[g];
                sm_l[warp][g] = l[g];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) sm_acc[warp][g][4 * lane + j] = acc[g][j];
        }
        __syncthreads();
        for (int idx = tid; idx < p.group * kHeadDim; idx += kThreads) {
            const int g = idx / kHeadDim;
            const int d = idx % kHeadDim;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][g]);
            float lt = 0.f, at = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    const float sc = exp2f(sm_m[w][g] - M);
                    lt += sc * sm_l[w][g];
                    at += sc * sm_acc[w][g][d];
                }
            }
            const int h = kvh * p.group + g;
            if (direct) {
                p.out[((int64_t)r * p.hq + h) * kHeadDim + d] = __float2half_rn(lt > 0.f ? at / lt : 0.f);
            } else {
                const int64_t base = ((int64_t)r * p.nsplit_max + s) * p.hq + h;
                p.ws_acc[base * kHeadDim + d] = at;
                if (d == 0) {
                    p.ws_m[base] = M;
                    p.ws_l[base] = lt;
                }
            }
        }
        __syncthreads();
    }
    if (direct) return;

    // Last split of this row to arrive merges all splits.
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int prev = atomicAdd(&p.counters[r], 1);
        sm_last = prev == nsplit - 1;
        if (sm_last) p.counters[r] = 0;  // every split of this row has arrived
    }
    __syncthreads();
    if (!sm_last) return;
    __threadfence();
    for (int idx = tid; idx < p.hq * kHeadDim; idx += kThreads) {
        const int h = idx / kHeadDim;
        const int d = idx % kHeadDim;
        const int64_t row0 = (int64_t)r * p.nsplit_max;
        float M = -INFINITY;
        for (int s2 = 0; s2 < nsplit; ++s2) M = fmaxf(M, __ldcg(p.ws_m + (row0 + s2) * p.hq + h));
        float lt = 0.f, at = 0.f;
        if (M != -INFINITY) {
            for (int s2 = 0; s2 < nsplit; ++s2) {
                const int64_t base = (row0 + s2) * p.hq + h;
                const float sc = exp2f(__ldcg(p.ws_m + base) - M);
                lt += sc * __ldcg(p.ws_l + base);
                at += sc * __ldcg(p.ws_acc + base * kHeadDim + d);
            }
        }
        p.out[((int64_t)r * p.hq + h) * kHeadDim + d] = __float2half_rn(lt > 0.f ? at / lt : 0.f);
    }
}

static int check_heads(int q_heads, int kv_heads, int head_dim) {
    if (q_heads <= 0 || kv_heads <= 0 || head_dim <= 0) return PKV_ERR_INVALID_ARG;
    if (q_heads % kv_heads) return PKV_ERR_INVALID_ARG;
    if (head_dim != kHeadDim || q_heads / kv_heads > kMaxGroup) return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

static DecodeParams make_params(void* out, const void* q, const void* k, const void* v,
                                const int32_t* tables, const int32_t* seq_lens, int rows,
                                int q_heads, int kv_heads, int block_size, int mbpr, int nb,
                                int limit, int width, float scale, int nsplit_max, void* workspace,
                                int32_t* dev_err) {
    DecodeParams p{};
    p.out = static_cast<__half*>(out);
    p.q = static_cast<const __half*>(q);
    p.k = static_cast<const __half*>(k);
    p.v = static_cast<const __half*>(v);
    p.tables = tables;
    p.seq_lens = seq_lens;
    p.rows = rows;
    p.hq = q_heads;
    p.hk = kv_heads;
    p.group = q_heads / kv_heads;
    p.bs = block_size;
    p.mbpr = mbpr;
    p.nb = nb;
    p.limit = limit;
    p.width = width;
    p.nsplit_max = nsplit_max;
    p.scale_log2 = scale * kLog2e;
    const WorkspaceLayout w = workspace_layout(rows, q_heads, nsplit_max);
    char* base = static_cast<char*>(workspace);
    p.counters = reinterpret_cast<int*>(base + w.counters);
    p.ws_m = reinterpret_cast<float*>(base + w.m);
    p.ws_l = reinterpret_cast<float*>(base + w.l);
    p.ws_acc = reinterpret_cast<float*>(base + w.acc);
    p.dev_err = dev_err;
    return p;
}

}  // namespace pkv

namespace pkv {
// Leading bytes of a decode workspace that must be zero when a call starts
// (the arrival counters); everything after them is written before it is read.
size_t decode_workspace_zero_bytes(int rows, int q_heads, int kv_heads, int head_dim,
                                   int max_seq_len, int block_size) {
    if (rows <= 0) return 0;
    if (tma_decode_supported(rows, q_heads, kv_heads, head_dim, block_size))
        return tma_workspace_zero_bytes(rows, kv_heads, max_seq_len);
    return workspace_layout(rows, 1, 1).m;
}
}  // namespace pkv

extern "C" size_t paged_attention_workspace_size(int rows, int q_heads, int kv_heads, int head_dim,
                                                 int max_seq_len, int block_size) {
    if (rows < 0 || pkv::check_heads(q_heads, kv_heads, head_dim) != PKV_OK || max_seq_len < 0 ||
        block_size <= 0)
        return 0;
    if (pkv::tma_decode_supported(rows, q_heads, kv_heads, head_dim, block_size))
        return pkv::tma_workspace_bytes(rows, q_heads, kv_heads, max_seq_len);
    return pkv::workspace_layout(rows, q_heads, pkv::splits_for(max_seq_len)).total;
}

extern "C" int paged_attention_decode(void* out, const void* q, const void* k_pool,
                                      const void* v_pool, const int32_t* block_tables,
                                      const int32_t* seq_lens, int rows, int q_heads, int kv_heads,
                                      int head_dim, int block_size, float scale,
                                      int max_blocks_per_row, int num_blocks, int max_seq_len,
                                      void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                      cudaStream_t stream) {
    using namespace pkv;
    const int hs = check_heads(q_heads, kv_heads, head_dim);
    if (hs != PKV_OK) return hs;
    if (rows < 0 || block_size <= 0 || block_size > 1024 || max_blocks_per_row <= 0 ||
        num_blocks <= 0 || max_seq_len < 0 || !isfinite(scale))
        return PKV_ERR_INVALID_ARG;
    if ((int64_t)max_seq_len > (int64_t)max_blocks_per_row * block_size) return PKV_ERR_INVALID_ARG;
    if (rows > 65535) return PKV_ERR_UNSUPPORTED;
    if (rows == 0) return PKV_OK;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !seq_lens) return PKV_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
        return PKV_ERR_INVALID_ARG;
    if (tma_decode_supported(rows, q_heads, kv_heads, head_dim, block_size)) {
        if (!workspace || workspace_bytes < tma_workspace_bytes(rows, q_heads, kv_heads, max_seq_len))
            return PKV_ERR_WORKSPACE;
        const int st = tma_decode_launch(out, q, k_pool, v_pool, block_tables, seq_lens, rows,
                                         q_heads, kv_heads, block_size, scale, max_blocks_per_row,
                                         num_blocks, max_seq_len, 0, workspace, dev_err, stream);
        if (st != PKV_ERR_UNSUPPORTED) return st;
    }
    const int nsplit = splits_for(max_seq_len);
    if (!workspace || workspace_bytes < workspace_layout(rows, q_heads, nsplit).total)
        return PKV_ERR_WORKSPACE;
    const DecodeParams p = make_params(out, q, k_pool, v_pool, block_tables, seq_lens, rows,
                                       q_heads, kv_heads, block_size, max_blocks_per_row,
                                       num_blocks, max_seq_len, 0, scale, nsplit, workspace,
                                       dev_err);
    decode_split_kernel<true><<<dim3(nsplit, rows), kThreads, 0, stream>>>(p);
    return launch_status();
}

extern "C" int paged_attention_padded_decode(void* out, const void* q, const void* k_slab,
                                             const void* v_slab, const int32_t* seq_lens, int rows,
                                             int width, int q_heads, int kv_heads, int head_dim,
                                             float scale, void* workspace, size_t workspace_bytes,
                                             int32_t* dev_err, cudaStream_t stream) {
    using namespace pkv;
    const int hs = check_heads(q_heads, kv_heads, head_dim);
    if (hs != PKV_OK) return hs;
    if (rows < 0 || width < 0 || !isfinite(scale)) return PKV_ERR_INVALID_ARG;
    if (rows > 65535) return PKV_ERR_UNSUPPORTED;
    if (rows == 0) return PKV_OK;
    if (!out || !q || !seq_lens || (width > 0 && (!k_slab || !v_slab))) return PKV_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_slab) || !aligned16(v_slab))
        return PKV_ERR_INVALID_ARG;
    // The staged kernel when the workspace is sized for it (block size 16),
    // else the split kernel.
    if (width > 0 && tma_decode_supported(rows, q_heads, kv_heads, head_dim, 16) && workspace &&
        workspace_bytes >= tma_workspace_bytes(rows, q_heads, kv_heads, width)) {
        return tma_decode_launch(out, q, k_slab, v_slab, nullptr, seq_lens, rows, q_heads,
                                 kv_heads, 16, scale, 1, 1, width, width, workspace, dev_err,
                                 stream);
    }
    const int nsplit = splits_for(width);
    if (!workspace || workspace_bytes < workspace_layout(rows, q_heads, nsplit).total)
        return PKV_ERR_WORKSPACE;
    const DecodeParams p = make_params(out, q, k_slab, v_slab, nullptr, seq_lens, rows, q_heads,
                                       kv_heads, 1, 1, 1, width, width, scale, nsplit, workspace,
                                       dev_err);
    decode_split_kernel<false><<<dim3(nsplit, rows), kThreads, 0, stream>>>(p);
    return launch_status();
}

extern "C" int paged_attention_append_decode(
    void* out, const void* q, void* k_pool, void* v_pool, const int32_t* block_tables,
    const int32_t* seq_lens, const int32_t* positions, const void* k_new, const void* v_new, int rows,
    int q_heads, int kv_heads, int head_dim, int block_size, float scale, int max_blocks_per_row,
    int num_blocks, int max_seq_len, void* workspace, size_t workspace_bytes, unsigned flags,
    int32_t* dev_err, cudaStream_t stream) {
    using namespace pkv;
    const int hs = check_heads(q_heads, kv_heads, head_dim);
    if (hs != PKV_OK) return hs;
    if (rows < 0 || block_size <= 0 || block_size > 1024 || max_blocks_per_row <= 0 ||
        num_blocks <= 0 || max_seq_len < 0 || !isfinite(scale) || (flags & ~PKV_FLAG_PDL))
        return PKV_ERR_INVALID_ARG;
    if ((int64_t)max_seq_len > (int64_t)max_blocks_per_row * block_size) return PKV_ERR_INVALID_ARG;
    if (rows == 0) return PKV_OK;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !seq_lens || !positions || !k_new ||
        !v_new)
        return PKV_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) ||
        !aligned16(k_new) || !aligned16(v_new))
        return PKV_ERR_INVALID_ARG;
    if (tma_decode_supported(rows, q_heads, kv_heads, head_dim, block_size)) {
        if (!workspace || workspace_bytes < tma_workspace_bytes(rows, q_heads, kv_heads, max_seq_len))
            return PKV_ERR_WORKSPACE;
        const AppendArgs app{positions, k_new, v_new};
        const int st = tma_decode_launch(out, q, k_pool, v_pool, block_tables, seq_lens, rows,
                                         q_heads, kv_heads, block_size, scale, max_blocks_per_row,
                                         num_blocks, max_seq_len, 0, workspace, dev_err, stream,
                                         &app, (flags & PKV_FLAG_PDL) != 0);
        if (st != PKV_ERR_UNSUPPORTED) return st;
    }
    // Shapes the staged kernel does not take: the two calls in sequence.
    const int st = paged_kv_append(k_pool, v_pool, block_tables, positions, k_new, v_new, rows,
                                   kv_heads, head_dim, block_size, max_blocks_per_row, num_blocks,
                                   dev_err, stream);
    if (st != PKV_OK) return st;
    return paged_attention_decode(out, q, k_pool, v_pool, block_tables, seq_lens, rows, q_heads,
                                  kv_heads, head_dim, block_size, scale, max_blocks_per_row,
                                  num_blocks, max_seq_len, workspace, workspace_bytes, dev_err,
                                  stream);
}

extern "C" size_t paged_attention_plan_size(int rows, int q_heads, int kv_heads, int head_dim,
                                            int max_seq_len, int block_size) {
    using namespace pkv;
    if (check_heads(q_heads, kv_heads, head_dim) != PKV_OK || rows <= 0 || max_seq_len < 0 ||
        block_size <= 0 || !tma_decode_supported(rows, q_heads, kv_heads, head_dim, block_size))
        return 0;
    return tma_plan_bytes(rows, kv_heads, max_seq_len);
}

extern "C" int paged_attention_plan(void* plan, size_t plan_bytes, const int32_t* block_tables,
                                    const int32_t* seq_lens, const int32_t* positions, int rows,
                                    int q_heads, int kv_heads, int head_dim, int block_size,
                                    int max_blocks_per_row, int num_blocks, int max_seq_len,
                                    int32_t* dev_err, cudaStream_t stream) {
    using namespace pkv;
    const int hs = check_heads(q_heads, kv_heads, head_dim);
    if (hs != PKV_OK) return hs;
    if (rows < 0 || block_size <= 0 || block_size > 1024 || max_blocks_per_row <= 0 ||
        num_blocks <= 0 || max_seq_len < 0)
        return PKV_ERR_INVALID_ARG;
    if ((int64_t)max_seq_len > (int64_t)max_blocks_per_row * block_size) return PKV_ERR_INVALID_ARG;
    if (!tma_decode_supported(rows, q_heads, kv_heads, head_dim, block_size))
        return PKV_ERR_UNSUPPORTED;
    if (rows == 0) return PKV_OK;
    if (!plan || !block_tables || !seq_lens) return PKV_ERR_INVALID_ARG;
    if (!aligned16(plan)) return PKV_ERR_INVALID_ARG;
    if (plan_bytes < tma_plan_bytes(rows, kv_heads, max_seq_len)) return PKV_ERR_WORKSPACE;
    return tma_plan_launch(plan, plan_bytes, block_tables, seq_lens, positions, rows, q_heads,
                           kv_heads, block_size, max_blocks_per_row, num_blocks, max_seq_len,
                           dev_err, stream);
}

extern "C" int paged_attention_decode_planned(
    void* out, const void* q, void* k_pool, void* v_pool, const float* k_scale,
    const float* v_scale, const int32_t* block_tables, const int32_t* seq_lens,
    const int32_t* positions, const void* k_new, const void* v_new, int rows, int q_heads,
    int kv_heads, int head_dim, int block_size, float scale, int max_blocks_per_row,
    int num_blocks, int max_seq_len, const void* plan, size_t plan_bytes, void* workspace,
    size_t workspace_bytes, unsigned flags, int32_t* dev_err, cudaStream_t stream) {
    using namespace pkv;
    const int hs = check_heads(q_heads, kv_heads, head_dim);
    if (hs != PKV_OK) return hs;
    if (rows < 0 || block_size <= 0 || block_size > 1024 || max_blocks_per_row <= 0 ||
        num_blocks <= 0 || max_seq_len < 0 || !isfinite(scale) || (flags & ~PKV_FLAG_PDL))
        return PKV_ERR_INVALID_ARG;
    if ((int64_t)max_seq_len > (int64_t)max_blocks_per_row * block_size) return PKV_ERR_INVALID_ARG;
    const bool fp8 = k_scale != nullptr || v_scale != nullptr;
    if (fp8 && (!k_scale || !v_scale)) return PKV_ERR_INVALID_ARG;
    if (!tma_decode_supported(rows, q_heads, kv_heads, head_dim, block_size) ||
        (fp8 && kv_heads > 16))
        return PKV_ERR_UNSUPPORTED;
    if (rows == 0) return PKV_OK;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !seq_lens || !plan)
        return PKV_ERR_INVALID_ARG;
    if (positions && (!k_new || !v_new)) return PKV_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) ||
        !aligned16(plan) || (positions && (!aligned16(k_new) || !aligned16(v_new))))
        return PKV_ERR_INVALID_ARG;
    if (plan_bytes < tma_plan_bytes(rows, kv_heads, max_seq_len)) return PKV_ERR_WORKSPACE;
    if (!workspace || workspace_bytes < tma_workspace_bytes(rows, q_heads, kv_heads, max_seq_len))
        return PKV_ERR_WORKSPACE;
    const AppendArgs app{positions, k_new, v_new};
    return tma_decode_launch(out, q, k_pool, v_pool, block_tables, seq_lens, rows, q_heads,
                             kv_heads, block_size, scale, max_blocks_per_row, num_blocks,
                             max_seq_len, 0, workspace, dev_err, stream, positions ? &app : nullptr,
                             (flags & PKV_FLAG_PDL) != 0, k_scale, v_scale, plan);
}
