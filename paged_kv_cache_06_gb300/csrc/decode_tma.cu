// Paged decode attention for sm_103a: TMA-staged, tensor-core, stream-K.
//
// "PagedAttention" (deepconcepts.dev), sections "PagedAttention" and "What
// the block table costs": the kernel walks each sequence's block table and
// gathers the listed blocks; closing note on FlashAttention: the softmax sum
// split over blocks and recombined through running maxima and log-sum-exp is
// exact.  "Paged attention" (danielfleming.xyz), section "What changed": each
// row is read only at its own length.  "SLM paged attention", section "The
// architecture": blocks are moved in coalesced chunks.
//
// Work split.  A unit is one (row, KV head); its tokens are cut into 16-token
// granules.  All granules of all units, in (row, head, token) order, are cut
// into gridDim.x equal contiguous ranges, one per thread block (one block per
// SM), so every SM moves the same number of bytes whatever the length mix.
// Each block derives the partition itself from seq_lens (a block-wide scan),
// so the host never reads device lengths.  The part of a unit inside one
// block is a piece; a unit with several pieces is merged by a fan-in-8 tree
// of last-arriving blocks (per-node atomic counters, re-armed by the merger).
//
// Block layout.  Warp 4 is the producer: it resolves each granule's physical
// block from the table and issues TMA tiled copies (a 16-token x 64-dim box,
// 128-byte swizzle, never crossing a physical block) into a 3-stage mbarrier
// pipeline; the first tile of a piece also brings the unit's query heads by
// a bulk copy.  Warps 0-3 consume one granule each per stage:
//   S^T[16 tok][8 heads] = K[16 tok][128] . Q^T        (mma.sync m16n8k16)
//   online softmax per head in fp32, base-2 exponent
//   O^T[128][8 heads]   += V^T[128][16 tok] . P^T      (P transposed in
//                                                       registers by movmatrix)
// The grouped query heads (up to 8) are the MMA's N = 8 columns, so every K
// and V byte is read once and feeds all heads of its group.
//
// Safety: table entries are range-checked before any copy is issued (a bad
// entry is skipped and flagged); every mbarrier wait is bounded and a timeout
// sets PKV_DEV_ERR_TIMEOUT, stops the block and drains its copies in flight.
#include <cuda.h>

#include <mutex>
#include <unordered_map>

#include "pkv_internal.cuh"

namespace pkv {
namespace tma {

constexpr int kGranule = 16;        // tokens per box and per consumer warp step
constexpr int kTileGranules = 4;    // granules per pipeline stage (64 tokens)
constexpr int kStages = 3;
constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kMaxCtas = 1024;
constexpr int kMaxRows = 1024;
constexpr int kRecHead = 16;   // per record: m[8], l[8], then o[group][128]
constexpr int kMaxPieces = 32; // append positions prefetched for a block's first pieces
constexpr int kMergeBatch = 8; // children merged per register batch
constexpr uint32_t kBoxBytes = kGranule * 128;                // 16 rows x 128 B
constexpr uint32_t kHalfBytes = kTileGranules * kBoxBytes;    // one 64-dim half of 64 tokens
constexpr uint32_t kStageK = 0;
constexpr uint32_t kStageV = 2 * kHalfBytes;
constexpr uint32_t kStageQ = 4 * kHalfBytes;
constexpr uint32_t kStageBytes = 4 * kHalfBytes + 8 * 256;    // K, V, Q (8 heads x 256 B)
constexpr int kCombStride = 68;                               // 64 dims + 4 pad (floats)
constexpr uint32_t kSpinLimit = 1u << 22;
constexpr float kLog2e = 1.4426950408889634f;

static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment for 128B swizzle");
static_assert(2 * kStages * 8 + 8 <= 64, "barrier area");

struct Params {
    __half* out;
    const __half* q;
    const int32_t* tables;
    const int32_t* seq_lens;
    int rows, hq, hk, group, bs, mbpr, nb;
    int limit;      // largest valid seq_len (paged); width (padded)
    int width;      // padded comparator: columns per row (0 = paged)
    float scale_log2;
    int rec_floats; // floats per record: 16 + group * 128
    int* counters;  // [units]: pieces arrived per split unit (zero between calls)
    float* records; // [slots][rec_floats]: partial results of split units
    int32_t* dev_err;
    // fused append (all null when the kernel only decodes)
    const int32_t* positions;
    const __half* k_new;
    const __half* v_new;
    __half* kpool;
    __half* vpool;
};

// Shared memory carve-up (offsets from a 1024-aligned base).
struct Smem {
    static constexpr uint32_t stages = 0;
    static constexpr uint32_t comb = kStages * kStageBytes;                         // [4][8][68] f32
    static constexpr uint32_t ml = comb + kConsumerWarps * 8 * kCombStride * 4;     // [4][8] m, [4][8] l
    static constexpr uint32_t bars = ml + 2 * kConsumerWarps * 8 * 4;               // full[S], empty[S], merge
    static constexpr uint32_t desc = bars + 64;                                     // TileDesc[S]
    static constexpr uint32_t flags = desc + kStages * 64;                          // misc ints
    static constexpr uint32_t ppos = flags + 16 * 4;                                // piece positions [32]
    static constexpr uint32_t part = comb;  // scan partials: prologue only, aliases comb
    static constexpr uint32_t prefix = ppos + kMaxPieces * 4;                       // rows + 1 ints
    __host__ __device__ static uint32_t lens(int rows) { return prefix + (uint32_t)(rows + 1) * 4; }
    __host__ __device__ static uint32_t total(int rows) { return lens(rows) + (uint32_t)rows * 4 + 1024; }
};

// ---------------------------------------------------------------------------
// PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait by a whole warp: every lane polls and a vote decides, so the
// warp leaves together (true) or gives up together after kSpinLimit polls.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (uint32_t i = 0; i < kSpinLimit; ++i)
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    return false;
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& a0, uint32_t& a1, uint32_t& a2,
                                        uint32_t& a3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& a0, uint32_t& a1, uint32_t& a2,
                                          uint32_t& a3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}
// 2^x by the hardware approximation (relative error about 2^-22; 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Per-stage tile descriptor: written by the producer before the stage's
// full barrier is armed, read by the consumers after it completes.
struct TileDesc {
    int ustart;                 // unit's first granule (global index)
    int pend;                   // end of this block's piece of the unit (global, exclusive)
    int flags;                  // kFirst | kLast | kEnd
    int r, kvh, ng;             // unit (row, KV head), granules in this tile
    int tok0;                   // unit-local token index of the tile's first granule
    int n;                      // unit's granule count
    int valid[kTileGranules];   // valid tokens per granule (0 = skipped block)
    int pad[4];
};
static_assert(sizeof(TileDesc) == 64, "descriptor size");
constexpr int kFirst = 1, kLast = 2, kEnd = 4, kBlockLast = 8;

__device__ __forceinline__ int granules_of(int L) { return (L + kGranule - 1) / kGranule; }

// Index c of the block whose range holds granule g (partition b_c = c*W/G).
__device__ __forceinline__ int owner_of(int g, int W, int G) {
    // largest c with floor(c*W/G) <= g  <=>  c*W <= (g+1)*G - 1, i.e.
    // c = floor(x / W) with x = (g+1)*G - 1.  A float quotient is within one
    // of it (x / W <= G <= 1024); exact integer checks fix the last unit.
    const int64_t x = (int64_t)(g + 1) * G - 1;
    int c = (int)__fdividef((float)x, (float)W);
    if ((int64_t)(c + 1) * W <= x) ++c;
    if ((int64_t)c * W > x) --c;
    return c;
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Log-sum-exp merge of P partial records (children j = 0..P-1, rec_floats
// apart) for head mh, dims md..md+7: M = max_j m_j, then
// L = sum_j 2^(m_j - M) l_j and o = sum_j 2^(m_j - M) o_j, summed in child order
// into two accumulator sets (even / odd j) added at the end.  The arithmetic
// is the same whether the records are read from shared or global memory, so
// the result never depends on which block merges.
__device__ __forceinline__ void merge_children(const float* base, int P, int rec_floats, int mh,
                                               int md, bool global, float& Ls_out, float* acc) {
    auto ld1 = [&](const float* a) { return global ? __ldcg(a) : *a; };
    auto ld4 = [&](const float* a) {
        return global ? __ldcg(reinterpret_cast<const float4*>(a)) : *reinterpret_cast<const float4*>(a);
    };
    float M = -INFINITY;
    for (int j = 0; j < P; ++j) M = fmaxf(M, ld1(base + (int64_t)j * rec_floats + mh));
    float acc2[8], Ls = 0.f, Ls2 = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = acc2[i] = 0.f;
    if (M != -INFINITY) {
        for (int j0 = 0; j0 < P; j0 += kMergeBatch) {
            float w[kMergeBatch], l[kMergeBatch];
            float4 x[kMergeBatch], y[kMergeBatch];
#pragma unroll
            for (int c = 0; c < kMergeBatch; ++c) {  // a batch's loads are in flight together
                if (j0 + c < P) {
                    const float* cr = base + (int64_t)(j0 + c) * rec_floats;
                    w[c] = ld1(cr + mh);
                    l[c] = ld1(cr + 8 + mh);
                    x[c] = ld4(cr + kRecHead + mh * kHeadDim + md);
                    y[c] = ld4(cr + kRecHead + mh * kHeadDim + md + 4);
                } else {
                    w[c] = -INFINITY;
                    l[c] = 0.f;
                    x[c] = y[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int c = 0; c < kMergeBatch; ++c) {
                const float wt = fast_exp2(w[c] - M);
                float* a = (c & 1) ? acc2 : acc;
                float& L = (c & 1) ? Ls2 : Ls;
                L += wt * l[c];
                a[0] += wt * x[c].x; a[1] += wt * x[c].y; a[2] += wt * x[c].z; a[3] += wt * x[c].w;
                a[4] += wt * y[c].x; a[5] += wt * y[c].y; a[6] += wt * y[c].z; a[7] += wt * y[c].w;
            }
        }
    }
    Ls_out = Ls + Ls2;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += acc2[i];
}

template <bool kPaged>
__global__ void __launch_bounds__(kThreads, 2)
    decode_tma_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const Params p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    float* sm_comb = reinterpret_cast<float*>(smem + Smem::comb);
    float* sm_m = reinterpret_cast<float*>(smem + Smem::ml);
    float* sm_l = sm_m + kConsumerWarps * 8;
    const uint32_t bar_full = sbase + Smem::bars;
    const uint32_t bar_empty = bar_full + kStages * 8;
    const uint32_t bar_merge = bar_full + 2 * kStages * 8;
    int* sm_ppos = reinterpret_cast<int*>(smem + Smem::ppos);
    TileDesc* sm_desc = reinterpret_cast<TileDesc*>(smem + Smem::desc);
    volatile int* sm_flags = reinterpret_cast<volatile int*>(smem + Smem::flags);
    int* sm_part = reinterpret_cast<int*>(smem + Smem::part);
    int* sm_pre = reinterpret_cast<int*>(smem + Smem::prefix);
    int* sm_len = reinterpret_cast<int*>(smem + Smem::lens(p.rows));

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int G = gridDim.x;  // blocks launched; the partition uses Geff <= G
    const int cta = blockIdx.x;
    const int hk = p.hk;
    const int rows = p.rows;

    // The next kernel in the stream (launched with programmatic serialization)
    // may start its own prologue now; it waits for this grid before touching
    // anything this grid writes.
    if (tid == 0) griddep_launch();

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kConsumerWarps);
        }
        mbar_init(bar_merge, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        sm_flags[0] = 0;  // abort
        sm_flags[3] = 0;  // split pieces recorded ([4..13]: their unit, first block, pieces, row, head)
    }

    // ---- granule prefix over rows: sm_pre[r] = first granule of row r ----
    const int per = (rows + kThreads - 1) / kThreads;
    bool bad_len = false;
    int sum = 0;
    for (int i = 0; i < per; ++i) {
        const int r = tid * per + i;
        if (r < rows) {
            int L = p.seq_lens[r];
            if (L < 0 || L > p.limit) {
                if (kPaged) bad_len = true;
                L = L < 0 ? 0 : p.limit;
            }
            sm_len[r] = L;  // tokens that count (clamped)
            const int c = hk * granules_of(kPaged ? L : p.width);
            sm_pre[r] = c;
            sum += c;
        }
    }
    sm_part[tid] = sum;
    if (bad_len && cta == 0) flag_error(p.dev_err, PKV_DEV_ERR_SEQ_LEN);
    __syncthreads();
    if (warp == 0) {
        constexpr int kPer = (kThreads + 31) / 32;
        int v[kPer];
        int acc = 0;
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

    // Partition over Geff = min(grid, W) blocks so every participating block
    // owns at least one granule (a merge counts on one piece per block).
    const int W = sm_pre[rows];
    const int Geff = W < G ? W : G;
    const int g0 = cta < Geff ? (int)((int64_t)W * cta / Geff) : 0;
    const int g1 = cta < Geff ? (int)((int64_t)W * (cta + 1) / Geff) : 0;

    if (warp == kConsumerWarps) {
        // ============================ producer ============================
        if (g0 >= g1) return;
        int tile = 0;
        bool waited = false;
        bool aborted = false;
        // Query copies of tiles armed before the dependency wait (lane 0).
        uint32_t pq_dst[kStages], pq_bar[kStages];
        const __half* pq_src[kStages];
        int npq = 0;
        const uint32_t qbytes = (uint32_t)p.group * 256u;
        auto wait_and_flush = [&]() {
            if (waited) return;
            griddep_wait();
            waited = true;
            if (lane == 0)
                for (int i = 0; i < npq; ++i) bulk_load(pq_dst[i], pq_src[i], qbytes, pq_bar[i]);
            npq = 0;
        };
        for (int bg = g0; bg < g1 && !aborted; bg += 32) {
            const int nbat = min(32, g1 - bg);
            // Lane j resolves granule bg + j: unit, valid tokens, physical row.
            int u = -1, r = 0, kvh = 0, n = 1, ustart = 0, tok = 0, valid = 0, zrow = 0;
            bool issue = false;
            if (lane < nbat) {
                const int gg = bg + lane;
                int lo = 0, hi = rows - 1;
                while (lo < hi) {  // largest row with sm_pre[row] <= gg
                    const int mid = (lo + hi + 1) >> 1;
                    if (sm_pre[mid] <= gg) lo = mid; else hi = mid - 1;
                }
                r = lo;
                n = (sm_pre[r + 1] - sm_pre[r]) / hk;
                kvh = (gg - sm_pre[r]) / n;
                ustart = sm_pre[r] + kvh * n;
                u = r * hk + kvh;
                tok = (gg - ustart) * kGranule;
                valid = min(kGranule, sm_len[r] - tok);
                if (valid < 0) valid = 0;
                if (kPaged) {
                    const int pb = p.tables[(int64_t)r * p.mbpr + tok / p.bs];
                    if (pb < 0 || pb >= p.nb) {
                        flag_error(p.dev_err, PKV_DEV_ERR_BLOCK_ID);
                        valid = 0;
                    } else {
                        zrow = pb * p.bs + tok % p.bs;
                        issue = true;
                    }
                } else {
                    zrow = r * p.width + tok;
                    issue = true;
                }
            }
            int j = 0;
            while (j < nbat) {
                // A tile: up to 4 consecutive granules of one unit.
                const int uj = __shfl_sync(0xffffffffu, u, j);
                const unsigned same = __ballot_sync(0xffffffffu, lane < nbat && u == uj) >> j;
                const unsigned gap = ~same;
                int ng = gap == 0 ? 32 : __ffs(gap) - 1;
                ng = min(min(ng, kTileGranules), nbat - j);
                const int r_j = __shfl_sync(0xffffffffu, r, j);
                const int kvh_j = __shfl_sync(0xffffffffu, kvh, j);
                const int n_j = __shfl_sync(0xffffffffu, n, j);
                const int us_j = __shfl_sync(0xffffffffu, ustart, j);
                const int tok_j = __shfl_sync(0xffffffffu, tok, j);
                const int gstart = bg + j;
                const int pend = min(g1, us_j + n_j);
                const int pstart = max(g0, us_j);
                const bool first = gstart == pstart;
                const bool last = gstart + ng == pend;
                if (!waited && tile >= kStages) wait_and_flush();
                const int s = tile % kStages;
                const uint32_t round = (uint32_t)tile / kStages;
                if (!mbar_wait(bar_empty + 8 * s, (round & 1) ^ 1)) {
                    if (lane == 0) {
                        sm_flags[0] = 1;
                        flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
                    }
                    aborted = true;
                    break;
                }
                const bool mine = lane >= j && lane < j + ng;
                TileDesc* d = sm_desc + s;
                if (lane == 0) {
                    d->ustart = us_j;
                    d->pend = pend;
                    d->flags = (first ? kFirst : 0) | (last ? kLast : 0) |
                               (last && pend == g1 ? kBlockLast : 0);
                    d->r = r_j;
                    d->kvh = kvh_j;
                    d->ng = ng;
                    d->tok0 = tok_j;
                    d->n = n_j;
                }
                if (lane < kTileGranules && lane >= ng) d->valid[lane] = 0;
                if (mine) d->valid[lane - j] = valid;
                const uint32_t nissue = __popc(__ballot_sync(0xffffffffu, mine && issue));
                __syncwarp();
                const uint32_t fb = bar_full + 8 * s;
                if (lane == 0) mbar_arrive_expect_tx(fb, nissue * 4u * kBoxBytes + (first ? qbytes : 0u));
                __syncwarp();
                const uint32_t stage = sbase + Smem::stages + s * kStageBytes;
                if (mine && issue) {
                    const uint32_t dk = stage + kStageK + (lane - j) * kBoxBytes;
                    const uint32_t dv = stage + kStageV + (lane - j) * kBoxBytes;
                    tma_load_3d(dk, &kmap, 0, kvh, zrow, fb);
                    tma_load_3d(dk + kHalfBytes, &kmap, 64, kvh, zrow, fb);
                    tma_load_3d(dv, &vmap, 0, kvh, zrow, fb);
                    tma_load_3d(dv + kHalfBytes, &vmap, 64, kvh, zrow, fb);
                }
                if (first && lane == 0) {
                    const __half* src = p.q + ((int64_t)r_j * p.hq + kvh_j * p.group) * kHeadDim;
                    if (waited) {
                        bulk_load(stage + kStageQ, src, qbytes, fb);
                    } else {
                        pq_dst[npq] = stage + kStageQ;
                        pq_src[npq] = src;
                        pq_bar[npq] = fb;
                        ++npq;
                    }
                }
                npq = __shfl_sync(0xffffffffu, npq, 0);
                ++tile;
                j += ng;
            }
        }
        wait_and_flush();
        if (!aborted) {
            // End marker: an empty stage whose descriptor says "no more tiles".
            const int s = tile % kStages;
            const uint32_t round = (uint32_t)tile / kStages;
            if (mbar_wait(bar_empty + 8 * s, (round & 1) ^ 1)) {
                if (lane == 0) {
                    sm_desc[s].flags = kEnd;
                    mbar_arrive(bar_full + 8 * s);
                }
                ++tile;
            } else if (lane == 0) {
                sm_flags[0] = 1;
                flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
            }
        }
        // Drain: the copies of every armed stage land before the block exits.
        for (int t = tile - kStages; t < tile; ++t) {
            if (t < 0) continue;
            if (!mbar_wait(bar_full + 8 * (t % kStages), (uint32_t)(t / kStages) & 1) && lane == 0)
                flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
        }
        return;
    }

    // ============================== consumers ==============================
    // Everything below may read what the preceding kernel wrote (query,
    // positions, new tokens, workspace) or write what it reads.
    griddep_wait();

    if (kPaged) {
        for (int r = cta; r < rows; r += G) {
            // Rows with nothing to read get zeros.
            if (sm_pre[r + 1] == sm_pre[r])
                for (int i = tid; i < p.hq * kHeadDim / 8; i += kConsumers)
                    reinterpret_cast<uint4*>(p.out + (int64_t)r * p.hq * kHeadDim)[i] =
                        make_uint4(0, 0, 0, 0);
            // Fused append: this block stores row r's new token into its slot.
            if (p.positions) {
                const int pos = p.positions[r];
                if (pos >= 0) {
                    const int lb = pos / p.bs;
                    int pb = -1;
                    if (lb >= p.mbpr) {
                        if (tid == 0) flag_error(p.dev_err, PKV_DEV_ERR_POSITION);
                    } else {
                        pb = p.tables[(int64_t)r * p.mbpr + lb];
                        if ((pb < 0 || pb >= p.nb) && tid == 0) flag_error(p.dev_err, PKV_DEV_ERR_BLOCK_ID);
                    }
                    if (pb >= 0 && pb < p.nb) {
                        const int vecs = hk * kHeadDim / 8;
                        const int64_t dst = ((int64_t)pb * p.bs + pos % p.bs) * vecs;
                        for (int i = tid; i < 2 * vecs; i += kConsumers) {
                            if (i < vecs)
                                reinterpret_cast<uint4*>(p.kpool)[dst + i] =
                                    reinterpret_cast<const uint4*>(p.k_new)[(int64_t)r * vecs + i];
                            else
                                reinterpret_cast<uint4*>(p.vpool)[dst + i - vecs] =
                                    reinterpret_cast<const uint4*>(p.v_new)[(int64_t)r * vecs + i - vecs];
                        }
                    }
                }
            }
        }
    }
    if (g0 >= g1) return;

    // Append positions of this block's first pieces, read once right after
    // the wait, so a piece never starts with a dependent global load.
    const bool fused = kPaged && p.positions != nullptr;
    if (fused) {
        if (tid == 0) {
            int lo = 0, hi = rows - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (sm_pre[mid] <= g0) lo = mid; else hi = mid - 1;
            }
            int r = lo, n = (sm_pre[r + 1] - sm_pre[r]) / hk;
            int kvh = (g0 - sm_pre[r]) / n, us = sm_pre[r] + kvh * n, k = 0;
            for (int g = g0; g < g1 && k < kMaxPieces;) {
                sm_ppos[k++] = r;  // row of piece k (replaced by its position below)
                g = min(g1, us + n);
                if (g >= g1) break;
                if (kvh + 1 < hk) {
                    ++kvh;
                    us += n;
                } else {
                    ++r;
                    while (r < rows - 1 && sm_pre[r + 1] == sm_pre[r]) ++r;
                    kvh = 0;
                    n = (sm_pre[r + 1] - sm_pre[r]) / hk;
                    us = sm_pre[r];
                }
            }
            sm_flags[2] = k;
        }
        consumer_sync();
    }
    // Each thread's position load stays in flight while the first tile lands;
    // it is published to shared memory after the first full barrier.
    const int npp = fused ? sm_flags[2] : 0;
    const int my_pos = tid < npp ? p.positions[sm_ppos[tid]] : 0;
    bool pos_published = !fused;
    int piece = 0;

    const int gq = lane >> 2;  // MMA group id: token row (QK) / dim row (PV) / head (B frag)
    const int tq = lane & 3;   // thread in group
    uint32_t qb[16];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[8][4];
    int patch_tok = -1;        // unit-local token this piece must take from k_new / v_new
    uint4 patch_val = make_uint4(0, 0, 0, 0);
    int tile = 0;
    while (true) {
        const int s = tile % kStages;
        const uint32_t round = (uint32_t)tile / kStages;
        if (!mbar_wait(bar_full + 8 * s, round & 1)) {
            if (lane == 0) {
                sm_flags[0] = 1;
                flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
            }
            break;
        }
        if (!pos_published) {
            if (tid < npp) sm_ppos[tid] = my_pos;
            consumer_sync();
            pos_published = true;
        }
        const TileDesc* d = sm_desc + s;
        const int flags = d->flags;
        if (flags & kEnd) break;
        const int r = d->r, kvh = d->kvh, ng = d->ng, tok0 = d->tok0;
        const int ustart = d->ustart, n = d->n, pend = d->pend;
        const int valid = warp < ng ? d->valid[warp] : 0;
        const uint32_t stage = sbase + Smem::stages + s * kStageBytes;
        unsigned char* stage_ptr = smem + Smem::stages + s * kStageBytes;
        if (flags & kFirst) {
            // B fragments of Q^T: b0 = Q[head gq][16ks + 2tq..], b1 = Q[head gq][16ks + 8 + 2tq..]
            const uint32_t* qrow = reinterpret_cast<const uint32_t*>(stage_ptr + kStageQ + gq * 256);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                qb[2 * ks] = gq < p.group ? qrow[ks * 8 + tq] : 0u;
                qb[2 * ks + 1] = gq < p.group ? qrow[ks * 8 + 4 + tq] : 0u;
            }
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
            patch_tok = -1;
            const int this_piece = piece++;
            if (fused) {
                // The appended token, if it falls inside this piece, is taken from
                // k_new / v_new (its slot may be written concurrently).
                const int pos = this_piece < kMaxPieces ? sm_ppos[this_piece] : p.positions[r];
                const int pg = pos >= 0 ? ustart + pos / kGranule : -1;
                if (pos >= 0 && pg >= ustart + tok0 / kGranule && pg < pend) {
                    patch_tok = pos;
                    const int chunk = lane & 15;
                    const uint4* src = reinterpret_cast<const uint4*>(
                        (lane < 16 ? p.k_new : p.v_new) + ((int64_t)r * hk + kvh) * kHeadDim);
                    patch_val = src[chunk];
                }
            }
        }
        if (warp < ng) {
            const int gtok = tok0 + warp * kGranule;  // unit-local token of this granule
            const uint32_t kb = stage + kStageK + warp * kBoxBytes;
            const uint32_t vb = stage + kStageV + warp * kBoxBytes;
            bool wrote = false;
            if (valid < kGranule) {
                // Rows past the row's length (or of a skipped block) may hold
                // anything, NaN included: zero them so 0 * V stays 0.
                uint4* v0 = reinterpret_cast<uint4*>(stage_ptr + kStageV + warp * kBoxBytes);
                for (int i = lane; i < (kGranule - valid) * 8; i += 32) {
                    const int row = valid + (i >> 3);
                    v0[row * 8 + (i & 7)] = make_uint4(0, 0, 0, 0);
                    v0[kHalfBytes / 16 + row * 8 + (i & 7)] = make_uint4(0, 0, 0, 0);
                }
                wrote = true;
            }
            if (patch_tok >= gtok && patch_tok < gtok + valid) {
                // Overwrite the staged row with the new token (swizzled layout).
                const int row = patch_tok - gtok;
                const int c16 = lane & 15;  // 16-byte chunk of the 128 dims
                unsigned char* box = stage_ptr + (lane < 16 ? kStageK : kStageV) + warp * kBoxBytes +
                                     (c16 >> 3) * kHalfBytes;
                *reinterpret_cast<uint4*>(box + row * 128 + (((c16 & 7) ^ (row & 7)) << 4)) = patch_val;
                wrote = true;
            }
            if (wrote) __syncwarp();
            // ---- S^T = K . Q^T ----
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
            {
                // two independent accumulation chains (even / odd k-steps)
                float sd[4] = {0.f, 0.f, 0.f, 0.f};
                const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const int chunk = (ks & 3) * 2 + (lane >> 4);
                    const uint32_t addr =
                        kb + (ks >> 2) * kHalfBytes + row * 128 + ((chunk ^ (row & 7)) << 4);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(addr, a0, a1, a2, a3);
                    mma16816((ks & 1) ? sd : sc, a0, a1, a2, a3, qb[2 * ks], qb[2 * ks + 1]);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) sc[i] += sd[i];
            }
            // scores: sc0 = (tok gq, head 2tq), sc1 = (gq, 2tq+1), sc2/3 = tok gq+8
            const float s0 = gq < valid ? sc[0] * p.scale_log2 : -INFINITY;
            const float s1 = gq < valid ? sc[1] * p.scale_log2 : -INFINITY;
            const float s2 = gq + 8 < valid ? sc[2] * p.scale_log2 : -INFINITY;
            const float s3 = gq + 8 < valid ? sc[3] * p.scale_log2 : -INFINITY;
            float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
            const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
            const float al0 = fast_exp2(m0 - mu0), al1 = fast_exp2(m1 - mu1);
            m0 = mn0;
            m1 = mn1;
            const uint32_t px = pack_half2(fast_exp2(s0 - mu0), fast_exp2(s1 - mu1));
            const uint32_t py = pack_half2(fast_exp2(s2 - mu0), fast_exp2(s3 - mu1));
            {
                const float2 fx = __half22float2(*reinterpret_cast<const __half2*>(&px));
                const float2 fy = __half22float2(*reinterpret_cast<const __half2*>(&py));
                l0 = l0 * al0 + fx.x + fy.x;
                l1 = l1 * al1 + fx.y + fy.y;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                o[i][0] *= al0;
                o[i][1] *= al1;
                o[i][2] *= al0;
                o[i][3] *= al1;
            }
            // B fragments of P^T (token x head) by transposing in registers.
            const uint32_t pb0 = movmatrix_t(px);
            const uint32_t pb1 = movmatrix_t(py);
            // ---- O^T += V^T . P^T ----
            {
                const int row = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    const int chunk = (mt & 3) * 2 + ((lane >> 3) & 1);
                    const uint32_t addr =
                        vb + (mt >> 2) * kHalfBytes + row * 128 + ((chunk ^ (row & 7)) << 4);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(addr, a0, a1, a2, a3);
                    mma16816(o[mt], a0, a1, a2, a3, pb0, pb1);
                }
            }
            // Generic-proxy writes must be ordered before TMA reuses the stage.
            if (wrote) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * s);
        ++tile;
        if (!(flags & kLast)) continue;

        // ---- end of a piece: combine the four warps' partial softmax states ----
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
        if (gq == 0) {
            sm_m[warp * 8 + 2 * tq] = m0;
            sm_m[warp * 8 + 2 * tq + 1] = m1;
            sm_l[warp * 8 + 2 * tq] = l0;
            sm_l[warp * 8 + 2 * tq + 1] = l1;
        }
        const int uend = ustart + n;
        const int cstart = owner_of(ustart, W, Geff);
        const int P = owner_of(uend - 1, W, Geff) - cstart + 1;
        const int u = r * hk + kvh;
        const int my_slot = cta + u;  // piece slot: block + unit is unique
        consumer_sync();
        const int ch = tid >> 4;        // head this thread combines
        float Mh = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) Mh = fmaxf(Mh, sm_m[w * 8 + ch]);
        float wsc[kConsumerWarps];
        float Lh = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            wsc[w] = Mh == -INFINITY ? 0.f : fast_exp2(sm_m[w * 8 + ch] - Mh);
            Lh += wsc[w] * sm_l[w * 8 + ch];
        }
        float* rec = p.records + (int64_t)my_slot * p.rec_floats;
        if (P > 1 && (tid & 15) == 0 && ch < p.group) {
            rec[ch] = Mh;
            rec[8 + ch] = Lh;
        }
        const float inv = Lh > 0.f ? 1.f / Lh : 0.f;
        const int cq = (tid & 15) * 4;  // four dims within a 64-dim pass
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            // warp writes its O^T fragments for dims [64 pass, 64 pass + 64)
            float* base = sm_comb + warp * 8 * kCombStride;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int mt = 4 * pass + k;
                base[(2 * tq) * kCombStride + 16 * k + gq] = o[mt][0];
                base[(2 * tq + 1) * kCombStride + 16 * k + gq] = o[mt][1];
                base[(2 * tq) * kCombStride + 16 * k + gq + 8] = o[mt][2];
                base[(2 * tq + 1) * kCombStride + 16 * k + gq + 8] = o[mt][3];
            }
            consumer_sync();
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float4 x =
                    *reinterpret_cast<const float4*>(sm_comb + (w * 8 + ch) * kCombStride + cq);
                v.x += wsc[w] * x.x;
                v.y += wsc[w] * x.y;
                v.z += wsc[w] * x.z;
                v.w += wsc[w] * x.w;
            }
            const int dd = 64 * pass + cq;
            if (ch < p.group) {
                if (P == 1) {
                    uint2 pk;
                    pk.x = pack_half2(v.x * inv, v.y * inv);
                    pk.y = pack_half2(v.z * inv, v.w * inv);
                    *reinterpret_cast<uint2*>(
                        p.out + ((int64_t)r * p.hq + kvh * p.group + ch) * kHeadDim + dd) = pk;
                } else {
                    *reinterpret_cast<float4*>(rec + kRecHead + ch * kHeadDim + dd) = v;
                }
            }
            consumer_sync();
        }
        if (P == 1) continue;
        // A split piece: its record is published; its arrival is counted once
        // per block, after the block's last piece (a contiguous range has at
        // most two split pieces: its first and its last).
        if (tid == 0) {
            const int k = sm_flags[3];
            sm_flags[4 + 5 * k] = u;
            sm_flags[5 + 5 * k] = cstart;
            sm_flags[6 + 5 * k] = P;
            sm_flags[7 + 5 * k] = r;
            sm_flags[8 + 5 * k] = kvh;
            sm_flags[3] = k + 1;
        }
    }

    // ---- arrivals of this block's split pieces; the last arriver of a unit
    // merges its pieces through their log-sum-exp and writes the output ----
    consumer_sync();
    const int nsplit = sm_flags[3];
    if (nsplit == 0 || sm_flags[0]) return;
    __threadfence();  // the records are visible before the arrivals count
    consumer_sync();
    if (tid < nsplit) {
        const int u = sm_flags[4 + 5 * tid];
        const int P = sm_flags[6 + 5 * tid];
        const int prev = atomicAdd(p.counters + u, 1);
        const int last = prev == P - 1;
        if (last) p.counters[u] = 0;  // every piece has arrived: re-arm for the next call
        sm_flags[14 + tid] = last;
    }
    consumer_sync();
    __threadfence();
    const uint32_t rec_bytes = (uint32_t)p.rec_floats * 4u;
    uint32_t land_total = 0;
    for (int k = 0; k < nsplit; ++k)
        if (sm_flags[14 + k]) land_total += (uint32_t)sm_flags[6 + 5 * k] * rec_bytes;
    if (land_total == 0) return;
    // The stages are idle once the block's tiles are consumed: every child
    // record of the units merged here comes in by bulk copies at once.
    const bool landing = land_total <= (uint32_t)(kStages * kStageBytes);
    if (landing) {
        if (warp == 0) {
            asm volatile("fence.proxy.async.global;" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if (lane == 0) mbar_arrive_expect_tx(bar_merge, land_total);
            __syncwarp();
            uint32_t off = 0;
            for (int k = 0; k < nsplit; ++k) {
                if (!sm_flags[14 + k]) continue;
                const int u = sm_flags[4 + 5 * k], cs = sm_flags[5 + 5 * k], P = sm_flags[6 + 5 * k];
                for (int j = lane; j < P; j += 32)
                    bulk_load(sbase + Smem::stages + off + j * rec_bytes,
                              p.records + (int64_t)(cs + j + u) * p.rec_floats, rec_bytes, bar_merge);
                off += (uint32_t)P * rec_bytes;
            }
        }
        if (!mbar_wait(bar_merge, 0)) {
            if (lane == 0) flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
            return;
        }
    }
    const int mh = tid >> 4;        // head
    const int md = (tid & 15) * 8;  // eight dims
    uint32_t off = 0;
    for (int k = 0; k < nsplit; ++k) {
        if (!sm_flags[14 + k]) continue;
        const int u = sm_flags[4 + 5 * k], cs = sm_flags[5 + 5 * k], P = sm_flags[6 + 5 * k];
        const int r = sm_flags[7 + 5 * k], kvh = sm_flags[8 + 5 * k];
        if (mh < p.group) {
            float Ls = 0.f, acc[8];
            const float* land = reinterpret_cast<const float*>(smem + Smem::stages + off);
            const float* glob = p.records + (int64_t)(cs + u) * p.rec_floats;
            if (landing)
                merge_children(land, P, p.rec_floats, mh, md, false, Ls, acc);
            else
                merge_children(glob, P, p.rec_floats, mh, md, true, Ls, acc);
            const float iv = Ls > 0.f ? 1.f / Ls : 0.f;
            uint4 pk;
            pk.x = pack_half2(acc[0] * iv, acc[1] * iv);
            pk.y = pack_half2(acc[2] * iv, acc[3] * iv);
            pk.z = pack_half2(acc[4] * iv, acc[5] * iv);
            pk.w = pack_half2(acc[6] * iv, acc[7] * iv);
            *reinterpret_cast<uint4*>(p.out + ((int64_t)r * p.hq + kvh * p.group + mh) * kHeadDim + md) = pk;
        }
        off += (uint32_t)P * rec_bytes;
    }
}

// ---------------------------------------------------------------------------
// Host side

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeFn encode_fn() {
    static EncodeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(f);
    });
    return fn;
}

struct MapKey {
    const void* base;
    int64_t rows;
    int hk;
    bool operator==(const MapKey& o) const { return base == o.base && rows == o.rows && hk == o.hk; }
};
struct MapKeyHash {
    size_t operator()(const MapKey& k) const {
        return std::hash<const void*>()(k.base) ^ (std::hash<int64_t>()(k.rows) * 31) ^ k.hk;
    }
};

// Tensor map over a pool viewed as [rows][hk][128] fp16: box 64 dims x 1 head
// x 16 tokens, 128-byte swizzle.
static int pool_map(const void* base, int64_t rows, int hk, CUtensorMap* out) {
    static std::mutex mu;
    static std::unordered_map<MapKey, CUtensorMap, MapKeyHash> cache;
    const MapKey key{base, rows, hk};
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
        *out = it->second;
        return PKV_OK;
    }
    EncodeFn enc = encode_fn();
    if (!enc) return PKV_ERR_CUDA;
    CUtensorMap m;
    const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)hk, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)hk * kHeadDim * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)kGranule};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return PKV_ERR_CUDA;
    if (cache.size() > 4096) cache.clear();
    cache.emplace(key, m);
    *out = m;
    return PKV_OK;
}

struct DeviceInfo {
    int sms = 0;
    bool attr_set[2] = {false, false};
};

static int device_info(DeviceInfo** out) {
    static std::mutex mu;
    static DeviceInfo infos[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    DeviceInfo& d = infos[dev];
    if (d.sms == 0) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return PKV_ERR_CUDA;
    }
    *out = &d;
    return PKV_OK;
}

}  // namespace tma

bool tma_decode_supported(int rows, int q_heads, int kv_heads, int head_dim, int block_size) {
    return head_dim == kHeadDim && kv_heads > 0 && q_heads % kv_heads == 0 &&
           q_heads / kv_heads <= kMaxGroup && block_size % tma::kGranule == 0 && rows >= 0 &&
           rows <= tma::kMaxRows;
}

static int64_t tma_slots(int rows, int kv_heads, int max_seq_len) {
    const int64_t units = (int64_t)rows * kv_heads;
    const int64_t granules = units * ((max_seq_len + tma::kGranule - 1) / tma::kGranule);
    const int64_t ctas = granules < tma::kMaxCtas ? (granules > 0 ? granules : 1) : tma::kMaxCtas;
    return ctas + units;  // piece slot = block + unit
}

static size_t tma_counter_bytes(int rows, int kv_heads) {
    return align_up(sizeof(int) * (size_t)rows * (size_t)kv_heads, 256);
}

size_t tma_workspace_bytes(int rows, int q_heads, int kv_heads, int max_seq_len) {
    const int group = kv_heads > 0 ? q_heads / kv_heads : 0;
    return tma_counter_bytes(rows, kv_heads) +
           align_up(sizeof(float) * (size_t)(tma::kRecHead + group * kHeadDim) *
                        (size_t)tma_slots(rows, kv_heads, max_seq_len),
                    256);
}

size_t tma_workspace_zero_bytes(int rows, int kv_heads, int max_seq_len) {
    (void)max_seq_len;
    return tma_counter_bytes(rows, kv_heads);  // the per-unit arrival counters
}

int tma_decode_launch(void* out, const void* q, const void* k_base, const void* v_base,
                      const int32_t* tables, const int32_t* seq_lens, int rows, int q_heads,
                      int kv_heads, int block_size, float scale, int mbpr, int num_blocks,
                      int max_seq_len, int width, void* workspace, int32_t* dev_err,
                      cudaStream_t stream, const AppendArgs* append, bool pdl) {
    using namespace tma;
    const bool paged = width == 0;
    const int64_t pool_rows = paged ? (int64_t)num_blocks * block_size : (int64_t)rows * width;
    if (pool_rows >= (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;
    const int limit = paged ? max_seq_len : width;
    const int64_t units = (int64_t)rows * kv_heads;
    const int64_t granules = units * ((limit + kGranule - 1) / kGranule);
    if (granules >= (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;
    DeviceInfo* info = nullptr;
    int st = device_info(&info);
    if (st != PKV_OK) return st;
    CUtensorMap km, vm;
    if ((st = pool_map(k_base, pool_rows, kv_heads, &km)) != PKV_OK) return st;
    if ((st = pool_map(v_base, pool_rows, kv_heads, &vm)) != PKV_OK) return st;

    int64_t ctas = info->sms;
    if (ctas > kMaxCtas) ctas = kMaxCtas;
    if (ctas > granules) ctas = granules > 0 ? granules : 1;

    Params prm{};
    prm.out = static_cast<__half*>(out);
    prm.q = static_cast<const __half*>(q);
    prm.tables = tables;
    prm.seq_lens = seq_lens;
    prm.rows = rows;
    prm.hq = q_heads;
    prm.hk = kv_heads;
    prm.group = q_heads / kv_heads;
    prm.bs = block_size;
    prm.mbpr = mbpr;
    prm.nb = num_blocks;
    prm.limit = limit;
    prm.width = paged ? 0 : width;
    prm.scale_log2 = scale * kLog2e;
    prm.rec_floats = kRecHead + prm.group * kHeadDim;
    prm.counters = static_cast<int*>(workspace);
    prm.records = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                           tma_counter_bytes(rows, kv_heads));
    prm.dev_err = dev_err;
    if (append) {
        prm.positions = append->positions;
        prm.k_new = static_cast<const __half*>(append->k_new);
        prm.v_new = static_cast<const __half*>(append->v_new);
        prm.kpool = static_cast<__half*>(const_cast<void*>(k_base));
        prm.vpool = static_cast<__half*>(const_cast<void*>(v_base));
    }

    const uint32_t smem = Smem::total(rows);
    const int which = paged ? 0 : 1;
    auto kernel = paged ? decode_tma_kernel<true> : decode_tma_kernel<false>;
    if (!info->attr_set[which]) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Smem::total(kMaxRows)) != cudaSuccess)
            return PKV_ERR_CUDA;
        info->attr_set[which] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, kernel, km, vm, prm) != cudaSuccess) return PKV_ERR_CUDA;
    return launch_status();
}

}  // namespace pkv
