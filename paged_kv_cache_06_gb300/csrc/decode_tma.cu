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
constexpr int kFanIn = 8;
constexpr int kLevels = 4;          // 8^4 leaves >= kMaxCtas
constexpr int kMaxCtas = 1024;
constexpr int kMaxRows = 1024;
constexpr int kRecFloats = 16 + 8 * kHeadDim;  // m[8], l[8], o[8][128]
constexpr uint32_t kBoxBytes = kGranule * 128;                // 16 rows x 128 B
constexpr uint32_t kHalfBytes = kTileGranules * kBoxBytes;    // one 64-dim half of 64 tokens
constexpr uint32_t kStageK = 0;
constexpr uint32_t kStageV = 2 * kHalfBytes;
constexpr uint32_t kStageQ = 4 * kHalfBytes;
constexpr uint32_t kStageBytes = 4 * kHalfBytes + 8 * 256;    // K, V, Q (8 heads x 256 B)
constexpr int kCombStride = 36;                               // 32 dims + 4 pad (floats)
constexpr uint32_t kSpinLimit = 1u << 22;
constexpr float kLog2e = 1.4426950408889634f;

static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment for 128B swizzle");

struct Params {
    __half* out;
    const __half* q;
    const int32_t* tables;
    const int32_t* seq_lens;
    int rows, hq, hk, group, bs, mbpr, nb;
    int limit;      // largest valid seq_len (paged); width (padded)
    int width;      // padded comparator: columns per row (0 = paged)
    float scale_log2;
    int slots;      // records / counters per level
    int* counters;  // [kLevels][slots]
    float* records; // [slots][kRecFloats]
    int32_t* dev_err;
};

// Shared memory carve-up (offsets from a 1024-aligned base).
struct Smem {
    static constexpr uint32_t stages = 0;
    static constexpr uint32_t comb = kStages * kStageBytes;                         // [4][8][36] f32
    static constexpr uint32_t ml = comb + kConsumerWarps * 8 * kCombStride * 4;     // [4][8] m, [4][8] l
    static constexpr uint32_t bars = ml + 2 * kConsumerWarps * 8 * 4;               // full[S], empty[S]
    static constexpr uint32_t meta = bars + 2 * kStages * 8;                        // valid[S][4]
    static constexpr uint32_t flags = meta + kStages * kTileGranules * 4;           // misc ints
    static constexpr uint32_t part = flags + 16 * 4;                                // scan partials
    static constexpr uint32_t prefix = part + kThreads * 4;                         // rows + 1 ints
    static uint32_t total(int rows) { return prefix + (uint32_t)(rows + 1) * 4 + 1024; }
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
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Granule count of one unit of row r (seq_len clamped; padded: the width).
__device__ __forceinline__ int row_len(const Params& p, int r, bool* bad) {
    int L = p.seq_lens[r];
    if (L < 0 || L > p.limit) {
        *bad = true;
        L = L < 0 ? 0 : p.limit;
    }
    return L;
}

// Cursor over the pieces of one block's granule range [g0, g1).
struct Cursor {
    int r, kvh, n;       // current unit and its granule count
    int64_t ustart;      // unit's first granule (global)
};

__device__ __forceinline__ int granules_of(int L) { return (L + kGranule - 1) / kGranule; }

// Index c of the block whose range holds granule g (partition b_c = c*W/G).
__device__ __forceinline__ int owner_of(int64_t g, int64_t W, int G) {
    // largest c with floor(c*W/G) <= g  <=>  c < (g+1)*G/W
    return (int)(((g + 1) * (int64_t)G + W - 1) / W) - 1;
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
    int* sm_valid = reinterpret_cast<int*>(smem + Smem::meta);
    volatile int* sm_flags = reinterpret_cast<volatile int*>(smem + Smem::flags);
    int* sm_part = reinterpret_cast<int*>(smem + Smem::part);
    int* sm_pre = reinterpret_cast<int*>(smem + Smem::prefix);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int G = gridDim.x;  // blocks launched; the partition uses Geff <= G
    const int cta = blockIdx.x;
    const int hk = p.hk;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        sm_flags[0] = 0;  // abort
        sm_flags[1] = 0;  // last-arriver broadcast
    }

    // ---- granule prefix over rows: sm_pre[r] = first granule of row r ----
    const int rows = p.rows;
    const int per = (rows + kThreads - 1) / kThreads;
    bool bad_len = false;
    int sum = 0;
    for (int i = 0; i < per; ++i) {
        const int r = tid * per + i;
        if (r < rows) {
            const int L = kPaged ? row_len(p, r, &bad_len) : p.width;
            const int c = hk * granules_of(L);
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
        int s = 0;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int idx = lane * kPer + j;
            v[j] = idx < kThreads ? sm_part[idx] : 0;
            s += v[j];
        }
        int incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        int run = incl - s;
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
    const int64_t W = sm_pre[rows];
    const int Geff = (int)(W < G ? W : G);
    const int64_t g0 = cta < Geff ? W * cta / Geff : 0;
    const int64_t g1 = cta < Geff ? W * (cta + 1) / Geff : 0;

    // Rows with nothing to read get zeros (spread over the blocks).
    if (kPaged && tid < kConsumers) {
        for (int r = cta; r < rows; r += G) {
            if (sm_pre[r + 1] == sm_pre[r]) {
                for (int i = tid; i < p.hq * kHeadDim / 8; i += kConsumers)
                    reinterpret_cast<uint4*>(p.out + (int64_t)r * p.hq * kHeadDim)[i] =
                        make_uint4(0, 0, 0, 0);
            }
        }
    }
    if (g0 >= g1) return;

    // Locate the unit holding g0: last row with sm_pre[r] <= g0 and a granule.
    auto locate = [&](int64_t g, Cursor& cur) {
        int lo = 0, hi = rows - 1;
        while (lo < hi) {  // largest r with sm_pre[r] <= g
            const int mid = (lo + hi + 1) >> 1;
            if (sm_pre[mid] <= g) lo = mid; else hi = mid - 1;
        }
        // skip empty rows (equal prefixes) forward
        while (lo < rows - 1 && sm_pre[lo + 1] <= g) ++lo;
        cur.r = lo;
        cur.n = (sm_pre[lo + 1] - sm_pre[lo]) / hk;
        cur.kvh = (int)((g - sm_pre[lo]) / cur.n);
        cur.ustart = sm_pre[lo] + (int64_t)cur.kvh * cur.n;
    };
    auto advance = [&](Cursor& cur) {
        if (cur.kvh + 1 < hk) {
            ++cur.kvh;
            cur.ustart += cur.n;
            return;
        }
        int r = cur.r + 1;
        while (r < rows - 1 && sm_pre[r + 1] == sm_pre[r]) ++r;
        cur.r = r;
        cur.kvh = 0;
        cur.n = (sm_pre[r + 1] - sm_pre[r]) / hk;
        cur.ustart = sm_pre[r];
    };

    if (warp == kConsumerWarps) {
        // ============================ producer ============================
        Cursor cur;
        locate(g0, cur);
        int64_t g = g0;
        int tile = 0;
        while (g < g1 && !sm_flags[0]) {
            const int64_t uend = cur.ustart + cur.n;
            const int64_t pend = g1 < uend ? g1 : uend;
            const int L = kPaged ? min(max(p.seq_lens[cur.r], 0), p.limit) : min(max(p.seq_lens[cur.r], 0), p.width);
            bool first = true;
            for (int64_t tg = g; tg < pend; tg += kTileGranules, ++tile) {
                const int s = tile % kStages;
                const uint32_t round = tile / kStages;
                if (!mbar_wait(bar_empty + 8 * s, (round & 1) ^ 1)) {
                    sm_flags[0] = 1;
                    flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
                    break;
                }
                const int ng = (int)(pend - tg < kTileGranules ? pend - tg : kTileGranules);
                // Lane j < ng resolves granule j of this tile.
                int valid = 0, zrow = 0;
                bool issue = false;
                if (lane < ng) {
                    const int tok = (int)(tg + lane - cur.ustart) * kGranule;
                    valid = min(kGranule, L - tok);
                    if (valid < 0) valid = 0;
                    if (kPaged) {
                        const int pb = p.tables[(int64_t)cur.r * p.mbpr + tok / p.bs];
                        if (pb < 0 || pb >= p.nb) {
                            flag_error(p.dev_err, PKV_DEV_ERR_BLOCK_ID);
                            valid = 0;
                        } else {
                            zrow = pb * p.bs + tok % p.bs;
                            issue = true;
                        }
                    } else {
                        zrow = cur.r * p.width + tok;
                        issue = true;
                    }
                }
                const uint32_t nissue = __popc(__ballot_sync(0xffffffffu, issue));
                const uint32_t qbytes = first ? (uint32_t)p.group * 256u : 0u;
                const uint32_t stage = sbase + Smem::stages + s * kStageBytes;
                // publish valid counts (lane j writes granule j)
                if (lane < kTileGranules) sm_valid[s * kTileGranules + lane] = lane < ng ? valid : 0;
                __syncwarp();
                if (lane == 0) mbar_arrive_expect_tx(bar_full + 8 * s, nissue * 4u * kBoxBytes + qbytes);
                __syncwarp();
                if (issue) {
                    const uint32_t dk = stage + kStageK + lane * kBoxBytes;
                    const uint32_t dv = stage + kStageV + lane * kBoxBytes;
                    tma_load_3d(dk, &kmap, 0, cur.kvh, zrow, bar_full + 8 * s);
                    tma_load_3d(dk + kHalfBytes, &kmap, 64, cur.kvh, zrow, bar_full + 8 * s);
                    tma_load_3d(dv, &vmap, 0, cur.kvh, zrow, bar_full + 8 * s);
                    tma_load_3d(dv + kHalfBytes, &vmap, 64, cur.kvh, zrow, bar_full + 8 * s);
                }
                if (first && lane == 0)
                    bulk_load(stage + kStageQ,
                              p.q + ((int64_t)cur.r * p.hq + cur.kvh * p.group) * kHeadDim, qbytes,
                              bar_full + 8 * s);
                first = false;
            }
            g = pend;
            if (g < g1) advance(cur);
        }
        // Drain: every issued stage's copies must land before the block exits.
        const int issued = tile;
        for (int t = issued - kStages; t < issued; ++t) {
            if (t < 0) continue;
            const int s = t % kStages;
            if (!mbar_wait(bar_full + 8 * s, (uint32_t)(t / kStages) & 1)) {
                flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
            }
        }
        return;
    }

    // ============================== consumers ==============================
    const int gq = lane >> 2;  // MMA group id: token row (QK) / dim row (PV) / head (B frag)
    const int tq = lane & 3;   // thread in group
    Cursor cur;
    locate(g0, cur);
    int64_t g = g0;
    int tile = 0;
    bool aborted = false;
    while (g < g1 && !aborted) {
        const int64_t uend = cur.ustart + cur.n;
        const int64_t pend = g1 < uend ? g1 : uend;
        uint32_t qb[16];
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        float o[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        bool first = true;
        for (int64_t tg = g; tg < pend; tg += kTileGranules, ++tile) {
            const int s = tile % kStages;
            const uint32_t round = tile / kStages;
            if (!mbar_wait(bar_full + 8 * s, round & 1)) {
                if (lane == 0) {
                    sm_flags[0] = 1;
                    flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
                }
                aborted = true;
                break;
            }
            const uint32_t stage = sbase + Smem::stages + s * kStageBytes;
            const unsigned char* stage_ptr = smem + Smem::stages + s * kStageBytes;
            if (first) {
                // B fragments of Q^T: b0 = Q[head gq][16ks + 2tq..], b1 = Q[head gq][16ks + 8 + 2tq..]
                const uint32_t* qrow =
                    reinterpret_cast<const uint32_t*>(stage_ptr + kStageQ + gq * 256);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    qb[2 * ks] = gq < p.group ? qrow[ks * 8 + tq] : 0u;
                    qb[2 * ks + 1] = gq < p.group ? qrow[ks * 8 + 4 + tq] : 0u;
                }
                first = false;
            }
            const int ng = (int)(pend - tg < kTileGranules ? pend - tg : kTileGranules);
            if (warp < ng) {
                const int valid = sm_valid[s * kTileGranules + warp];
                const uint32_t kb = stage + kStageK + warp * kBoxBytes;
                const uint32_t vb = stage + kStageV + warp * kBoxBytes;
                if (valid < kGranule) {
                    // Rows past the row's length (or of a skipped block) may hold
                    // anything, NaN included: zero them so 0 * V stays 0.
                    uint4* v0 = reinterpret_cast<uint4*>(const_cast<unsigned char*>(stage_ptr) +
                                                         kStageV + warp * kBoxBytes);
                    for (int i = lane; i < (kGranule - valid) * 8; i += 32) {
                        const int row = valid + (i >> 3);
                        v0[row * 8 + (i & 7)] = make_uint4(0, 0, 0, 0);
                        v0[kHalfBytes / 16 + row * 8 + (i & 7)] = make_uint4(0, 0, 0, 0);
                    }
                    __syncwarp();
                }
                // ---- S^T = K . Q^T ----
                float sc[4] = {0.f, 0.f, 0.f, 0.f};
                {
                    const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const int chunk = (ks & 3) * 2 + (lane >> 4);
                        const uint32_t addr = kb + (ks >> 2) * kHalfBytes + row * 128 +
                                              ((chunk ^ (row & 7)) << 4);
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4(addr, a0, a1, a2, a3);
                        mma16816(sc, a0, a1, a2, a3, qb[2 * ks], qb[2 * ks + 1]);
                    }
                }
                // scores: sc0 = (tok gq, head 2tq), sc1 = (gq, 2tq+1), sc2/3 = tok gq+8
                float s0 = gq < valid ? sc[0] * p.scale_log2 : -INFINITY;
                float s1 = gq < valid ? sc[1] * p.scale_log2 : -INFINITY;
                float s2 = gq + 8 < valid ? sc[2] * p.scale_log2 : -INFINITY;
                float s3 = gq + 8 < valid ? sc[3] * p.scale_log2 : -INFINITY;
                float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                }
                const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
                const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
                const float al0 = exp2f(m0 - mu0), al1 = exp2f(m1 - mu1);
                m0 = mn0;
                m1 = mn1;
                const uint32_t px = pack_half2(exp2f(s0 - mu0), exp2f(s1 - mu1));
                const uint32_t py = pack_half2(exp2f(s2 - mu0), exp2f(s3 - mu1));
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
                        const uint32_t addr = vb + (mt >> 2) * kHalfBytes + row * 128 +
                                              ((chunk ^ (row & 7)) << 4);
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4_t(addr, a0, a1, a2, a3);
                        mma16816(o[mt], a0, a1, a2, a3, pb0, pb1);
                    }
                }
                if (valid < kGranule) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * s);
        }
        if (aborted) break;

        // ---- combine the four warps' partial softmax states ----
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
        const int P = owner_of(uend - 1, W, Geff) - owner_of(cur.ustart, W, Geff) + 1;
        const int cstart = owner_of(cur.ustart, W, Geff);
        const int u = cur.r * hk + cur.kvh;
        const int my_slot = cstart + (cta - cstart) + u;  // leaf slot id = block + unit
        consumer_sync();
        const int ch = tid >> 4;                 // head this thread combines
        const int cd = (tid & 15) * 2;           // two dims within a 32-dim pass
        float Mh = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) Mh = fmaxf(Mh, sm_m[w * 8 + ch]);
        float wsc[kConsumerWarps];
        float Lh = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            wsc[w] = Mh == -INFINITY ? 0.f : exp2f(sm_m[w * 8 + ch] - Mh);
            Lh += wsc[w] * sm_l[w * 8 + ch];
        }
        float* rec = p.records + (int64_t)my_slot * kRecFloats;
        if (P > 1 && (tid & 15) == 0) {
            rec[ch] = Mh;
            rec[8 + ch] = Lh;
        }
#pragma unroll
        for (int pass = 0; pass < 4; ++pass) {
            // warp writes its O^T fragments for dims [32 pass, 32 pass + 32)
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int mt = 2 * pass + k;
                float* base = sm_comb + warp * 8 * kCombStride;
                base[(2 * tq) * kCombStride + 16 * k + gq] = o[mt][0];
                base[(2 * tq + 1) * kCombStride + 16 * k + gq] = o[mt][1];
                base[(2 * tq) * kCombStride + 16 * k + gq + 8] = o[mt][2];
                base[(2 * tq + 1) * kCombStride + 16 * k + gq + 8] = o[mt][3];
            }
            consumer_sync();
            float v0 = 0.f, v1 = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float* src = sm_comb + (w * 8 + ch) * kCombStride + cd;
                v0 += wsc[w] * src[0];
                v1 += wsc[w] * src[1];
            }
            const int d = 32 * pass + cd;
            if (P == 1) {
                if (ch < p.group) {
                    const float inv = Lh > 0.f ? 1.f / Lh : 0.f;
                    *reinterpret_cast<__half2*>(
                        p.out + ((int64_t)cur.r * p.hq + cur.kvh * p.group + ch) * kHeadDim + d) =
                        __floats2half2_rn(v0 * inv, v1 * inv);
                }
            } else {
                *reinterpret_cast<float2*>(rec + 16 + ch * kHeadDim + d) = make_float2(v0, v1);
            }
            consumer_sync();
        }

        // ---- merge tree over the unit's pieces (last arriver merges) ----
        if (P > 1) {
            int level = 0, idx = cta - cstart, count = P;
            int stride = 1;  // leaves between siblings at this level
            while (true) {
                const int parent = idx / kFanIn;
                const int firstc = parent * kFanIn;
                const int nch = min(kFanIn, count - firstc);
                const int pslot = cstart + u + firstc * stride;  // parent's leftmost leaf slot
                __threadfence();
                consumer_sync();
                if (tid == 0) {
                    int* ctr = p.counters + (int64_t)level * p.slots + pslot;
                    const int prev = atomicAdd(ctr, 1);
                    const int last = prev == nch - 1;
                    if (last) *ctr = 0;
                    sm_flags[1] = last;
                }
                consumer_sync();
                if (!sm_flags[1]) break;
                __threadfence();
                // merge children firstc .. firstc + nch - 1 (slots cstart + u + c * stride)
                const int mh = tid >> 4;
                const int md = (tid & 15) * 8;
                float M = -INFINITY;
                for (int c = 0; c < nch; ++c) {
                    const float* cr = p.records + (int64_t)(cstart + u + (firstc + c) * stride) * kRecFloats;
                    M = fmaxf(M, __ldcg(cr + mh));
                }
                float Lm = 0.f, acc[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] = 0.f;
                for (int c = 0; c < nch; ++c) {
                    const float* cr = p.records + (int64_t)(cstart + u + (firstc + c) * stride) * kRecFloats;
                    const float w = M == -INFINITY ? 0.f : exp2f(__ldcg(cr + mh) - M);
                    Lm += w * __ldcg(cr + 8 + mh);
                    const float4 x = __ldcg(reinterpret_cast<const float4*>(cr + 16 + mh * kHeadDim + md));
                    const float4 y = __ldcg(reinterpret_cast<const float4*>(cr + 16 + mh * kHeadDim + md + 4));
                    acc[0] += w * x.x; acc[1] += w * x.y; acc[2] += w * x.z; acc[3] += w * x.w;
                    acc[4] += w * y.x; acc[5] += w * y.y; acc[6] += w * y.z; acc[7] += w * y.w;
                }
                const int next = (count + kFanIn - 1) / kFanIn;
                consumer_sync();  // all reads of the children done before the slot is reused
                if (next == 1) {
                    if (mh < p.group) {
                        const float inv = Lm > 0.f ? 1.f / Lm : 0.f;
                        uint4 pk;
                        pk.x = pack_half2(acc[0] * inv, acc[1] * inv);
                        pk.y = pack_half2(acc[2] * inv, acc[3] * inv);
                        pk.z = pack_half2(acc[4] * inv, acc[5] * inv);
                        pk.w = pack_half2(acc[6] * inv, acc[7] * inv);
                        *reinterpret_cast<uint4*>(
                            p.out + ((int64_t)cur.r * p.hq + cur.kvh * p.group + mh) * kHeadDim + md) = pk;
                    }
                    break;
                }
                float* pr = p.records + (int64_t)pslot * kRecFloats;
                if ((tid & 15) == 0) {
                    pr[mh] = M;
                    pr[8 + mh] = Lm;
                }
                *reinterpret_cast<float4*>(pr + 16 + mh * kHeadDim + md) = make_float4(acc[0], acc[1], acc[2], acc[3]);
                *reinterpret_cast<float4*>(pr + 16 + mh * kHeadDim + md + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
                idx = parent;
                count = next;
                stride *= kFanIn;
                ++level;
            }
        }
        g = pend;
        if (g < g1) advance(cur);
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

size_t tma_workspace_bytes(int rows, int q_heads, int kv_heads, int max_seq_len) {
    (void)q_heads;
    const int64_t units = (int64_t)rows * kv_heads;
    const int64_t granules = units * ((max_seq_len + tma::kGranule - 1) / tma::kGranule);
    const int64_t ctas = granules < tma::kMaxCtas ? (granules > 0 ? granules : 1) : tma::kMaxCtas;
    const int64_t slots = ctas + units;
    const size_t counters = align_up(sizeof(int) * (size_t)(tma::kLevels * slots), 256);
    return counters + align_up(sizeof(float) * (size_t)tma::kRecFloats * (size_t)slots, 256);
}

size_t tma_workspace_zero_bytes(int rows, int kv_heads, int max_seq_len) {
    const int64_t units = (int64_t)rows * kv_heads;
    const int64_t granules = units * ((max_seq_len + tma::kGranule - 1) / tma::kGranule);
    const int64_t ctas = granules < tma::kMaxCtas ? (granules > 0 ? granules : 1) : tma::kMaxCtas;
    return align_up(sizeof(int) * (size_t)(tma::kLevels * (ctas + units)), 256);
}

int tma_decode_launch(void* out, const void* q, const void* k_base, const void* v_base,
                      const int32_t* tables, const int32_t* seq_lens, int rows, int q_heads,
                      int kv_heads, int block_size, float scale, int mbpr, int num_blocks,
                      int max_seq_len, int width, void* workspace, int32_t* dev_err,
                      cudaStream_t stream) {
    using namespace tma;
    const bool paged = width == 0;
    const int64_t pool_rows = paged ? (int64_t)num_blocks * block_size : (int64_t)rows * width;
    if (pool_rows >= (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;
    DeviceInfo* info = nullptr;
    int st = device_info(&info);
    if (st != PKV_OK) return st;
    CUtensorMap km, vm;
    if ((st = pool_map(k_base, pool_rows, kv_heads, &km)) != PKV_OK) return st;
    if ((st = pool_map(v_base, pool_rows, kv_heads, &vm)) != PKV_OK) return st;

    const int limit = paged ? max_seq_len : width;
    const int64_t units = (int64_t)rows * kv_heads;
    const int64_t granules = units * ((limit + kGranule - 1) / kGranule);
    int64_t ctas = info->sms;
    if (ctas > kMaxCtas) ctas = kMaxCtas;
    if (ctas > granules) ctas = granules > 0 ? granules : 1;
    const int64_t slots_cap = (granules < kMaxCtas ? (granules > 0 ? granules : 1) : kMaxCtas) + units;

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
    prm.slots = (int)slots_cap;
    prm.counters = static_cast<int*>(workspace);
    prm.records = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                           align_up(sizeof(int) * (size_t)(kLevels * slots_cap), 256));
    prm.dev_err = dev_err;

    const uint32_t smem = Smem::total(rows);
    const int which = paged ? 0 : 1;
    if (!info->attr_set[which]) {
        cudaError_t e = paged ? cudaFuncSetAttribute(decode_tma_kernel<true>,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     Smem::total(kMaxRows))
                              : cudaFuncSetAttribute(decode_tma_kernel<false>,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     Smem::total(kMaxRows));
        if (e != cudaSuccess) return PKV_ERR_CUDA;
        info->attr_set[which] = true;
    }
    if (paged)
        decode_tma_kernel<true><<<(int)ctas, kThreads, smem, stream>>>(km, vm, prm);
    else
        decode_tma_kernel<false><<<(int)ctas, kThreads, smem, stream>>>(km, vm, prm);
    return launch_status();
}

}  // namespace pkv
