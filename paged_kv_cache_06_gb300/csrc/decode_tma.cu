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
// block is a piece.  A unit with pieces in several blocks is merged by the
// block that holds its last piece: every piece publishes a partial record
// (running max, sum and unnormalised output) and counts itself on a per-unit
// counter with a release; the merging block waits (bounded) until the others
// have all counted, lands every record and combines them through their
// log-sum-exp, then re-arms the counter.  A block merges at most one unit.
//
// Block layout.  Warp 4 is the producer: it resolves each granule's physical
// block from the table and issues TMA tiled copies (a 16-token x 64-dim box,
// 128-byte swizzle, never crossing a physical block) into a ring of twelve
// 8 KB granule slots.  Warps 0-3 consume, in one of two modes:
//   * burst: the block's whole range fits the ring and covers at most four
//     pieces.  Every copy is issued before the dependency wait, warps are
//     dealt to pieces in proportion to their size, and each warp attends to
//     its granules; the warps' partial states are then combined for all
//     pieces together.
//   * stream: the ring runs as three stages of four granules, one granule
//     per warp per stage, and pieces are combined as they end.
// Per granule (16 tokens) and group of query heads (up to 8):
//   S^T[16 tok][8 heads] = K[16 tok][128] . Q^T        (mma.sync m16n8k16)
//   online softmax per head in fp32, base-2 exponent
//   O^T[128][8 heads]   += V^T[128][16 tok] . P^T      (P transposed in
//                                                       registers by movmatrix)
// The grouped query heads are the MMA's N = 8 columns, so every K and V byte
// is read once and feeds all heads of its group.
//
// Safety: table entries are range-checked before any copy is issued (a bad
// entry is skipped and flagged); every mbarrier wait is bounded and a timeout
// sets PKV_DEV_ERR_TIMEOUT, stops the block and drains its copies in flight.
#include <cuda.h>

#include <mutex>

#include "fp8_codec.cuh"
#include "pkv_internal.cuh"
#include "ptx.cuh"

namespace pkv {
namespace tma {

constexpr int kGranule = 16;        // tokens per box and per consumer warp step
constexpr int kTileGranules = 4;    // stream mode: granules per stage (one per consumer warp)
constexpr int kStages = 3;
constexpr int kRing = kStages * kTileGranules;  // granule slots
constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kMaxCtas = 1024;
constexpr int kMaxRows = 1024;
constexpr int kRecHead = 16;   // per record: m[8], l[8], then o[group][128]
constexpr int kMaxPieces = 32; // append positions prefetched for a block's first pieces
constexpr int kMergeBatch = 8; // children merged per register batch
constexpr int kMergeBars = 4;  // landing barriers, one per batch
constexpr int kLandMax = kMergeBars * kMergeBatch;  // most records a landed merge takes
constexpr int kBurstPieces = 4;
constexpr int kBatch = 1;      // burst mode: granules per attend step (larger batches measured slower)
constexpr int kCounterStride = 32;  // ints between the arrival counters of two units
constexpr uint32_t kPollLimit = 1u << 21;  // polls of a merge wait (about a second)
constexpr uint32_t kBoxBytes = kGranule * 128;   // 16 rows x 128 B (64 dims)
constexpr uint32_t kSlotBytes = 4 * kBoxBytes;   // K dims 0-63, K 64-127, V 0-63, V 64-127
constexpr uint32_t kSlotV = 2 * kBoxBytes;
constexpr int kFp8MaxKvHeads = 16;                // FP8 pools: per-head scales kept in shared memory
constexpr uint32_t kQBytes = 8 * 256;            // up to 8 query heads x 128 dims
constexpr int kCombStride = 68;                  // stream combine: 64 dims + 4 pad (floats)
constexpr int kDumpStride = 132;                 // burst dump: 128 dims + 4 pad (floats)
constexpr float kLog2e = 1.4426950408889634f;

static_assert(kSlotBytes % 1024 == 0, "slots must keep 1024-byte alignment for 128B swizzle");
static_assert((kRecHead + 8 * kDumpStride) * 4 <= (int)kSlotBytes, "a dumped partial fits one slot");

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
    int* counters;  // [units][kCounterStride]: pieces arrived per split unit (zero between calls)
    float* records; // [slots][rec_floats]: partial results of split units
    int32_t* dev_err;
    // fused append (all null when the kernel only decodes)
    const int32_t* positions;
    const __half* k_new;
    const __half* v_new;
    __half* kpool;
    __half* vpool;
    // FP8 pools: one scale per KV head (null for fp16 pools)
    const float* k_scale;
    const float* v_scale;
};

// Burst-mode plan of one block, written by thread 0 after the prologue.
struct Plan {
    int burst, npieces;
    int r[kBurstPieces], kvh[kBurstPieces], ustart[kBurstPieces], n[kBurstPieces];
    int P[kBurstPieces], cstart[kBurstPieces], w0[kBurstPieces], wn[kBurstPieces];
    int wpiece[kConsumerWarps], wa[kConsumerWarps], wb[kConsumerWarps];
    int valid[kRing];
};

// Shared memory carve-up (offsets from a 1024-aligned base).
struct Smem {
    static constexpr uint32_t ring = 0;
    static constexpr uint32_t q = ring + kRing * kSlotBytes;                        // [stages] stream queries
    static constexpr uint32_t comb = q + kStages * kQBytes;                         // [4][8][68] f32
    static constexpr uint32_t ml = comb + kConsumerWarps * 8 * kCombStride * 4;     // [4][8] m, [4][8] l
    static constexpr uint32_t bars = ml + 2 * kConsumerWarps * 8 * 4;               // full[S], empty[S], slot[R], merge
    static constexpr uint32_t desc = bars + (2 * kStages + kRing + 1 + kMergeBars) * 8;  // TileDesc[S]
    static constexpr uint32_t plan = desc + kStages * 64;
    static constexpr uint32_t flags = plan + ((sizeof(Plan) + 15) / 16) * 16;       // misc ints
    static constexpr uint32_t scales = flags + 16 * 4;                              // FP8: k, v scale [2][16]
    static constexpr uint32_t ppos = scales + 2 * kFp8MaxKvHeads * 4;               // piece positions [32]
    static constexpr uint32_t part = comb;  // scan partials: prologue only, aliases comb
    static constexpr uint32_t prefix = ppos + kMaxPieces * 4;                       // rows + 1 ints
    __host__ __device__ static constexpr uint32_t lens(int rows) { return prefix + (uint32_t)(rows + 1) * 4; }
    __host__ __device__ static constexpr uint32_t total(int rows) { return lens(rows) + (uint32_t)rows * 4 + 1024; }
};
// Two blocks per SM (this layer's and the next one's, under programmatic
// dependent launch) at batch 32: 228 KB per SM, 1 KB reserved per block.
static_assert(Smem::total(32) + 1024 <= 233472 / 2, "two blocks per SM at 32 rows");

// ---------------------------------------------------------------------------
// PTX wrappers (shared ones in ptx.cuh)

using namespace ptx;

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

// Stream-mode tile descriptor: written by the producer before the stage's
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


// Running softmax state of one warp: per lane, heads 2tq and 2tq+1
// (tq = lane & 3) and the O^T fragments of all eight 16-dim row groups.
struct Soft {
    float m0, m1, l0, l1;
    float o[8][4];
    __device__ __forceinline__ void reset() {
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    }
};

// One online-softmax step of a warp over kB granules staged in slots
// slot[0..kB-1] (K dims 0-63 at +0, K 64-127 at +2 KB, V at +4 KB / +6 KB,
// 128-byte swizzled rows), valid[j] tokens each.  Rows past valid[j] must
// hold finite values (zeroed by the caller) so that 0 * V stays 0.
template <int kB>
__device__ __forceinline__ void attend(Soft& st, const uint32_t (&qb)[16], const uint32_t* slot,
                                       const int* valid, float scale_log2, int lane) {
    const int gq = lane >> 2;
    float s[kB][4];
    {
        // S^T = K . Q^T; per granule two independent chains (even / odd k-steps)
        const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
        float c0[kB][4], c1[kB][4];
#pragma unroll
        for (int j = 0; j < kB; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i) c0[j][i] = c1[j][i] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int chunk = (ks & 3) * 2 + (lane >> 4);
            const uint32_t off = (ks >> 2) * kBoxBytes + row * 128 + ((chunk ^ (row & 7)) << 4);
#pragma unroll
            for (int j = 0; j < kB; ++j) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(slot[j] + off, a0, a1, a2, a3);
                mma16816((ks & 1) ? c1[j] : c0[j], a0, a1, a2, a3, qb[2 * ks], qb[2 * ks + 1]);
            }
        }
#pragma unroll
        for (int j = 0; j < kB; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i) s[j][i] = c0[j][i] + c1[j][i];
    }
    // scores: s0 = (tok gq, head 2tq), s1 = (gq, 2tq+1), s2/3 = tok gq+8
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < kB; ++j) {
        const int v = valid[j];
        s[j][0] = gq < v ? s[j][0] * scale_log2 : -INFINITY;
        s[j][1] = gq < v ? s[j][1] * scale_log2 : -INFINITY;
        s[j][2] = gq + 8 < v ? s[j][2] * scale_log2 : -INFINITY;
        s[j][3] = gq + 8 < v ? s[j][3] * scale_log2 : -INFINITY;
        mx0 = fmaxf(mx0, fmaxf(s[j][0], s[j][2]));
        mx1 = fmaxf(mx1, fmaxf(s[j][1], s[j][3]));
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(st.m0, mx0), mn1 = fmaxf(st.m1, mx1);
    const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
    const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = fast_exp2(st.m0 - mu0), al1 = fast_exp2(st.m1 - mu1);
    st.m0 = mn0;
    st.m1 = mn1;
    uint32_t pb0[kB], pb1[kB];
    float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
    for (int j = 0; j < kB; ++j) {
        const uint32_t px = pack_half2(fast_exp2(s[j][0] - mu0), fast_exp2(s[j][1] - mu1));
        const uint32_t py = pack_half2(fast_exp2(s[j][2] - mu0), fast_exp2(s[j][3] - mu1));
        // the sum takes the fp16 weights the MMA multiplies by
        const float2 fx = __half22float2(*reinterpret_cast<const __half2*>(&px));
        const float2 fy = __half22float2(*reinterpret_cast<const __half2*>(&py));
        ls0 += fx.x + fy.x;
        ls1 += fx.y + fy.y;
        // B fragments of P^T (token x head) by transposing in registers
        pb0[j] = movmatrix_t(px);
        pb1[j] = movmatrix_t(py);
    }
    st.l0 = st.l0 * al0 + ls0;
    st.l1 = st.l1 * al1 + ls1;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        st.o[i][0] *= al0;
        st.o[i][1] *= al1;
        st.o[i][2] *= al0;
        st.o[i][3] *= al1;
    }
    // O^T += V^T . P^T
    const int row = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        const int chunk = (mt & 3) * 2 + ((lane >> 3) & 1);
        const uint32_t off = kSlotV + (mt >> 2) * kBoxBytes + row * 128 + ((chunk ^ (row & 7)) << 4);
#pragma unroll
        for (int j = 0; j < kB; ++j) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(slot[j] + off, a0, a1, a2, a3);
            mma16816(st.o[mt], a0, a1, a2, a3, pb0[j], pb1[j]);
        }
    }
}

// Prepares a staged granule for attend: zeroes V rows past `valid` (they may
// hold anything, NaN included) and overwrites row patch_row with the new
// token (lanes 0-15 carry its K, lanes 16-31 its V, 16 bytes each).  Returns
// whether shared memory was written.
__device__ __forceinline__ bool prepare_granule(unsigned char* slot_ptr, int valid, int patch_row,
                                                const uint4& patch_val, int lane) {
    bool wrote = false;
    if (valid < kGranule) {
        uint4* v0 = reinterpret_cast<uint4*>(slot_ptr + kSlotV);
        for (int i = lane; i < (kGranule - valid) * 8; i += 32) {
            const int row = valid + (i >> 3);
            v0[row * 8 + (i & 7)] = make_uint4(0, 0, 0, 0);
            v0[kBoxBytes / 16 + row * 8 + (i & 7)] = make_uint4(0, 0, 0, 0);
        }
        wrote = true;
    }
    if (patch_row >= 0 && patch_row < valid) {
        const int c16 = lane & 15;  // 16-byte chunk of the 128 dims
        unsigned char* box = slot_ptr + (lane < 16 ? 0u : kSlotV) + (c16 >> 3) * kBoxBytes;
        *reinterpret_cast<uint4*>(box + patch_row * 128 + (((c16 & 7) ^ (patch_row & 7)) << 4)) =
            patch_val;
        wrote = true;
    }
    return wrote;
}

// FP8 pools: the producer lands a granule's E4M3 K box (16 tokens x 128
// bytes, 128-byte swizzle) at +0 and its V box at +2 KB of the slot; the
// owning warp widens both in place to the fp16 slot layout attend expects
// (exact: every E4M3 value is an fp16 value; the per-head scales are applied
// to the scores and to the output instead).  All of the warp's reads happen
// before any of its writes.
__device__ __forceinline__ void widen_fp8_slot(unsigned char* slot, int lane) {
    uint4 kc[4], vc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int i = lane + 32 * k, r = i >> 3, c = i & 7;
        const uint32_t off = r * 128 + ((c ^ (r & 7)) << 4);
        kc[k] = *reinterpret_cast<const uint4*>(slot + off);
        vc[k] = *reinterpret_cast<const uint4*>(slot + kBoxBytes + off);
    }
    __syncwarp();
    auto widen = [](uint32_t w, uint32_t& lo, uint32_t& hi) { widen4(w, lo, hi); };
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int i = lane + 32 * k, r = i >> 3, c = i & 7;
        // 16 dims 16c..16c+15: fp16 chunks 2(c%4), 2(c%4)+1 of box c/4
        const uint32_t j0 = (c & 3) * 2;
        const uint32_t b0 = (c >> 2) * kBoxBytes + r * 128;
        const uint32_t o0 = b0 + ((j0 ^ (r & 7)) << 4), o1 = b0 + (((j0 + 1) ^ (r & 7)) << 4);
        uint4 a, b;
        widen(kc[k].x, a.x, a.y);
        widen(kc[k].y, a.z, a.w);
        widen(kc[k].z, b.x, b.y);
        widen(kc[k].w, b.z, b.w);
        *reinterpret_cast<uint4*>(slot + o0) = a;
        *reinterpret_cast<uint4*>(slot + o1) = b;
        widen(vc[k].x, a.x, a.y);
        widen(vc[k].y, a.z, a.w);
        widen(vc[k].z, b.x, b.y);
        widen(vc[k].w, b.z, b.w);
        *reinterpret_cast<uint4*>(slot + kSlotV + o0) = a;
        *reinterpret_cast<uint4*>(slot + kSlotV + o1) = b;
    }
    __syncwarp();
}

// One batch of the log-sum-exp merge of P partial records (children j0 ..
// j0 + kMergeBatch - 1 of P, rec_floats apart) for head mh, dims md..md+3 and
// md+64..md+67, merged online: M is the running maximum of the children's m;
// when a batch raises it, what is summed so far is scaled by 2^(M_old - M),
// then L += 2^(m_j - M) l_j and o += 2^(m_j - M) o_j in child order, into two
// accumulator sets (even / odd j) added at the end.  The arithmetic is the
// same whether the records are read from shared or global memory, so the
// result never depends on which block merges.  The sixteen threads of a head
// read 256 contiguous bytes per load.
template <bool kGlobal>
__device__ __forceinline__ void merge_batch(const float* base, int j0, int P, int rec_floats, int mh,
                                            int md, float& M, float& Ls, float& Ls2, float* acc,
                                            float* acc2) {
    auto ld1 = [&](const float* a) { return kGlobal ? __ldcg(a) : *a; };
    auto ld4 = [&](const float* a) {
        return kGlobal ? __ldcg(reinterpret_cast<const float4*>(a)) : *reinterpret_cast<const float4*>(a);
    };
    float w[kMergeBatch], l[kMergeBatch];
    float4 x[kMergeBatch], y[kMergeBatch];
#pragma unroll
    for (int c = 0; c < kMergeBatch; ++c) {  // a batch's loads are in flight together
        if (j0 + c < P) {
            const float* cr = base + (int64_t)(j0 + c) * rec_floats;
            w[c] = ld1(cr + mh);
            l[c] = ld1(cr + 8 + mh);
            x[c] = ld4(cr + kRecHead + mh * kHeadDim + md);
            y[c] = ld4(cr + kRecHead + mh * kHeadDim + md + 64);
        } else {
            w[c] = -INFINITY;
            l[c] = 0.f;
            x[c] = y[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    float Mb = M;
#pragma unroll
    for (int c = 0; c < kMergeBatch; ++c) Mb = fmaxf(Mb, w[c]);
    if (Mb == -INFINITY) return;
    if (Mb > M) {
        const float sc = M == -INFINITY ? 0.f : fast_exp2(M - Mb);
        Ls *= sc;
        Ls2 *= sc;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            acc[i] *= sc;
            acc2[i] *= sc;
        }
        M = Mb;
    }
#pragma unroll
    for (int c = 0; c < kMergeBatch; c += 2) {
        const float wa = fast_exp2(w[c] - M), wb = fast_exp2(w[c + 1] - M);
        Ls += wa * l[c];
        Ls2 += wb * l[c + 1];
        acc[0] += wa * x[c].x; acc[1] += wa * x[c].y; acc[2] += wa * x[c].z; acc[3] += wa * x[c].w;
        acc[4] += wa * y[c].x; acc[5] += wa * y[c].y; acc[6] += wa * y[c].z; acc[7] += wa * y[c].w;
        acc2[0] += wb * x[c + 1].x; acc2[1] += wb * x[c + 1].y; acc2[2] += wb * x[c + 1].z;
        acc2[3] += wb * x[c + 1].w; acc2[4] += wb * y[c + 1].x; acc2[5] += wb * y[c + 1].y;
        acc2[6] += wb * y[c + 1].z; acc2[7] += wb * y[c + 1].w;
    }
}

// Burst plan for the block's range [g0, g1): its pieces (at most four) and
// the warps dealt to them.  Every piece gets one warp; each further warp goes
// to the piece whose busiest warp has the most granules, while that is more
// than one.  A piece's warps take near-equal contiguous shares of it.
__device__ void make_plan(Plan& pl, volatile int* flags, const int* sm_pre, const int* sm_len, int rows,
                          int hk, int g0, int g1, int W, int Geff) {
    pl.burst = 0;
    pl.npieces = 0;
    for (int w = 0; w < kConsumerWarps; ++w) pl.wpiece[w] = -1;
    if (g0 >= g1 || g1 - g0 > kRing) return;
    int lo = 0, hi = rows - 1;
    while (lo < hi) {  // largest row with sm_pre[row] <= g0
        const int mid = (lo + hi + 1) >> 1;
        if (sm_pre[mid] <= g0) lo = mid; else hi = mid - 1;
    }
    int r = lo, n = (sm_pre[r + 1] - sm_pre[r]) / hk;
    int kvh = (g0 - sm_pre[r]) / n, us = sm_pre[r] + kvh * n;
    int k = 0;
    for (int g = g0; g < g1;) {
        if (k == kBurstPieces) return;  // too many pieces: stream mode
        const int pend = min(g1, us + n);
        pl.r[k] = r;
        pl.kvh[k] = kvh;
        pl.ustart[k] = us;
        pl.n[k] = n;
        pl.cstart[k] = owner_of(us, W, Geff);
        pl.P[k] = owner_of(us + n - 1, W, Geff) - pl.cstart[k] + 1;
        pl.w0[k] = g;  // piece range [w0, wn) until the warps are dealt below
        pl.wn[k] = pend;
        ++k;
        g = pend;
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
    // wc counts the warps of each piece (registers: the loops are unrolled)
    int wc[kBurstPieces] = {1, 1, 1, 1};
#pragma unroll
    for (int e = 1; e < kConsumerWarps; ++e) {
        if (e < k) continue;
        int best = -1, bc = 1;
#pragma unroll
        for (int i = 0; i < kBurstPieces; ++i) {
            if (i >= k) break;
            const int c = (pl.wn[i] - pl.w0[i] + wc[i] - 1) / wc[i];
            if (c > bc) {
                bc = c;
                best = i;
            }
        }
#pragma unroll
        for (int i = 0; i < kBurstPieces; ++i)
            if (i == best) ++wc[i];
    }
    int w = 0;
#pragma unroll
    for (int i = 0; i < kBurstPieces; ++i) {
        if (i >= k) break;
        const int a = pl.w0[i], len = pl.wn[i] - a;
        pl.w0[i] = w;
        pl.wn[i] = wc[i];
        for (int j = 0; j < wc[i]; ++j, ++w) {
            pl.wpiece[w] = i;
            pl.wa[w] = a + j * len / wc[i];
            pl.wb[w] = a + (j + 1) * len / wc[i];
        }
    }
    for (; w < kConsumerWarps; ++w) pl.wpiece[w] = -1;
    pl.npieces = k;
    pl.burst = 1;
    // the split pieces, recorded now for the tail (their unit, first block,
    // pieces, row, head)
    int ks = 0;
    for (int i = 0; i < k; ++i) {
        if (pl.P[i] == 1) continue;
        flags[4 + 5 * ks] = pl.r[i] * hk + pl.kvh[i];
        flags[5 + 5 * ks] = pl.cstart[i];
        flags[6 + 5 * ks] = pl.P[i];
        flags[7 + 5 * ks] = pl.r[i];
        flags[8 + 5 * ks] = pl.kvh[i];
        ++ks;
    }
    flags[3] = ks;
}

// Per-row work of block cta, done by its producer warp after the dependency
// wait (off the consumers' critical path): rows cta, cta + G, ... with nothing
// to read get zero outputs, and in the fused form their new token is stored
// into its slot (as E4M3 codes for FP8 pools, quantised exactly as
// paged_kv_append_fp8 does).  The block that stages the slot's granule takes
// the token from k_new / v_new directly, so the order of this store and that
// copy does not matter.
template <bool kFp8>
__device__ void row_work(const Params& p, const int* sm_pre, int cta, int G, int lane) {
    for (int r = cta; r < p.rows; r += G) {
        if (sm_pre[r + 1] == sm_pre[r])
            for (int i = lane; i < p.hq * kHeadDim / 8; i += 32)
                reinterpret_cast<uint4*>(p.out + (int64_t)r * p.hq * kHeadDim)[i] = make_uint4(0, 0, 0, 0);
        if (!p.positions) continue;
        const int pos = p.positions[r];
        if (pos < 0) continue;
        const int lb = pos / p.bs;
        if (lb >= p.mbpr) {
            if (lane == 0) flag_error(p.dev_err, PKV_DEV_ERR_POSITION);
            continue;
        }
        const int pb = p.tables[(int64_t)r * p.mbpr + lb];
        if (pb < 0 || pb >= p.nb) {
            if (lane == 0) flag_error(p.dev_err, PKV_DEV_ERR_BLOCK_ID);
            continue;
        }
        const int vecs = p.hk * kHeadDim / 8;  // 8-element vectors per token and pool
        const int64_t dst = ((int64_t)pb * p.bs + pos % p.bs) * vecs;
        for (int i = lane; i < 2 * vecs; i += 32) {
            const bool is_v = i >= vecs;
            const int j = is_v ? i - vecs : i;
            const uint4 x = reinterpret_cast<const uint4*>(is_v ? p.v_new : p.k_new)[(int64_t)r * vecs + j];
            if (kFp8) {
                const float sc = (is_v ? p.v_scale : p.k_scale)[j / (kHeadDim / 8)];
                reinterpret_cast<uint2*>(is_v ? p.vpool : p.kpool)[dst + j] = quantize8(x, sc);
            } else {
                reinterpret_cast<uint4*>(is_v ? p.vpool : p.kpool)[dst + j] = x;
            }
        }
    }
}

template <bool kPaged, bool kFp8>
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
    const uint32_t bar_slot = bar_full + 2 * kStages * 8;
    const uint32_t bar_merge = bar_slot + kRing * 8;
    int* sm_ppos = reinterpret_cast<int*>(smem + Smem::ppos);
    TileDesc* sm_desc = reinterpret_cast<TileDesc*>(smem + Smem::desc);
    Plan* sm_plan = reinterpret_cast<Plan*>(smem + Smem::plan);
    volatile int* sm_flags = reinterpret_cast<volatile int*>(smem + Smem::flags);
    int* sm_part = reinterpret_cast<int*>(smem + Smem::part);
    int* sm_pre = reinterpret_cast<int*>(smem + Smem::prefix);
    int* sm_len = reinterpret_cast<int*>(smem + Smem::lens(p.rows));
    float* sm_ks = reinterpret_cast<float*>(smem + Smem::scales);  // FP8 only
    float* sm_vs = sm_ks + kFp8MaxKvHeads;
    // bytes the producer lands per granule
    constexpr uint32_t kGranuleLoad = kFp8 ? 2 * kBoxBytes : kSlotBytes;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int G = gridDim.x;  // blocks launched; the partition uses Geff <= G
    const int cta = blockIdx.x;
    const int hk = p.hk;
    const int rows = p.rows;


    if (warp == kConsumerWarps && lane == 0) {
        // fetch the tensor-map descriptors now; the first copy would wait for them
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kmap)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&vmap)) : "memory");
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kConsumerWarps);
        }
        for (int s = 0; s < kRing; ++s) mbar_init(bar_slot + 8 * s, 1);
        for (int b = 0; b < kMergeBars; ++b) mbar_init(bar_merge + 8 * b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        sm_flags[0] = 0;  // abort
        sm_flags[3] = 0;  // split pieces recorded ([4..13]: their unit, first block, pieces, row, head)
    }
    if (kFp8 && tid < 2 * p.hk) sm_ks[tid < p.hk ? tid : kFp8MaxKvHeads + tid - p.hk] =
        tid < p.hk ? p.k_scale[tid] : p.v_scale[tid - p.hk];

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
        if (g0 >= g1) {
            griddep_wait();
            if (kPaged) row_work<kFp8>(p, sm_pre, cta, G, lane);
            return;
        }
        // Burst mode when the range fits the ring and covers at most
        // kBurstPieces units (the consumers' plan, made concurrently, takes
        // the same decision).
        bool burst = false;
        if (g1 - g0 <= kRing) {
            int u = -1;
            if (lane < g1 - g0) {
                const int gg = g0 + lane;
                int lo = 0, hi = rows - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (sm_pre[mid] <= gg) lo = mid; else hi = mid - 1;
                }
                const int n = (sm_pre[lo + 1] - sm_pre[lo]) / hk;
                u = lo * hk + (gg - sm_pre[lo]) / n;
            }
            const int up = __shfl_up_sync(0xffffffffu, u, 1);
            const int pieces = __popc(__ballot_sync(0xffffffffu, u >= 0 && (lane == 0 || u != up)));
            burst = pieces <= kBurstPieces;
        }
        if (burst) {
            // Every granule of the range goes to its own slot now, before the
            // dependency wait; lane j handles granule g0 + j.
            const int ng = g1 - g0;
            if (lane < ng) {
                const int gg = g0 + lane;
                int lo = 0, hi = rows - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (sm_pre[mid] <= gg) lo = mid; else hi = mid - 1;
                }
                const int r = lo;
                const int n = (sm_pre[r + 1] - sm_pre[r]) / hk;
                const int kvh = (gg - sm_pre[r]) / n;
                const int tok = (gg - sm_pre[r] - kvh * n) * kGranule;
                int valid = min(kGranule, sm_len[r] - tok);
                if (valid < 0) valid = 0;
                bool issue = false;
                int zrow = 0;
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
                sm_plan->valid[lane] = valid;
                const uint32_t fb = bar_slot + 8 * lane;
                mbar_arrive_expect_tx(fb, issue ? kGranuleLoad : 0u);
                if (issue) {
                    const uint32_t dst = sbase + Smem::ring + lane * kSlotBytes;
                    if (kFp8) {
                        tma_load_3d(dst, &kmap, 0, kvh, zrow, fb);
                        tma_load_3d(dst + kBoxBytes, &vmap, 0, kvh, zrow, fb);
                    } else {
                        tma_load_3d(dst, &kmap, 0, kvh, zrow, fb);
                        tma_load_3d(dst + kBoxBytes, &kmap, 64, kvh, zrow, fb);
                        tma_load_3d(dst + kSlotV, &vmap, 0, kvh, zrow, fb);
                        tma_load_3d(dst + kSlotV + kBoxBytes, &vmap, 64, kvh, zrow, fb);
                    }
                }
            }
            griddep_wait();
            if (kPaged) row_work<kFp8>(p, sm_pre, cta, G, lane);
            // Drain: every copy lands before the block exits.
            for (int j = 0; j < ng; ++j)
                if (!mbar_wait(bar_slot + 8 * j, 0) && lane == 0) flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
            return;
        }
        int tile = 0;
        bool waited = false;
        bool aborted = false;
        const uint32_t qbytes = (uint32_t)p.group * 256u;
        // Stages armed before the dependency wait get their query copies
        // after it (the query may be written by the preceding kernel).
        auto wait_and_flush = [&]() {
            if (waited) return;
            griddep_wait();
            waited = true;
            if (lane == 0)
                for (int t = 0; t < tile && t < kStages; ++t) {
                    const TileDesc* d = sm_desc + t;
                    if (d->flags & kFirst)
                        bulk_load(sbase + Smem::q + t * kQBytes,
                                  p.q + ((int64_t)d->r * p.hq + d->kvh * p.group) * kHeadDim, qbytes,
                                  bar_full + 8 * t);
                }
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
                if (lane == 0) mbar_arrive_expect_tx(fb, nissue * kGranuleLoad + (first ? qbytes : 0u));
                __syncwarp();
                if (mine && issue) {
                    const uint32_t dst =
                        sbase + Smem::ring + (s * kTileGranules + lane - j) * kSlotBytes;
                    if (kFp8) {
                        tma_load_3d(dst, &kmap, 0, kvh, zrow, fb);
                        tma_load_3d(dst + kBoxBytes, &vmap, 0, kvh, zrow, fb);
                    } else {
                        tma_load_3d(dst, &kmap, 0, kvh, zrow, fb);
                        tma_load_3d(dst + kBoxBytes, &kmap, 64, kvh, zrow, fb);
                        tma_load_3d(dst + kSlotV, &vmap, 0, kvh, zrow, fb);
                        tma_load_3d(dst + kSlotV + kBoxBytes, &vmap, 64, kvh, zrow, fb);
                    }
                }
                if (first && lane == 0 && waited)
                    bulk_load(sbase + Smem::q + s * kQBytes,
                              p.q + ((int64_t)r_j * p.hq + kvh_j * p.group) * kHeadDim, qbytes, fb);
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
        if (kPaged) row_work<kFp8>(p, sm_pre, cta, G, lane);
        // Drain: the copies of every armed stage land before the block exits.
        for (int t = tile - kStages; t < tile; ++t) {
            if (t < 0) continue;
            if (!mbar_wait(bar_full + 8 * (t % kStages), (uint32_t)(t / kStages) & 1) && lane == 0)
                flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
        }
        return;
    }

    // ============================== consumers ==============================
    if (tid == 0) make_plan(*sm_plan, sm_flags, sm_pre, sm_len, rows, hk, g0, g1, W, Geff);
    consumer_sync();
    const bool burst = sm_plan->burst != 0;
    if (burst && sm_plan->wpiece[warp] >= 0) {
        // Warm L2 with this warp's query rows and new token.  A prefetch reads
        // nothing into the block, so it may precede the dependency wait: the
        // values used are loaded after it.
        const int pi = sm_plan->wpiece[warp];
        const int r = sm_plan->r[pi], kvh = sm_plan->kvh[pi];
        const char* qrow = reinterpret_cast<const char*>(p.q + ((int64_t)r * p.hq + kvh * p.group) * kHeadDim);
        if (lane < 2 * p.group)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(qrow + lane * 128));
        if (kPaged && p.positions && lane < 8) {
            const char* nt = reinterpret_cast<const char*>(
                (lane < 4 ? p.k_new : p.v_new) + ((int64_t)r * hk + kvh) * kHeadDim);
            asm volatile("prefetch.global.L2 [%0];" ::"l"(nt + (lane & 3) * 64));
        }
        if (kPaged && p.positions && lane == 8)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(p.positions + r));
    }
    // Everything below may read what the preceding kernel wrote (query,
    // positions, new tokens, workspace) or write what it reads.
    griddep_wait();

    if (g0 >= g1) return;

    const bool fused = kPaged && p.positions != nullptr;
    const int gq = lane >> 2;  // MMA group id: token row (QK) / dim row (PV) / head (B frag)
    const int tq = lane & 3;   // thread in group

    if (burst) {
        // ============================ burst mode ============================
        const Plan& pl = *sm_plan;
        const int pi = pl.wpiece[warp];
        if (pi >= 0) {
            const int r = pl.r[pi], kvh = pl.kvh[pi], us = pl.ustart[pi];
            const int a = pl.wa[warp], b = pl.wb[warp];
            // Query fragments straight from global memory: b0 = Q[head gq][16ks + 2tq..],
            // b1 = Q[head gq][16ks + 8 + 2tq..].
            uint32_t qb[16];
            {
                const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
                    p.q + ((int64_t)r * p.hq + kvh * p.group + gq) * kHeadDim);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    qb[2 * ks] = gq < p.group ? qrow[ks * 8 + tq] : 0u;
                    qb[2 * ks + 1] = gq < p.group ? qrow[ks * 8 + 4 + tq] : 0u;
                }
            }
            // The appended token, if it falls inside this warp's granules, is
            // taken from k_new / v_new (its slot may be written concurrently).
            int patch_tok = -1;
            uint4 patch_val = make_uint4(0, 0, 0, 0);
            if (fused) {
                const uint4* src = reinterpret_cast<const uint4*>(
                    (lane < 16 ? p.k_new : p.v_new) + ((int64_t)r * hk + kvh) * kHeadDim);
                patch_val = src[lane & 15];
                // FP8 pools hold the token as codes: take their exact fp16 values
                if (kFp8) patch_val = widen8(quantize8(patch_val, lane < 16 ? sm_ks[kvh] : sm_vs[kvh]));
                const int pos = p.positions[r];
                if (pos >= 0 && us + pos / kGranule >= a && us + pos / kGranule < b) patch_tok = pos;
            }
            Soft st;
            st.reset();
            bool ok = true;
            for (int bs = a; bs < b && ok; bs += kBatch) {
                const int nb = min(kBatch, b - bs);
                uint32_t slot[kBatch];
                int valid[kBatch];
                bool wrote = false;
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    slot[j] = sbase;
                    valid[j] = 0;
                    if (j >= nb || !ok) continue;
                    const int si = bs + j - g0;
                    if (!mbar_wait(bar_slot + 8 * si, 0)) {
                        if (lane == 0) {
                            sm_flags[0] = 1;
                            flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
                        }
                        ok = false;
                        continue;
                    }
                    slot[j] = sbase + Smem::ring + si * kSlotBytes;
                    valid[j] = pl.valid[si];
                    const int gtok = (bs + j - us) * kGranule;
                    if (kFp8) {
                        widen_fp8_slot(smem + Smem::ring + si * kSlotBytes, lane);
                        wrote = true;
                    }
                    wrote |= prepare_granule(smem + Smem::ring + si * kSlotBytes, valid[j],
                                             patch_tok >= 0 ? patch_tok - gtok : -1, patch_val, lane);
                }
                if (!ok) break;
                if (wrote) __syncwarp();
                const float sl2 = kFp8 ? p.scale_log2 * sm_ks[kvh] : p.scale_log2;
                attend<1>(st, qb, slot, valid, sl2, lane);
            }
            // Dump the warp's state into its first slot: m[8], l[8], o[8][132].
            __syncwarp();
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, off);
                st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, off);
            }
            float* dump = reinterpret_cast<float*>(smem + Smem::ring + (a - g0) * kSlotBytes);
            if (gq == 0) {
                dump[2 * tq] = st.m0;
                dump[2 * tq + 1] = st.m1;
                dump[8 + 2 * tq] = st.l0;
                dump[8 + 2 * tq + 1] = st.l1;
            }
            float* o0 = dump + kRecHead;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const int dim = mt * 16 + gq;
                o0[(2 * tq) * kDumpStride + dim] = st.o[mt][0];
                o0[(2 * tq + 1) * kDumpStride + dim] = st.o[mt][1];
                o0[(2 * tq) * kDumpStride + dim + 8] = st.o[mt][2];
                o0[(2 * tq + 1) * kDumpStride + dim + 8] = st.o[mt][3];
            }
        }
        consumer_sync();
        // The next kernel in the stream (launched with programmatic
        // serialization) may start now that this block's queries have
        // arrived: its prefetch then no longer competes with them.  It waits
        // for this grid before touching anything this grid writes.
        if (tid == 0) griddep_launch();
        if (sm_flags[0]) return;
        // Combine every piece's warp states.  Thread (head h, dims 8c..8c+7)
        // reads all four warps' states at once, then finishes each piece.
        {
            const int gsz = p.group;
            const int h = tid >> 4, c = tid & 15;
            float mw[kConsumerWarps], lw[kConsumerWarps];
            float4 xw[kConsumerWarps], yw[kConsumerWarps];
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                mw[w] = -INFINITY;
                lw[w] = 0.f;
                xw[w] = yw[w] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (pl.wpiece[w] >= 0 && h < gsz) {
                    const float* dw = reinterpret_cast<const float*>(smem + Smem::ring +
                                                                     (pl.wa[w] - g0) * kSlotBytes);
                    mw[w] = dw[h];
                    lw[w] = dw[8 + h];
                    xw[w] = *reinterpret_cast<const float4*>(dw + kRecHead + h * kDumpStride + 8 * c);
                    yw[w] = *reinterpret_cast<const float4*>(dw + kRecHead + h * kDumpStride + 8 * c + 4);
                }
            }
            int pw0[kBurstPieces], pwn[kBurstPieces], pr[kBurstPieces], pkv[kBurstPieces], pP[kBurstPieces];
#pragma unroll
            for (int pc = 0; pc < kBurstPieces; ++pc) {
                pw0[pc] = pl.w0[pc];
                pwn[pc] = pl.wn[pc];
                pr[pc] = pl.r[pc];
                pkv[pc] = pl.kvh[pc];
                pP[pc] = pl.P[pc];
            }
            const int npc = h < gsz ? pl.npieces : 0;
#pragma unroll
            for (int pc = 0; pc < kBurstPieces; ++pc) {
                if (pc >= npc) break;
                const int w0 = pw0[pc], w1 = w0 + pwn[pc];
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w)
                    if (w >= w0 && w < w1) M = fmaxf(M, mw[w]);
                float L = 0.f, acc[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) {
                    if (w < w0 || w >= w1) continue;
                    const float wt = M == -INFINITY ? 0.f : fast_exp2(mw[w] - M);
                    L += wt * lw[w];
                    acc[0] += wt * xw[w].x; acc[1] += wt * xw[w].y; acc[2] += wt * xw[w].z; acc[3] += wt * xw[w].w;
                    acc[4] += wt * yw[w].x; acc[5] += wt * yw[w].y; acc[6] += wt * yw[w].z; acc[7] += wt * yw[w].w;
                }
                const int r = pr[pc], kvh = pkv[pc];
                if (pP[pc] == 1) {
                    const float inv = L > 0.f ? __fdividef(kFp8 ? sm_vs[kvh] : 1.f, L) : 0.f;
                    uint4 pk;
                    pk.x = pack_half2(acc[0] * inv, acc[1] * inv);
                    pk.y = pack_half2(acc[2] * inv, acc[3] * inv);
                    pk.z = pack_half2(acc[4] * inv, acc[5] * inv);
                    pk.w = pack_half2(acc[6] * inv, acc[7] * inv);
                    *reinterpret_cast<uint4*>(p.out + ((int64_t)r * p.hq + kvh * gsz + h) * kHeadDim + 8 * c) = pk;
                } else {
                    float* rec = p.records + (int64_t)(cta + r * hk + kvh) * p.rec_floats;
                    if (c == 0) {
                        rec[h] = M;
                        rec[8 + h] = L;
                    }
                    *reinterpret_cast<float4*>(rec + kRecHead + h * kHeadDim + 8 * c) =
                        make_float4(acc[0], acc[1], acc[2], acc[3]);
                    *reinterpret_cast<float4*>(rec + kRecHead + h * kHeadDim + 8 * c + 4) =
                        make_float4(acc[4], acc[5], acc[6], acc[7]);
                }
            }
        }
    } else {
        // ============================ stream mode ============================
        // Append positions of this block's first pieces, read once right after
        // the wait, so a piece never starts with a dependent global load.
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

        uint32_t qb[16];
        Soft st;
        st.reset();
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
            if (flags & kFirst) {
                // B fragments of Q^T: b0 = Q[head gq][16ks + 2tq..], b1 = Q[head gq][16ks + 8 + 2tq..]
                const uint32_t* qrow =
                    reinterpret_cast<const uint32_t*>(smem + Smem::q + s * kQBytes + gq * 256);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    qb[2 * ks] = gq < p.group ? qrow[ks * 8 + tq] : 0u;
                    qb[2 * ks + 1] = gq < p.group ? qrow[ks * 8 + 4 + tq] : 0u;
                }
                st.reset();
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
                        if (kFp8) patch_val = widen8(quantize8(patch_val, lane < 16 ? sm_ks[kvh] : sm_vs[kvh]));
                    }
                }
            }
            if (warp < ng) {
                const int gtok = tok0 + warp * kGranule;  // unit-local token of this granule
                const int si = s * kTileGranules + warp;
                if (kFp8) widen_fp8_slot(smem + Smem::ring + si * kSlotBytes, lane);
                const bool wrote = kFp8 | prepare_granule(smem + Smem::ring + si * kSlotBytes, valid,
                                                   patch_tok >= 0 ? patch_tok - gtok : -1, patch_val, lane);
                if (wrote) __syncwarp();
                const uint32_t slot[1] = {sbase + Smem::ring + si * kSlotBytes};
                const int vv[1] = {valid};
                attend<1>(st, qb, slot, vv, kFp8 ? p.scale_log2 * sm_ks[kvh] : p.scale_log2, lane);
                // Generic-proxy writes must be ordered before TMA reuses the slot.
                if (wrote) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * s);
            if (tile == 0 && tid == 0) griddep_launch();  // as in burst mode
            ++tile;
            if (!(flags & kLast)) continue;

            // ---- end of a piece: combine the four warps' partial softmax states ----
            float l0 = st.l0, l1 = st.l1;
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, off);
                l1 += __shfl_xor_sync(0xffffffffu, l1, off);
            }
            if (gq == 0) {
                sm_m[warp * 8 + 2 * tq] = st.m0;
                sm_m[warp * 8 + 2 * tq + 1] = st.m1;
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
            const float inv = Lh > 0.f ? __fdividef(kFp8 ? sm_vs[kvh] : 1.f, Lh) : 0.f;
            const int cq = (tid & 15) * 4;  // four dims within a 64-dim pass
#pragma unroll
            for (int pass = 0; pass < 2; ++pass) {
                // warp writes its O^T fragments for dims [64 pass, 64 pass + 64)
                float* base = sm_comb + warp * 8 * kCombStride;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int mt = 4 * pass + k;
                    base[(2 * tq) * kCombStride + 16 * k + gq] = st.o[mt][0];
                    base[(2 * tq + 1) * kCombStride + 16 * k + gq] = st.o[mt][1];
                    base[(2 * tq) * kCombStride + 16 * k + gq + 8] = st.o[mt][2];
                    base[(2 * tq + 1) * kCombStride + 16 * k + gq + 8] = st.o[mt][3];
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
    }

    // ---- split pieces.  Every piece publishes its record and counts itself
    // on the unit's counter with a release.  The block holding the unit's
    // last piece waits (bounded) until all P pieces have counted, lands their
    // records and combines them through their log-sum-exp, then re-arms the
    // counter.  A block merges at most one unit: the one whose end is its
    // first piece.  (Splitting a long unit's merge over several blocks, one
    // query head each, measured slower.) ----
    // Shared memory written through the generic proxy (partials, patches) is
    // ordered before the bulk copies that may land records over it, and the
    // records written here before the bulk copies that may read them back.
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("fence.proxy.async.global;" ::: "memory");
    consumer_sync();
    const int nsplit = sm_flags[3];
    if (nsplit == 0 || sm_flags[0]) return;
    if (tid < nsplit) {
        // The barrier above orders every thread's record stores before this
        // thread's release.
        const int u = sm_flags[4 + 5 * tid];
        const int cs = sm_flags[5 + 5 * tid];
        const int P = sm_flags[6 + 5 * tid];
        int* ctr = p.counters + (int64_t)u * kCounterStride;
        asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(ctr) : "memory");
        int merge = 0;
        if (cta == cs + P - 1) {
            // the acquire makes every piece's record visible to this block
            // after the next barrier
            int seen = 0;
            for (uint32_t i = 0; i < kPollLimit; ++i) {
                asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(seen) : "l"(ctr) : "memory");
                if (seen >= P) break;
                __nanosleep(32);
            }
            if (seen >= P) {
                *ctr = 0;  // every piece has arrived: re-arm for the next call
                merge = 1;
            } else {
                sm_flags[0] = 1;
                flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
            }
        }
        sm_flags[14 + tid] = merge;
    }
    consumer_sync();
    if (sm_flags[0]) return;
    int job = -1;
    for (int k = 0; k < nsplit; ++k)
        if (sm_flags[14 + k]) job = k;
    if (job < 0) return;
    const int u = sm_flags[4 + 5 * job], cs = sm_flags[5 + 5 * job], P = sm_flags[6 + 5 * job];
    const int r = sm_flags[7 + 5 * job], kvh = sm_flags[8 + 5 * job];
    const float vs = kFp8 ? sm_vs[kvh] : 1.f;
    const uint32_t rec_bytes = (uint32_t)p.rec_floats * 4u;
    // The ring is idle once the block's granules are consumed: the records
    // land there by bulk copies issued at once, in batches of kMergeBatch
    // with a barrier each, and each batch is merged as soon as it has landed.
    // A unit with more records than the ring or the barriers take is merged
    // from the workspace directly.
    const bool landing =
        P <= kLandMax && (uint32_t)P * rec_bytes <= (uint32_t)(kRing * kSlotBytes);
    if (landing && warp == 0) {
        // a unit's records sit in consecutive workspace slots: one copy per batch
        const int nbat = (P + kMergeBatch - 1) / kMergeBatch;
        if (lane < nbat) {
            const uint32_t bytes = (uint32_t)min(kMergeBatch, P - lane * kMergeBatch) * rec_bytes;
            mbar_arrive_expect_tx(bar_merge + 8 * lane, bytes);
            bulk_load(sbase + Smem::ring + lane * kMergeBatch * rec_bytes,
                      p.records + (int64_t)(cs + u + lane * kMergeBatch) * p.rec_floats, bytes,
                      bar_merge + 8 * lane);
        }
    }
    const int mh = tid >> 4;        // head
    const int md = (tid & 15) * 4;  // dims md..md+3 and md+64..md+67
    const bool mine = mh < p.group;
    float M = -INFINITY, Ls = 0.f, Ls2 = 0.f, acc[8], acc2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = acc2[i] = 0.f;
    for (int j0 = 0; j0 < P; j0 += kMergeBatch) {
        if (landing) {
            if (!mbar_wait(bar_merge + 8 * (j0 / kMergeBatch), 0)) {
                if (lane == 0) flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
                return;
            }
            if (mine)
                merge_batch<false>(reinterpret_cast<const float*>(smem + Smem::ring), j0, P,
                                   p.rec_floats, mh, md, M, Ls, Ls2, acc, acc2);
        } else if (mine) {
            merge_batch<true>(p.records + (int64_t)(cs + u) * p.rec_floats, j0, P, p.rec_floats, mh,
                              md, M, Ls, Ls2, acc, acc2);
        }
    }
    if (mine) {
        const float L = Ls + Ls2;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += acc2[i];
        const float iv = L > 0.f ? __fdividef(vs, L) : 0.f;
        __half* orow = p.out + ((int64_t)r * p.hq + kvh * p.group + mh) * kHeadDim;
        *reinterpret_cast<uint2*>(orow + md) =
            make_uint2(pack_half2(acc[0] * iv, acc[1] * iv), pack_half2(acc[2] * iv, acc[3] * iv));
        *reinterpret_cast<uint2*>(orow + md + 64) =
            make_uint2(pack_half2(acc[4] * iv, acc[5] * iv), pack_half2(acc[6] * iv, acc[7] * iv));
    }
}

// ---------------------------------------------------------------------------
// Host side

// Tensor map over a pool viewed as [rows][hk][128] elements, 128-byte swizzle:
// fp16, box 64 dims x 1 head x 16 tokens; FP8 (bytes), box 128 dims x 1 head
// x 16 tokens.  Either way a box row is 128 bytes.
static int pool_map(const void* base, int64_t rows, int hk, bool fp8, CUtensorMap* out) {
    const int64_t esize = fp8 ? 1 : 2;
    const int64_t dims[3] = {kHeadDim, hk, rows};
    const int64_t strides[2] = {kHeadDim * esize, hk * kHeadDim * esize};
    const int box[3] = {fp8 ? 128 : 64, 1, kGranule};
    return tiled_map_3d(base, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        dims, strides, box, out);
}

struct DeviceInfo {
    int sms = 0;
    bool attr_set[3] = {false, false, false};
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
    // one counter per 128-byte line: arrivals on different units never
    // queue on the same L2 line
    return align_up((size_t)tma::kCounterStride * sizeof(int) * (size_t)rows * (size_t)kv_heads, 256);
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
                      cudaStream_t stream, const AppendArgs* append, bool pdl,
                      const float* k_scale, const float* v_scale) {
    using namespace tma;
    const bool paged = width == 0;
    const bool fp8 = k_scale != nullptr;
    if (fp8 && (!paged || !v_scale || kv_heads > kFp8MaxKvHeads)) return PKV_ERR_UNSUPPORTED;
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
    if ((st = pool_map(k_base, pool_rows, kv_heads, fp8, &km)) != PKV_OK) return st;
    if ((st = pool_map(v_base, pool_rows, kv_heads, fp8, &vm)) != PKV_OK) return st;

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

    prm.k_scale = k_scale;
    prm.v_scale = v_scale;

    const uint32_t smem = Smem::total(rows);
    const int which = fp8 ? 2 : paged ? 0 : 1;
    auto kernel = fp8 ? decode_tma_kernel<true, true>
                      : paged ? decode_tma_kernel<true, false> : decode_tma_kernel<false, false>;
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
