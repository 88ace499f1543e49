// Paged decode attention for sm_103a: asynchronously staged, tensor-core, stream-K.
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
// The host never reads device lengths: the split of a step (each block's
// range, pieces, warp shares and the physical rows of its granules) is a
// plan, made on the device from seq_lens and the block tables, either by
// each block in its prologue or once per step by paged_attention_plan for
// all the layers of the step.  The part of a unit inside one block is a
// piece.
//
// Block layout.  Warps 0-6 consume; warp 7 does the block's row work (the
// fused append) after the dependency wait.  Two modes, chosen per block:
//   * burst: the block's whole range fits the ring of twelve 8 KB granule
//     slots and covers at most four pieces.  The seven consumer warps are
//     dealt to pieces in proportion to their size; before the dependency
//     wait each stages its own granules, each then attends to its granules,
//     and the warps of a piece combine their states.
//   * stream: warps 0-3 each stream an equal contiguous share of the range
//     through three slots of their own, two granules' copies in flight; a
//     unit wholly inside one share is finished by its warp, the others are
//     combined by the warps holding their states once every share is done.
// Granules are staged with 16-byte cp.async copies (rows past the length
// zero-filled) in the 128-byte-swizzled layout of a tiled copy.  Plain
// asynchronous copies are used because, in a grid launched with programmatic
// stream serialization, tiled bulk copies issued before the dependency wait
// complete only after the preceding grid has completed, while cp.async
// proceeds at once; and because a single thread's tiled copies issue at a
// lower rate than a warp's cp.async.
// Per granule (16 tokens) and group of query heads (up to 8):
//   S^T[16 tok][8 heads] = K[16 tok][128] . Q^T        (mma.sync m16n8k16)
//   online softmax per head in fp32, base-2 exponent
//   O^T[128][8 heads]   += V^T[128][16 tok] . P^T      (P transposed in
//                                                       registers by movmatrix)
// The grouped query heads are the MMA's N = 8 columns, so every K and V byte
// is read once and feeds all heads of its group.
//
// A warp's softmax state is kept, dumped and published in the MMA fragment
// layout: per lane the running max and sum of heads 2t, 2t+1 (t = lane % 4)
// and eight float4 chunks, chunk c holding O^T rows 16c + lane/4 and
// 16c + 8 + lane/4 of those heads.  Chunk c of all lanes (512 bytes) is the
// output's dims 16c..16c+15 for every head of the group.
//
// Split units.  A unit with pieces in P > 1 blocks is merged in slices: the
// unit's first K = min(P, 8) pieces are its participants, participant k
// merging the chunks c with c % K == k.  Every piece writes its combined
// state as a record into the unit's region of the workspace (chunk-major
// over the unit's pieces, so a participant's slice of all P records is
// contiguous), each float stored as the complement of its bits so that a
// zero word means "not yet written".  A participant polls (bounded) its
// slice of the P records, merges them through their log-sum-exp in piece
// order, so the result never depends on timing, and clears the words it
// read.
//
// Safety: table entries are range-checked before any copy is issued (a bad
// entry is skipped and flagged); every record poll is bounded, and a poll
// that runs out sets PKV_DEV_ERR_TIMEOUT and stops the block (its copies have
// all landed by then).
#include <cuda.h>

#include <mutex>

#include "fp8_codec.cuh"
#include "pkv_internal.cuh"
#include "ptx.cuh"

namespace pkv {
namespace tma {

constexpr int kGranule = 16;        // tokens per box and per consumer warp step
constexpr int kRing = 12;           // granule slots
constexpr int kConsumerWarps = 7;   // burst mode
constexpr int kStreamWarps = 4;     // stream mode: warps 0-3 stream, each through three slots
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kMaxCtas = 1024;
constexpr int kMaxRows = 1024;
constexpr int kBurstPieces = 4;
constexpr int kMaxTasks = 2;   // split pieces of a block: its first and its last
constexpr int kMergeWays = 8;  // most participants of a split unit's merge
constexpr uint32_t kPollLimit = 1u << 22;  // polls of a record batch (well over a second)
constexpr uint32_t kBoxBytes = kGranule * 128;   // 16 rows x 128 B (64 dims)
constexpr uint32_t kSlotBytes = 4 * kBoxBytes;   // K dims 0-63, K 64-127, V 0-63, V 64-127
constexpr uint32_t kSlotV = 2 * kBoxBytes;
constexpr uint32_t kChunkBytes = 512;            // one chunk of a state: 32 lanes x float4
constexpr uint32_t kMlBytes = 64;                // m[8], l[8]
constexpr uint32_t kStateBytes = kMlBytes + 8 * kChunkBytes;  // a dumped state
constexpr uint32_t kLandBytes = kRing * kSlotBytes / kMaxTasks;  // merge partials per task
constexpr int kModeIdle = 0, kModeBurst = 1, kModeStream = 2;
constexpr uint32_t kPlanBytes = 512;             // one block's plan
constexpr int kPlanThreads = 1024;               // threads of the plan kernel
constexpr int kFp8MaxKvHeads = 16;                // FP8 pools: per-head scales kept in shared memory
constexpr float kLog2e = 1.4426950408889634f;

// named barriers (0 is __syncthreads)
constexpr int kBarConsumers = 1;  // burst: the seven consumer warps
constexpr int kBarStream = 2;     // stream: warps 0-3
constexpr int kBarPiece = 4;      // burst: 4 + piece, the piece's warps
constexpr int kBarMerge = 8;      // 8 + task, the task's warps

static_assert(kSlotBytes % 1024 == 0, "slots must keep 1024-byte alignment for 128B swizzle");
static_assert(kStateBytes <= kSlotBytes, "a dumped state fits one slot");

struct Params {
    __half* out;
    const __half* q;
    const int32_t* tables;
    const int32_t* seq_lens;
    int rows, hq, hk, group, bs, mbpr, nb;
    int limit;      // largest valid seq_len (paged); width (padded)
    int width;      // padded comparator: columns per row (0 = paged)
    float scale_log2;
    uint32_t poll_limit;  // polls of a record batch before a merge gives up
    const uint32_t* stuck;  // test hook: a word every merge poll also waits on (null: none)
    const unsigned char* plan;  // [grid][kPlanBytes] step plan, or null: each block makes its own
    unsigned char* records;  // unit regions of split-piece records (zero between calls)
    int32_t* dev_err;
    // fused append (all null when the kernel only decodes)
    const int32_t* positions;
    const __half* k_new;
    const __half* v_new;
    __half* kpool;
    __half* vpool;
    // pools (or padded slabs) as the consumers' plain copies read them
    const void* kbase;
    const void* vbase;
    // FP8 pools: one scale per KV head (null for fp16 pools)
    const float* k_scale;
    const float* v_scale;
};

static_assert(sizeof(Params) <= 256 && sizeof(Params) % 8 == 0, "Params fit their shared-memory copy");

// A split piece of this block: its unit, the unit's first block and piece
// count, this piece's index among them, and the unit's row and head.
struct Task {
    int u, cs, P, idx, r, kvh;
};

// One block's plan.  Burst blocks get their slots (physical row of each
// granule's first token, or -1 for no copy; KV head; valid tokens), pieces
// (row, head, unit's first granule, blocks holding the unit and the first of
// them, first granule and size in this block, the appended token's unit-local
// index when it falls in the piece), the warps dealt to each piece with their
// granule ranges, and the split pieces as merge tasks.  Other blocks only get
// their mode and range.
struct BlockPlan {
    int mode, g0, g1, G;  // G: the grid the plan was made for
    int npieces, ntasks, W, Geff;
    int pr[kBurstPieces], pkvh[kBurstPieces], pus[kBurstPieces], pP[kBurstPieces];
    int pcs[kBurstPieces], pw0[kBurstPieces], pwn[kBurstPieces], ppatch[kBurstPieces];
    int pfirst[kBurstPieces], psize[kBurstPieces];
    int wpiece[8], wa[8], wb[8];
    int szrow[kRing], skvh[kRing], svalid[kRing];
    Task tasks[kMaxTasks];
    int pad[8];
};
static_assert(sizeof(BlockPlan) == kPlanBytes, "a plan is 32 lanes x 16 bytes");
static_assert(kConsumerWarps <= 8, "warp shares fit the plan");

// Shared memory carve-up (offsets from a 1024-aligned base).
struct Smem {
    static constexpr uint32_t ring = 0;
    static constexpr uint32_t sinfo = ring + kRing * kSlotBytes;                    // stream: unit of each slot [kRing]
    static constexpr uint32_t plan = sinfo + kRing * 4;                             // BlockPlan (16-byte aligned)
    static constexpr uint32_t flags = plan + kPlanBytes;                            // misc ints
    static constexpr uint32_t scales = flags + 16 * 4;                              // FP8: k, v scale [2][16]
    static constexpr uint32_t part = scales + 2 * kFp8MaxKvHeads * 4;               // scan partials [kThreads]
    static constexpr uint32_t prefix = part + kThreads * 4;                         // rows + 1 ints
    __host__ __device__ static constexpr uint32_t lens(int rows) { return prefix + (uint32_t)(rows + 1) * 4; }
    __host__ __device__ static constexpr uint32_t total(int rows) { return lens(rows) + (uint32_t)rows * 4 + 1024; }
};
// Two blocks per SM (this layer's and the next one's, under programmatic
// dependent launch) at batch 32: 228 KB per SM, 1 KB reserved per block.
static_assert(Smem::total(32) + 1024 <= 233472 / 2, "two blocks per SM at 32 rows");


// ---------------------------------------------------------------------------
// PTX wrappers (shared ones in ptx.cuh)

using namespace ptx;

__device__ __forceinline__ void named_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

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
// l0 / l1 are per-lane partial sums until reduce_l() folds the lanes.
struct Soft {
    float m0, m1, l0, l1;
    float o[8][4];
    __device__ __forceinline__ void reset() {
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    }
    // sums over the eight lanes sharing tq (the token rows of a fragment)
    __device__ __forceinline__ void reduce_l() {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
    }
};

// Writes the appended token's row `prow` into a staged slot: lanes 0-15
// carry its K, lanes 16-31 its V, each lane one 16-byte chunk of fp16 dims
// 8c..8c+7 (c = lane % 16), or, for FP8 pools, those dims' 8 codes in the
// low 8 bytes.
template <bool kFp8>
__device__ __forceinline__ void patch_row(unsigned char* sp, int prow, const uint4& v, int lane) {
    const int c16 = lane & 15;
    if (kFp8) {
        unsigned char* box = sp + (lane < 16 ? 0u : kBoxBytes);
        *reinterpret_cast<uint2*>(box + prow * 128 + ((((c16 >> 1) ^ (prow & 7)) << 4) | ((c16 & 1) << 3))) =
            make_uint2(v.x, v.y);
    } else {
        unsigned char* box = sp + (lane < 16 ? 0u : kSlotV) + (c16 >> 3) * kBoxBytes;
        *reinterpret_cast<uint4*>(box + prow * 128 + (((c16 & 7) ^ (prow & 7)) << 4)) = v;
    }
}

// The online-softmax step of a warp on its granule's scores S^T (s0 = token
// gq, head 2tq; s1 = gq, 2tq+1; s2, s3 = token gq+8) with `valid` tokens:
// updates the running max and sum, rescales O and returns the B fragments
// of P^T (token x head) for the PV product.
__device__ __forceinline__ void softmax_step(Soft& st, float (&s)[4], int valid, float scale_log2,
                                             int lane, uint32_t& pb0, uint32_t& pb1) {
    const int gq = lane >> 2;
    s[0] = gq < valid ? s[0] * scale_log2 : -INFINITY;
    s[1] = gq < valid ? s[1] * scale_log2 : -INFINITY;
    s[2] = gq + 8 < valid ? s[2] * scale_log2 : -INFINITY;
    s[3] = gq + 8 < valid ? s[3] * scale_log2 : -INFINITY;
    float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
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
    const uint32_t px = pack_half2(fast_exp2(s[0] - mu0), fast_exp2(s[1] - mu1));
    const uint32_t py = pack_half2(fast_exp2(s[2] - mu0), fast_exp2(s[3] - mu1));
    // the sum takes the fp16 weights the MMA multiplies by
    const float2 fx = __half22float2(*reinterpret_cast<const __half2*>(&px));
    const float2 fy = __half22float2(*reinterpret_cast<const __half2*>(&py));
    st.l0 = st.l0 * al0 + (fx.x + fy.x);
    st.l1 = st.l1 * al1 + (fx.y + fy.y);
    // B fragments of P^T (token x head) by transposing in registers
    pb0 = movmatrix_t(px);
    pb1 = movmatrix_t(py);
    // O rescaled by (al0, al1) per head pair, two lanes per packed multiply
    const uint64_t al2 = f32x2(al0, al1);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
            f32x2_split(mul_f32x2(f32x2(st.o[i][2 * h], st.o[i][2 * h + 1]), al2), st.o[i][2 * h],
                        st.o[i][2 * h + 1]);
    }
}

// One online-softmax step of a warp over the fp16 granule staged at `slot`
// (K dims 0-63 at +0, K 64-127 at +2 KB, V at +4 KB / +6 KB, 128-byte
// swizzled rows) with `valid` tokens.  Rows past `valid` hold zeros.
__device__ __forceinline__ void attend(Soft& st, const uint32_t (&qb)[16], uint32_t slot, int valid,
                                       float scale_log2, int lane) {
    float s[4];
    {
        // S^T = K . Q^T; two independent chains (even / odd k-steps)
        const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int chunk = (ks & 3) * 2 + (lane >> 4);
            const uint32_t off = (ks >> 2) * kBoxBytes + row * 128 + ((chunk ^ (row & 7)) << 4);
            uint32_t a0, a1, a2, a3;
            ldsm_x4(slot + off, a0, a1, a2, a3);
            mma16816((ks & 1) ? c1 : c0, a0, a1, a2, a3, qb[2 * ks], qb[2 * ks + 1]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) s[i] = c0[i] + c1[i];
    }
    uint32_t pb0, pb1;
    softmax_step(st, s, valid, scale_log2, lane, pb0, pb1);
    // O^T += V^T . P^T
    const int row = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        const int chunk = (mt & 3) * 2 + ((lane >> 3) & 1);
        const uint32_t off = kSlotV + (mt >> 2) * kBoxBytes + row * 128 + ((chunk ^ (row & 7)) << 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(slot + off, a0, a1, a2, a3);
        mma16816(st.o[mt], a0, a1, a2, a3, pb0, pb1);
    }
}

// The same over an FP8 granule at `slot` (E4M3 K box at +0, V box at +2 KB,
// 16 rows x 128 bytes, 128-byte swizzled), converting E4M3 to fp16 in
// registers (exact) as the fragments are built.  The dot product runs over
// the dims in a per-lane order: k-step ks of lane (g, t) takes dims 32t + 4ks
// .. 32t + 4ks + 3 (its 4-byte word ks of K rows g and g + 8), so the queries
// come in the same order (load_q_fp8).  The output dims are ordered per lane
// too: row g of m-tile i is dim 16g + 2i and row g + 8 is 16g + 2i + 1, so
// lane (g, t) reads one 16-byte chunk of each of its four V rows
// (store_chunk_fp8 writes the result back in natural order).
__device__ __forceinline__ void attend8(Soft& st, const uint32_t (&qb)[16], const unsigned char* slot,
                                        int valid, float scale_log2, int lane) {
    const int g = lane >> 2, t = lane & 3;
    float s[4];
    {
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            // bytes 32t + 16h .. +15 of K rows g and g + 8 (chunk 2t + h; (g + 8) & 7 == g)
            const uint32_t off = ((uint32_t)(2 * t + h) ^ (uint32_t)g) << 4;
            const uint4 r0 = *reinterpret_cast<const uint4*>(slot + g * 128 + off);
            const uint4 r1 = *reinterpret_cast<const uint4*>(slot + (g + 8) * 128 + off);
            const uint32_t w0[4] = {r0.x, r0.y, r0.z, r0.w}, w1[4] = {r1.x, r1.y, r1.z, r1.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int ks = 4 * h + j;
                uint32_t a0, a1, a2, a3;
                widen4(w0[j], a0, a2);  // row g: dims 2t, 2t+1 | 8+2t, 9+2t of the k-step
                widen4(w1[j], a1, a3);  // row g + 8
                mma16816((ks & 1) ? c1 : c0, a0, a1, a2, a3, qb[2 * ks], qb[2 * ks + 1]);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) s[i] = c0[i] + c1[i];
    }
    uint32_t pb0, pb1;
    softmax_step(st, s, valid, scale_log2, lane, pb0, pb1);
    // O^T += V^T . P^T: chunk g (dims 16g .. 16g+15) of V rows 2t, 2t+1, 8+2t, 9+2t
    const unsigned char* vb = slot + kBoxBytes;
    const int ra = 2 * t;  // rows ra, ra + 1, ra + 8, ra + 9 share ra & 7 up to the low bit
    const uint4 X = *reinterpret_cast<const uint4*>(vb + ra * 128 + (((uint32_t)g ^ (uint32_t)(ra & 7)) << 4));
    const uint4 Y = *reinterpret_cast<const uint4*>(vb + (ra + 1) * 128 + (((uint32_t)g ^ (uint32_t)((ra + 1) & 7)) << 4));
    const uint4 Z = *reinterpret_cast<const uint4*>(vb + (ra + 8) * 128 + (((uint32_t)g ^ (uint32_t)(ra & 7)) << 4));
    const uint4 W = *reinterpret_cast<const uint4*>(vb + (ra + 9) * 128 + (((uint32_t)g ^ (uint32_t)((ra + 1) & 7)) << 4));
    const uint32_t xs[4] = {X.x, X.y, X.z, X.w}, ys[4] = {Y.x, Y.y, Y.z, Y.w};
    const uint32_t zs[4] = {Z.x, Z.y, Z.z, Z.w}, ws[4] = {W.x, W.y, W.z, W.w};
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        // bytes 2mt, 2mt+1 of each row: (x, y) pairs for tokens 2t, 2t+1 and
        // (z, w) pairs for tokens 8+2t, 9+2t
        const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
        const uint32_t xy = __byte_perm(xs[mt >> 1], ys[mt >> 1], sel);
        const uint32_t zw = __byte_perm(zs[mt >> 1], ws[mt >> 1], sel);
        uint32_t a0, a1, a2, a3;
        widen4(xy, a0, a1);  // dim 16g+2mt (row g) | dim 16g+2mt+1 (row g+8), tokens 2t, 2t+1
        widen4(zw, a2, a3);  // the same, tokens 8+2t, 9+2t
        mma16816(st.o[mt], a0, a1, a2, a3, pb0, pb1);
    }
}

// Query fragments of the heads of a group, from global memory, for the
// group's first head row `q0`: b0 = Q[head gq][16ks + 2tq..], b1 = Q[head
// gq][16ks + 8 + 2tq..]; heads past the group repeat its last head (every head
// is its own MMA column, so those columns are computed and never stored).
__device__ __forceinline__ void load_q_global(uint32_t (&qb)[16], const __half* q0, int group, int lane) {
    const int h = (lane >> 2) < group ? (lane >> 2) : group - 1;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(q0 + h * kHeadDim) + (lane & 3);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        qb[2 * ks] = qrow[ks * 8];
        qb[2 * ks + 1] = qrow[ks * 8 + 4];
    }
}
// The same in the FP8 dim order (attend8): lane (g, t) takes dims 32t ..
// 32t + 31 of head g, so its word i is k-step i / 2's pair (i even: dims
// 2t, 2t+1 of the step; odd: 8+2t, 9+2t).
__device__ __forceinline__ void load_q_fp8(uint32_t (&qb)[16], const __half* q0, int group, int lane) {
    const int h = (lane >> 2) < group ? (lane >> 2) : group - 1;
    const uint4* qrow = reinterpret_cast<const uint4*>(q0 + h * kHeadDim + 32 * (lane & 3));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = qrow[i];
        qb[4 * i] = v.x;
        qb[4 * i + 1] = v.y;
        qb[4 * i + 2] = v.z;
        qb[4 * i + 3] = v.w;
    }
}

// The copies of stage_granule, from the byte offset `row0` of the granule's
// first token (for its KV head) in both pools, rows `rstride` bytes apart.
template <bool kFp8>
__device__ __forceinline__ void stage_rows(uint32_t slot, const unsigned char* kpool,
                                           const unsigned char* vpool, int64_t row0, uint32_t rstride,
                                           int valid, int lane) {
    const int c = lane & 7, r0 = lane >> 3;  // chunk; first of the rows r0, r0 + 4, ...
    const unsigned char* kb = kpool + row0 + c * 16;
    const unsigned char* vb = vpool + row0 + c * 16;
#pragma unroll
    for (int k = 0; k < (kFp8 ? 8 : 16); ++k) {
        const int r = r0 + 4 * (k & 3), b = k >> 2;  // row, box
        const unsigned char* src = ((kFp8 ? b : b >> 1) ? vb : kb) + (r < valid ? r : 0) * rstride +
                                   (kFp8 ? 0 : (b & 1) * 128);
        const uint32_t dst = slot + b * kBoxBytes + r * 128 + ((c ^ (r & 7)) << 4);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                     "r"(r < valid ? 16 : 0)
                     : "memory");
    }
}

// Stages one granule into `slot` (shared address) with 16-byte cp.async
// copies by one warp, in the layout the tiled copies produce: fp16 pools as
// four boxes (K dims 0-63, K 64-127, V 0-63, V 64-127) of 16 rows x 128 B,
// FP8 pools as a K box and a V box of 16 rows x 128 B; chunk c of row r at
// r*128 + ((c ^ (r & 7)) << 4) (128-byte swizzle).  Rows at or past `valid`
// are zero-filled without reading the pool.  Plain asynchronous copies are
// used, not tiled bulk copies, because they run before the dependency wait
// of a programmatically launched grid: bulk copies issued there complete
// only once the preceding grid has completed.
template <bool kFp8>
__device__ __forceinline__ void stage_granule(uint32_t slot, const unsigned char* kpool,
                                              const unsigned char* vpool, int64_t zrow, int hk,
                                              int kvh, int valid, int lane) {
    constexpr int kRowBytes = kFp8 ? 128 : 256;  // one token of one KV head
    stage_rows<kFp8>(slot, kpool, vpool, (zrow * hk + kvh) * kRowBytes, (uint32_t)hk * kRowBytes, valid,
                     lane);
}
// ---------------------------------------------------------------------------
// States in the fragment layout: dump, output, records, merge.

// Writes a warp's state (l reduced) at `dump`: per head pair tq one float4
// (m[2tq], m[2tq+1], l[2tq], l[2tq+1]) at 16tq, then chunk c at 64 + 512c,
// lane-major (conflict-free 16-byte stores).
__device__ __forceinline__ void dump_state(const Soft& st, unsigned char* dump, int lane) {
    if (lane < 4) *reinterpret_cast<float4*>(dump + 16 * lane) = make_float4(st.m0, st.m1, st.l0, st.l1);
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4*>(dump + kMlBytes + c * kChunkBytes + lane * 16) =
            make_float4(st.o[c][0], st.o[c][1], st.o[c][2], st.o[c][3]);
}

// Stores chunk c (dims 16c..16c+15) of a normalised state as fp16 into the
// group's output rows `ob` (head h at ob + 128h).  movmatrix turns the
// (dim, head-pair) fragment into (head, dim-pair) words.
__device__ __forceinline__ void store_chunk(__half* ob, int c, const float (&o)[4], float inv0,
                                            float inv1, int group, int lane) {
    const uint32_t x = movmatrix_t(pack_half2(o[0] * inv0, o[1] * inv1));
    const uint32_t y = movmatrix_t(pack_half2(o[2] * inv0, o[3] * inv1));
    const int h = lane >> 2, d = 16 * c + 2 * (lane & 3);
    if (h < group) {
        *reinterpret_cast<uint32_t*>(ob + h * kHeadDim + d) = x;
        *reinterpret_cast<uint32_t*>(ob + h * kHeadDim + d + 8) = y;
    }
}
// The same for a state in the FP8 dim order (attend8): chunk c of lane
// (g, t) holds dims 16g + 2c (o[0], o[1]) and 16g + 2c + 1 (o[2], o[3]) of
// heads 2t, 2t + 1.
__device__ __forceinline__ void store_chunk_fp8(__half* ob, int c, const float (&o)[4], float inv0,
                                                float inv1, int group, int lane) {
    const int t = lane & 3, d = 16 * (lane >> 2) + 2 * c;
    if (2 * t < group) *reinterpret_cast<uint32_t*>(ob + 2 * t * kHeadDim + d) = pack_half2(o[0] * inv0, o[2] * inv0);
    if (2 * t + 1 < group)
        *reinterpret_cast<uint32_t*>(ob + (2 * t + 1) * kHeadDim + d) = pack_half2(o[1] * inv1, o[3] * inv1);
}

// ---------------------------------------------------------------------------
// Split-unit records.  Every float of a record is stored as the bitwise
// complement of its bits in a 4-byte word, so a zero word means "not written
// yet": the only value that would encode as zero is the all-ones NaN pattern,
// which the GPU's arithmetic never produces (its NaN results are canonical).
// Naturally aligned 4-byte relaxed accesses are single-copy atomic, element
// by element of a vector access, so a reader that sees a word non-zero sees
// its value: the writer needs no fence or release and the reader no separate
// arrival counter or second read.  The reader clears the words it took, so
// the workspace is all zero between calls.
//
// Region of unit u (pieces in blocks cs .. cs+P-1) at slot cs + u: chunk c of
// piece i at (c*P + i) * 512 B, lane-major (16 bytes per lane: a warp's store
// fills whole sectors), then m/l of piece i for participant k at 8*P*512 +
// (k*P + i)*64: m[2tq], m[2tq+1], l[2tq], l[2tq+1] at 16*tq.  Participant k
// reads chunks c = k, k + K, ... of every piece and its own m/l copies, so no
// word is read by two blocks.
constexpr uint32_t kLLChunk = 32 * 16;      // one chunk of a state: 512 B
constexpr uint32_t kLLMl = 4 * 16;          // m/l of one piece for one participant
constexpr uint32_t kRecBytes = 8 * kLLChunk + kMergeWays * kLLMl;  // per record slot

__device__ __forceinline__ unsigned char* unit_region(const Params& p, int u, int cs) {
    return p.records + (int64_t)(cs + u) * kRecBytes;
}
__device__ __forceinline__ void st_rec(unsigned char* a, float x, float y, float z, float w) {
    asm volatile("st.relaxed.gpu.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(a),
                 "r"(~__float_as_uint(x)), "r"(~__float_as_uint(y)), "r"(~__float_as_uint(z)),
                 "r"(~__float_as_uint(w))
                 : "memory");
}
__device__ __forceinline__ void clear_rec(unsigned char* a) {
    asm volatile("st.relaxed.gpu.global.v4.b32 [%0], {%1, %1, %1, %1};" ::"l"(a), "r"(0u) : "memory");
}
__device__ __forceinline__ uint4 ld_rec(const unsigned char* a) {
    uint4 v;
    asm volatile("ld.relaxed.gpu.global.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(a)
                 : "memory");
    return v;
}
__device__ __forceinline__ bool rec_written(const uint4& v) { return v.x && v.y && v.z && v.w; }
__device__ __forceinline__ float rec_value(uint32_t w) { return __uint_as_float(~w); }

// Where a piece's combined state goes: its unit's fp16 output rows (P == 1),
// or its record (P > 1, piece idx of the unit, K participants).
struct PieceOut {
    __half* ob;             // output rows of the unit's query heads
    unsigned char* region;  // the unit's record region
    int P, idx, K, group;
    float vs;               // FP8 V scale (1 for fp16 pools)
};
__device__ __forceinline__ PieceOut piece_out(const Params& p, int r, int kvh, int cs, int P, int cta,
                                              float vs) {
    PieceOut po;
    po.ob = p.out + ((int64_t)r * p.hq + kvh * p.group) * kHeadDim;
    po.region = unit_region(p, r * p.hk + kvh, cs);
    po.P = P;
    po.idx = cta - cs;
    po.K = P < kMergeWays ? P : kMergeWays;
    po.group = p.group;
    po.vs = vs;
    return po;
}

// Chunk c of a piece's combined state (unnormalised acc, sums L0 / L1): the
// fp16 output dims 16c.. when the unit is whole, else the record words.
template <bool kFp8>
__device__ __forceinline__ void emit_chunk(const PieceOut& po, int c, const float (&acc)[4], float L0,
                                           float L1, int lane) {
    if (po.P == 1) {
        const float inv0 = L0 > 0.f ? __fdividef(po.vs, L0) : 0.f;
        const float inv1 = L1 > 0.f ? __fdividef(po.vs, L1) : 0.f;
        if (kFp8)  // the state is in the FP8 dim order
            store_chunk_fp8(po.ob, c, acc, inv0, inv1, po.group, lane);
        else
            store_chunk(po.ob, c, acc, inv0, inv1, po.group, lane);
    } else {
        st_rec(po.region + (uint32_t)(c * po.P + po.idx) * kLLChunk + lane * 16, acc[0], acc[1], acc[2],
               acc[3]);
    }
}
// m/l of a split piece, one copy per participant (lanes 0-3).
__device__ __forceinline__ void emit_ml(const PieceOut& po, float M0, float M1, float L0, float L1,
                                        int lane) {
    if (po.P == 1 || lane >= 4) return;
#pragma unroll 1
    for (int k = 0; k < po.K; ++k)
        st_rec(po.region + 8u * po.P * kLLChunk + (uint32_t)(k * po.P + po.idx) * kLLMl + lane * 16, M0,
               M1, L0, L1);
}

// Stream mode, warp j of the k stream warps (k <= kStreamWarps) holding a
// unit's states, dumped in ring slots slot[0 .. k-1]: combines them through
// their log-sum-exp for chunks c = j, j + k, ... and emits those; warp 0 also
// emits the m/l.  Every
// state's offset, maximum and sum is loaded up front, the weights are
// computed once, and each chunk's k loads are issued together, so the chains
// overlap.
template <bool kFp8>
__device__ void combine_dumps(const PieceOut& po, const unsigned char* ring,
                              const int (&slot)[kStreamWarps], int k, int j, int lane) {
    const int tq = lane & 3;
    uint32_t off[kStreamWarps];
#pragma unroll
    for (int s = 0; s < kStreamWarps; ++s) off[s] = (uint32_t)slot[s < k ? s : 0] * kSlotBytes;
    float4 ml[kStreamWarps];
#pragma unroll
    for (int s = 0; s < kStreamWarps; ++s)
        ml[s] = s < k ? *reinterpret_cast<const float4*>(ring + off[s] + 16 * tq)
                      : make_float4(-INFINITY, -INFINITY, 0.f, 0.f);
    float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
    for (int s = 0; s < kStreamWarps; ++s) {
        M0 = fmaxf(M0, ml[s].x);
        M1 = fmaxf(M1, ml[s].y);
    }
    float L0 = 0.f, L1 = 0.f;
#pragma unroll
    for (int s = 0; s < kStreamWarps; ++s) {  // ml[s].x / .y become the weights
        ml[s].x = M0 == -INFINITY ? 0.f : fast_exp2(ml[s].x - M0);
        ml[s].y = M1 == -INFINITY ? 0.f : fast_exp2(ml[s].y - M1);
        L0 += ml[s].x * ml[s].z;
        L1 += ml[s].y * ml[s].w;
    }
#pragma unroll 1
    for (int c = j; c < 8; c += k) {
        float4 v[kStreamWarps];
#pragma unroll
        for (int s = 0; s < kStreamWarps; ++s)
            v[s] = s < k ? *reinterpret_cast<const float4*>(ring + off[s] + kMlBytes + c * kChunkBytes + lane * 16)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s = 0; s < kStreamWarps; ++s) {
            acc[0] += ml[s].x * v[s].x;
            acc[1] += ml[s].y * v[s].y;
            acc[2] += ml[s].x * v[s].z;
            acc[3] += ml[s].y * v[s].w;
        }
        emit_chunk<kFp8>(po, c, acc, L0, L1, lane);
    }
    if (j == 0) emit_ml(po, M0, M1, L0, L1, lane);
}

// Merge of a split unit's slice by participant t.idx (< K): chunks
// c_m = idx + m*K for m < nch.  The task's nw warps form min(nch, nw) chunk
// groups of gsz = nw / groups warps; the warp of rank q in group g merges
// chunks m = g, g + groups, ... over records j = q, q + gsz, ..., polled in
// batches of four, each batch taken once all its words are written, absorbed
// in order (running maximum) and cleared.  Every warp leaves its partial of
// each chunk in shared memory at `part`; after the task's barrier the rank-0
// warp of each group combines its group's partials in rank order and stores
// the chunk, so the result never depends on timing.  Returns false if a poll
// gave up.
__device__ __forceinline__ void absorb(float& M0, float& M1, float& L0, float& L1, float (&acc)[4],
                                       float m0, float m1, float l0, float l1, float x0, float x1,
                                       float x2, float x3) {
    const float N0 = fmaxf(M0, m0), N1 = fmaxf(M1, m1);
    const float a0 = N0 == -INFINITY ? 0.f : fast_exp2(M0 - N0);
    const float a1 = N1 == -INFINITY ? 0.f : fast_exp2(M1 - N1);
    const float w0 = N0 == -INFINITY ? 0.f : fast_exp2(m0 - N0);
    const float w1 = N1 == -INFINITY ? 0.f : fast_exp2(m1 - N1);
    L0 = L0 * a0 + w0 * l0;
    L1 = L1 * a1 + w1 * l1;
    acc[0] = acc[0] * a0 + w0 * x0;
    acc[1] = acc[1] * a1 + w1 * x1;
    acc[2] = acc[2] * a0 + w0 * x2;
    acc[3] = acc[3] * a1 + w1 * x3;
    M0 = N0;
    M1 = N1;
}

template <bool kFp8>
__device__ __forceinline__ bool merge_task(const Params& p, const Task& t, int lw, int nw,
                                           unsigned char* part, int bar_id, float vs,
                                           volatile int* fail, int lane) {
    const int P = t.P;
    const int K = P < kMergeWays ? P : kMergeWays;
    if (t.idx >= K) return true;  // not a participant
    int nch = 0;  // chunks idx, idx + K, ... below 8
    for (int c = t.idx; c < 8; c += K) ++nch;
    const int groups = nch < nw ? nch : nw;
    int gsz = 0, g = lw, q = 0;  // nw / groups, lw % groups, lw / groups
    for (int x = groups; x <= nw; x += groups) ++gsz;
    while (g >= groups) {
        g -= groups;
        ++q;
    }
    const int tq = lane & 3;
    unsigned char* reg = unit_region(p, t.u, t.cs);
    unsigned char* mlb = reg + 8u * P * kLLChunk + (uint32_t)t.idx * P * kLLMl + tq * 16;
    bool ok = true;
#pragma unroll 1
    for (int m = g; q < gsz && m < nch && ok; m += groups) {
        unsigned char* cb = reg + (uint32_t)(t.idx + m * K) * P * kLLChunk + lane * 16;
        float M0 = -INFINITY, M1 = -INFINITY, L0 = 0.f, L1 = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
        for (int j0 = q; j0 < P; j0 += 4 * gsz) {
            uint4 wm[4], wc[4];
            uint32_t it = 0;
            bool all;
            do {
                all = true;
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int j = j0 + b * gsz < P ? j0 + b * gsz : j0;  // past P: record j0 again
                    wm[b] = ld_rec(mlb + j * kLLMl);
                    wc[b] = ld_rec(cb + j * kLLChunk);
                    all &= rec_written(wm[b]) & rec_written(wc[b]);
                }
                if (p.stuck) all &= *reinterpret_cast<const volatile uint32_t*>(p.stuck) != 0u;
            } while (!__all_sync(0xffffffffu, all) && ++it < p.poll_limit);
            if (it >= p.poll_limit) {
                ok = false;
                break;
            }
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int j = j0 + b * gsz;
                if (j >= P) break;
                absorb(M0, M1, L0, L1, acc, rec_value(wm[b].x), rec_value(wm[b].y), rec_value(wm[b].z),
                       rec_value(wm[b].w), rec_value(wc[b].x), rec_value(wc[b].y), rec_value(wc[b].z),
                       rec_value(wc[b].w));
                // taken: clear the chunk words (read by this warp alone) for the
                // next call; the m/l words are shared by the task's warps
                clear_rec(cb + j * kLLChunk);
            }
        }
        if (gsz == 1) {
            const float inv0 = L0 > 0.f ? __fdividef(vs, L0) : 0.f;
            const float inv1 = L1 > 0.f ? __fdividef(vs, L1) : 0.f;
            __half* ob = p.out + ((int64_t)t.r * p.hq + t.kvh * p.group) * kHeadDim;
            if (kFp8)
                store_chunk_fp8(ob, t.idx + m * K, acc, inv0, inv1, p.group, lane);
            else
                store_chunk(ob, t.idx + m * K, acc, inv0, inv1, p.group, lane);
        } else {
            unsigned char* pw = part + (q * nch + m) * 1024 + lane * 16;
            *reinterpret_cast<float4*>(pw) = make_float4(M0, M1, L0, L1);
            *reinterpret_cast<float4*>(pw + 512) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        }
    }
    if (!ok && lane == 0) *fail = 1;
    named_sync(bar_id, nw * 32);
    if (*fail) {
        if (lane == 0 && lw == 0) flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
        return false;
    }
    // every warp of the task is past the m/l words: clear them for the next call
#pragma unroll 1
    for (int j = lw; j < P; j += nw) clear_rec(mlb + j * kLLMl);
    if (q != 0 || gsz == 1) return true;
    __half* ob = p.out + ((int64_t)t.r * p.hq + t.kvh * p.group) * kHeadDim;
#pragma unroll 1
    for (int m = g; m < nch; m += groups) {
        // the group's partials of chunk m, in rank order
        float M0 = -INFINITY, M1 = -INFINITY, L0 = 0.f, L1 = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
        for (int r = 0; r < gsz; ++r) {
            const unsigned char* pw = part + (r * nch + m) * 1024 + lane * 16;
            const float4 pm = *reinterpret_cast<const float4*>(pw);
            const float4 pv = *reinterpret_cast<const float4*>(pw + 512);
            absorb(M0, M1, L0, L1, acc, pm.x, pm.y, pm.z, pm.w, pv.x, pv.y, pv.z, pv.w);
        }
        const float inv0 = L0 > 0.f ? __fdividef(vs, L0) : 0.f;
        const float inv1 = L1 > 0.f ? __fdividef(vs, L1) : 0.f;
        if (kFp8)
            store_chunk_fp8(ob, t.idx + m * K, acc, inv0, inv1, p.group, lane);
        else
            store_chunk(ob, t.idx + m * K, acc, inv0, inv1, p.group, lane);
    }
    return true;
}

// Granule prefix over rows, by all NT threads of a block: sm_pre[r] = first
// granule of row r (its KV heads' granules in head order), sm_pre[rows] = W;
// sm_len[r] = the row's tokens, clamped to the bound (a length outside
// [0, limit] is flagged when `flag` is set).  Returns W.
template <int NT>
__device__ int scan_lengths(const Params& p, bool paged, int* sm_pre, int* sm_len, int* sm_part,
                            bool flag) {
    const int tid = threadIdx.x, lane = tid & 31, rows = p.rows;
    const int per = (rows + NT - 1) / NT;
    bool bad_len = false;
    int sum = 0;
#pragma unroll 1
    for (int i = 0; i < per; ++i) {
        const int r = tid * per + i;
        if (r < rows) {
            int L = p.seq_lens[r];
            if (L < 0 || L > p.limit) {
                if (paged) bad_len = true;
                L = L < 0 ? 0 : p.limit;
            }
            sm_len[r] = L;  // tokens that count (clamped)
            const int c = p.hk * granules_of(paged ? L : p.width);
            sm_pre[r] = c;
            sum += c;
        }
    }
    sm_part[tid] = sum;
    if (bad_len && flag) flag_error(p.dev_err, PKV_DEV_ERR_SEQ_LEN);
    __syncthreads();
    if (tid < 32) {
        constexpr int kPer = (NT + 31) / 32;  // partials per lane
        int acc = 0;
#pragma unroll 1
        for (int j = 0; j < kPer; ++j) acc += sm_part[lane * kPer + j];
        int incl = acc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        int run = incl - acc;
#pragma unroll 1
        for (int j = 0; j < kPer; ++j) {
            const int v = sm_part[lane * kPer + j];
            sm_part[lane * kPer + j] = run;
            run += v;
        }
    }
    __syncthreads();
    {
        int run = sm_part[tid];
#pragma unroll 1
        for (int i = 0; i < per; ++i) {
            const int r = tid * per + i;
            if (r < rows) {
                const int c = sm_pre[r];
                sm_pre[r] = run;
                run += c;
            }
        }
        if (tid == NT - 1) sm_pre[rows] = run;
    }
    __syncthreads();
    return sm_pre[rows];
}

// One warp writes block b's plan into bp (shared memory), from the granule
// prefix of a scan_lengths.  The W granules are cut into Geff = min(G, W)
// equal contiguous ranges; block b's range is burst when it fits the ring
// and covers at most four pieces.  Lane j resolves granule g0 + j (row, KV
// head, valid tokens, physical row through the table).  Every piece gets one
// warp; each further warp goes to the piece whose busiest warp has the most
// granules, while that is more than one, and a piece's warps take near-equal
// contiguous shares of it.
__device__ void build_block_plan(BlockPlan* bp, const Params& p, bool paged, int b, int G, int W,
                                 int Geff, const int* sm_pre, const int* sm_len, int lane) {
    const int hk = p.hk, rows = p.rows;
    int g0 = 0, g1 = 0;
    if (b < Geff) {
        g0 = (int)((int64_t)W * b / Geff);
        g1 = (int)((int64_t)W * (b + 1) / Geff);
    }
    const int ng = g1 - g0;
    const bool fits = ng > 0 && ng <= kRing;
    int u = -1, r = 0, kvh = 0, n = 1, us = 0, valid = 0, zrow = -1;
    if (fits && lane < ng) {
        const int gg = g0 + lane;
        int lo = 0, hi = rows - 1;
#pragma unroll 1
        while (lo < hi) {  // largest row with sm_pre[row] <= gg
            const int mid = (lo + hi + 1) >> 1;
            if (sm_pre[mid] <= gg) lo = mid; else hi = mid - 1;
        }
        r = lo;
        n = (sm_pre[r + 1] - sm_pre[r]) / hk;
        kvh = (gg - sm_pre[r]) / n;
        us = sm_pre[r] + kvh * n;
        u = r * hk + kvh;
        const int tok = (gg - us) * kGranule;
        valid = min(kGranule, sm_len[r] - tok);
        if (valid < 0) valid = 0;
        if (paged) {
            const int pb = p.tables[(int64_t)r * p.mbpr + tok / p.bs];
            if (pb < 0 || pb >= p.nb) {
                flag_error(p.dev_err, PKV_DEV_ERR_BLOCK_ID);
                valid = 0;
            } else {
                zrow = pb * p.bs + tok % p.bs;
            }
        } else {
            zrow = r * p.width + tok;  // the comparator reads every column
        }
    }
    const int up = __shfl_up_sync(0xffffffffu, u, 1);
    const unsigned starts = __ballot_sync(0xffffffffu, u >= 0 && (lane == 0 || u != up));
    const int np = __popc(starts);
    const int mode = ng <= 0 ? kModeIdle : (fits && np <= kBurstPieces) ? kModeBurst : kModeStream;
    if (lane == 0) {
        bp->mode = mode;
        bp->g0 = g0;
        bp->g1 = g1;
        bp->G = G;
        bp->W = W;
        bp->Geff = Geff;
        bp->npieces = mode == kModeBurst ? np : 0;
        bp->ntasks = 0;
    }
    if (lane < 8) bp->wpiece[lane] = -1;
    if (mode != kModeBurst) {
        __syncwarp();
        return;
    }
    if (lane < ng) {
        bp->szrow[lane] = zrow;
        bp->skvh[lane] = kvh;
        bp->svalid[lane] = valid;
    }
    if (u >= 0 && ((starts >> lane) & 1u)) {
        const int k = __popc(starts & ((1u << lane) - 1u));
        const unsigned later = lane == 31 ? 0u : (starts >> (lane + 1));
        const int end = later ? lane + __ffs(later) : ng;  // the next piece's first lane
        const int cs = owner_of(us, W, Geff);
        bp->pr[k] = r;
        bp->pkvh[k] = kvh;
        bp->pus[k] = us;
        bp->pcs[k] = cs;
        bp->pP[k] = owner_of(us + n - 1, W, Geff) - cs + 1;
        bp->pfirst[k] = g0 + lane;
        bp->psize[k] = end - lane;
        int patch = -1;
        if (paged && p.positions) {
            const int pos = p.positions[r];
            if (pos >= 0) {
                const int pg = us + pos / kGranule;
                if (pg >= g0 + lane && pg < g0 + end) patch = pos;
            }
        }
        bp->ppatch[k] = patch;
    }
    __syncwarp();
    // deal the consumer warps: lane k < np holds piece k
    const int sz = lane < np ? bp->psize[lane] : 0;
    int wc = lane < np ? 1 : 0;
#pragma unroll 1
    for (int e = np; e < kConsumerWarps; ++e) {
        const int c = lane < np ? (sz + wc - 1) / wc : 0;
        int best = c;
        best = max(best, __shfl_xor_sync(0xffffffffu, best, 1));
        best = max(best, __shfl_xor_sync(0xffffffffu, best, 2));
        best = __shfl_sync(0xffffffffu, best, 0);  // lanes 0-3 hold the pieces
        if (best <= 1) break;
        const unsigned who = __ballot_sync(0xffffffffu, lane < np && c == best);
        if (lane == __ffs(who) - 1) ++wc;
    }
    int w0 = 0;
#pragma unroll
    for (int j = 0; j < kBurstPieces; ++j) {
        const int wj = __shfl_sync(0xffffffffu, wc, j);
        if (j < lane) w0 += wj;
    }
    if (lane < np) {
        bp->pw0[lane] = w0;
        bp->pwn[lane] = wc;
        const int a = bp->pfirst[lane];
#pragma unroll 1
        for (int j = 0; j < wc; ++j) {
            bp->wpiece[w0 + j] = lane;
            bp->wa[w0 + j] = a + j * sz / wc;
            bp->wb[w0 + j] = a + (j + 1) * sz / wc;
        }
    }
    __syncwarp();
    if (lane == 0) {
        // split pieces: a contiguous range has at most two, its first and its last
        int nt = 0;
#pragma unroll 1
        for (int k = 0; k < np; ++k) {
            if (bp->pP[k] == 1 || nt == kMaxTasks) continue;
            Task& t = bp->tasks[nt++];
            t.u = bp->pr[k] * hk + bp->pkvh[k];
            t.cs = bp->pcs[k];
            t.P = bp->pP[k];
            t.idx = b - bp->pcs[k];
            t.r = bp->pr[k];
            t.kvh = bp->pkvh[k];
        }
        bp->ntasks = nt;
    }
    __syncwarp();
}

// Per-row work of block cta, done by its warp 7 after the dependency wait
// (off the consumers' critical path): rows cta, cta + G, ... with nothing
// to read get zero outputs, and in the fused form their new token is stored
// into its slot (as E4M3 codes for FP8 pools, quantised exactly as
// paged_kv_append_fp8 does).  The block that stages the slot's granule takes
// the token from k_new / v_new directly, so the order of this store and that
// copy does not matter.
template <bool kFp8>
__device__ void row_work(const Params& p, int cta, int G, int lane) {
#pragma unroll 1
    for (int r = cta; r < p.rows; r += G) {
        if (p.seq_lens[r] <= 0)
#pragma unroll 1
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
#pragma unroll 1
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

// Shared-memory views of a decode block, handed to the out-of-line stream
// functions.
struct Ctx {
    unsigned char* smem;
    uint32_t sbase;
    BlockPlan* bp;
    volatile int* flags;
    int* pre;   // granule prefix over rows
    int* len;   // clamped lengths
    const float* ks;  // FP8 scales (shared memory)
    const float* vs;
    int W, Geff;
};

// Stream mode: warps 0 .. kSWarps-1 each stream an equal contiguous share
// [wa, wb) of the block's range through their own kSSlots ring slots, with
// kSSlots - 1 granules' copies in flight (16-byte cp.async; the first ones go
// out before the dependency wait).  A unit that lies wholly in one warp's
// share is finished by that warp (fp16 output straight from registers).  A
// unit that a warp shares with other warps or blocks leaves a state: at the
// warp's end in its slot 0, or, when it is the warp's first unit and ends
// before the warp's share does, in the warp's global scratch slot (reloaded
// into its slot 1 at the end).  After a barrier of the stream warps each such
// unit is combined by the warps that hold its states and emitted (fp16
// output, or the block's record of a split unit), as in burst mode.
constexpr int kSWarps = kStreamWarps;      // stream warps
constexpr int kSSlots = kRing / kSWarps;   // ring slots per stream warp
constexpr int kSDepth = kSSlots - 1;       // copies in flight ahead of the granule consumed
static_assert(kSSlots >= 2 && kSWarps * kSSlots == kRing, "stream slots");
static_assert(kSWarps <= kConsumerWarps, "stream warps are consumer warps");

// A granule's unit (row, KV head, first granule, granules) and valid tokens.
struct SInfo {
    int r, kvh, us, n, valid;
};

// Byte offset of the stream warps' scratch states in the workspace (after
// the record slots of the grid's blocks and the units).
__device__ __forceinline__ size_t stream_scratch_offset(const Params& p) {
    const size_t rec = (size_t)kRecBytes * ((size_t)gridDim.x + (size_t)p.rows * p.hk);
    return (rec + 255) / 256 * 256;
}

// Granule gg's unit, valid tokens and physical row (-1: a bad table entry,
// flagged; nothing is read for it).
__device__ __forceinline__ void resolve_granule(const Params& p, bool paged, const int* sm_pre,
                                                const int* sm_len, int gg, SInfo& gi, int& zrow) {
    int lo = 0, hi = p.rows - 1;
#pragma unroll 1
    while (lo < hi) {  // largest row with sm_pre[row] <= gg
        const int mid = (lo + hi + 1) >> 1;
        if (sm_pre[mid] <= gg) lo = mid; else hi = mid - 1;
    }
    const int r = lo;
    const int n = (sm_pre[r + 1] - sm_pre[r]) / p.hk;
    const int kvh = (gg - sm_pre[r]) / n;
    const int us = sm_pre[r] + kvh * n;
    const int tok = (gg - us) * kGranule;
    int valid = min(kGranule, sm_len[r] - tok);
    if (valid < 0) valid = 0;
    if (paged) {
        const int pb = p.tables[(int64_t)r * p.mbpr + tok / p.bs];
        if (pb < 0 || pb >= p.nb) {
            flag_error(p.dev_err, PKV_DEV_ERR_BLOCK_ID);
            valid = 0;
            zrow = -1;
        } else {
            zrow = pb * p.bs + tok % p.bs;
        }
    } else {
        zrow = r * p.width + tok;
    }
    gi.r = r;
    gi.kvh = kvh;
    gi.us = us;
    gi.n = n;
    gi.valid = valid;
}

// Writes a warp's state (l reduced) to global memory in the dump layout.
__device__ __forceinline__ void dump_state_global(const Soft& st, unsigned char* dump, int lane) {
    if (lane < 4) *reinterpret_cast<float4*>(dump + 16 * lane) = make_float4(st.m0, st.m1, st.l0, st.l1);
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4*>(dump + kMlBytes + c * kChunkBytes + lane * 16) =
            make_float4(st.o[c][0], st.o[c][1], st.o[c][2], st.o[c][3]);
}

// The granule share [wa, wb) of stream warp w.
__device__ __forceinline__ void stream_share(int g0, int g1, int w, int& wa, int& wb) {
    const int ng = g1 - g0;
    wa = g0 + (int)((int64_t)ng * w / kSWarps);
    wb = g0 + (int)((int64_t)ng * (w + 1) / kSWarps);
}

template <bool kPaged, bool kFp8>
__device__ __noinline__ void stream_warp(const Params& p, const Ctx& cx, int cta, int warp, int lane,
                                         unsigned char* scratch) {
    constexpr int kRowBytes = kFp8 ? 128 : 256;  // one token of one KV head
    BlockPlan* bp = cx.bp;
    const int g0 = bp->g0, g1 = bp->g1, hk = p.hk;
    const int* sm_pre = cx.pre;
    const int* sm_len = cx.len;
    unsigned char* smem = cx.smem;
    int* sinfo = reinterpret_cast<int*>(smem + Smem::sinfo) + warp * kSSlots;  // packed unit of each slot
    const uint32_t slot0 = cx.sbase + Smem::ring + warp * kSSlots * kSlotBytes;
    const unsigned char* kpool = reinterpret_cast<const unsigned char*>(p.kbase);
    const unsigned char* vpool = reinterpret_cast<const unsigned char*>(p.vbase);
    const uint32_t rstride = (uint32_t)hk * kRowBytes;
    const bool fused = kPaged && p.positions != nullptr;
    int wa, wb;
    stream_share(g0, g1, warp, wa, wb);

    // Lane j resolves granule bb + j of the share, 32 at a time: the byte
    // offset of its first token's row for its KV head (-1: a bad table entry)
    // and its row | KV head << 16 | valid tokens << 24.
    int bb = wa, pinfo = 0;
    long long koff = 0;
    auto resolve = [&]() {
        if (lane < wb - bb) {
            SInfo x;
            int zrow = 0;
            resolve_granule(p, kPaged, sm_pre, sm_len, bb + lane, x, zrow);
            koff = zrow < 0 ? -1ll : ((long long)zrow * hk + x.kvh) * kRowBytes;
            pinfo = x.r | (x.kvh << 16) | ((zrow < 0 ? 0 : x.valid) << 24);
        }
    };
    resolve();
    const int fpi = __shfl_sync(0xffffffffu, pinfo, 0);
    const int fr = fpi & 0xffff, fkvh = (fpi >> 16) & 0xff;
    const int fn = (sm_pre[fr + 1] - sm_pre[fr]) / hk, fus = sm_pre[fr] + fkvh * fn;
    auto issue = [&](int g) {
        if (g >= bb + 32) {  // the next 32 granules
            bb += 32;
            resolve();
        }
        const int j = g - bb;
        const long long off = __shfl_sync(0xffffffffu, koff, j);
        const int pi = __shfl_sync(0xffffffffu, pinfo, j);
        const int s = (g - wa) % kSSlots;
        stage_rows<kFp8>(slot0 + s * kSlotBytes, kpool, vpool, off < 0 ? 0 : off, rstride, pi >> 24, lane);
        if (lane == 0) sinfo[s] = pi;
    };
    // the first granules' copies go out before the dependency wait
#pragma unroll 1
    for (int g = wa; g < wa + kSDepth; ++g) {
        if (g < wb) issue(g);
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    {
        // warm L2 with the first unit's query rows (read after the wait)
        const char* qrow = reinterpret_cast<const char*>(p.q + ((int64_t)fr * p.hq + fkvh * p.group) * kHeadDim);
        if (lane < 2 * p.group) asm volatile("prefetch.global.L2 [%0];" ::"l"(qrow + lane * 128));
    }
    // Everything below may read what the preceding kernel wrote (query,
    // positions, new tokens, workspace) or write what it reads.
    griddep_wait();

    Soft st;
    int cu = -1, cr = 0, ckvh = 0, cus = 0, cn = 0;  // the unit being accumulated
    bool parked = false;  // this warp's first unit waits in its scratch slot
    uint32_t qb[16];
    int patch_tok = -1;
    uint4 patch_val = make_uint4(0, 0, 0, 0);
    float sl2 = p.scale_log2;
    auto finish = [&](bool at_end) {
        st.reduce_l();
        __syncwarp();
        if (cus >= wa && cus + cn <= wb) {
            // the whole unit lies in this share: its output, straight from registers
            const PieceOut po = piece_out(p, cr, ckvh, 0, 1, 0, kFp8 ? cx.vs[ckvh] : 1.f);
#pragma unroll
            for (int c = 0; c < 8; ++c) emit_chunk<kFp8>(po, c, st.o[c], st.l0, st.l1, lane);
        } else if (!at_end) {
            dump_state_global(st, scratch, lane);  // the first unit, shared with earlier warps or blocks
            parked = true;
        } else {
            dump_state(st, smem + Smem::ring + warp * kSSlots * kSlotBytes, lane);
        }
    };
#pragma unroll 1
    for (int g = wa; g < wb; ++g) {
        if (g + kSDepth < wb) issue(g + kSDepth);
        asm volatile("cp.async.commit_group;" ::: "memory");
        asm volatile("cp.async.wait_group %0;" ::"n"(kSDepth) : "memory");
        __syncwarp();
        const int s = (g - wa) % kSSlots;
        const int pi = sinfo[s];
        const int u = pi & 0xffffff;  // row | KV head << 16
        const int valid = pi >> 24;
        if (u != cu) {
            if (cu >= 0) finish(false);
            cu = u;
            cr = pi & 0xffff;
            ckvh = (pi >> 16) & 0xff;
            cn = (sm_pre[cr + 1] - sm_pre[cr]) / hk;
            cus = sm_pre[cr] + ckvh * cn;
            st.reset();
            if (kFp8)
                load_q_fp8(qb, p.q + ((int64_t)cr * p.hq + ckvh * p.group) * kHeadDim, p.group, lane);
            else
                load_q_global(qb, p.q + ((int64_t)cr * p.hq + ckvh * p.group) * kHeadDim, p.group, lane);
            if (kFp8) sl2 = p.scale_log2 * cx.ks[ckvh];
            patch_tok = -1;
            if (fused) {
                // the appended token, if its granule is in this share, comes from k_new / v_new
                const int pos = p.positions[cr];
                const int pg = pos >= 0 ? cus + pos / kGranule : -1;
                if (pos >= 0 && pg >= (cus > wa ? cus : wa) && pg < (cus + cn < wb ? cus + cn : wb)) {
                    patch_tok = pos;
                    const uint4* src = reinterpret_cast<const uint4*>(
                        (lane < 16 ? p.k_new : p.v_new) + ((int64_t)cr * hk + ckvh) * kHeadDim);
                    patch_val = src[lane & 15];
                    if (kFp8) {  // FP8 pools hold the token as codes
                        const uint2 c8 = quantize8(patch_val, lane < 16 ? cx.ks[ckvh] : cx.vs[ckvh]);
                        patch_val = make_uint4(c8.x, c8.y, 0u, 0u);
                    }
                }
            }
        }
        unsigned char* sp = smem + Smem::ring + (warp * kSSlots + s) * kSlotBytes;
        const int prow = patch_tok >= 0 ? patch_tok - (g - cus) * kGranule : -1;
        if (prow >= 0 && prow < valid) patch_row<kFp8>(sp, prow, patch_val, lane);
        __syncwarp();
        if (kFp8)
            attend8(st, qb, sp, valid, sl2, lane);
        else
            attend(st, qb, slot0 + s * kSlotBytes, valid, sl2, lane);
        __syncwarp();  // the slot is read before its next copy is issued
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    if (cu >= 0) finish(true);
    if (parked) {
        // back into slot 1 for the combine (written by this warp above)
        __syncwarp();
        const uint4* src = reinterpret_cast<const uint4*>(scratch);
        uint4* dst = reinterpret_cast<uint4*>(smem + Smem::ring + (warp * kSSlots + 1) * kSlotBytes);
#pragma unroll 1
        for (int i = lane; i < (int)(kStateBytes / 16); i += 32) dst[i] = src[i];
    }
    named_sync(kBarStream, kSWarps * 32);

    // ---- combine: every unit of the block that is not whole in one share,
    // by the warps that hold its states ----
#pragma unroll 1
    for (int side = 0; side < 2; ++side) {
        // this warp's first unit, then its last one
        const int xr = side ? cr : fr, xkvh = side ? ckvh : fkvh;
        const int xus = side ? cus : fus, xn = side ? cn : fn;
        if (side == 1 && xus == fus && xr == fr && xkvh == fkvh) continue;  // the same unit
        if (xus >= wa && xus + xn <= wb) continue;                          // whole: done
        // warps a .. b hold the unit's states
        int a = 0, b = kSWarps - 1;
#pragma unroll 1
        for (int w = 0; w < kSWarps; ++w) {
            int xa, xb;
            stream_share(g0, g1, w, xa, xb);
            if (xb <= xus) a = w + 1;
            if (xa >= xus + xn && b == kSWarps - 1 && w > 0) b = w - 1;
        }
        int slot[kSWarps];
#pragma unroll
        for (int i = 0; i < kSWarps; ++i) slot[i] = 0;
#pragma unroll 1
        for (int w = a; w <= b; ++w) {
            int xa, xb;
            stream_share(g0, g1, w, xa, xb);
            // a unit that started before the warp's share and ends inside it
            // is the warp's first unit, finished early and parked
            const bool early = xus < xa && xus + xn < xb;
            slot[w - a] = w * kSSlots + (early ? 1 : 0);
        }
        const int cs = owner_of(xus, cx.W, cx.Geff);
        const int P = owner_of(xus + xn - 1, cx.W, cx.Geff) - cs + 1;
        const PieceOut po = piece_out(p, xr, xkvh, cs, P, cta, kFp8 ? cx.vs[xkvh] : 1.f);
        combine_dumps<kFp8>(po, smem + Smem::ring, slot, b - a + 1, warp - a, lane);
        if (P > 1 && warp == a && lane == 0) {
            // the block's split pieces (its first and its last) are its merge tasks
            const int k = atomicAdd(&bp->ntasks, 1);
            if (k < kMaxTasks) {
                Task& t = bp->tasks[k];
                t.u = xr * hk + xkvh;
                t.cs = cs;
                t.P = P;
                t.idx = cta - cs;
                t.r = xr;
                t.kvh = xkvh;
            }
        }
    }
    named_sync(kBarStream, kSWarps * 32);
}

// Burst mode, warp j of piece k's n warps (n > 1): chunks c = j, j + n, ...
// of the piece.  Combines the states the piece's warps dumped into their
// first slots through their log-sum-exp and emits each chunk (fp16 output of
// a whole unit, or the piece's record); warp 0 also emits a split piece's m/l.
template <bool kFp8>
__device__ void burst_emit(const PieceOut& po, const BlockPlan* bp, const unsigned char* ring, int k,
                           int j, int lane) {
    const int n = bp->pwn[k], w0 = bp->pw0[k], g0 = bp->g0, tq = lane & 3;
    uint32_t off[kConsumerWarps];
    float4 ml[kConsumerWarps];
#pragma unroll
    for (int s = 0; s < kConsumerWarps; ++s) {
        off[s] = (uint32_t)(bp->wa[w0 + (s < n ? s : 0)] - g0) * kSlotBytes;
        ml[s] = *reinterpret_cast<const float4*>(ring + off[s] + 16 * tq);
    }
    float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
    for (int s = 0; s < kConsumerWarps; ++s)
        if (s < n) {
            M0 = fmaxf(M0, ml[s].x);
            M1 = fmaxf(M1, ml[s].y);
        }
    float L0 = 0.f, L1 = 0.f;
#pragma unroll
    for (int s = 0; s < kConsumerWarps; ++s) {  // ml[s].x / .y become the weights
        ml[s].x = s < n && M0 != -INFINITY ? fast_exp2(ml[s].x - M0) : 0.f;
        ml[s].y = s < n && M1 != -INFINITY ? fast_exp2(ml[s].y - M1) : 0.f;
        L0 += ml[s].x * ml[s].z;
        L1 += ml[s].y * ml[s].w;
    }
#pragma unroll 1
    for (int c = j; c < 8; c += n) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s = 0; s < kConsumerWarps; ++s) {
            const float4 v = *reinterpret_cast<const float4*>(ring + off[s] + kMlBytes + c * kChunkBytes + lane * 16);
            acc[0] += ml[s].x * v.x;
            acc[1] += ml[s].y * v.y;
            acc[2] += ml[s].x * v.z;
            acc[3] += ml[s].y * v.w;
        }
        emit_chunk<kFp8>(po, c, acc, L0, L1, lane);
    }
    if (j == 0) emit_ml(po, M0, M1, L0, L1, lane);
}

template <bool kPaged, bool kFp8>
__global__ void __launch_bounds__(kThreads, 2)
    decode_tma_kernel(const __grid_constant__ Params prm) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Params& p = prm;
    const uint32_t sbase = smem_u32(smem);
    BlockPlan* bp = reinterpret_cast<BlockPlan*>(smem + Smem::plan);
    volatile int* sm_flags = reinterpret_cast<volatile int*>(smem + Smem::flags);
    int* sm_part = reinterpret_cast<int*>(smem + Smem::part);
    int* sm_pre = reinterpret_cast<int*>(smem + Smem::prefix);
    int* sm_len = reinterpret_cast<int*>(smem + Smem::lens(prm.rows));
    float* sm_ks = reinterpret_cast<float*>(smem + Smem::scales);  // FP8 only
    float* sm_vs = sm_ks + kFp8MaxKvHeads;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int G = gridDim.x;
    const int cta = blockIdx.x;
    const int hk = prm.hk;

    // The next kernel in the stream (launched with programmatic stream
    // serialization) may be scheduled as soon as every block has started:
    // its blocks then take the SMs' second slots as the blocks of the kernel
    // before this one leave, and prefetch their own work.  It waits for this
    // grid to complete before touching anything this grid writes.
    griddep_launch();
    if (warp == kConsumerWarps) {
        // the step's plan for this block: one 16-byte load per lane
        if (prm.plan)
            reinterpret_cast<uint4*>(bp)[lane] =
                __ldg(reinterpret_cast<const uint4*>(prm.plan + (size_t)cta * kPlanBytes) + lane);
    }
    if (tid == 0) {
        sm_flags[0] = 0;  // abort
        sm_flags[4] = sm_flags[5] = 0;  // a merge task's poll gave up
    }
    if (kFp8 && tid < 2 * hk) sm_ks[tid < hk ? tid : kFp8MaxKvHeads + tid - hk] =
        tid < hk ? prm.k_scale[tid] : prm.v_scale[tid - hk];
    __syncthreads();

    // ---- the block's plan: loaded (made for this grid), or made here ----
    int W, Geff;
    if (p.plan) {
        if (bp->G != G) {  // made for another grid: nothing is read or written
            if (tid == 0) flag_error(p.dev_err, PKV_DEV_ERR_PLAN);
            return;
        }
        W = bp->W;
        Geff = bp->Geff;
        // stream blocks walk their range through the granule prefix
        if (bp->mode == kModeStream) scan_lengths<kThreads>(p, kPaged, sm_pre, sm_len, sm_part, false);
    } else {
        W = scan_lengths<kThreads>(p, kPaged, sm_pre, sm_len, sm_part, cta == 0);
        Geff = W < G ? W : G;
        if (warp == kConsumerWarps) build_block_plan(bp, p, kPaged, cta, G, W, Geff, sm_pre, sm_len, lane);
        __syncthreads();
    }
    const int mode = bp->mode;
    const int g0 = bp->g0;
    Ctx cx;
    cx.smem = smem;
    cx.sbase = sbase;
    cx.bp = bp;
    cx.flags = sm_flags;
    cx.pre = sm_pre;
    cx.len = sm_len;
    cx.ks = sm_ks;
    cx.vs = sm_vs;
    cx.W = W;
    cx.Geff = Geff;

    if (warp == kConsumerWarps) {
        // ============================ row work ============================
        // Burst (or idle): the consumer warps stage their own granules; this
        // warp only does the block's row work after the dependency wait.
        griddep_wait();
        if (kPaged) row_work<kFp8>(p, cta, G, lane);
        return;
    }

    // ============================== consumers ==============================
    if (mode == kModeStream) {
        if (warp >= kSWarps) return;  // stream mode runs on warps 0 .. kSWarps-1
        stream_warp<kPaged, kFp8>(p, cx, cta, warp, lane,
                                  p.records + stream_scratch_offset(p) + ((size_t)cta * kSWarps + warp) * kStateBytes);
    } else {
        // ============================ burst mode ============================
        const int pi = bp->wpiece[warp];
        if (pi >= 0) {
            // This warp's granules go to their slots now, before the
            // dependency wait (the cached tokens are not written by the
            // preceding kernel; the appended one is patched in after it).
            const unsigned char* kpool = reinterpret_cast<const unsigned char*>(p.kbase);
            const unsigned char* vpool = reinterpret_cast<const unsigned char*>(p.vbase);
#pragma unroll 1
            for (int g = bp->wa[warp]; g < bp->wb[warp]; ++g) {
                const int si = g - g0, zrow = bp->szrow[si];
                stage_granule<kFp8>(sbase + Smem::ring + si * kSlotBytes, kpool, vpool, zrow < 0 ? 0 : zrow, hk,
                                    bp->skvh[si], zrow < 0 ? 0 : bp->svalid[si], lane);
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
            // Warm L2 with this warp's query rows and new token.  A prefetch
            // reads nothing into the block, so it may precede the dependency
            // wait: the values used are loaded after it.
            const int r = bp->pr[pi], kvh = bp->pkvh[pi];
            const char* qrow = reinterpret_cast<const char*>(p.q + ((int64_t)r * p.hq + kvh * p.group) * kHeadDim);
            if (lane < 2 * p.group)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(qrow + lane * 128));
            if (kPaged && p.positions && lane < 8) {
                const char* nt = reinterpret_cast<const char*>(
                    (lane < 4 ? p.k_new : p.v_new) + ((int64_t)r * hk + kvh) * kHeadDim);
                asm volatile("prefetch.global.L2 [%0];" ::"l"(nt + (lane & 3) * 64));
            }
        }
        // Everything below may read what the preceding kernel wrote (query,
        // positions, new tokens, workspace) or write what it reads.
        griddep_wait();
        if (mode == kModeIdle) return;
        const bool fused = kPaged && p.positions != nullptr;
        if (pi >= 0) {
            Soft st;
            st.reset();
            const int r = bp->pr[pi], kvh = bp->pkvh[pi], us = bp->pus[pi];
            const int a = bp->wa[warp], b = bp->wb[warp];
            uint32_t qb[16];
            if (kFp8)
                load_q_fp8(qb, p.q + ((int64_t)r * p.hq + kvh * p.group) * kHeadDim, p.group, lane);
            else
                load_q_global(qb, p.q + ((int64_t)r * p.hq + kvh * p.group) * kHeadDim, p.group, lane);
            // The appended token, if it falls inside this warp's granules, is
            // taken from k_new / v_new (its slot may be written concurrently).
            int patch_tok = -1;
            uint4 patch_val = make_uint4(0, 0, 0, 0);
            const int pos = fused ? bp->ppatch[pi] : -1;
            if (pos >= 0 && us + pos / kGranule >= a && us + pos / kGranule < b) {
                patch_tok = pos;
                const uint4* src = reinterpret_cast<const uint4*>(
                    (lane < 16 ? p.k_new : p.v_new) + ((int64_t)r * hk + kvh) * kHeadDim);
                patch_val = src[lane & 15];
                if (kFp8) {  // FP8 pools hold the token as codes
                    const uint2 c8 = quantize8(patch_val, lane < 16 ? sm_ks[kvh] : sm_vs[kvh]);
                    patch_val = make_uint4(c8.x, c8.y, 0u, 0u);
                }
            }
            const float sl2 = kFp8 ? p.scale_log2 * sm_ks[kvh] : p.scale_log2;
            // this lane's copies have landed; then every lane's
            asm volatile("cp.async.wait_group 0;" ::: "memory");
            __syncwarp();
#pragma unroll 1
            for (int g = a; g < b; ++g) {
                const int si = g - g0;
                unsigned char* sp = smem + Smem::ring + si * kSlotBytes;
                const int prow = patch_tok >= 0 ? patch_tok - (g - us) * kGranule : -1;
                if (prow >= 0 && prow < bp->svalid[si]) patch_row<kFp8>(sp, prow, patch_val, lane);
                __syncwarp();
                if (kFp8)
                    attend8(st, qb, sp, bp->svalid[si], sl2, lane);
                else
                    attend(st, qb, sbase + Smem::ring + si * kSlotBytes, bp->svalid[si], sl2, lane);
            }
            st.reduce_l();
            __syncwarp();
            // A piece of several warps: each dumps its state into its first
            // slot, and after the piece's barrier each combines a share of
            // the chunks of all of them.
            const int k = bp->pwn[pi];
            if (k > 1) {
                dump_state(st, smem + Smem::ring + (a - g0) * kSlotBytes, lane);
                named_sync(kBarPiece + pi, k * 32);
            }
            if (!sm_flags[0]) {
                const PieceOut po = piece_out(p, r, kvh, bp->pcs[pi], bp->pP[pi], cta, kFp8 ? sm_vs[kvh] : 1.f);
                if (k == 1) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) emit_chunk<kFp8>(po, c, st.o[c], st.l0, st.l1, lane);
                    emit_ml(po, st.m0, st.m1, st.l0, st.l1, lane);
                } else {
                    burst_emit<kFp8>(po, bp, smem + Smem::ring, pi, warp - bp->pw0[pi], lane);
                }
            }
        }
        // every dump has been read: the ring is free for the merges
        named_sync(kBarConsumers, kConsumers);
    }

    // ---- merges: the block's split pieces that make it a participant (the
    // first min(P, 8) pieces of their unit); with two such tasks the
    // consumer warps are halved between them ----
    if (sm_flags[0]) return;
    int ntask = 0, first = 0;
#pragma unroll
    for (int k = 0; k < kMaxTasks; ++k) {
        if (k >= bp->ntasks) break;
        const Task& tk = bp->tasks[k];
        if (tk.idx < (tk.P < kMergeWays ? tk.P : kMergeWays)) {
            if (ntask == 0) first = k;
            ++ntask;
        }
    }
    if (ntask == 0) return;
    const bool burst = mode == kModeBurst;
    const int nc = burst ? kConsumerWarps : kSWarps;
    const int half = nc / 2;
    const int t = ntask == 1 ? first : (warp < half ? 0 : 1);
    const int lw = (ntask == 1 || warp < half) ? warp : warp - half;
    const int nw = ntask == 1 ? nc : (t == 0 ? half : nc - half);
    const Task task = bp->tasks[t];
    merge_task<kFp8>(p, task, lw, nw, smem + Smem::ring + t * kLandBytes, kBarMerge + t,
               kFp8 ? sm_vs[task.kvh] : 1.f, sm_flags + 4 + t, lane);
}

// The plan of a step: every block scans the lengths, then warp w of block i
// makes the plan of decode block 32 i + w (and of those a grid stride
// further) and copies it out as 32 x 16 bytes.
__global__ void __launch_bounds__(kPlanThreads, 1)
    decode_plan_kernel(const Params p, unsigned char* plan, int G) {
    extern __shared__ __align__(16) unsigned char psm[];
    BlockPlan* bps = reinterpret_cast<BlockPlan*>(psm);
    int* part = reinterpret_cast<int*>(psm + (kPlanThreads / 32) * kPlanBytes);
    int* pre = part + kPlanThreads;
    int* len = pre + p.rows + 1;
    const int W = scan_lengths<kPlanThreads>(p, true, pre, len, part, blockIdx.x == 0);
    const int Geff = W < G ? W : G;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int b = blockIdx.x * (kPlanThreads / 32) + warp; b < G; b += gridDim.x * (kPlanThreads / 32)) {
        build_block_plan(bps + warp, p, true, b, G, W, Geff, pre, len, lane);
        reinterpret_cast<uint4*>(plan + (size_t)b * kPlanBytes)[lane] =
            reinterpret_cast<const uint4*>(bps + warp)[lane];
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------
// Host side

// Test hooks for the bounded waits of the split-unit merge (see
// pkv_debug_set_decode_hooks); zero / null in normal use.
static std::mutex g_hook_mutex;
static uint32_t g_hook_poll_limit = 0;
static const void* g_hook_stuck = nullptr;

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

// Blocks of a decode launch: one per SM, at most kMaxCtas and at most one per
// granule the sizes allow.  The plan and the decode launch agree on it.
static int decode_grid(int rows, int kv_heads, int limit, int* grid) {
    DeviceInfo* info = nullptr;
    const int st = device_info(&info);
    if (st != PKV_OK) return st;
    const int64_t granules = (int64_t)rows * kv_heads * ((limit + kGranule - 1) / kGranule);
    int64_t ctas = info->sms;
    if (ctas > kMaxCtas) ctas = kMaxCtas;
    if (ctas > granules) ctas = granules > 0 ? granules : 1;
    *grid = (int)ctas;
    return PKV_OK;
}

}  // namespace tma

bool tma_decode_supported(int rows, int q_heads, int kv_heads, int head_dim, int block_size) {
    return head_dim == kHeadDim && kv_heads > 0 && q_heads % kv_heads == 0 &&
           q_heads / kv_heads <= kMaxGroup && block_size % tma::kGranule == 0 && rows >= 0 &&
           rows <= tma::kMaxRows;
}

// Record slots a launch may use: one per block plus one per unit (a unit's
// records start at slot first block + unit).  Blocks are one per SM of the
// current device, so a workspace sized here serves any device with at most as
// many SMs.
static int64_t tma_slots(int rows, int kv_heads, int max_seq_len) {
    const int64_t units = (int64_t)rows * kv_heads;
    int ctas = tma::kMaxCtas;
    if (tma::decode_grid(rows, kv_heads, max_seq_len, &ctas) != PKV_OK) ctas = tma::kMaxCtas;
    return ctas + units;
}

size_t tma_workspace_bytes(int rows, int q_heads, int kv_heads, int max_seq_len) {
    (void)q_heads;
    // the records, then one parked state per stream warp of every block
    int ctas = tma::kMaxCtas;
    if (tma::decode_grid(rows, kv_heads, max_seq_len, &ctas) != PKV_OK) ctas = tma::kMaxCtas;
    return align_up((size_t)tma::kRecBytes * (size_t)tma_slots(rows, kv_heads, max_seq_len), 256) +
           (size_t)ctas * tma::kSWarps * tma::kStateBytes;
}

size_t tma_plan_bytes(int rows, int kv_heads, int max_seq_len) {
    const int64_t granules = (int64_t)rows * kv_heads * ((max_seq_len + tma::kGranule - 1) / tma::kGranule);
    const int64_t ctas = granules < tma::kMaxCtas ? (granules > 0 ? granules : 1) : tma::kMaxCtas;
    return (size_t)ctas * tma::kPlanBytes;
}

int tma_plan_launch(void* plan, size_t plan_bytes, const int32_t* tables, const int32_t* seq_lens,
                    const int32_t* positions, int rows, int q_heads, int kv_heads, int block_size,
                    int mbpr, int num_blocks, int max_seq_len, int32_t* dev_err,
                    cudaStream_t stream) {
    using namespace tma;
    if ((int64_t)num_blocks * block_size >= (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;
    int G = 0;
    int st = decode_grid(rows, kv_heads, max_seq_len, &G);
    if (st != PKV_OK) return st;
    if (plan_bytes < (size_t)G * kPlanBytes) return PKV_ERR_WORKSPACE;
    Params prm{};
    prm.tables = tables;
    prm.seq_lens = seq_lens;
    prm.rows = rows;
    prm.hq = q_heads;
    prm.hk = kv_heads;
    prm.group = q_heads / kv_heads;
    prm.bs = block_size;
    prm.mbpr = mbpr;
    prm.nb = num_blocks;
    prm.limit = max_seq_len;
    prm.dev_err = dev_err;
    prm.positions = positions;
    const size_t smem = (kPlanThreads / 32) * kPlanBytes + kPlanThreads * 4 + (size_t)(2 * rows + 1) * 4;
    decode_plan_kernel<<<(G + kPlanThreads / 32 - 1) / (kPlanThreads / 32), kPlanThreads, smem, stream>>>(
        prm, static_cast<unsigned char*>(plan), G);
    return launch_status();
}

size_t tma_workspace_zero_bytes(int rows, int kv_heads, int max_seq_len) {
    // every record word starts cleared (and each call leaves them so)
    return align_up((size_t)tma::kRecBytes * (size_t)tma_slots(rows, kv_heads, max_seq_len), 256);
}

int tma_decode_launch(void* out, const void* q, const void* k_base, const void* v_base,
                      const int32_t* tables, const int32_t* seq_lens, int rows, int q_heads,
                      int kv_heads, int block_size, float scale, int mbpr, int num_blocks,
                      int max_seq_len, int width, void* workspace, int32_t* dev_err,
                      cudaStream_t stream, const AppendArgs* append, bool pdl,
                      const float* k_scale, const float* v_scale, const void* plan) {
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
    int ctas = 0;
    if ((st = decode_grid(rows, kv_heads, limit, &ctas)) != PKV_OK) return st;
    if (plan && !paged) return PKV_ERR_UNSUPPORTED;

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
    {
        std::lock_guard<std::mutex> lock(g_hook_mutex);
        prm.poll_limit = g_hook_poll_limit ? g_hook_poll_limit : kPollLimit;
        prm.stuck = static_cast<const uint32_t*>(g_hook_stuck);
    }
    prm.plan = static_cast<const unsigned char*>(plan);
    prm.records = static_cast<unsigned char*>(workspace);
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
    prm.kbase = k_base;
    prm.vbase = v_base;

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
    if (cudaLaunchKernelEx(&cfg, kernel, prm) != cudaSuccess) return PKV_ERR_CUDA;
    return launch_status();
}

}  // namespace pkv

extern "C" int pkv_debug_set_decode_hooks(unsigned poll_limit, const void* stuck_word) {
    std::lock_guard<std::mutex> lock(pkv::tma::g_hook_mutex);
    pkv::tma::g_hook_poll_limit = poll_limit;
    pkv::tma::g_hook_stuck = stuck_word;
    return PKV_OK;
}
