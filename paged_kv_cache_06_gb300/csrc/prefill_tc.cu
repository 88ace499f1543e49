// Chunked-prefill paged attention on the 5th-generation tensor cores
// (tcgen05, accumulators and the probabilities in tensor memory), sm_103a.
//
// What it computes is paged_attention_prefill's definition ("Paged
// attention", danielfleming.xyz, closing sections: long prompts broken
// into fixed-size pieces with decode steps in between; "PagedAttention", deepconcepts.dev,
// section "PagedAttention": keys gathered through the row's block table):
// query i of row r's chunk sits at position seq_lens[r] - C_r + i and attends
// causally to the row's tokens 0 .. that position.
//
// Work.  A unit is 128 queries of one row and one query head; it walks the
// row's keys in 128-token tiles, one step per tile.  All steps of all units,
// in (row, head, query tile, key tile) order, are cut into one contiguous
// range per block, and one block runs per SM (persistent, stream-K), so every
// SM does the same number of steps whatever the number of units.  A unit
// inside one range is done by one block; a unit cut by range boundaries is
// done in pieces, each giving a partial result (row maxima, row sums, the
// unnormalised 128 x 128 output in fp32), and merged through their
// log-sum-exp ("PagedAttention", deepconcepts.dev, closing note on
// FlashAttention: the split softmax recombined exactly).  A block walks its
// segments from the last to the first: the piece that ends a split unit is
// the first segment of its block's range, so it is processed last, while the
// unit's other pieces are the last segments of the blocks before, processed
// first.  The end piece's block merges: once its S products are done, its
// S-issue thread waits (bounded) until the other pieces have counted
// themselves on its arrival word and lands the first other piece's partial in
// the idle K ring with one bulk copy; the softmax warps then combine the
// partials with their own state before they normalise and store.
//
// Warp roles (each walks the same segments):
//   warps 0-7  softmax: warps w and w + 4 share query rows 32 (w % 4) .. (TMEM
//              lanes); warp half hf = w / 4 takes tokens 64 hf .. 64 hf + 63 of
//              each tile and head dims 64 hf .. 64 hf + 63 of the output;
//   warp 8     TMA: K tiles into a 3-slot ring;
//   warp 9     TMA: V in 64-token halves into a 5-slot ring;
//              each K/V copy moves one box of 16, 32, 64 or 128 consecutive
//              tokens of one page (the largest that divides the page size),
//              its pool rows found through the block table;
//   warp 10    S issue: each segment's queries (once the previous segment's
//              products no longer read them), then
//              S_t[128 q][128 tok] = Q . K_t^T (both from shared memory);
//   warp 11    PV issue: O[128 q][128 dims] += P_t . V_t, P read from TMEM;
//              a segment's first product overwrites O only after the softmax
//              warps have read the previous segment's O out.
// One thread of each issuing warp drives tcgen05.mma (f16 in, f32
// accumulate) and commits each group to an mbarrier.  S is triple-buffered
// in TMEM and each softmax half stores its fp16 probabilities over the first
// half of its own S columns, so S_{t+3} reuses a buffer only after PV_t has
// read P_t.  Per tile a softmax thread reads its half S row, applies the
// causal mask, agrees on the row maximum with its partner warp, rescales its
// half O row in TMEM when the maximum moved, and stores its P.  The producer
// and issuer loops keep slots, parities and descriptors as running values:
// each of those warps runs alone, so its loop is a chain of dependent
// instructions.  Every wait sleeps in mbarrier.try_wait and is bounded in
// wall time; a block that gives up flags the error, tells its other warps to
// stop, and lets its copies in flight land before it frees tensor memory.
#include <mutex>

#include "pkv_internal.cuh"
#include "ptx.cuh"

namespace pkv {
namespace prefill_tc {
using namespace ptx;

constexpr int kQTile = 128;
constexpr int kKTile = 128;
constexpr int kGranule = 16;  // the k-step of the PV product and the smallest copy box
constexpr int kKSlots = 3;     // K ring, 128 tokens a slot; free once its S product is done
constexpr int kVSlots = 5;     // V ring, 64 tokens a slot; free once its PV product is done
constexpr int kSBufs = 3;      // S buffers in TMEM
constexpr int kSoftWarps = 8;
constexpr int kThreads = (kSoftWarps + 4) * 32;  // softmax, K TMA, V TMA, S issue, PV issue
constexpr int kMaxRows = 1024;
constexpr int kMaxGrid = 192;   // persistent blocks: one per SM, at most this many
constexpr int kCountStride = 32;  // ints between two blocks' arrival words
constexpr uint32_t kHalfQ = kQTile * 128;        // 128 queries x 64 dims
constexpr uint32_t kKHalf = kKTile * 128;        // 128 tokens x 64 dims
constexpr uint32_t kKSlot = 2 * kKHalf;          // K lo, K hi
constexpr uint32_t kVHalf = 64 * 128;            // 64 tokens x 64 dims
constexpr uint32_t kVSlot = 2 * kVHalf;          // V lo, V hi
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // S buffers [0, 128), [128, 256), [256, 384); P over [0, 32) and [64, 96) of each
constexpr uint32_t kColO = 384;  // O [384, 512)
// A partial: m[128], l[128], then O as [32 groups of 4 dims][128 rows][4], so
// that a warp's 32 rows of one group are 512 contiguous bytes.
constexpr int kPartFloats = 2 * kQTile + kQTile * kHeadDim;
constexpr float kLog2e = 1.4426950408889634f;

struct Params {
    const __half* q;
    __half* out;
    const int32_t* tables;
    const int32_t* seq_lens;
    const int32_t* q_start;
    int rows, hq, group, bs, mbpr, nb, limit;
    int kbox, vbox;  // tokens per K and V copy
    float scale_log2;
    int out_v8;      // out is 32-byte aligned: 32-byte stores
    float* part;     // [grid][kPartFloats]: the partial of each block's cut unit
    int* count;      // [grid][kCountStride]: pieces arrived for the unit a block merges (zero between calls)
    int32_t* dev_err;
};

struct Smem {
    static constexpr uint32_t q = 0;                               // Q lo, Q hi
    static constexpr uint32_t kring = q + 2 * kHalfQ;              // [K slots]
    static constexpr uint32_t vring = kring + kKSlots * kKSlot;    // [V slots]
    static constexpr uint32_t bars = vring + kVSlots * kVSlot;     // 35 mbarriers
    static constexpr uint32_t tmem = bars + 40 * 8;                // allocated TMEM address
    static constexpr uint32_t misc = tmem + 16;                    // start unit, abort flag [8]
    static constexpr uint32_t xch = misc + 32;                     // row maxima [2][2][128], sums [2][128]
    static constexpr uint32_t rowc = xch + 6 * kQTile * 4;         // per row: chunk length C [rows]
    static constexpr uint32_t rowp = rowc + kMaxRows * 4;          // per row: first query position [rows]
    static constexpr uint32_t rowq = rowp + kMaxRows * 4;          // per row: q_start [rows]
    // The scan's scratch (partials [threads], step prefix [rows + 1]) lives
    // in the K ring: it is read before the first copy is issued.
    static constexpr uint32_t part = kring;
    static constexpr uint32_t pre = part + kThreads * 4;
    __host__ __device__ static constexpr uint32_t total() { return rowq + kMaxRows * 4 + 1024; }
};
static_assert(Smem::kring % 1024 == 0 && Smem::vring % 1024 == 0 && (Smem::q + kHalfQ) % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(Smem::pre + (kMaxRows + 1) * 4 <= Smem::kring + kKSlots * kKSlot, "scan scratch fits the K ring");
static_assert(Smem::total() <= 232448, "shared memory per block");
static_assert(kQTile == kKTile, "a unit's key tiles line up with its query tile");

// Key tiles of query tile t of a row whose chunk has C queries, the first at
// position pos0: keys 0 .. pos0 + min(128 (t + 1), C) - 1 are visible to it.
__device__ __forceinline__ int tiles_of(int pos0, int C, int t) {
    return (pos0 + min(kQTile * (t + 1), C) + kKTile - 1) / kKTile;
}

// A block's position in its range: the unit (row r, head h, query tile t)
// starting at step U with nkt steps, and the end e of the segment in it.
struct Walk {
    int r, h, t, U, nkt, e, s0, hq;
    const int* C;
    const int* pos0;
    __device__ __forceinline__ int k0() const { return s0 > U ? s0 - U : 0; }
    __device__ __forceinline__ int k1() const { return min(e - U, nkt); }
    // Step back to the previous unit; false once the range is done.
    __device__ __forceinline__ bool prev() {
        if (U <= s0) return false;
        e = U;
        if (t > 0) {
            --t;
        } else if (h > 0) {
            --h;
            t = (C[r] + kQTile - 1) / kQTile - 1;
        } else {
            do --r; while (C[r] == 0);
            h = hq - 1;
            t = (C[r] + kQTile - 1) / kQTile - 1;
        }
        nkt = tiles_of(pos0[r], C[r], t);
        U -= nkt;
        return true;
    }
};
// Shared-memory matrix descriptor: 128-byte swizzle, version 1.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: f16 A and B, f32 D, M x N, B major-ness.
__device__ __forceinline__ uint32_t idesc(int M, int N, int b_mn_major) {
    return (1u << 4) | ((uint32_t)b_mn_major << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}
// D (TMEM) (+)= A (shared memory) . B (shared memory)
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(id), "r"(accumulate));
}
// D (TMEM) (+)= A (TMEM: row m in lane m, column c holds k = 2c, 2c + 1) . B (shared memory)
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t id,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(id), "r"(accumulate));
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Columns c .. c + 31 of this warp's 32 lanes; the wait is part of the same
// statement, so no use of v can be scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t addr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(addr)
        : "memory");
}
// Columns c .. c + 63: two loads, one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t addr, uint32_t (&v)[32], uint32_t (&w)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]),
          "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7]), "=r"(w[8]), "=r"(w[9]), "=r"(w[10]), "=r"(w[11]), "=r"(w[12]), "=r"(w[13]), "=r"(w[14]), "=r"(w[15]), "=r"(w[16]), "=r"(w[17]), "=r"(w[18]), "=r"(w[19]), "=r"(w[20]), "=r"(w[21]), "=r"(w[22]), "=r"(w[23]), "=r"(w[24]), "=r"(w[25]), "=r"(w[26]), "=r"(w[27]), "=r"(w[28]), "=r"(w[29]), "=r"(w[30]), "=r"(w[31])
        : "r"(addr), "r"(addr + 32)
        : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t addr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(addr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
        "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
        "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// Waits that sleep: try_wait with a suspend-time hint parks the thread
// until the phase completes (or the hint runs out) instead of spinning, so a
// waiting warp leaves the issue slots to the warps that share its
// scheduler.  Each wait gives up after kWaitLimitNs of wall time.
constexpr uint32_t kSuspendNs = 1000000;
constexpr uint64_t kWaitLimitNs = 1000000000ull;
__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}
// One thread's bounded wait (the issuing threads wait alone).  It also gives
// up once another warp of the block has raised the abort flag.
__device__ __forceinline__ bool mbar_wait1(uint32_t bar, uint32_t parity, const volatile int* abort) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    const uint64_t t0 = now_ns();
    while (now_ns() - t0 < kWaitLimitNs) {
        if (*abort) return false;
        if (mbar_try_wait_sleep(bar, parity)) return true;
    }
    return false;
}
// The whole warp waits and leaves together (true) or gives up together.
__device__ __forceinline__ bool mbar_waitw(uint32_t bar, uint32_t parity, const volatile int* abort) {
    if (__all_sync(0xffffffffu, mbar_try_wait_sleep(bar, parity))) return true;
    const uint64_t t0 = __shfl_sync(0xffffffffu, now_ns(), 0);
    for (;;) {
        if (__any_sync(0xffffffffu, *abort != 0)) return false;
        if (__all_sync(0xffffffffu, mbar_try_wait_sleep(bar, parity))) return true;
        const bool late = __shfl_sync(0xffffffffu, now_ns(), 0) - t0 >= kWaitLimitNs;
        if (late) return false;
    }
}
// A wait for copies or products already issued, which complete whatever the
// other warps do: used before the block exits, so it ignores the abort flag.
__device__ __forceinline__ bool mbar_drain1(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = now_ns();
    do {
        if (mbar_try_wait_sleep(bar, parity)) return true;
    } while (now_ns() - t0 < kWaitLimitNs);
    return false;
}

// Sixteen fp16 outputs (8 words) to a 32-byte-aligned address.
__device__ __forceinline__ void st_v8(void* dst, const uint32_t (&u)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst), "r"(u[0]), "r"(u[1]),
                 "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]), "r"(u[6]), "r"(u[7])
                 : "memory");
}

// Bring one box of a tensor map into L2 ahead of its load.
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// Block that holds step s of W steps cut into Ge equal ranges.
__device__ __forceinline__ int owner_of(int s, int W, int Ge) {
    return (int)(((int64_t)(s + 1) * Ge + W - 1) / W) - 1;
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap,
                      const __grid_constant__ CUtensorMap qmap, const Params p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_q = sbase + Smem::bars;               // queries landed
    const uint32_t bar_kfull = bar_q + 8;                    // [K slots]
    const uint32_t bar_kempty = bar_kfull + kKSlots * 8;     // [K slots]
    const uint32_t bar_vfull = bar_kempty + kKSlots * 8;     // [V slots]
    const uint32_t bar_vempty = bar_vfull + kVSlots * 8;     // [V slots]
    const uint32_t bar_s = bar_vempty + kVSlots * 8;  // [3]: S buffer b computed (tiles b, b + 3, ...)
    const uint32_t bar_p = bar_s + 8 * kSBufs;  // [3]: P of S buffer b written
    const uint32_t bar_o = bar_p + 8 * kSBufs;  // [3]: PV product of buffer b done
    const uint32_t bar_x = bar_o + 8 * kSBufs;  // [2]: both halves' row maxima of a tile written
    const uint32_t bar_l = bar_x + 16;          // both halves' row sums written
    const uint32_t bar_qfree = bar_l + 8;       // a segment's S products are done with its queries
    const uint32_t bar_odrained = bar_qfree + 8;  // the softmax warps have read a segment's O out
    const uint32_t bar_sfin = bar_odrained + 8;   // the S issuer's last products are complete
    const uint32_t bar_pfin = bar_sfin + 8;       // the PV issuer's last products are complete
    const uint32_t bar_pub = bar_pfin + 8;        // the softmax warps have written the block's partial
    const uint32_t bar_mrg = bar_pub + 8;         // the pieces of the unit this block merges have arrived
    uint32_t* sm_tmem = reinterpret_cast<uint32_t*>(smem + Smem::tmem);
    volatile int* sm_misc = reinterpret_cast<volatile int*>(smem + Smem::misc);
    const volatile int* abort = sm_misc + 4;
    int* sm_part = reinterpret_cast<int*>(smem + Smem::part);
    int* sm_pre = reinterpret_cast<int*>(smem + Smem::pre);
    int* sm_C = reinterpret_cast<int*>(smem + Smem::rowc);
    int* sm_p0 = reinterpret_cast<int*>(smem + Smem::rowp);
    int* sm_qs = reinterpret_cast<int*>(smem + Smem::rowq);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rows = p.rows, hq = p.hq;

    // ---- per row: chunk length, first query position, steps; their prefix ----
    // A row's query tile t sees tiles_of(pos0, C, t) key tiles: ceil(pos0 / 128)
    // + t + 1 for every tile but the last, which sees all ceil(L / 128).
    const int per = (rows + kThreads - 1) / kThreads;
    int sum = 0;
    for (int i = 0; i < per; ++i) {
        const int r = tid * per + i;
        if (r < rows) {
            const int q0 = p.q_start[r];
            int C = p.q_start[r + 1] - q0;
            const int L = p.seq_lens[r];
            if (C < 0 || L < C || L > p.limit) {
                if (blockIdx.x == 0) flag_error(p.dev_err, PKV_DEV_ERR_SEQ_LEN);
                C = 0;
            }
            const int pos0 = L - C;
            sm_C[r] = C;
            sm_p0[r] = pos0;
            sm_qs[r] = q0;
            int64_t steps = 0;
            if (C > 0) {
                const int64_t nt = (C + kQTile - 1) / kQTile, a = (pos0 + kKTile - 1) / kKTile;
                steps = (nt - 1) * nt / 2 + (nt - 1) * a + (L + kKTile - 1) / kKTile;
            }
            sm_pre[r] = (int)(steps * hq);  // below 2^31 in total (checked by the host)
            sum += sm_pre[r];
        }
    }
    sm_part[tid] = sum;
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

    // ---- this block's range [s0, s1) of the W steps, over Ge <= grid blocks
    // (every participating block gets at least one step) ----
    const int W = sm_pre[rows];
    const int Ge = W < (int)gridDim.x ? W : (int)gridDim.x;
    const int cta = blockIdx.x;
    if (cta >= Ge) return;
    const int s0 = (int)((int64_t)W * cta / Ge);
    const int s1 = (int)((int64_t)W * (cta + 1) / Ge);
    if (tid == 0) {
        // the unit holding step s1 - 1: row, head, then query tile, whose
        // steps start at t (t + 1) / 2 + t a (a = ceil(pos0 / 128)) in the head
        const int x = s1 - 1;
        int lo = 0, hi = rows - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (sm_pre[mid] <= x) lo = mid; else hi = mid - 1;
        }
        const int r = lo;
        const int wh = (sm_pre[r + 1] - sm_pre[r]) / hq;
        const int off = x - sm_pre[r];
        const int h = off / wh, o2 = off - h * wh;
        const int64_t a = (sm_p0[r] + kKTile - 1) / kKTile;
        int tl = 0, th = (sm_C[r] + kQTile - 1) / kQTile - 1;
        while (tl < th) {
            const int tm = (tl + th + 1) >> 1;
            if ((int64_t)tm * (tm + 1) / 2 + tm * a <= o2) tl = tm; else th = tm - 1;
        }
        sm_misc[0] = r;
        sm_misc[1] = h;
        sm_misc[2] = tl;
        sm_misc[3] = sm_pre[r] + h * wh + (int)((int64_t)tl * (tl + 1) / 2 + tl * a);
        sm_misc[4] = 0;  // abort
        sm_misc[5] = 0;  // merge: the other pieces arrived
    }

    // ---- barriers and tensor memory (the scan scratch is dead from here) ----
    if (tid == 0) {
        mbar_init(bar_q, 1);
        for (int s = 0; s < kKSlots; ++s) {
            mbar_init(bar_kfull + 8 * s, 1);
            mbar_init(bar_kempty + 8 * s, 1);
        }
        for (int s = 0; s < kVSlots; ++s) {
            mbar_init(bar_vfull + 8 * s, 1);
            mbar_init(bar_vempty + 8 * s, 1);
        }
        mbar_init(bar_l, kSoftWarps);
        for (int b2 = 0; b2 < 2; ++b2) mbar_init(bar_x + 8 * b2, kSoftWarps);
        for (int b3 = 0; b3 < kSBufs; ++b3) {
            mbar_init(bar_s + 8 * b3, 1);
            mbar_init(bar_p + 8 * b3, kSoftWarps);
            mbar_init(bar_o + 8 * b3, 1);
        }
        mbar_init(bar_qfree, 1);
        mbar_init(bar_odrained, kSoftWarps);
        mbar_init(bar_sfin, 1);
        mbar_init(bar_pfin, 1);
        mbar_init(bar_pub, kSoftWarps);
        mbar_init(bar_mrg, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         sbase + Smem::tmem),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sm_tmem;
    auto raise_abort = [&]() { sm_misc[4] = 1; };

    // Every role walks the block's segments, last to first.
    Walk w;
    w.r = sm_misc[0];
    w.h = sm_misc[1];
    w.t = sm_misc[2];
    w.U = sm_misc[3];
    w.e = s1;
    w.s0 = s0;
    w.hq = hq;
    w.C = sm_C;
    w.pos0 = sm_p0;
    w.nkt = tiles_of(sm_p0[w.r], sm_C[w.r], w.t);

    if (warp == kSoftWarps || warp == kSoftWarps + 1) {
        // ============================== TMA ==============================
        // Warp kSoftWarps streams K tiles, the next warp V halves; each
        // granule's pool rows come from the block table.
        const bool is_v = warp == kSoftWarps + 1;
        const int nslots = is_v ? kVSlots : kKSlots;
        const int unit_tok = is_v ? 64 : kKTile;
        const uint32_t full0 = is_v ? bar_vfull : bar_kfull;
        const uint32_t empty0 = is_v ? bar_vempty : bar_kempty;
        const uint32_t ring = sbase + (is_v ? Smem::vring : Smem::kring);
        const uint32_t slot_bytes = is_v ? kVSlot : kKSlot;
        const uint32_t half_bytes = is_v ? kVHalf : kKHalf;
        const CUtensorMap* map = is_v ? &vmap : &kmap;
        // Block-table entries are fetched a batch ahead: lane l handles box
        // l % gpu of unit l / gpu of a batch of 32 / gpu units, so the
        // table's latency is paid once per batch and hidden behind the
        // previous one.  Slots, parities and addresses advance by increments:
        // this warp runs alone, and its loop is a chain of dependent
        // instructions.
        const int box = is_v ? p.vbox : p.kbox;
        const int gpu = unit_tok / box;        // boxes per unit
        const int upb = 32 / gpu;              // units per batch
        const int my_j = lane / gpu, my_g = lane % gpu;
        const uint32_t box_bytes = (uint32_t)box * 128;
        int s = 0, armed = 0;
        uint32_t ph = 0, fb = full0, eb = empty0, slot = ring;
        bool ok = true;
        do {
            const int r = w.r, C = sm_C[r];
            const int kend = sm_p0[r] + w.t * kQTile + min(kQTile, C - w.t * kQTile);
            const int kvh = w.h / p.group;
            const int ua = is_v ? 2 * w.k0() : w.k0();
            const int ue = is_v ? min(2 * w.k1(), (kend + 63) / 64) : w.k1();
            const int32_t* trow = p.tables + (int64_t)r * p.mbpr;
            auto fetch = [&](int ub) -> int {  // raw block id of this lane's box in the batch at unit ub
                const int tok0 = (ub + my_j) * unit_tok + my_g * box;
                return tok0 < kend ? __ldg(trow + tok0 / p.bs) : 0;
            };
            auto to_row = [&](int ub, int pb) -> int {  // its pool row, or -1 for no copy
                const int tok0 = (ub + my_j) * unit_tok + my_g * box;
                if (tok0 >= kend) return -1;
                if (pb < 0 || pb >= p.nb) {
                    flag_error(p.dev_err, PKV_DEV_ERR_BLOCK_ID);
                    return -1;
                }
                return pb * p.bs + tok0 % p.bs;
            };
            int pb_next = fetch(ua);
            int row = to_row(ua, pb_next);
            pb_next = fetch(ua + upb);
            int j = 0;
            for (int u = ua; u < ue; ++u) {
                if (!mbar_waitw(eb, ph ^ 1, abort)) {
                    ok = false;
                    break;
                }
                const bool issue = my_j == j && row >= 0;
                const uint32_t nissue = __popc(__ballot_sync(0xffffffffu, issue));
                if (lane == 0) mbar_arrive_expect_tx(fb, nissue * 2 * box_bytes);
                __syncwarp();
                if (issue) {
                    const uint32_t st = slot + my_g * box_bytes;
                    tma_load_3d(st, map, 0, kvh, row, fb);
                    tma_load_3d(st + half_bytes, map, 64, kvh, row, fb);
                }
                ++armed;
                if (++j == upb) {
                    j = 0;
                    row = to_row(u + 1, pb_next);
                    pb_next = fetch(u + 1 + upb);
                }
                if (++s == nslots) {
                    s = 0;
                    ph ^= 1;
                    fb = full0;
                    eb = empty0;
                    slot = ring;
                } else {
                    fb += 8;
                    eb += 8;
                    slot += slot_bytes;
                }
            }
        } while (ok && w.prev());
        if (!ok && lane == 0) {
            raise_abort();
            flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
        }
        // every armed slot's copies have landed before the block exits
        for (int u = max(0, armed - nslots); u < armed; ++u)
            if (!mbar_drain1(full0 + 8 * (u % nslots), (uint32_t)(u / nslots) & 1) && lane == 0)
                flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
        __syncwarp();
    } else if (warp == kSoftWarps + 2) {
        // ============================ S issue ============================
        // Per segment: its queries, once the previous segment's products are
        // done with the buffer; then S_t = Q . K_t^T into S buffer t % 3, once
        // K_t has landed and PV_{t-3} has read P_{t-3} out of that buffer.
        if (lane == 0) {
            const uint32_t id_s = idesc(kQTile, kKTile, 0);
            const uint64_t kd0 = sdesc(sbase + Smem::kring, 16, 1024);
            uint64_t kd = kd0;
            const uint64_t qd = sdesc(sbase + Smem::q, 16, 1024);
            uint32_t kf = bar_kfull, ke = bar_kempty, ph = 0;
            int s = 0, sb = 0, gt = 0, seg = 0;
            uint32_t sph = 0;  // use parity of S buffer sb
            bool ok = true, q_pending = false;
            do {
                if (seg > 0 && !(ok = mbar_wait1(bar_qfree, (uint32_t)(seg - 1) & 1, abort))) break;
                const int qrow0 = sm_qs[w.r] + w.t * kQTile;
                mbar_arrive_expect_tx(bar_q, 2 * kHalfQ);
                tma_load_3d(sbase + Smem::q, &qmap, 0, w.h, qrow0, bar_q);
                tma_load_3d(sbase + Smem::q + kHalfQ, &qmap, 64, w.h, qrow0, bar_q);
                q_pending = true;
                if (!(ok = mbar_wait1(bar_q, (uint32_t)seg & 1, abort))) break;
                q_pending = false;
                {
                    // the next segment's queries come from L2 when it starts
                    Walk nx = w;
                    if (nx.prev()) {
                        const int nrow = sm_qs[nx.r] + nx.t * kQTile;
                        tma_prefetch_l2_3d(&qmap, 0, nx.h, nrow);
                        tma_prefetch_l2_3d(&qmap, 64, nx.h, nrow);
                    }
                }
                const int k1 = w.k1();
                for (int kt = w.k0(); kt < k1; ++kt, ++gt) {
                    if (!(ok = mbar_wait1(kf, ph, abort))) break;
                    if (gt >= kSBufs && !(ok = mbar_wait1(bar_o + 8 * sb, sph ^ 1, abort))) break;
                    tc_fence_after();
                    const uint32_t d = tmem + kColS + sb * kKTile;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t off = (uint32_t)((((ks >> 2) * kHalfQ) + (ks & 3) * 32) >> 4);
                        umma_ss(d, qd + off, kd + off, id_s, ks > 0);
                    }
                    umma_commit(bar_s + 8 * sb);
                    umma_commit(ke);  // K_t is no longer read
                    if (++sb == kSBufs) {
                        sb = 0;
                        sph ^= 1;
                    }
                    if (++s == kKSlots) {
                        s = 0;
                        ph ^= 1;
                        kd = kd0;
                        kf = bar_kfull;
                        ke = bar_kempty;
                    } else {
                        kd += kKSlot >> 4;
                        kf += 8;
                        ke += 8;
                    }
                }
                if (!ok) break;
                umma_commit(bar_qfree);  // the queries are free once these products are done
                ++seg;
            } while (w.prev());
            if (!ok) {
                raise_abort();
                flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
            }
            // the block exits only after its copies and products are complete
            if (q_pending && !mbar_drain1(bar_q, (uint32_t)seg & 1)) flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
            umma_commit(bar_sfin);
            if (!mbar_drain1(bar_sfin, 0)) flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
            // The block's last segment ends a unit cut over blocks cf .. cta:
            // once the K ring is idle, wait (bounded) until the other pieces
            // have counted, then land block cf's partial there while the
            // softmax warps finish their last tiles.
            if (w.k0() > 0 && w.k1() == w.nkt) {
                const int cf = owner_of(w.U, W, Ge);
                int* word = p.count + (int64_t)cta * kCountStride;
                int seen = 0;
                const uint64_t t0 = now_ns();
                if (ok) {
                    do {
                        asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(seen) : "l"(word) : "memory");
                        if (seen >= cta - cf) break;
                        __nanosleep(64);
                    } while (now_ns() - t0 < kWaitLimitNs && !*abort);
                }
                if (ok && seen >= cta - cf) {
                    *word = 0;  // re-armed for the next call
                    sm_misc[5] = 1;
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    mbar_arrive_expect_tx(bar_mrg, (uint32_t)kPartFloats * 4u);
                    bulk_load(sbase + Smem::kring, p.part + (int64_t)cf * kPartFloats,
                              (uint32_t)kPartFloats * 4u, bar_mrg);
                    if (!mbar_drain1(bar_mrg, 0)) flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
                } else {
                    if (ok) flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
                    mbar_arrive(bar_mrg);  // sm_misc[5] stays 0: the softmax warps give up
                }
            }
        }
        __syncwarp();
    } else if (warp == kSoftWarps + 3) {
        // ============================ PV issue ===========================
        // O += P_kt . V_kt once both V halves have landed and the softmax
        // has stored P_kt; a segment's first product starts O afresh, after
        // the softmax warps have read the previous segment's O.  K-steps past
        // the last visible key are skipped and rows of the last granule past
        // it are zeroed (0 * V must stay 0 whatever the pool holds there).
        if (lane == 0) {
            const uint32_t id_o = idesc(kQTile, 128, 1);
            const uint64_t vd0 = sdesc(sbase + Smem::vring, kVHalf, 1024);
            int va = 0;        // V slot of half 2 kt
            uint32_t vph = 0;  // its fill parity
            int pb = 0;        // S buffer holding P_kt
            uint32_t pph = 0;  // its use parity
            int seg = 0;
            bool ok = true;
            do {
                const int r = w.r, C = sm_C[r];
                const int kend = sm_p0[r] + w.t * kQTile + min(kQTile, C - w.t * kQTile);
                const int nvh = (kend + 63) / 64;
                const int k0 = w.k0(), k1 = w.k1();
                for (int kt = k0; kt < k1; ++kt) {
                    int vb = va + 1;
                    uint32_t vphb = vph;
                    if (vb == kVSlots) {
                        vb = 0;
                        vphb ^= 1;
                    }
                    const bool two = 2 * kt + 1 < nvh;
                    const int vrows = min(kKTile, kend - kt * kKTile);
                    const int nsteps = (vrows + 15) / 16;
                    if (!(ok = mbar_wait1(bar_vfull + 8 * va, vph, abort))) break;
                    if (two && !(ok = mbar_wait1(bar_vfull + 8 * vb, vphb, abort))) break;
                    if (vrows < nsteps * 16) {
                        const int zr0 = vrows, zn = nsteps * 16 - vrows;
                        unsigned char* vs = smem + Smem::vring + (zr0 >= 64 ? vb : va) * kVSlot;
                        for (int i = 0; i < zn * 16; ++i) {
                            const int row = (zr0 & 63) + (i >> 4), c = i & 15;
                            *reinterpret_cast<uint4*>(vs + (c >> 3) * kVHalf + row * 128 +
                                                      (((c & 7) ^ (row & 7)) << 4)) = make_uint4(0, 0, 0, 0);
                        }
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    }
                    if (!(ok = mbar_wait1(bar_p + 8 * pb, pph, abort))) break;
                    if (kt == k0 && seg > 0 &&
                        !(ok = mbar_wait1(bar_odrained, (uint32_t)(seg - 1) & 1, abort)))
                        break;
                    tc_fence_after();
                    const uint32_t pa = tmem + kColS + pb * kKTile;
                    const uint64_t da = vd0 + (uint64_t)(va * (kVSlot >> 4));
                    const uint64_t db = vd0 + (uint64_t)(vb * (kVSlot >> 4));
                    // tokens 64 e .. 64 e + 63 sit in columns 64 e .. 64 e + 31
                    if (nsteps == 8 && kt > k0) {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            umma_ts(tmem + kColO, pa + (kk >> 2) * 64 + (kk & 3) * 8,
                                    (kk < 4 ? da : db) + (uint64_t)((kk & 3) * 128), id_o, 1u);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            if (kk < nsteps)
                                umma_ts(tmem + kColO, pa + (kk >> 2) * 64 + (kk & 3) * 8,
                                        (kk < 4 ? da : db) + (uint64_t)((kk & 3) * 128), id_o,
                                        (kt > k0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    umma_commit(bar_o + 8 * pb);
                    umma_commit(bar_vempty + 8 * va);
                    if (two) umma_commit(bar_vempty + 8 * vb);
                    // the next tile's first half follows this tile's last one
                    va = two ? vb + 1 : vb;
                    vph = vphb;
                    if (va == kVSlots) {
                        va = 0;
                        vph ^= 1;
                    }
                    if (++pb == kSBufs) {
                        pb = 0;
                        pph ^= 1;
                    }
                }
                ++seg;
            } while (ok && w.prev());
            if (!ok) {
                raise_abort();
                flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
            }
            umma_commit(bar_pfin);
            if (!mbar_drain1(bar_pfin, 0)) flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
        }
        __syncwarp();
    } else {
        // ============================ softmax =============================
        // The two halves of a row agree on its maximum through shared memory
        // (bounded mbarrier waits), so both use one reference.
        const int quarter = warp & 3, hf = warp >> 2;
        const int i = quarter * 32 + lane;  // query row of the tile, TMEM lane
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        float* xmax = reinterpret_cast<float*>(smem + Smem::xch);  // [2][2][128]
        float* xsum = xmax + 4 * kQTile;                            // [2][128]
        bool ok = true;
        int sb = 0, psb = 0;          // S buffer of this tile and of the previous one
        uint32_t sph = 0, psph = 0;   // their use parities
        int gt = 0, seg = 0;          // tiles and segments done by this block
        do {
            const int r = w.r, C = sm_C[r], h = w.h;
            const int i_first = w.t * kQTile;
            const int nq = min(kQTile, C - i_first);
            const int pos0 = sm_p0[r];
            const int kend = pos0 + i_first + nq;  // keys 0 .. kend-1 are visible to someone
            const int vis = min(pos0 + i_first + i, kend - 1);
            const int k0 = w.k0(), k1 = w.k1();
            float m = -INFINITY, l = 0.f;
            for (int kt = k0; kt < k1; ++kt, ++gt) {
                if (!(ok = mbar_waitw(bar_s + 8 * sb, sph, abort))) break;
                tc_fence_after();
                float s[64];
                {
                    uint32_t v0[32], v1[32];
                    tmem_ld64(tmem + lane_base + kColS + sb * kKTile + hf * 64, v0, v1);
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        s[c] = __uint_as_float(v0[c]);
                        s[32 + c] = __uint_as_float(v1[c]);
                    }
                }
                const int t0 = kt * kKTile + hf * 64;
                if (t0 + 63 > vis) {
#pragma unroll
                    for (int c = 0; c < 64; ++c) s[c] = t0 + c <= vis ? s[c] : -INFINITY;
                }
                float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < 64; ++c) mx4[c & 3] = fmaxf(mx4[c & 3], s[c]);
                const float pm = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
                xmax[((gt & 1) * 2 + hf) * kQTile + i] = pm;
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_x + 8 * (gt & 1));
                if (!(ok = mbar_waitw(bar_x + 8 * (gt & 1), ((uint32_t)gt >> 1) & 1, abort))) break;
                const float mx = fmaxf(pm, xmax[((gt & 1) * 2 + (hf ^ 1)) * kQTile + i]) * p.scale_log2;
                // Lazy rescaling: the reference maximum m only moves when a score
                // exceeds it by more than 2^8 (weights stay <= 256, exact enough in
                // fp16).  A piece that starts past some query's last key leaves that
                // row at m = -inf (and zero weights) until a visible key comes.
                float alpha = 1.f;
                bool moved = false;
                if (mx > m + 8.f) {
                    alpha = fast_exp2(m - mx);  // 0 while m is -inf
                    m = mx;
                    moved = kt > k0;
                }
                const float mneg = m == -INFINITY ? 0.f : -m;
                uint32_t pk[32];
                // scores in pairs: one packed FMA for the exponents, one
                // packed add for the row sums (two pairs of partial sums)
                const uint64_t sc2 = f32x2(p.scale_log2, p.scale_log2), mn2 = f32x2(mneg, mneg);
                uint64_t rs2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    float x0, x1;
                    f32x2_split(fma_f32x2(f32x2(s[2 * c], s[2 * c + 1]), sc2, mn2), x0, x1);
                    const float e0 = fast_exp2(x0);
                    const float e1 = fast_exp2(x1);
                    pk[c] = pack_half2(e0, e1);
                    rs2[c & 1] = add_f32x2(rs2[c & 1], f32x2(e0, e1));
                }
                float r0, r1, r2, r3;
                f32x2_split(rs2[0], r0, r1);
                f32x2_split(rs2[1], r2, r3);
                l = l * alpha + ((r0 + r1) + (r2 + r3));
                // O is rescaled only after the previous PV product is complete.
                if (__any_sync(0xffffffffu, moved)) {
                    if (!(ok = mbar_waitw(bar_o + 8 * psb, psph, abort))) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c0 = 0; c0 < 64; c0 += 32) {
                        uint32_t v[32];
                        tmem_ld32(tmem + lane_base + kColO + hf * 64 + c0, v);
#pragma unroll
                        for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * alpha);
                        tmem_st32(tmem + lane_base + kColO + hf * 64 + c0, v);
                    }
                }
                // P over the first 32 of this half's own 64 S columns (already read)
                tmem_st32(tmem + lane_base + kColS + sb * kKTile + hf * 64, pk);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_p + 8 * sb);
                psb = sb;
                psph = sph;
                if (++sb == kSBufs) {
                    sb = 0;
                    sph ^= 1;
                }
            }
            if (!ok) break;
            // ---- end of the segment: wait for its last PV product, add the
            // two halves' row sums ----
            if (!(ok = mbar_waitw(bar_o + 8 * psb, psph, abort))) break;
            xsum[hf * kQTile + i] = l;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_l);
            if (!(ok = mbar_waitw(bar_l, (uint32_t)seg & 1, abort))) break;
            tc_fence_after();
            const float L = l + xsum[(hf ^ 1) * kQTile + i];
            __half* orow = p.out + ((int64_t)(sm_qs[r] + i_first + i) * hq + h) * kHeadDim + hf * 64;
            if (k0 == 0 && k1 == w.nkt) {
                // ---- a whole unit: normalise and store ----
                // O is read out and released to the next segment's products
                // before the stores
                const float inv = L > 0.f ? __fdividef(1.f, L) : 0.f;
                uint32_t v[32], v2[32];
                tmem_ld64(tmem + lane_base + kColO + hf * 64, v, v2);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_odrained);
                if (i < nq && p.out_v8) {
#pragma unroll
                    for (int c = 0; c < 64; c += 16) {
                        const uint32_t* u = c < 32 ? v + c : v2 + (c - 32);
                        uint32_t w8[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            w8[e] = pack_half2(__uint_as_float(u[2 * e]) * inv, __uint_as_float(u[2 * e + 1]) * inv);
                        st_v8(orow + c, w8);
                    }
                } else if (i < nq) {
#pragma unroll
                    for (int c = 0; c < 64; c += 8) {
                        const uint32_t* u = c < 32 ? v + c : v2 + (c - 32);
                        uint4 q4;
                        q4.x = pack_half2(__uint_as_float(u[0]) * inv, __uint_as_float(u[1]) * inv);
                        q4.y = pack_half2(__uint_as_float(u[2]) * inv, __uint_as_float(u[3]) * inv);
                        q4.z = pack_half2(__uint_as_float(u[4]) * inv, __uint_as_float(u[5]) * inv);
                        q4.w = pack_half2(__uint_as_float(u[6]) * inv, __uint_as_float(u[7]) * inv);
                        *reinterpret_cast<uint4*>(orow + c) = q4;
                    }
                }
            } else if (k1 < w.nkt) {
                // ---- a piece that does not end its unit: publish the partial
                // (reference maxima, row sums, unnormalised O) in this block's
                // slot and count it on the arrival word of the unit's last block ----
                float* slot = p.part + (int64_t)cta * kPartFloats;
                uint32_t v[32], v2[32];
                tmem_ld64(tmem + lane_base + kColO + hf * 64, v, v2);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_odrained);  // O is free for the next segment
                if (hf == 0) {
                    __stcg(slot + i, m);
                    __stcg(slot + kQTile + i, L);
                }
                float4* po = reinterpret_cast<float4*>(slot + 2 * kQTile) + hf * 16 * kQTile + i;
#pragma unroll
                for (int g = 0; g < 16; ++g) {
                    const uint32_t* u = g < 8 ? v + 4 * g : v2 + 4 * (g - 8);
                    __stcg(po + g * kQTile, make_float4(__uint_as_float(u[0]), __uint_as_float(u[1]),
                                                        __uint_as_float(u[2]), __uint_as_float(u[3])));
                }
                // The mbarrier orders every softmax warp's stores before thread
                // 0's release (release and acquire are cumulative).
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_pub);
                if (tid == 0) {
                    // every softmax warp's stores are ordered before this release
                    if (mbar_wait1(bar_pub, 0, abort)) {
                        int* word = p.count + (int64_t)owner_of(w.U + w.nkt - 1, W, Ge) * kCountStride;
                        asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(word) : "memory");
                    } else {
                        ok = false;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);  // one decision per warp
            } else {
                // ---- the piece that ends a unit cut over blocks cf .. cta: the S
                // issuer has landed block cf's partial in the K ring once all
                // cta - cf other pieces counted; merge the partials (in block
                // order, any beyond cf's from the workspace) with this block's
                // state ----
                const int cf = owner_of(w.U, W, Ge);
                if (!(ok = mbar_waitw(bar_mrg, 0, abort) && sm_misc[5] != 0)) break;
                const float* lp = reinterpret_cast<const float*>(smem + Smem::kring);  // block cf's partial
                float M = fmaxf(m, lp[i]);
                for (int j = cf + 1; j < cta; ++j) M = fmaxf(M, __ldcg(p.part + (int64_t)j * kPartFloats + i));
                const float ws = m == -INFINITY ? 0.f : fast_exp2(m - M);
                const float wf = lp[i] == -INFINITY ? 0.f : fast_exp2(lp[i] - M);
                float Lt = L * ws + lp[kQTile + i] * wf;
                for (int j = cf + 1; j < cta; ++j) {
                    const float* pj = p.part + (int64_t)j * kPartFloats;
                    const float mj = __ldcg(pj + i);
                    Lt += (mj == -INFINITY ? 0.f : fast_exp2(mj - M)) * __ldcg(pj + kQTile + i);
                }
                const float inv = Lt > 0.f ? __fdividef(1.f, Lt) : 0.f;
#pragma unroll 1
                for (int c0 = 0; c0 < 64; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_base + kColO + hf * 64 + c0, v);
                    float acc[32];
                    const float4* of = reinterpret_cast<const float4*>(lp + 2 * kQTile) +
                                       (hf * 16 + c0 / 4) * kQTile + i;
#pragma unroll
                    for (int c = 0; c < 32; c += 4) {
                        const float4 x = of[(c / 4) * kQTile];
                        acc[c] = __uint_as_float(v[c]) * ws + wf * x.x;
                        acc[c + 1] = __uint_as_float(v[c + 1]) * ws + wf * x.y;
                        acc[c + 2] = __uint_as_float(v[c + 2]) * ws + wf * x.z;
                        acc[c + 3] = __uint_as_float(v[c + 3]) * ws + wf * x.w;
                    }
                    for (int j = cf + 1; j < cta; ++j) {
                        const float* pj = p.part + (int64_t)j * kPartFloats;
                        const float mj = __ldcg(pj + i);
                        const float wj = mj == -INFINITY ? 0.f : fast_exp2(mj - M);
                        const float4* oj = reinterpret_cast<const float4*>(pj + 2 * kQTile) +
                                           (hf * 16 + c0 / 4) * kQTile + i;
#pragma unroll
                        for (int c = 0; c < 32; c += 4) {
                            const float4 x = __ldcg(oj + (c / 4) * kQTile);
                            acc[c] += wj * x.x;
                            acc[c + 1] += wj * x.y;
                            acc[c + 2] += wj * x.z;
                            acc[c + 3] += wj * x.w;
                        }
                    }
                    if (i < nq && p.out_v8) {
#pragma unroll
                        for (int c = 0; c < 32; c += 16) {
                            uint32_t w8[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) w8[e] = pack_half2(acc[c + 2 * e] * inv, acc[c + 2 * e + 1] * inv);
                            st_v8(orow + c0 + c, w8);
                        }
                    } else if (i < nq) {
#pragma unroll
                        for (int c = 0; c < 32; c += 8) {
                            uint4 q4;
                            q4.x = pack_half2(acc[c] * inv, acc[c + 1] * inv);
                            q4.y = pack_half2(acc[c + 2] * inv, acc[c + 3] * inv);
                            q4.z = pack_half2(acc[c + 4] * inv, acc[c + 5] * inv);
                            q4.w = pack_half2(acc[c + 6] * inv, acc[c + 7] * inv);
                            *reinterpret_cast<uint4*>(orow + c0 + c) = q4;
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_odrained);
            }
            ++seg;
        } while (ok && w.prev());
        if (!ok && lane == 0) {
            raise_abort();
            flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
        }
    }

    // ---- release tensor memory ----
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
}

}  // namespace prefill_tc

}  // namespace pkv

namespace {

// Partials of cut units and the merging blocks' arrival words, one slot per
// persistent block, for launches made without a caller workspace; shared by
// all such launches on a device, so those must run one after another (one
// stream, or streams the caller orders).  Each such launch clears the arrival
// words first.
static __device__ __align__(256) float g_prefill_part[pkv::prefill_tc::kMaxGrid * pkv::prefill_tc::kPartFloats];
static __device__ __align__(256) int g_prefill_count[pkv::prefill_tc::kMaxGrid * pkv::prefill_tc::kCountStride];

constexpr int kMaxDevices = 64;
std::mutex g_prefill_mutex;
struct PrefillDevice {
    float* part = nullptr;
    int* count = nullptr;
    int sms = 0;
};
PrefillDevice g_prefill_dev[kMaxDevices];

// The scratch addresses and SM count of the current device (looked up once).
int prefill_device(PrefillDevice* out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_prefill_mutex);
    PrefillDevice& d = g_prefill_dev[dev];
    if (!d.part) {
        void* a = nullptr;
        void* b = nullptr;
        int sms = 0;
        if (cudaGetSymbolAddress(&a, g_prefill_part) != cudaSuccess || !a ||
            cudaGetSymbolAddress(&b, g_prefill_count) != cudaSuccess || !b ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
            return PKV_ERR_CUDA;
        d.count = static_cast<int*>(b);
        d.sms = sms;
        d.part = static_cast<float*>(a);
    }
    *out = d;
    return PKV_OK;
}

}  // namespace

namespace pkv {

// Launch of the tcgen05 prefill kernel; the caller has validated the
// arguments (paged_attention_prefill).
size_t prefill_workspace_bytes() {
    using namespace prefill_tc;
    return prefill_count_bytes() + (size_t)kMaxGrid * kPartFloats * sizeof(float);
}

size_t prefill_count_bytes() {
    using namespace prefill_tc;
    return align_up((size_t)kMaxGrid * kCountStride * sizeof(int), 256);
}

int prefill_tc_launch(void* out, const void* q, const void* k_pool, const void* v_pool,
                      const int32_t* block_tables, const int32_t* seq_lens,
                      const int32_t* q_start, int rows, int total_q, int q_heads, int kv_heads,
                      int block_size, float scale, int max_blocks_per_row, int num_blocks,
                      int max_seq_len, void* workspace, int32_t* dev_err, cudaStream_t stream) {
    using namespace prefill_tc;
    const int64_t pool_rows = (int64_t)num_blocks * block_size;
    int kbox = kGranule;
    while (kbox < kKTile && block_size % (2 * kbox) == 0) kbox *= 2;
    const int vbox = kbox < 64 ? kbox : 64;
    // Steps of all units (key tiles summed over query tiles and heads) must
    // stay below 2^31: bounded by heads x query tiles x key tiles per tile.
    const int64_t max_steps = (int64_t)q_heads * (((int64_t)total_q + kQTile - 1) / kQTile + rows) *
                              (((int64_t)max_seq_len + kKTile - 1) / kKTile);
    if (pool_rows >= (int64_t(1) << 31) || max_steps >= (int64_t(1) << 31) || rows > kMaxRows)
        return PKV_ERR_UNSUPPORTED;
    PrefillDevice dv;
    int st = prefill_device(&dv);
    if (st != PKV_OK) return st;
    CUtensorMap km, vm, qm;
    {
        const int64_t dims[3] = {kHeadDim, kv_heads, pool_rows};
        const int64_t strides[2] = {kHeadDim * 2, (int64_t)kv_heads * kHeadDim * 2};
        const int kb[3] = {64, 1, kbox}, vb[3] = {64, 1, vbox};
        if ((st = tiled_map_3d(k_pool, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, dims, strides, kb, &km)) != PKV_OK)
            return st;
        if ((st = tiled_map_3d(v_pool, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, dims, strides, vb, &vm)) != PKV_OK)
            return st;
    }
    {
        const int64_t dims[3] = {kHeadDim, q_heads, total_q};
        const int64_t strides[2] = {kHeadDim * 2, (int64_t)q_heads * kHeadDim * 2};
        const int box[3] = {64, 1, kQTile};
        if ((st = tiled_map_3d(q, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, dims, strides, box, &qm)) != PKV_OK)
            return st;
    }
    Params prm{};
    prm.q = static_cast<const __half*>(q);
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
    prm.kbox = kbox;
    prm.vbox = vbox;
    prm.scale_log2 = scale * kLog2e;
    prm.out_v8 = (reinterpret_cast<uintptr_t>(out) & 31) == 0;
    const int grid = dv.sms < kMaxGrid ? dv.sms : kMaxGrid;
    if (workspace) {
        // caller-owned: arrival words first (zero between calls), then the partials
        prm.count = static_cast<int*>(workspace);
        prm.part = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + prefill_count_bytes());
    } else {
        // library-owned: its arrival words are cleared here, so a launch that
        // timed out leaves nothing behind for the next one
        prm.part = dv.part;
        prm.count = dv.count;
        if (cudaMemsetAsync(dv.count, 0, (size_t)grid * kCountStride * sizeof(int), stream) != cudaSuccess)
            return PKV_ERR_CUDA;
    }
    prm.dev_err = dev_err;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Smem::total()) != cudaSuccess)
            return PKV_ERR_CUDA;
        attr_set = true;
    }
    // One block per SM: every block is resident at once, so a merging block
    // never waits on a block that has not started.
    prefill_tc_kernel<<<grid, kThreads, Smem::total(), stream>>>(km, vm, qm, prm);
    return launch_status();
}

}  // namespace pkv
