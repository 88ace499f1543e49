// Chunked-prefill paged attention on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory), sm_103a.
//
// What it computes is paged_attention_prefill's definition ("Paged
// attention", danielfleming.xyz, closing sections: long prompts split into
// fixed chunks so decode steps interleave; "PagedAttention", deepconcepts.dev,
// section "PagedAttention": keys gathered through the row's block table):
// query i of row r's chunk sits at position seq_lens[r] - C_r + i and attends
// causally to the row's tokens 0 .. that position.
//
// A block takes 128 queries of one row and one query head.  Warp roles:
//   warps 0-3  softmax: thread i owns query row i, which is also TMEM lane i;
//   warp 4     TMA: the queries once, then 64-token K/V tiles (four 16-token
//              granules gathered through the block table) into a 3-stage ring;
//   warp 5     MMA: one thread issues tcgen05.mma, f16 in / f32 accumulate:
//                S_j[128 q][64 tok]  = Q[128][128] . K_j^T   (TMEM, double-buffered)
//                O[128 q][128 dims] += P_j[128][64] . V_j    (TMEM)
//              and commits each group to an mbarrier.
// Per tile a softmax thread reads its S row from TMEM, applies the causal
// mask, updates its running maximum and sum, rescales its O row in TMEM when
// the maximum moved, and writes its fp16 P row (128-byte swizzled) to shared
// memory for the PV product.  All waits are bounded.
#include "pkv_internal.cuh"
#include "ptx.cuh"

namespace pkv {
namespace prefill_tc {

using namespace ptx;

constexpr int kQTile = 128;
constexpr int kKTile = 64;
constexpr int kGranule = 16;
constexpr int kStages = 3;
constexpr int kSoftWarps = 4;
constexpr int kThreads = (kSoftWarps + 2) * 32;  // softmax, TMA, MMA
constexpr int kMaxRows = 1024;
constexpr uint32_t kHalfQ = kQTile * 128;         // 128 queries x 64 dims
constexpr uint32_t kHalfKV = kKTile * 128;        // 64 tokens x 64 dims
constexpr uint32_t kStageBytes = 4 * kHalfKV;     // K lo, K hi, V lo, V hi
constexpr uint32_t kBox = kGranule * 128;         // one granule box
constexpr uint32_t kTmemCols = 256;               // S0 [0,64), S1 [64,128), O [128,256)
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
    static constexpr uint32_t q = 0;                                 // Q lo, Q hi
    static constexpr uint32_t kv = q + 2 * kHalfQ;                   // [stages]
    static constexpr uint32_t pbuf = kv + kStages * kStageBytes;     // P [2][128][64] fp16
    static constexpr uint32_t bars = pbuf + 2 * kQTile * 128;        // q, full[3], empty[3], s[2], p[2], o[2]
    static constexpr uint32_t tmem = bars + 16 * 8;                  // allocated TMEM address
    static constexpr uint32_t part = tmem + 16;                      // scan partials [threads]
    static constexpr uint32_t pre = part + kThreads * 4;             // tile prefix [rows + 1]
    __host__ __device__ static constexpr uint32_t total(int rows) {
        return pre + (uint32_t)(rows + 1) * 4 + 1024;
    }
};
static_assert(Smem::kv % 1024 == 0 && Smem::pbuf % 1024 == 0, "swizzled tiles need 1024-byte alignment");

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
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                     uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(id), "r"(accumulate));
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
// 32 consecutive columns of this warp's 32 lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t addr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
          "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
          "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(addr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
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
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const Params p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_q = sbase + Smem::bars;
    const uint32_t bar_full = bar_q + 8;                 // [3]
    const uint32_t bar_empty = bar_full + kStages * 8;   // [3]
    const uint32_t bar_s = bar_empty + kStages * 8;      // [2]
    const uint32_t bar_p = bar_s + 16;  // [2]: P buffer b written (tiles b, b + 2, ...)
    const uint32_t bar_o = bar_p + 16;  // [2]: PV product of P buffer b done
    uint32_t* sm_tmem = reinterpret_cast<uint32_t*>(smem + Smem::tmem);
    int* sm_part = reinterpret_cast<int*>(smem + Smem::part);
    int* sm_pre = reinterpret_cast<int*>(smem + Smem::pre);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rows = p.rows;
    const int h = blockIdx.y, kvh = h / p.group;

    // ---- tiles of 128 queries per row, their prefix, this block's tile ----
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
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sm_pre[mid] <= b) lo = mid; else hi = mid - 1;
    }
    const int r = lo;
    const int tile = b - sm_pre[r];
    const int C = p.q_start[r + 1] - p.q_start[r];
    const int L = p.seq_lens[r];
    const int pos0 = L - C;
    const int i_first = tile * kQTile;
    const int nq = min(kQTile, C - i_first);
    const int kend = pos0 + i_first + nq;  // keys 0 .. kend-1 are visible to someone
    const int nkt = (kend + kKTile - 1) / kKTile;
    const int qrow0 = p.q_start[r] + i_first;

    // ---- barriers and tensor memory ----
    if (tid == 0) {
        mbar_init(bar_q, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int b2 = 0; b2 < 2; ++b2) {
            mbar_init(bar_s + 8 * b2, 1);
            mbar_init(bar_p + 8 * b2, kSoftWarps);
            mbar_init(bar_o + 8 * b2, 1);
        }
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
    const uint32_t t_o = tmem + 128;  // O columns

    if (warp == kSoftWarps) {
        // ============================== TMA ==============================
        if (lane == 0) {
            mbar_arrive_expect_tx(bar_q, 2 * kHalfQ);
            tma_load_3d(sbase + Smem::q, &qmap, 0, h, qrow0, bar_q);
            tma_load_3d(sbase + Smem::q + kHalfQ, &qmap, 64, h, qrow0, bar_q);
        }
        for (int kt = 0; kt < nkt; ++kt) {
            const int s = kt % kStages;
            if (!mbar_wait(bar_empty + 8 * s, (((uint32_t)kt / kStages) & 1) ^ 1)) {
                if (lane == 0) flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
                break;
            }
            int zrow = 0;
            bool issue = false;
            if (lane < 4) {
                const int tok0 = kt * kKTile + lane * kGranule;
                if (tok0 < kend) {
                    const int pb = p.tables[(int64_t)r * p.mbpr + tok0 / p.bs];
                    if (pb < 0 || pb >= p.nb) {
                        flag_error(p.dev_err, PKV_DEV_ERR_BLOCK_ID);
                    } else {
                        zrow = pb * p.bs + tok0 % p.bs;
                        issue = true;
                    }
                }
            }
            const uint32_t nissue = __popc(__ballot_sync(0xffffffffu, issue));
            const uint32_t fb = bar_full + 8 * s;
            if (lane == 0) mbar_arrive_expect_tx(fb, nissue * 4 * kBox);
            __syncwarp();
            if (issue) {
                const uint32_t st = sbase + Smem::kv + s * kStageBytes + lane * kBox;
                tma_load_3d(st, &kmap, 0, kvh, zrow, fb);
                tma_load_3d(st + kHalfKV, &kmap, 64, kvh, zrow, fb);
                tma_load_3d(st + 2 * kHalfKV, &vmap, 0, kvh, zrow, fb);
                tma_load_3d(st + 3 * kHalfKV, &vmap, 64, kvh, zrow, fb);
            }
        }
    } else if (warp == kSoftWarps + 1) {
        // ============================== MMA ==============================
        const uint32_t id_s = idesc(kQTile, kKTile, 0);
        const uint32_t id_o = idesc(kQTile, 128, 1);
        bool ok = mbar_wait(bar_q, 0);
        for (int kt = 0; ok && kt <= nkt; ++kt) {
            if (kt < nkt) {
                const int s = kt % kStages;
                if (!(ok = mbar_wait(bar_full + 8 * s, ((uint32_t)kt / kStages) & 1))) break;
                unsigned char* stp = smem + Smem::kv + s * kStageBytes;
                // V rows past the last visible key may hold anything (or be
                // unloaded): zero them so that 0 * V stays 0 in the PV product.
                const int vrow0 = kend - kt * kKTile;
                if (vrow0 < kKTile) {
                    for (int i = lane; i < (kKTile - vrow0) * 16; i += 32) {
                        const int row = vrow0 + (i >> 4), c = i & 15;
                        *reinterpret_cast<uint4*>(stp + 2 * kHalfKV + (c >> 3) * kHalfKV + row * 128 +
                                                  (((c & 7) ^ (row & 7)) << 4)) = make_uint4(0, 0, 0, 0);
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                }
                if (lane == 0) {
                    tc_fence_after();
                    const uint32_t st = sbase + Smem::kv + s * kStageBytes;
                    const uint32_t d = tmem + (kt & 1) * kKTile;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint64_t a = sdesc(sbase + Smem::q + (ks >> 2) * kHalfQ + (ks & 3) * 32, 16, 1024);
                        const uint64_t bk = sdesc(st + (ks >> 2) * kHalfKV + (ks & 3) * 32, 16, 1024);
                        umma(d, a, bk, id_s, ks > 0);
                    }
                    umma_commit(bar_s + 8 * (kt & 1));
                }
                __syncwarp();
            }
            if (kt > 0) {
                // O += P_{kt-1} . V_{kt-1} once the softmax has written P_{kt-1}
                const int j = kt - 1, s = j % kStages, pb = j & 1;
                if (!(ok = mbar_wait(bar_p + 8 * pb, ((uint32_t)j >> 1) & 1))) break;
                if (lane == 0) {
                    tc_fence_after();
                    const uint32_t vb = sbase + Smem::kv + s * kStageBytes + 2 * kHalfKV;
                    const uint32_t pa = sbase + Smem::pbuf + pb * (kQTile * 128);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t a = sdesc(pa + kk * 32, 16, 1024);
                        const uint64_t bv = sdesc(vb + kk * 2048, kHalfKV, 1024);
                        umma(t_o, a, bv, id_o, (j > 0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(bar_o + 8 * pb);
                    umma_commit(bar_empty + 8 * s);  // K_j and V_j are no longer read
                }
                __syncwarp();
            }
        }
        if (!ok && lane == 0) flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
    } else {
        // ============================ softmax =============================
        const int i = tid;  // query row of the tile, TMEM lane
        const int pos = pos0 + i_first + i;
        const int vis = min(pos, kend - 1);
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int kt = 0; kt < nkt && ok; ++kt) {
            if (!(ok = mbar_wait(bar_s + 8 * (kt & 1), ((uint32_t)kt >> 1) & 1))) break;
            tc_fence_after();
            float s[64];
            {
                uint32_t v[32];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    tmem_ld32(tmem + lane_base + (kt & 1) * kKTile + half * 32, v);
#pragma unroll
                    for (int c = 0; c < 32; ++c) s[half * 32 + c] = __uint_as_float(v[c]);
                }
            }
            const int t0 = kt * kKTile;
            // Mask only where the tile reaches past this query's position
            // (the diagonal tiles); scores stay unscaled until the exponent.
            if (t0 + kKTile - 1 > vis) {
#pragma unroll
                for (int c = 0; c < 64; ++c) s[c] = t0 + c <= vis ? s[c] : -INFINITY;
            }
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < 64; ++c) mx4[c & 3] = fmaxf(mx4[c & 3], s[c]);
            const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * p.scale_log2;
            // Lazy rescaling: the reference maximum m only moves when a score
            // exceeds it by more than 2^8 (weights stay <= 256, exact enough in
            // fp16); the first tile sets it (key 0 is visible to every query).
            float alpha = 1.f;
            bool moved = false;
            if (mx > m + 8.f) {
                alpha = fast_exp2(m - mx);  // 0 on the first tile
                m = mx;
                moved = kt > 0;
            }
            const float mneg = -m;
            uint32_t pk[32];
            float rs4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float e0 = fast_exp2(fmaf(s[2 * c], p.scale_log2, mneg));
                const float e1 = fast_exp2(fmaf(s[2 * c + 1], p.scale_log2, mneg));
                pk[c] = pack_half2(e0, e1);
                rs4[c & 3] += e0 + e1;
            }
            l = l * alpha + ((rs4[0] + rs4[1]) + (rs4[2] + rs4[3]));
            // O is rescaled only after the previous PV product is complete.
            if (__any_sync(0xffffffffu, moved)) {
                if (!(ok = mbar_wait(bar_o + 8 * ((kt - 1) & 1), ((uint32_t)(kt - 1) >> 1) & 1))) break;
                tc_fence_after();
                {
#pragma unroll 1
                    for (int c0 = 0; c0 < 128; c0 += 32) {
                        uint32_t v[32];
                        tmem_ld32(t_o + lane_base + c0, v);
#pragma unroll
                        for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * alpha);
                        tmem_st32(t_o + lane_base + c0, v);
                    }
                }
            }
            // P buffer kt & 1 was last read by the PV product of tile kt - 2.
            if (kt >= 2) {
                if (!(ok = mbar_wait(bar_o + 8 * (kt & 1), ((uint32_t)(kt - 2) >> 1) & 1))) break;
            }
            unsigned char* prow = smem + Smem::pbuf + (kt & 1) * (kQTile * 128) + i * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(prow + ((c ^ (i & 7)) << 4)) =
                    make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_p + 8 * (kt & 1));
        }
        // ---- finish: wait for the last PV product, normalise, store ----
        if (ok) ok = mbar_wait(bar_o + 8 * ((nkt - 1) & 1), ((uint32_t)(nkt - 1) >> 1) & 1);
        if (ok) {
            tc_fence_after();
            const float inv = l > 0.f ? __fdividef(1.f, l) : 0.f;
            __half* orow = p.out + ((int64_t)(qrow0 + i) * p.hq + h) * kHeadDim;
#pragma unroll 1
            for (int c0 = 0; c0 < 128; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(t_o + lane_base + c0, v);
                if (i < nq) {
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        uint4 q4;
                        q4.x = pack_half2(__uint_as_float(v[c]) * inv, __uint_as_float(v[c + 1]) * inv);
                        q4.y = pack_half2(__uint_as_float(v[c + 2]) * inv, __uint_as_float(v[c + 3]) * inv);
                        q4.z = pack_half2(__uint_as_float(v[c + 4]) * inv, __uint_as_float(v[c + 5]) * inv);
                        q4.w = pack_half2(__uint_as_float(v[c + 6]) * inv, __uint_as_float(v[c + 7]) * inv);
                        *reinterpret_cast<uint4*>(orow + c0 + c) = q4;
                    }
                }
            }
        } else if (lane == 0) {
            flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
        }
    }

    // ---- drain and release tensor memory ----
    tc_fence_before();
    __syncthreads();
    if (warp == kSoftWarps) {
        // every armed stage's copies have landed before the block exits
        for (int kt = max(0, nkt - kStages); kt < nkt; ++kt)
            if (!mbar_wait(bar_full + 8 * (kt % kStages), ((uint32_t)kt / kStages) & 1) && lane == 0)
                flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
        if (!mbar_wait(bar_q, 0) && lane == 0) flag_error(p.dev_err, PKV_DEV_ERR_TIMEOUT);
    }
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
}

}  // namespace prefill_tc

// Launch of the tcgen05 prefill kernel; the caller has validated the
// arguments (paged_attention_prefill).
int prefill_tc_launch(void* out, const void* q, const void* k_pool, const void* v_pool,
                      const int32_t* block_tables, const int32_t* seq_lens,
                      const int32_t* q_start, int rows, int total_q, int q_heads, int kv_heads,
                      int block_size, float scale, int max_blocks_per_row, int num_blocks,
                      int max_seq_len, int32_t* dev_err, cudaStream_t stream) {
    using namespace prefill_tc;
    const int64_t pool_rows = (int64_t)num_blocks * block_size;
    const int64_t grid_x = ((int64_t)total_q + kQTile - 1) / kQTile + rows;
    if (pool_rows >= (int64_t(1) << 31) || grid_x >= (int64_t(1) << 31) || rows > kMaxRows)
        return PKV_ERR_UNSUPPORTED;
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
        if (cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Smem::total(kMaxRows)) != cudaSuccess)
            return PKV_ERR_CUDA;
        attr_set = true;
    }
    prefill_tc_kernel<<<dim3((unsigned)grid_x, (unsigned)q_heads), kThreads, Smem::total(rows), stream>>>(
        qm, km, vm, prm);
    return launch_status();
}

}  // namespace pkv
