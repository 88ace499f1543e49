/*
 * paged_kv.h -- C ABI of libpagedkv: paged KV-cache append and decode
 * attention for GB300 (sm_103a), plus a host-side block manager.
 *
 * Terms (from the pages this library implements):
 *   - "PagedAttention" (deepconcepts.dev), section "PagedAttention": the KV
 *     cache is cut into fixed-size blocks; each sequence keeps a block table
 *     mapping its logical block n to the physical block holding it, and the
 *     attention kernel walks that table instead of striding a slab.
 *     Section "What the block table costs": the tables of all rows form a
 *     single dense int32 matrix, a row per request and a column per possible
 *     logical block.
 *   - "Paged attention" (danielfleming.xyz), section "What changed": decode
 *     touches, for each row, just the blocks named in that row's table, up to
 *     the row's true length; a request takes its blocks from a free list when
 *     it is admitted (reserve on admit).
 *   - "SLM paged attention" (aicassindra.com), section "The architecture":
 *     the pool is allocated once and divided into fixed-size blocks; token
 *     position p lives in logical block p / block_size; the final block fills
 *     one slot at a time; blocks shared by a prefix are reference-counted and
 *     copied before a write.
 *
 * Data layout (all device buffers, row-major, contiguous, 16-byte aligned):
 *   k_pool, v_pool   fp16 [num_blocks][block_size][kv_heads][head_dim]
 *   block_tables     int32 [rows][max_blocks_per_row]; entries past a row's
 *                    ceil(seq_len / block_size) are never read (-1 by
 *                    convention)
 *   seq_lens         int32 [rows]: tokens a row attends to, including the
 *                    token appended in this step
 *   q, out           fp16 [rows][q_heads][head_dim]
 *   k_new, v_new     fp16 [rows][kv_heads][head_dim]
 * Query head h reads KV head h / (q_heads / kv_heads) (contiguous groups).
 *
 * Ownership: the caller allocates and owns every buffer (including the
 * decode workspace).  The library never allocates, frees or synchronises,
 * except pkv_check_error, which synchronises the given stream to read the
 * device error word.
 *
 * Asynchrony: kernel entry points enqueue work on `stream` and return.
 *
 * Errors: every call returns a pkv_status.  Problems visible on the host
 * (null pointers, bad sizes, unsupported shapes, small workspace) are
 * returned before anything is launched.  Problems only visible on the device
 * (a table entry outside [0, num_blocks), a seq_len above the bound, an
 * append position past the row's table) never fault: the offending block,
 * row or token is skipped, and when `dev_err` is non-null a PKV_DEV_ERR_*
 * bit is OR-ed into *dev_err.  Kernels never trap and never spin-wait.
 */
#ifndef PAGED_KV_H
#define PAGED_KV_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,  /* null pointer, negative/zero size, bad combination */
    PKV_ERR_UNSUPPORTED = 2,  /* valid but not built: head_dim != 128, group > 8, ... */
    PKV_ERR_WORKSPACE = 3,    /* workspace null or smaller than required */
    PKV_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    PKV_ERR_BAD_TABLE = 5,    /* (block manager) inconsistent table / id */
    PKV_ERR_NO_BLOCKS = 6,    /* (block manager) free list cannot cover the request */
    PKV_ERR_NOT_FOUND = 7,    /* (block manager) unknown sequence or prefix id */
    PKV_ERR_STATE = 8         /* (block manager) operation not valid in this state */
} pkv_status;

/* Bits OR-ed into the optional device error word. */
#define PKV_DEV_ERR_BLOCK_ID 0x1 /* a table entry that had to be read is outside [0, num_blocks) */
#define PKV_DEV_ERR_SEQ_LEN 0x2  /* seq_len < 0, > max_seq_len or > max_blocks_per_row * block_size */
#define PKV_DEV_ERR_POSITION 0x4 /* append position's logical block >= max_blocks_per_row */
#define PKV_DEV_ERR_TIMEOUT 0x8  /* a bounded wait inside a kernel gave up (the call's output is invalid) */
#define PKV_DEV_ERR_PLAN 0x10    /* a decode plan made for another launch size was passed (nothing was done) */

/* Human-readable name of a pkv_status.  Never null; static storage. */
const char* pkv_status_string(int status);

/* ABI version of this header (increments on incompatible changes). */
int pkv_abi_version(void);

/*
 * paged_kv_append -- write this step's new K and V token of every row into
 * its slot.  Defining passage: "SLM paged attention", section "The
 * architecture" (logical block = position / block_size; the last block's
 * slots fill one at a time; growth is one block at a time).
 *
 * For each row r with positions[r] >= 0, with lb = positions[r] / block_size,
 * off = positions[r] % block_size and pb = block_tables[r][lb]:
 *     k_pool[pb][off][h][:] = k_new[r][h][:]   and likewise for V,
 * for every KV head h.  Rows with positions[r] < 0 are skipped.  The copy is
 * bit-exact.  Two rows naming the same slot is a caller error (the result is
 * one of the two writes).  lb >= max_blocks_per_row sets
 * PKV_DEV_ERR_POSITION, pb outside [0, num_blocks) sets PKV_DEV_ERR_BLOCK_ID;
 * either way that row is skipped.
 *
 * head_dim must be a multiple of 8; rows may be 0 (nothing is launched).
 */
int paged_kv_append(void* k_pool, void* v_pool, const int32_t* block_tables,
                    const int32_t* positions, const void* k_new, const void* v_new,
                    int rows, int kv_heads, int head_dim, int block_size,
                    int max_blocks_per_row, int num_blocks, int32_t* dev_err,
                    cudaStream_t stream);

/*
 * paged_kv_copy_blocks -- copy-on-write: for i < n, block dst_ids[i] of both
 * pools becomes a bit-exact copy of block src_ids[i].  Defining passage:
 * "SLM paged attention", sections "The architecture" and "End-to-end flow"
 * (a writer about to modify a block it shares receives a private copy of
 * that block alone, and its table entry then points at the copy).  The pairs come from
 * pkv_bm_append_slot.  The dst ids must be distinct and must not appear among
 * the src ids of the same call (pairs run concurrently).  An id outside
 * [0, num_blocks) skips its pair and sets PKV_DEV_ERR_BLOCK_ID.
 * src_ids, dst_ids: device int32 [n].  head_dim must be a multiple of 8.
 */
int paged_kv_copy_blocks(void* k_pool, void* v_pool, const int32_t* src_ids,
                         const int32_t* dst_ids, int n, int block_size, int kv_heads,
                         int head_dim, int num_blocks, int32_t* dev_err, cudaStream_t stream);

/*
 * paged_kv_prefill_scatter -- lay a batched prefill's K/V into the rows'
 * blocks with the padding dropped.  Defining passage: "Paged attention",
 * section "What changed" (requests admitted together are prefilled as one
 * batch, padded on the left to its longest prompt; each row's K/V then moves
 * into the row's blocks without the padding).
 *
 * k_src, v_src: fp16 [rows][width][kv_heads][head_dim].  For each row r with
 * lengths[r] > 0, source columns src_start[r] .. src_start[r] + lengths[r] - 1
 * go to logical positions dst_start[r] .. of the row (slot pos % block_size
 * of block block_tables[r][pos / block_size]); left padding is
 * src_start[r] = width - lengths[r].  A source range past the width sets
 * PKV_DEV_ERR_POSITION and skips the row; a position past the table or an id
 * out of range skips that token and sets PKV_DEV_ERR_POSITION /
 * PKV_DEV_ERR_BLOCK_ID.  Bit-exact copy.
 */
int paged_kv_prefill_scatter(void* k_pool, void* v_pool, const int32_t* block_tables,
                             const int32_t* src_start, const int32_t* dst_start,
                             const int32_t* lengths, const void* k_src, const void* v_src,
                             int rows, int width, int kv_heads, int head_dim, int block_size,
                             int max_blocks_per_row, int num_blocks, int32_t* dev_err,
                             cudaStream_t stream);

/*
 * paged_attention_workspace_size -- bytes of device workspace that
 * paged_attention_decode needs for these sizes (the split-K partial results
 * and per-row arrival counters).  Pure host arithmetic; never fails (returns
 * 0 for invalid sizes).  max_seq_len is the caller's upper bound on every
 * seq_lens[r] of the calls the workspace will serve.
 *
 * The workspace must be zero-filled once after allocation.  Every decode
 * call that completes without PKV_DEV_ERR_TIMEOUT leaves it ready for the
 * next call (every split-K record word it read cleared back to zero), so it
 * may be reused by later calls on the same stream, including from a CUDA
 * graph; two decode calls that run at the same time need separate
 * workspaces.  After a call that flagged PKV_DEV_ERR_TIMEOUT, words may be
 * left set: zero-fill the workspace again before reusing it.
 */
size_t paged_attention_workspace_size(int rows, int q_heads, int kv_heads, int head_dim,
                                      int max_seq_len, int block_size);

/*
 * paged_attention_decode -- one decode step of attention over a paged KV
 * cache.  Defining passages: "PagedAttention" (deepconcepts.dev), sections
 * "PagedAttention" and "What the block table costs" (walk the table, gather
 * the listed blocks) and its closing note on FlashAttention (block-wise
 * softmax recombined exactly); "Paged attention" (danielfleming.xyz),
 * section "What changed" (read each row only at its true length).
 *
 * For every row r and query head h, with L = seq_lens[r],
 * kvh = h / (q_heads / kv_heads) and, for t < L,
 * K_t = k_pool[block_tables[r][t / block_size]][t % block_size][kvh][:]:
 *     out[r][h][:] = sum_t softmax_t(scale * q[r][h] . K_t) * V_t[:]
 * computed in fp32 and rounded to fp16 (round to nearest even).  Rows with
 * L == 0 produce zeros.  Long rows are split across thread blocks and the
 * partial results merged exactly through their log-sum-exp.
 *
 * Supported: head_dim == 128; q_heads % kv_heads == 0 with group size
 * q_heads / kv_heads <= 8; block_size in [1, 1024]; max_seq_len <=
 * max_blocks_per_row * block_size.  Anything else returns
 * PKV_ERR_UNSUPPORTED or PKV_ERR_INVALID_ARG before launch.
 * workspace must hold paged_attention_workspace_size(...) bytes (see there).
 * seq_lens[r] > max_seq_len is clamped to max_seq_len and flagged
 * (PKV_DEV_ERR_SEQ_LEN); bad table entries are skipped and flagged.
 */
int paged_attention_decode(void* out, const void* q, const void* k_pool, const void* v_pool,
                           const int32_t* block_tables, const int32_t* seq_lens, int rows,
                           int q_heads, int kv_heads, int head_dim, int block_size, float scale,
                           int max_blocks_per_row, int num_blocks, int max_seq_len,
                           void* workspace, size_t workspace_bytes, int32_t* dev_err,
                           cudaStream_t stream);

/* Flags of paged_attention_append_decode. */
#define PKV_FLAG_PDL 0x1u /* overlap this launch's start with the preceding kernel (see below) */

/*
 * paged_attention_append_decode -- one decode step of one layer: exactly
 * paged_kv_append(k_pool, v_pool, block_tables, positions, k_new, v_new, ...)
 * followed by paged_attention_decode(out, q, k_pool, v_pool, block_tables,
 * seq_lens, ...), with the same arguments, results and errors as those two
 * calls (the pools end bit-identical; the new token takes part in the
 * attention when positions[r] < seq_lens[r]).  Defining passages: as for the
 * two calls ("SLM paged attention", "The architecture": the new token goes to
 * slot position % block_size of block position / block_size; decode reads
 * every row at its true length).
 *
 * Where the decode kernel supports the shape (head_dim 128, group <= 8,
 * block_size a multiple of 16, rows <= 1024) this is ONE launch: the block
 * that stages the new token's granule takes it from k_new / v_new directly,
 * and the pool slot is written in the same kernel.  Otherwise the two calls
 * are made in sequence.
 *
 * flags: 0 or PKV_FLAG_PDL.  With PKV_FLAG_PDL the launch uses programmatic
 * stream serialization: its blocks may start while the preceding kernel in
 * `stream` is still running, and before that kernel completes they read
 * seq_lens, block_tables and the cached tokens of k_pool / v_pool.  q,
 * positions, k_new, v_new, out, the workspace and the appended slots are
 * touched only after it completes.  The caller guarantees that the preceding
 * kernel writes neither seq_lens, block_tables nor these pools (for example
 * the previous layer's call, or a projection kernel).  Without the flag the
 * launch is ordered after all earlier work as usual.
 */
int paged_attention_append_decode(void* out, const void* q, void* k_pool, void* v_pool,
                                  const int32_t* block_tables, const int32_t* seq_lens,
                                  const int32_t* positions, const void* k_new, const void* v_new,
                                  int rows, int q_heads, int kv_heads, int head_dim,
                                  int block_size, float scale, int max_blocks_per_row,
                                  int num_blocks, int max_seq_len, void* workspace,
                                  size_t workspace_bytes, unsigned flags, int32_t* dev_err,
                                  cudaStream_t stream);

/*
 * paged_attention_padded_decode -- the comparator the paged cache replaced:
 * attention over a contiguous slab that gives every row a slot as wide as
 * the widest row, computed across that whole width for every row with the
 * columns past the row's length masked out ("Continuous batching",
 * danielfleming.xyz, sections "What changed" and "Where the missing capacity
 * went": masking removes the padded values from the result, not their cost).  Used to measure what reading true lengths saves.
 *
 * k_slab, v_slab: fp16 [rows][width][kv_heads][head_dim].  Row r's result
 * equals paged_attention_decode's on the same tokens; every column of the
 * slab is read.  Masked columns must hold finite values.  workspace as for
 * paged_attention_decode with max_seq_len = width.
 */
int paged_attention_padded_decode(void* out, const void* q, const void* k_slab,
                                  const void* v_slab, const int32_t* seq_lens, int rows,
                                  int width, int q_heads, int kv_heads, int head_dim,
                                  float scale, void* workspace, size_t workspace_bytes,
                                  int32_t* dev_err, cudaStream_t stream);

/*
 * paged_attention_prefill -- chunked prefill: attention of several query
 * tokens per row, causal within the row's chunk.  Defining passages:
 * "Paged attention" (danielfleming.xyz), closing sections (long prompts
 * broken into fixed-size pieces of 512 tokens, with decode steps in between) and
 * "PagedAttention" (deepconcepts.dev), section "PagedAttention" (keys gathered
 * through the row's block table).
 *
 * q: fp16 [total_q][q_heads][head_dim], the rows' chunks packed in order;
 * q_start: device int32 [rows + 1], q_start[0] = 0, row r's queries are
 * q_start[r] .. q_start[r+1]-1 (C_r of them, possibly 0).  seq_lens[r] counts
 * the row's tokens including its chunk, whose K/V must already be in the
 * row's blocks (paged_kv_append / paged_kv_prefill_scatter); query i of the
 * chunk sits at position seq_lens[r] - C_r + i and attends to the row's
 * tokens 0 .. that position.  out: fp16, the shape of q.  total_q = q_start[rows]
 * (host value, sizes the launch).  A row with C_r > seq_lens[r] or
 * seq_lens[r] > max_seq_len is skipped (its outputs untouched) and flagged
 * PKV_DEV_ERR_SEQ_LEN; table entries as in paged_attention_decode.  Supported
 * for head_dim 128, block_size a multiple of 16, rows <= 1024, and at most
 * 2^31 key-tile steps in total (q_heads x 128-query tiles x 128-key tiles;
 * PKV_ERR_UNSUPPORTED beyond).
 *
 * Workspace: one block per SM splits the steps evenly, and a 128-query tile
 * cut between two blocks is merged through a partial result that goes
 * through `workspace`: paged_attention_prefill_workspace_size(...) bytes of
 * caller device memory, 256-byte aligned, zero-filled once after allocation
 * (a smaller or misaligned one returns PKV_ERR_WORKSPACE).  Every call that
 * completes without PKV_DEV_ERR_TIMEOUT leaves it ready for the next (its
 * arrival words back at zero); after one that timed out, zero-fill it again.
 * Calls on separate workspaces may overlap; calls that share one must not.
 * workspace == NULL uses library-owned device memory instead (about 13 MB per
 * device, held from load to exit), whose arrival words every such call clears
 * first on `stream`: calls without a workspace on one device must not overlap
 * each other (issue them on one stream, or order the streams).
 */
size_t paged_attention_prefill_workspace_size(int rows, int q_heads, int kv_heads, int head_dim,
                                              int block_size);
int paged_attention_prefill(void* out, const void* q, const void* k_pool, const void* v_pool,
                            const int32_t* block_tables, const int32_t* seq_lens,
                            const int32_t* q_start, int rows, int total_q, int q_heads,
                            int kv_heads, int head_dim, int block_size, float scale,
                            int max_blocks_per_row, int num_blocks, int max_seq_len,
                            void* workspace, size_t workspace_bytes, int32_t* dev_err,
                            cudaStream_t stream);

/*
 * FP8 KV pools.  "PagedAttention" (deepconcepts.dev), section "Checking it on
 * a real system", names FP8 KV as a way to change the bytes per token; the
 * pages fix no format.  Here a pool holds E4M3 codes (1 sign, 4 exponent bits
 * with bias 7, 3 mantissa bits; no infinities, 0x7F / 0xFF are NaN, 448 is
 * the largest value), laid out like the fp16 pools but one byte per element:
 * [num_blocks][block_size][kv_heads][head_dim].  k_scale, v_scale: device
 * float [kv_heads]; code c of head h stands for e4m3(c) * scale[h].
 *
 * paged_kv_append_fp8 -- paged_kv_append into FP8 pools: element x of head h
 * of the new token is stored as the nearest E4M3 value of the binary32
 * quotient x / scale[h], ties to even, magnitudes above 448 saturating to 448.
 * Bit-exact; errors and skipped rows as in paged_kv_append.  The pools need
 * 8-byte alignment, k_new / v_new 16-byte alignment; head_dim % 8 == 0.
 */
int paged_kv_append_fp8(void* k_pool, void* v_pool, const float* k_scale, const float* v_scale,
                        const int32_t* block_tables, const int32_t* positions, const void* k_new,
                        const void* v_new, int rows, int kv_heads, int head_dim, int block_size,
                        int max_blocks_per_row, int num_blocks, int32_t* dev_err,
                        cudaStream_t stream);

/*
 * paged_attention_decode_fp8 -- paged_attention_decode over FP8 pools: the
 * same attention with K and V dequantised as e4m3(code) * scale[kv head].
 * Arguments, workspace (paged_attention_workspace_size), errors and
 * device-side checks as in paged_attention_decode.  Supported for head_dim
 * 128, q_heads / kv_heads <= 8, kv_heads <= 16, block_size a multiple of 16
 * and rows <= 1024 (PKV_ERR_UNSUPPORTED otherwise).  The scales are read once
 * per launch.
 */
int paged_attention_decode_fp8(void* out, const void* q, const void* k_pool, const void* v_pool,
                               const float* k_scale, const float* v_scale,
                               const int32_t* block_tables, const int32_t* seq_lens, int rows,
                               int q_heads, int kv_heads, int head_dim, int block_size, float scale,
                               int max_blocks_per_row, int num_blocks, int max_seq_len,
                               void* workspace, size_t workspace_bytes, int32_t* dev_err,
                               cudaStream_t stream);

/*
 * paged_attention_append_decode_fp8 -- one decode step of one layer over FP8
 * pools: exactly paged_kv_append_fp8(k_pool, v_pool, k_scale, v_scale,
 * block_tables, positions, k_new, v_new, ...) followed by
 * paged_attention_decode_fp8(out, q, k_pool, v_pool, k_scale, v_scale,
 * block_tables, seq_lens, ...), with the same arguments, results and errors
 * as those two calls (the pools end bit-identical, the outputs equal those of
 * the two calls).  Defining passages as for paged_attention_append_decode and
 * the FP8 block above.  One launch: the new token is quantised and stored by
 * the decode kernel, and the block that stages its slot takes the token's
 * E4M3 values from k_new / v_new directly.  Supported shapes as for
 * paged_attention_decode_fp8 (PKV_ERR_UNSUPPORTED otherwise); k_pool, v_pool,
 * k_new and v_new need 16-byte alignment.
 *
 * flags: 0 or PKV_FLAG_PDL, as for paged_attention_append_decode; before the
 * preceding kernel completes, a PDL launch also reads k_scale and v_scale,
 * which that kernel must not write either.
 */
int paged_attention_append_decode_fp8(void* out, const void* q, void* k_pool, void* v_pool,
                                      const float* k_scale, const float* v_scale,
                                      const int32_t* block_tables, const int32_t* seq_lens,
                                      const int32_t* positions, const void* k_new,
                                      const void* v_new, int rows, int q_heads, int kv_heads,
                                      int head_dim, int block_size, float scale,
                                      int max_blocks_per_row, int num_blocks, int max_seq_len,
                                      void* workspace, size_t workspace_bytes, unsigned flags,
                                      int32_t* dev_err, cudaStream_t stream);

/*
 * Decode plans.  The work of a decode step is split over one thread block per
 * SM by cutting every row's tokens, in 16-token granules, into equal
 * contiguous ranges; each block then gathers the K/V blocks of its range
 * through the rows' block tables ("PagedAttention", deepconcepts.dev, section
 * "PagedAttention": walk the table, gather only the listed blocks), and rows
 * cut between blocks are merged exactly through their log-sum-exp (its
 * closing note on FlashAttention).  Every layer of a step reads the same rows
 * at the same lengths through the same tables, so that split -- each block's
 * range, the rows and heads it serves, the physical rows of its granules, and
 * which block holds each row's appended token -- is the same for all of them.
 * paged_attention_plan makes it once per step; paged_attention_decode_planned
 * then starts each layer's copies straight from it instead of re-deriving it
 * from seq_lens and the tables.
 *
 * paged_attention_plan_size -- bytes of a plan for these sizes (an upper
 * bound independent of the device), or 0 when the staged decode kernel does
 * not take the shape (then plan nothing and call the unplanned entry points).
 */
size_t paged_attention_plan_size(int rows, int q_heads, int kv_heads, int head_dim,
                                 int max_seq_len, int block_size);

/*
 * paged_attention_plan -- write the plan of one decode step into `plan`
 * (device buffer of paged_attention_plan_size(...) bytes, caller-owned).  One
 * small launch on `stream`.  block_tables, seq_lens, positions and the sizes
 * are those every planned call of the step will pass; positions may be null
 * when the step appends nothing.  A seq_len outside [0, max_seq_len] and table
 * entries outside [0, num_blocks) are flagged here (PKV_DEV_ERR_SEQ_LEN /
 * PKV_DEV_ERR_BLOCK_ID), and the granules concerned are planned as empty.
 * The plan stays valid while those inputs do not change.
 */
int paged_attention_plan(void* plan, size_t plan_bytes, const int32_t* block_tables,
                         const int32_t* seq_lens, const int32_t* positions, int rows, int q_heads,
                         int kv_heads, int head_dim, int block_size, int max_blocks_per_row,
                         int num_blocks, int max_seq_len, int32_t* dev_err, cudaStream_t stream);

/*
 * paged_attention_decode_planned -- one layer of a planned step: the same
 * result as paged_attention_append_decode (positions non-null) or
 * paged_attention_decode (positions null; k_new, v_new unused), over fp16
 * pools (k_scale == v_scale == null) or FP8 pools (both non-null, as in
 * paged_attention_append_decode_fp8 / paged_attention_decode_fp8).  `plan`
 * must come from paged_attention_plan with the same block_tables, seq_lens,
 * positions (null or not) and sizes; a plan made for a different launch size
 * sets PKV_DEV_ERR_PLAN and the call writes nothing.  Workspace as for
 * paged_attention_decode.  Supported for the staged kernel's shapes
 * (paged_attention_plan_size(...) > 0); PKV_ERR_UNSUPPORTED otherwise.
 *
 * flags: 0 or PKV_FLAG_PDL, as for paged_attention_append_decode; a PDL launch
 * also reads the plan before the preceding kernel completes, so the plan must
 * not be written by that kernel: launch the step's first planned call after
 * paged_attention_plan without PKV_FLAG_PDL (or with other work in between).
 */
int paged_attention_decode_planned(void* out, const void* q, void* k_pool, void* v_pool,
                                   const float* k_scale, const float* v_scale,
                                   const int32_t* block_tables, const int32_t* seq_lens,
                                   const int32_t* positions, const void* k_new, const void* v_new,
                                   int rows, int q_heads, int kv_heads, int head_dim,
                                   int block_size, float scale, int max_blocks_per_row,
                                   int num_blocks, int max_seq_len, const void* plan,
                                   size_t plan_bytes, void* workspace, size_t workspace_bytes,
                                   unsigned flags, int32_t* dev_err, cudaStream_t stream);

/* Bytes of the static device scratch behind paged_attention_decode_noalloc
 * (8 MiB, held by every GPU that loads the library until the process exits). */
#define PKV_NOALLOC_WORKSPACE_BYTES ((size_t)8 << 20)

/*
 * paged_attention_decode_noalloc -- paged_attention_decode for callers that
 * cannot allocate device memory, such as a plug-in inside a host framework
 * that owns all device memory through its own pool, or a serving loop that
 * forbids cudaMalloc after start-up because cudaMalloc / cudaFree can
 * synchronise the device and stall other streams.  (The pages have no
 * counterpart: this is an interface choice of this library.)
 *
 * Same arguments, layout and result as paged_attention_decode, minus the
 * workspace: the caller still passes every input and output buffer, and the
 * split-K scratch comes from one file-scope static device array of
 * PKV_NOALLOC_WORKSPACE_BYTES instead.  Allocates nothing: no cudaMalloc,
 * cudaFree or allocating library routine is called.
 *
 *  - Limit: sizes whose paged_attention_workspace_size(...) exceeds
 *    PKV_NOALLOC_WORKSPACE_BYTES return PKV_ERR_WORKSPACE before launch.
 *  - Set-up: the first call made on a device looks up the array's device
 *    address (cudaGetSymbolAddress, with that device current) and caches it;
 *    make that first call before any stream capture.  The cached address
 *    belongs to the device's context at that time: after cudaDeviceReset (or
 *    any other teardown of that context) the cached address is stale, so a
 *    process that resets a device must not call this entry point again.
 *  - Sharing: every call on a device uses the same array, which keeps the
 *    last call's contents.  Each call first clears the part that must start
 *    at zero (the split-K record words, by cudaMemsetAsync on `stream`); the
 *    rest is written before it is read.  Calls that overlap on the GPU (for
 *    example on two streams at once) race on the array and give wrong
 *    results: serialise them.
 */
int paged_attention_decode_noalloc(void* out, const void* q, const void* k_pool,
                                   const void* v_pool, const int32_t* block_tables,
                                   const int32_t* seq_lens, int rows, int q_heads, int kv_heads,
                                   int head_dim, int block_size, float scale,
                                   int max_blocks_per_row, int num_blocks, int max_seq_len,
                                   int32_t* dev_err, cudaStream_t stream);

/*
 * pkv_debug_set_decode_hooks -- test hook for the bounded waits of the
 * decode kernels' split-unit merge (no counterpart in the pages).  A merge
 * polls the records of a unit's other pieces; poll_limit (0 = the default,
 * about 2^22 polls) caps those polls, after which the merge gives up, flags
 * PKV_DEV_ERR_TIMEOUT and its block ends.  stuck_word, if non-null, is a
 * device word that every merge poll also waits to see non-zero: a word that
 * nothing writes makes every merge give up.  Both apply to launches made
 * after the call, from any thread, until changed; pass (0, NULL) to restore
 * normal operation.  After a timed-out call, zero-fill the workspace before
 * reusing it.  For tests of the failure path; not for production use.
 */
int pkv_debug_set_decode_hooks(unsigned poll_limit, const void* stuck_word);

/*
 * pkv_check_error -- synchronise `stream`, copy the device error word to
 * *host_err and clear it on the device.  Returns PKV_ERR_CUDA if the stream
 * reported an error.  The only library call that blocks.  If the word holds
 * PKV_DEV_ERR_TIMEOUT, the outputs of the calls that reported into it are
 * invalid, and every decode or prefill workspace those calls used must be
 * zero-filled again before its next use (the library's own scratch is
 * cleared by its next call).
 */
int pkv_check_error(int32_t* dev_err, cudaStream_t stream, int32_t* host_err);

/* ------------------------------------------------------------------------ */
/*
 * Host block manager.  Defining passages: "Paged attention"
 * (danielfleming.xyz), section "What changed" (a free list hands out blocks
 * at admission and takes them back at eviction with no copy; reserve on
 * admit: admit only if every block for prompt + full budget is free);
 * "SLM paged attention", section "The architecture" and "End-to-end flow"
 * (O(1) pop/push free list; growth one block at a time when nothing was
 * reserved; shared prefix blocks are reference counted, freed at count 0 and
 * copied on the first write into them); "PagedAttention" (deepconcepts.dev),
 * section "So what does block_size trade?" (blocks are shared whole: only
 * floor(prefix_tokens / block_size) blocks of a prefix are shareable).
 *
 * Host memory only, single-threaded (callers serialise access).  Block ids
 * are in [0, num_blocks).  Errors: PKV_ERR_INVALID_ARG for bad arguments,
 * PKV_ERR_NOT_FOUND for unknown ids, PKV_ERR_NO_BLOCKS when the free list
 * cannot cover a request (state unchanged: nothing is partially allocated),
 * PKV_ERR_STATE for a sequence that is already admitted / past its table.
 */
typedef struct pkv_block_manager pkv_block_manager;

typedef struct {
    int32_t num_blocks;      /* pool size */
    int32_t free_blocks;     /* on the free list */
    int32_t used_blocks;     /* num_blocks - free_blocks */
    int32_t shared_blocks;   /* used blocks with reference count > 1 */
    int32_t sequences;       /* admitted sequences */
    int32_t prefixes;        /* registered prefixes */
    int64_t live_tokens;     /* sum of sequence lengths */
    int64_t reserved_slots;  /* slots held by sequences but not yet written */
    int64_t cow_copies;      /* copy-on-write events so far */
} pkv_bm_stats_t;

/* Create a manager over a pool of num_blocks blocks of block_size tokens;
 * tables have max_blocks_per_row entries.  All blocks start free. */
int pkv_bm_create(int num_blocks, int block_size, int max_blocks_per_row,
                  pkv_block_manager** out);
void pkv_bm_destroy(pkv_block_manager* bm);

/* Register a shared prefix of prefix_tokens tokens: takes
 * floor(prefix_tokens / block_size) blocks from the free list (the partial
 * remainder is not shareable) and holds one reference on each.  Writes the
 * prefix id and (nullable) the block ids, in logical order, to block_ids_out
 * (capacity floor(prefix_tokens / block_size)). */
int pkv_bm_register_prefix(pkv_block_manager* bm, int prefix_tokens, int32_t* prefix_id_out,
                           int32_t* block_ids_out);
/* Drop the registration's own reference; blocks return to the free list once
 * no sequence references them. */
int pkv_bm_release_prefix(pkv_block_manager* bm, int32_t prefix_id);

/* Admit sequence seq_id with prompt_len tokens and a budget of up to
 * max_new_tokens further tokens.  With reserve != 0 (reserve on admit) every
 * block the sequence can ever need -- ceil((prompt_len + max_new_tokens) /
 * block_size) table entries, including the private copy a later write into a
 * shared block needs -- is taken now, or nothing is and PKV_ERR_NO_BLOCKS is
 * returned.  With reserve == 0 only the prompt's blocks are taken and later
 * blocks come one at a time from pkv_bm_append_slot.  prefix_id >= 0 points
 * the sequence's leading entries at that prefix's shared blocks (as many as
 * its prompt covers). */
int pkv_bm_admit(pkv_block_manager* bm, int64_t seq_id, int prompt_len, int max_new_tokens,
                 int32_t prefix_id, int reserve);

/* Claim the slot for the sequence's next token and advance its length by
 * one.  Writes the token's position to *position_out.  If that position
 * lies in a block the sequence shares, the block is copied on write: a
 * private block is taken (from the reservation, else the free list), the
 * table entry is repointed, and the copy the caller must perform on the
 * device is reported in *cow_src_out / *cow_dst_out (both -1 when no copy is
 * needed).  Returns PKV_ERR_NO_BLOCKS (length unchanged) if a new block is
 * needed and none is free, PKV_ERR_STATE past max_blocks_per_row. */
int pkv_bm_append_slot(pkv_block_manager* bm, int64_t seq_id, int32_t* position_out,
                       int32_t* cow_src_out, int32_t* cow_dst_out);

/* Release a finished sequence: every block it references loses one
 * reference; blocks at zero go back to the free list (no data moves). */
int pkv_bm_free(pkv_block_manager* bm, int64_t seq_id);

/* Copy the sequence's table (max_blocks_per_row int32, -1 past its blocks)
 * into row_out and its length into *seq_len_out (nullable). */
int pkv_bm_table(const pkv_block_manager* bm, int64_t seq_id, int32_t* row_out,
                 int32_t* seq_len_out);

/* Pool and sharing counters (the pages' operating metrics: memory in use,
 * blocks shared). */
int pkv_bm_stats(const pkv_block_manager* bm, pkv_bm_stats_t* out);

/* Reference count of a physical block (0 = free). */
int pkv_bm_refcount(const pkv_block_manager* bm, int32_t block_id, int32_t* count_out);

/* Host-side fault injection for tests: after `pops` more successful block
 * pops, every further pop fails as if the free list were empty (-1 turns it
 * off). */
int pkv_bm_inject_pop_failure(pkv_block_manager* bm, int pops);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_H */
